"""Seeded synthetic inputs for paged GQA attention.

This module is shared by the tests, the benchmark and the oracle's tests. It
builds inputs only: sequence/query lengths, a paged KV cache with a permuted
block table, Q, and the FP8 e4m3 quantisation of the synthetic values. It holds
none of the attention arithmetic.

Workload shapes follow the pages' problem statements:
  * "Optimize Qwen3.5 MTP unified attention on gfx950" (sglang #36330),
    Motivation / Benchmarking: q_len <= 4, 16 q heads per kv head, head size
    256, page size 16, bf16 Q, FP8 KV cache, per-tensor descales.
  * "asm FP8 FMHA for prefix-hit prefill" (ROCm/ATOM #2534), summary: 16k new
    tokens on a 32k total context, 8 q heads / 1 kv head, hd256, FP8 Q/K/V,
    bottom-right causal mask.
  * "gfx1250 GDN prefill kernels ...; DP points on unified attention"
    (ROCm/ATOM #2830), commit 6: 64-token KV blocks.

Recipe (the same for every config):
  * lengths come from a CPU torch.Generator seeded with ``seed``; "uniform in
    [a, b]" means integers a..b inclusive;
  * physical pages are a random permutation of all pages (plus the spare pages
    a config names); each sequence takes the next ceil(L/P) entries; the rest
    of its block-table row is -1;
  * Q, K and V values are N(0, 1) from a generator on the target device
    seeded with seed+1 (K), seed+2 (V), seed+3 (Q);
  * FP8 tensors use one fp32 scale = amax/448 over the whole tensor and
    x8 = RNE(clamp(x/scale, +-448)) through torch.float8_e4m3fn; the descale
    passed to the kernel is that scale;
  * FP8 Q's descale is folded into softmax_scale (the call has no q_descale);
  * with ``poison=True`` every cache slot no sequence reads (tails of last
    pages, spare pages) holds NaN, so a kernel that reads them fails parity.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import torch

HEAD_DIM = 256
E4M3_MAX = 448.0
E4M3_NAN_BYTE = 0x7F
BF16_NAN_BITS = 0x7FC0


@dataclasses.dataclass
class CaseSpec:
    """Shape recipe of one call: per-sequence (q_len, kv_len) and head layout."""

    name: str
    seqs: List[Tuple[int, int]]          # (q_len, L) per sequence, L = total K/V length
    num_q_heads: int
    num_kv_heads: int
    page_size: int
    q_dtype: str = "bf16"                # "bf16" | "e4m3"
    kv_dtype: str = "e4m3"               # "bf16" | "e4m3"
    spare_pages: int = 0
    softmax_scale: float = 1.0 / 16.0    # 1/sqrt(256)
    extra_table_cols: int = 0            # block-table width beyond the longest sequence

    @property
    def num_seqs(self) -> int:
        return len(self.seqs)

    @property
    def total_q(self) -> int:
        return sum(q for q, _ in self.seqs)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def pages_of(self, L: int) -> int:
        return (L + self.page_size - 1) // self.page_size

    @property
    def used_pages(self) -> int:
        return sum(self.pages_of(L) for _, L in self.seqs)

    @property
    def kv_bytes(self) -> int:
        """Algorithmic KV bytes: every valid token's K and V once per kv head."""
        esz = 1 if self.kv_dtype == "e4m3" else 2
        return sum(L for _, L in self.seqs) * self.num_kv_heads * HEAD_DIM * 2 * esz

    @property
    def flops(self) -> int:
        """Causal-exact FLOPs: 4*D per (query row, visible key) pair."""
        pairs = 0
        for q, L in self.seqs:
            # rows t = 0..q-1 see L - q + t + 1 keys
            pairs += q * (L - q + 1) + q * (q - 1) // 2
        return 4 * HEAD_DIM * self.num_q_heads * pairs


def _uniform_int(gen: torch.Generator, lo: int, hi: int, n: int) -> List[int]:
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


def config_spec(index: int, seed: int = 0) -> CaseSpec:
    """The five workloads of the benchmark, numbered 1..5."""
    gen = torch.Generator().manual_seed(seed)
    if index == 1:
        return CaseSpec("tiny_verify_b1_q2_h16x1_L600_p16_bf16", [(2, 600)], 16, 1, 16,
                        q_dtype="bf16", kv_dtype="bf16", spare_pages=64 - 38)
    if index == 2:
        Ls = _uniform_int(gen, 1024, 32768, 64)
        return CaseSpec("mtp_verify_b64_q4_h16x1_L1k-32k_p16_e4m3kv", [(4, L) for L in Ls], 16, 1, 16)
    if index == 3:
        qs = _uniform_int(gen, 2, 4, 256)
        return CaseSpec("verify_b256_q2-4_h32x2_L8192_p16_e4m3kv", [(q, 8192) for q in qs], 32, 2, 16)
    if index == 4:
        return CaseSpec("prefix_prefill_q16384_L32768_h8x1_p64_e4m3qkv", [(16384, 32768)], 8, 1, 64,
                        q_dtype="e4m3", kv_dtype="e4m3")
    if index == 5:
        Ls = _uniform_int(gen, 2048, 65536, 512)
        seqs = [(8192, 8192 + 24576)] * 8 + [(4, L) for L in Ls]
        return CaseSpec("mixed_8x(q8192,L32768)+512x(q4,L2k-64k)_h24x2_p64_e4m3kv", seqs, 24, 2, 64)
    raise ValueError(f"unknown config {index}")


SPARSE_TOPK = 2051  # selected tokens per row in "Tune sparse GQA prefill profile on gfx942 and gfx950"


def sparse_spec(tp: int = 1) -> CaseSpec:
    """Sparse prefill: 8192 new tokens on a 32768-token context, 64-token pages, FP8 K/V,
    bf16 Q; heads of the sparse page's TP1 (24 q / 2 kv) or TP2 (12 q / 1 kv) shapes."""
    heads = {1: (24, 2), 2: (12, 1), 4: (6, 1), 8: (3, 1)}[tp]
    return CaseSpec(f"sparse_prefill_q8192_L32768_h{heads[0]}x{heads[1]}_p64_top{SPARSE_TOPK}",
                    [(8192, 32768)], heads[0], heads[1], 64)


def sparse_indices(spec: CaseSpec, topk: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """[T, Hkv, topk] int32 selected positions per (token, kv head), ascending.

    Row (t, h) of a sequence of length L with q_len qn sees positions 0..n-1, n = L - qn +
    t + 1. If n <= topk it lists all of them and pads with -1; otherwise it takes one
    position uniformly from each of topk strata [j n / topk, (j + 1) n / topk) (integer
    bounds), so the positions are distinct and spread over the whole visible range.
    Draws come from a generator on ``device`` seeded with seed + 11.
    """
    gen = _device_generator(device, seed + 11)
    n_vis = []
    for q, L in spec.seqs:
        n_vis.append(torch.arange(L - q + 1, L + 1, dtype=torch.int64))
    n = torch.cat(n_vis).to(device) if n_vis else torch.zeros(0, dtype=torch.int64, device=device)
    T, H = n.shape[0], spec.num_kv_heads
    j = torch.arange(topk, dtype=torch.int64, device=device)
    out = torch.empty(T, H, topk, dtype=torch.int32, device=device)
    chunk = max(1, (1 << 24) // max(1, H * topk))
    for t0 in range(0, T, chunk):
        nn = n[t0:t0 + chunk].view(-1, 1, 1)
        lo = (j * nn) // topk
        hi = ((j + 1) * nn) // topk
        u = torch.rand(nn.shape[0], H, topk, generator=gen, device=device)
        pos = lo + torch.minimum((u * (hi - lo)).to(torch.int64), hi - lo - 1)
        full = nn <= topk
        pos = torch.where(full, torch.where(j < nn, j, -1), pos)
        out[t0:t0 + chunk] = pos.to(torch.int32)
    return out


def write_chunks_spec() -> CaseSpec:
    """A cache-write case that fits a profiler's memory budget but exceeds L2: 32 fresh
    prefill chunks of 4096 tokens, 2 kv heads, 64-token pages (403 MB written and read)."""
    return CaseSpec("write_chunks_b32_q4096_h2_p64", [(4096, 4096)] * 32, 16, 2, 64)


def random_small_spec(gen: torch.Generator, *, group: int, num_kv_heads: int, page_size: int,
                      q_lens: Sequence[int], max_ctx: int, kv_dtype: str = "e4m3",
                      q_dtype: str = "bf16", spare_pages: int = 3, name: str = "small") -> CaseSpec:
    """Random small varlen case: each sequence gets L in [max(q,1), max_ctx]."""
    seqs = []
    for q in q_lens:
        lo = max(q, 1)
        L = int(torch.randint(lo, max(lo, max_ctx) + 1, (1,), generator=gen))
        seqs.append((int(q), L))
    return CaseSpec(name, seqs, group * num_kv_heads, num_kv_heads, page_size,
                    q_dtype=q_dtype, kv_dtype=kv_dtype, spare_pages=spare_pages, extra_table_cols=2)


@dataclasses.dataclass
class Case:
    """One call's inputs. FP8 tensors are stored as torch.uint8 bit patterns."""

    spec: CaseSpec
    q: torch.Tensor              # [T, Hq, 256] bf16 or uint8(e4m3)
    k_cache: torch.Tensor        # [NB, P, Hkv, 256] bf16 or uint8(e4m3)
    v_cache: torch.Tensor
    block_table: torch.Tensor    # [num_seqs, W] int32
    seq_lens: torch.Tensor       # [num_seqs] int32
    query_start_loc: torch.Tensor  # [num_seqs+1] int32
    q_descale: float
    k_descale: float
    v_descale: float
    softmax_scale: float         # what the caller passes: includes q_descale for FP8 Q

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]


def _device_generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_quantised(shape, dtype: str, device, seed: int, chunk: int = 1 << 27):
    """N(0,1) values of ``shape``; FP8 -> (uint8 bits, scale), bf16 -> (bf16, 1.0).

    Generated in chunks so that very large caches never hold a full fp32 copy.
    Two passes over the same generator stream: amax, then quantise.
    """
    n = math.prod(shape)
    gen = _device_generator(device, seed)
    if dtype == "bf16":
        out = torch.empty(n, dtype=torch.bfloat16, device=device)
        for s in range(0, n, chunk):
            e = min(n, s + chunk)
            out[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
        return out.view(shape), 1.0
    assert dtype == "e4m3"
    state = gen.get_state()
    amax = 0.0
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        amax = max(amax, float(x.abs().max()))
    gen.set_state(state)
    scale = torch.tensor(amax / E4M3_MAX, dtype=torch.float32).item()
    out = torch.empty(n, dtype=torch.uint8, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        x8 = (x / scale).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
        out[s:e] = x8.view(torch.uint8)
    return out.view(shape), scale


def make_case(spec: CaseSpec, device="cpu", seed: int = 0, poison: bool = False) -> Case:
    """Materialise ``spec`` on ``device`` (values) with CPU-seeded structure."""
    gen = torch.Generator().manual_seed(seed + 7919)
    P, Hkv, Hq, D = spec.page_size, spec.num_kv_heads, spec.num_q_heads, HEAD_DIM
    n_pages = [spec.pages_of(L) for _, L in spec.seqs]
    NB = sum(n_pages) + spec.spare_pages
    NB = max(NB, 1)
    W = max([1] + n_pages) + spec.extra_table_cols
    perm = torch.randperm(NB, generator=gen)
    bt = torch.full((spec.num_seqs, W), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(n_pages):
        bt[s, :n] = perm[off:off + n].to(torch.int32)
        off += n
    seq_lens = torch.tensor([L for _, L in spec.seqs], dtype=torch.int32)
    qsl = torch.zeros(spec.num_seqs + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(torch.tensor([q for q, _ in spec.seqs], dtype=torch.int64), 0).to(torch.int32)
    T = int(qsl[-1])

    k_cache, k_scale = _randn_quantised((NB, P, Hkv, D), spec.kv_dtype, device, seed + 1)
    v_cache, v_scale = _randn_quantised((NB, P, Hkv, D), spec.kv_dtype, device, seed + 2)
    q, q_scale = _randn_quantised((T, Hq, D), spec.q_dtype, device, seed + 3)
    if spec.kv_dtype == "bf16":
        k_scale = v_scale = 1.0

    if poison:
        _poison_unused(spec, k_cache, v_cache, bt, perm, n_pages)

    softmax_scale = spec.softmax_scale * (q_scale if spec.q_dtype == "e4m3" else 1.0)
    return Case(spec, q, k_cache, v_cache, bt.to(device), seq_lens.to(device), qsl.to(device),
                q_scale, k_scale, v_scale, softmax_scale)


def _poison_unused(spec: CaseSpec, k_cache, v_cache, bt, perm, n_pages):
    """Fill every slot that no sequence may read with NaN."""
    P = spec.page_size
    nan = E4M3_NAN_BYTE if spec.kv_dtype == "e4m3" else None
    used = sum(n_pages)
    spare = perm[used:].tolist()

    def fill(t, idx, rows):
        if spec.kv_dtype == "e4m3":
            t[idx, rows] = nan
        else:
            t[idx, rows] = float("nan")

    for blk in spare:
        fill(k_cache, blk, slice(0, P))
        fill(v_cache, blk, slice(0, P))
    for s, (_, L) in enumerate(spec.seqs):
        n = n_pages[s]
        if n == 0:
            continue
        tail = L - (n - 1) * P
        if tail < P:
            blk = int(bt[s, n - 1])
            fill(k_cache, blk, slice(tail, P))
            fill(v_cache, blk, slice(tail, P))


def sample_rows(spec: CaseSpec, n_rows: int, seed: int = 0, whole_seqs: Sequence[int] = ()) -> torch.Tensor:
    """Deterministic sample of flat output rows (token*Hq + head) for large cases."""
    gen = torch.Generator().manual_seed(seed + 31)
    T, Hq = spec.total_q, spec.num_q_heads
    picks = torch.randint(0, T * Hq, (n_rows,), generator=gen)
    extra = []
    starts = [0]
    for q, _ in spec.seqs:
        starts.append(starts[-1] + q)
    for s in whole_seqs:
        for t in range(starts[s], starts[s + 1]):
            extra.extend(range(t * Hq, (t + 1) * Hq))
    rows = torch.cat([picks, torch.tensor(extra, dtype=torch.int64)]) if extra else picks
    return torch.unique(rows)


def to_device(case: Case, device="cuda") -> Case:
    return Case(case.spec, case.q.to(device), case.k_cache.to(device), case.v_cache.to(device),
                   case.block_table.to(device), case.seq_lens.to(device), case.query_start_loc.to(device),
                   case.q_descale, case.k_descale, case.v_descale, case.softmax_scale)


def subcase(case: Case, seq_ids) -> Case:
    """The listed sequences alone, with only their pages (sequences are independent)."""
    spec = case.spec
    P = spec.page_size
    qsl = case.query_start_loc.cpu().tolist()
    sl = case.seq_lens.cpu().tolist()
    bt = case.block_table.cpu()
    pages, q_parts, seqs, rows = [], [], [], []
    for s in seq_ids:
        n = (sl[s] + P - 1) // P
        rows.append(list(range(len(pages), len(pages) + n)))
        pages.extend(bt[s, :n].tolist())
        q_parts.append(case.q[qsl[s]:qsl[s + 1]].cpu())
        seqs.append((qsl[s + 1] - qsl[s], sl[s]))
    idx = torch.tensor(pages, dtype=torch.long, device=case.k_cache.device)
    k = case.k_cache.index_select(0, idx).cpu()
    v = case.v_cache.index_select(0, idx).cpu()
    W = max(1, max(len(r) for r in rows))
    nbt = torch.full((len(seq_ids), W), -1, dtype=torch.int32)
    for i, r in enumerate(rows):
        nbt[i, :len(r)] = torch.tensor(r, dtype=torch.int32)
    nsl = torch.tensor([L for _, L in seqs], dtype=torch.int32)
    nqsl = torch.zeros(len(seqs) + 1, dtype=torch.int32)
    nqsl[1:] = torch.cumsum(torch.tensor([q for q, _ in seqs]), 0).to(torch.int32)
    sub_spec = CaseSpec(spec.name + "_sub", seqs, spec.num_q_heads, spec.num_kv_heads, P,
                           q_dtype=spec.q_dtype, kv_dtype=spec.kv_dtype, softmax_scale=spec.softmax_scale)
    return Case(sub_spec, torch.cat(q_parts, 0), k, v, nbt, nsl, nqsl, case.q_descale, case.k_descale,
                   case.v_descale, case.softmax_scale)


