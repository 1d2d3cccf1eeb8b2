"""Sparse paged GQA on the GPU against the oracle, element by element."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


TC_MIN_KEYS = 64  # under path 2, lists at least this long run on the tcgen05 kernel (path bit 32)


def _run(case, idx, out=None, check=True):
    import paged_gqa_gb300 as pg
    T, Hq = case.q.shape[0], case.q.shape[1]
    if out is None:
        out = torch.full((T, Hq, wl.HEAD_DIM), float("nan"), dtype=torch.bfloat16, device="cuda")
    pg.paged_gqa_sparse_attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                             case.query_start_loc, idx, case.k_descale, case.v_descale, case.softmax_scale, out)
    if check:
        assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
    if T > 0 and idx.shape[2] > 0:
        bits = pg.paged_gqa_last_plan()["path_bits"]
        path = pg.paged_gqa_set_path(0)  # read the current selection, then put it back
        pg.paged_gqa_set_path(path)
        want = 32 if path == 2 and idx.shape[2] >= TC_MIN_KEYS else 64
        assert bits == want, f"path bits {bits}, expected {want}"
    return out


class kernel_path:
    """Calls inside run under paged_gqa_set_path(path): 1 = warp-level kernel everywhere,
    2 = the tcgen05 sparse kernel for lists of TC_MIN_KEYS or more."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        import paged_gqa_gb300 as pg
        self.prev = pg.paged_gqa_set_path(self.path)

    def __exit__(self, *exc):
        import paged_gqa_gb300 as pg
        pg.paged_gqa_set_path(self.prev)


@pytest.fixture(autouse=True)
def tcgen05_sparse():
    """Every sparse test runs with the tcgen05 sparse kernel selected (path 2) unless it
    selects another path itself; the default path's kernel is covered by the "auto" cases."""
    with kernel_path(2):
        yield


def _oracle(case, idx, rows=None):
    c = gu.to_device(case, "cpu")
    return oracle.sparse_attention(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens, c.query_start_loc,
                                   idx.cpu(), q_dtype="bf16", kv_dtype="e4m3", q_descale=1.0,
                                   k_descale=case.k_descale, v_descale=case.v_descale,
                                   softmax_scale=case.spec.softmax_scale, rows=rows)


def _random_lists(case, K, seed, junk=True):
    """Random positions in [-3, L + 5) per (token, kv head): in-range, padding, past the
    causal limit, and duplicates all occur."""
    g = torch.Generator().manual_seed(seed)
    T, Hkv = case.q.shape[0], case.spec.num_kv_heads
    Lmax = int(case.seq_lens.max())
    lo = -3 if junk else 0
    idx = torch.randint(lo, Lmax + (5 if junk else 0), (T, Hkv, K), generator=g, dtype=torch.int32)
    if K >= 4:
        idx[:, :, 1] = idx[:, :, 0]  # a duplicate in every list
    return idx.cuda()


SMALL = [
    # (group, kv heads, page, q_lens, max context, K)
    (12, 2, 64, [4, 1, 37], 500, 100),     # the sparse page's TP1 head layout, ragged K
    (12, 1, 16, [9, 2], 300, 33),          # TP2
    (6, 1, 32, [5, 16], 200, 64),          # TP4
    (3, 1, 16, [7], 90, 5),                # TP8, a short list
    (16, 1, 64, [3, 20], 400, 70),         # a full 16-head group
    (24, 1, 16, [6, 2], 250, 40),          # two head groups per kv head
]


@pytest.mark.parametrize("path", [2, 0, 1])
@pytest.mark.parametrize("i", range(len(SMALL)))
def test_small_cases_match_the_oracle(i, path):
    G, hkv, page, q_lens, ctx, K = SMALL[i]
    gen = torch.Generator().manual_seed(90 + i)
    spec = wl.random_small_spec(gen, group=G, num_kv_heads=hkv, page_size=page, q_lens=q_lens, max_ctx=ctx,
                                kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=90 + i, poison=True)
    idx = _random_lists(case, K, 90 + i)
    ref = _oracle(case, idx)
    with kernel_path(path):
        gu.compare(_run(case, idx), ref, f"sparse case {i}, path {path}")


# tcgen05 kernel shapes: units not a multiple of four (padding units), two head groups per
# kv head, several kv heads, lists that are not a multiple of 32, and one whole tile only
TC_CASES = [
    # (group, kv heads, page, q_lens, max context, K)
    (12, 2, 64, [3, 2], 700, 257),
    (24, 1, 16, [5, 1, 2], 600, 96),
    (3, 4, 32, [6, 1], 500, 64),
    (16, 1, 128, [7], 1200, 301),
    (6, 2, 16, [1, 1, 1, 1, 1], 900, 130),
]


@pytest.mark.parametrize("i", range(len(TC_CASES)))
def test_tcgen05_sparse_shapes_match_the_oracle(i):
    G, hkv, page, q_lens, ctx, K = TC_CASES[i]
    gen = torch.Generator().manual_seed(190 + i)
    spec = wl.random_small_spec(gen, group=G, num_kv_heads=hkv, page_size=page, q_lens=q_lens, max_ctx=ctx,
                                kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=190 + i, poison=True)
    idx = _random_lists(case, K, 190 + i)
    gu.compare(_run(case, idx), _oracle(case, idx), f"tcgen05 sparse case {i}")
    idx = wl.sparse_indices(case.spec, K, device="cuda", seed=190 + i)
    gu.compare(_run(case, idx), _oracle(case, idx), f"tcgen05 sparse case {i}, generated lists")


def test_generated_top_k_lists_and_empty_lists():
    gen = torch.Generator().manual_seed(97)
    spec = wl.random_small_spec(gen, group=12, num_kv_heads=2, page_size=64, q_lens=[40, 3], max_ctx=900,
                                kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=97, poison=True)
    idx = wl.sparse_indices(case.spec, 129, device="cuda", seed=97)
    gu.compare(_run(case, idx), _oracle(case, idx), "generated top-k lists")
    none = torch.full_like(idx, -1)
    out = _run(case, none)
    assert (out == 0).all()
    empty = torch.empty(idx.shape[0], idx.shape[1], 0, dtype=torch.int32, device="cuda")
    assert (_run(case, empty) == 0).all()


def test_full_lists_equal_the_dense_call():
    """Listing every position 0..L-1 is the dense attention: the sparse kernel against the
    dense oracle and against the dense GPU path on the same case."""
    gen = torch.Generator().manual_seed(98)
    spec = wl.random_small_spec(gen, group=12, num_kv_heads=1, page_size=16, q_lens=[4, 130], max_ctx=600,
                                kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=98, poison=True)
    Lmax = int(case.seq_lens.max())
    idx = torch.arange(Lmax, dtype=torch.int32, device="cuda").expand(case.q.shape[0], 1, Lmax).contiguous()
    got = _run(case, idx)
    gu.check_full(case, got, "full lists vs dense oracle")
    dense = gu.run_library(case)
    assert (got.float() - dense.float()).abs().max().item() < 1e-2


def test_bad_page_is_flagged_and_the_key_skipped():
    import paged_gqa_gb300 as pg
    gen = torch.Generator().manual_seed(99)
    spec = wl.random_small_spec(gen, group=6, num_kv_heads=1, page_size=16, q_lens=[3], max_ctx=200,
                                kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=99)
    idx = wl.sparse_indices(case.spec, 20, device="cuda", seed=99)
    bt = case.block_table.clone()
    bt[0, 0] = case.num_blocks + 7  # page of positions 0..15: out of range
    case_bad = wl.Case(case.spec, case.q, case.k_cache, case.v_cache, bt, case.seq_lens, case.query_start_loc,
                       case.q_descale, case.k_descale, case.v_descale, case.softmax_scale)
    got = _run(case_bad, idx, check=False)
    assert pg.paged_gqa_check_device_errors() == -5
    dropped = torch.where(idx < 16, torch.full_like(idx, -1), idx)  # what the kernel skipped
    gu.compare(got, _oracle(case, dropped), "bad page skipped")


@pytest.mark.parametrize("path", [2, 0])
def test_sparse_prefill_workload_sampled_rows(path):
    """The sparse page's TP1 shape: 8192 new tokens on a 32768-token context, 24 q / 2 kv
    heads, 2051 selected positions per (token, kv head); sampled rows and the end tokens."""
    spec = wl.sparse_spec(1)
    case = wl.make_case(spec, device="cuda", seed=0, poison=True)
    idx = wl.sparse_indices(spec, wl.SPARSE_TOPK, device="cuda", seed=0)
    with kernel_path(path):
        got = _run(case, idx).reshape(-1, wl.HEAD_DIM)
    Hq = spec.num_q_heads
    gen = torch.Generator().manual_seed(1)
    rows = torch.cat([torch.arange(Hq), torch.randperm(spec.total_q * Hq, generator=gen)[:400],
                      torch.arange((spec.total_q - 1) * Hq, spec.total_q * Hq)]).numpy().astype(np.int64)
    ref = _oracle(case, idx, rows=rows)
    gu.compare(got[torch.from_numpy(rows).cuda()], ref, "sparse prefill TP1 sampled rows")


@pytest.mark.parametrize("qscale", [1e5, 1e-6])
def test_q_beyond_the_f16_range(qscale):
    """bf16 q far outside f16's normal range (|q| ~ 1e5 overflows f16, ~1e-6 is subnormal
    there), with softmax_scale scaled the other way so that the scores are those of N(0, 1)
    inputs: the result must still match the oracle on the same bf16 q."""
    import dataclasses
    gen = torch.Generator().manual_seed(96)
    spec = wl.random_small_spec(gen, group=12, num_kv_heads=1, page_size=16, q_lens=[5, 2], max_ctx=300,
                                kv_dtype="e4m3", q_dtype="bf16")
    spec = dataclasses.replace(spec, softmax_scale=spec.softmax_scale / qscale)
    case = wl.make_case(spec, device="cuda", seed=96, poison=True)
    q = (case.q.float() * qscale).to(torch.bfloat16)
    assert (q.float().abs().max() > 65504) if qscale > 1 else (q.float().abs().max() < 6.1e-5)
    case = wl.Case(spec, q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, case.query_start_loc,
                   case.q_descale, case.k_descale, case.v_descale, spec.softmax_scale)
    idx = _random_lists(case, 60, 96)
    gu.compare(_run(case, idx), _oracle(case, idx), f"sparse, q x {qscale:g}")
