"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bar (bf16 output): max |diff| <= 1e-2, rel-L2 <= 5e-3, every value finite.
Unused cache slots are NaN-poisoned in every case, so a kernel that reads a tail
slot or a spare page fails.
"""
import pytest
import torch

import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

# auto: the tcgen05 kernels, the verify kernel planning its own class where it can;
# warp_mma: the warp-level MMA kernel everywhere; plan_kernel: as auto, but the plan kernel
# plans the verify class before its kernel runs.
PATHS = {"auto": 0, "warp_mma": 1, "plan_kernel": 3}


@pytest.fixture(params=list(PATHS))
def path(request):
    import paged_gqa_gb300 as pg
    prev = pg.paged_gqa_set_path(PATHS[request.param])
    yield request.param
    pg.paged_gqa_set_path(prev)


def _small(seed, **kw):
    gen = torch.Generator().manual_seed(seed)
    spec = wl.random_small_spec(gen, **kw)
    return wl.make_case(spec, device="cuda", seed=seed, poison=True)


SMALL_CASES = [
    # verify shapes (q_len*G <= 64): the MTP packing, several G, both page sizes
    dict(group=16, num_kv_heads=1, page_size=16, q_lens=[4, 2, 3, 1], max_ctx=700),
    dict(group=16, num_kv_heads=2, page_size=16, q_lens=[2, 4, 3], max_ctx=1500),
    dict(group=12, num_kv_heads=2, page_size=64, q_lens=[4, 4, 1, 5], max_ctx=3000),
    dict(group=8, num_kv_heads=1, page_size=64, q_lens=[8, 1, 0, 3], max_ctx=900),
    dict(group=1, num_kv_heads=4, page_size=32, q_lens=[1, 2, 4], max_ctx=400),
    dict(group=3, num_kv_heads=2, page_size=128, q_lens=[2, 6], max_ctx=1000),
    dict(group=6, num_kv_heads=1, page_size=16, q_lens=[4, 4, 4, 4, 4, 4], max_ctx=260),
    # prefill shapes (128-row blocks), ragged last block, cached prefix
    dict(group=8, num_kv_heads=1, page_size=64, q_lens=[300, 17], max_ctx=1200),
    dict(group=12, num_kv_heads=2, page_size=64, q_lens=[100, 4, 33], max_ctx=800),
    dict(group=16, num_kv_heads=1, page_size=16, q_lens=[65, 9], max_ctx=400),
    # bf16 cache
    dict(group=16, num_kv_heads=1, page_size=16, q_lens=[2, 4], max_ctx=600, kv_dtype="bf16"),
    dict(group=4, num_kv_heads=2, page_size=64, q_lens=[70, 3], max_ctx=500, kv_dtype="bf16"),
    # FP8 q
    dict(group=8, num_kv_heads=1, page_size=64, q_lens=[200, 4], max_ctx=700, q_dtype="e4m3"),
    dict(group=16, num_kv_heads=1, page_size=16, q_lens=[4, 3], max_ctx=900, q_dtype="e4m3"),
]


def _assert_tcgen05_only(path, case=None):
    """Under the automatic paths every class ran on a tcgen05 kernel (path bits 2 / 4), never on
    the warp-MMA kernel (8 / 16). With at most 512 verify blocks the automatic path's verify
    kernel (FP8 or bf16) planned its own class; under plan_kernel it never does."""
    import paged_gqa_gb300 as pg
    plan = pg.paged_gqa_last_plan()
    if path in ("auto", "plan_kernel"):
        bits = plan["path_bits"]
        assert bits & 6 and not bits & 24, f"path bits {bits}"
    if path == "plan_kernel" or path == "warp_mma":
        assert plan["verify_self_planned"] == 0
    elif case is not None:
        tc = case.k_cache.dtype != torch.bfloat16 or case.q.dtype == torch.bfloat16  # a tcgen05 verify kernel
        small = case.spec.num_seqs * case.spec.num_kv_heads <= 512
        single_prefill = case.spec.num_seqs == 1 and case.spec.total_q * case.spec.group > 64
        assert plan["verify_self_planned"] == int(tc and small and not single_prefill), plan


@pytest.mark.parametrize("i", range(len(SMALL_CASES)))
def test_small_cases_match_oracle(i, path):
    case = _small(1000 + i, **SMALL_CASES[i])
    got = gu.run_library(case)
    _assert_tcgen05_only(path, case)
    gu.check_full(case, got, f"case {i} path {path}")


BF16_CASES = [
    # bf16 q and caches (the tcgen05 bf16 kernel serves both classes): verify blocks of
    # several G on every page size, prefill blocks with a ragged last block and a cached
    # prefix, both classes in one call, a long sequence split across CTAs
    dict(group=16, num_kv_heads=1, page_size=32, q_lens=[4, 1, 3], max_ctx=2000),
    dict(group=8, num_kv_heads=2, page_size=128, q_lens=[2, 8, 5], max_ctx=1700),
    dict(group=3, num_kv_heads=4, page_size=64, q_lens=[1, 4], max_ctx=300),
    dict(group=8, num_kv_heads=1, page_size=16, q_lens=[300, 17, 4], max_ctx=1200),
    dict(group=12, num_kv_heads=2, page_size=128, q_lens=[100, 33], max_ctx=900),
    dict(group=32, num_kv_heads=1, page_size=64, q_lens=[1, 2, 3, 4], max_ctx=1300),
]


@pytest.mark.parametrize("i", range(len(BF16_CASES)))
def test_bf16_cache_cases_match_oracle(i, path):
    case = _small(1100 + i, kv_dtype="bf16", **BF16_CASES[i])
    got = gu.run_library(case)
    _assert_tcgen05_only(path, case)
    gu.check_full(case, got, f"bf16 case {i} path {path}")


def test_bf16_long_sequence_is_split(path):
    spec = wl.CaseSpec("long bf16", [(4, 30000)], 16, 1, 16, kv_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=14, poison=True)
    got = gu.run_library(case)
    _assert_tcgen05_only(path, case)
    gu.check_full(case, got, "long split bf16")


def test_config1_tiny_verify(path):
    case = wl.make_case(wl.config_spec(1), device="cuda", seed=0, poison=True)
    got = gu.run_library(case)
    _assert_tcgen05_only(path, case)
    gu.check_full(case, got, "config 1")


def test_page_edges_and_no_cache(path):
    """L exactly on, one past and one short of page boundaries; q_len == L."""
    seqs = [(4, 16), (4, 17), (4, 15), (3, 3), (1, 1), (4, 128), (4, 129), (2, 255), (40, 40), (4, 4)]
    spec = wl.CaseSpec("edges", seqs, 16, 1, 16, spare_pages=2)
    case = wl.make_case(spec, device="cuda", seed=5, poison=True)
    gu.check_full(case, gu.run_library(case), "page edges")


def test_many_short_sequences(path):
    """More sequences than CTAs, most blocks unsplit."""
    gen = torch.Generator().manual_seed(9)
    seqs = [(int(q), int(L)) for q, L in zip(torch.randint(1, 5, (400,), generator=gen),
                                                torch.randint(4, 300, (400,), generator=gen))]
    spec = wl.CaseSpec("many", seqs, 16, 1, 16)
    case = wl.make_case(spec, device="cuda", seed=9, poison=True)
    gu.check_full(case, gu.run_library(case), "many short")


def test_plan_beyond_shared_memory_caches(path):
    """More sequences (2600) and row blocks (~21000) than the plan kernel keeps in shared
    memory, with prefill sequences past the cached range: the plan's global-memory paths."""
    gen = torch.Generator().manual_seed(21)
    seqs = [(int(q), int(L)) for q, L in zip(torch.randint(1, 5, (2600,), generator=gen),
                                                torch.randint(4, 160, (2600,), generator=gen))]
    for i in (5, 2100, 2599):
        seqs[i] = (40, 300)  # 40 tokens x G=2 = 80 rows: prefill blocks
    spec = wl.CaseSpec("beyond caches", seqs, 16, 8, 16)
    case = wl.make_case(spec, device="cuda", seed=21, poison=True)
    gu.check_full(case, gu.run_library(case), "beyond plan caches")
    _assert_tcgen05_only(path, case)  # 20800 verify blocks: planned by the plan kernel


def test_self_planned_verify_at_its_limit(path):
    """512 verify blocks (256 sequences x 2 kv heads), the most a self-planning verify kernel
    takes, with short and long contexts, a few empty and a few prefill sequences between
    them, and 513 blocks (one more sequence), which the plan kernel plans."""
    gen = torch.Generator().manual_seed(23)
    for n in (256, 257):
        seqs = [(int(q), int(L)) for q, L in zip(torch.randint(1, 5, (n,), generator=gen),
                                                    torch.randint(1, 2000, (n,), generator=gen))]
        seqs[3] = (0, 70)
        seqs[100] = (20, 900)  # 20 tokens x G = 8: 160 rows, prefill blocks
        seqs[200] = (0, 0)
        seqs[-1] = (4, 9000)
        spec = wl.CaseSpec("limit", seqs, 16, 2, 16)
        case = wl.make_case(spec, device="cuda", seed=23 + n, poison=True)
        gu.check_full(case, gu.run_library(case), f"{n} sequences x 2 kv heads")
        _assert_tcgen05_only(path, case)


@pytest.mark.parametrize("i", range(6))
def test_self_planned_verify_matches_the_plan_kernel_bit_for_bit(i):
    """A verify kernel that plans its own class takes exactly the plan kernel's cut: the same
    pieces on the same CTAs, and merges that add every piece's partial in piece order
    whichever piece arrives last. So both planning paths give the same output bits, on
    random MTP batches from 1 to 200 sequences, contexts up to 40k keys (blocks split over
    many CTAs), one and two kv heads, e4m3 and bf16 caches."""
    import paged_gqa_gb300 as pg
    gen = torch.Generator().manual_seed(600 + i)
    n = [1, 7, 64, 150, 200, 40][i]
    hkv = [1, 2, 1, 1, 2, 1][i]
    Ls = torch.randint(1, 40000 if n <= 64 else 12000, (n,), generator=gen).tolist()
    qs = torch.randint(1, 5, (n,), generator=gen).tolist()
    spec = wl.CaseSpec(f"self-plan {i}", [(min(q, L), L) for q, L in zip(qs, Ls)], 16 * hkv, hkv, 16,
                       kv_dtype="bf16" if i == 5 else "e4m3")
    case = wl.make_case(spec, device="cuda", seed=600 + i, poison=True)
    outs = []
    for p in (0, 3):
        prev = pg.paged_gqa_set_path(p)
        try:
            outs.append(gu.run_library(case))
            assert pg.paged_gqa_last_plan()["verify_self_planned"] == (1 if p == 0 else 0)
        finally:
            pg.paged_gqa_set_path(prev)
    assert torch.isfinite(outs[0].float()).all()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16)), f"case {i}"


def test_decode_batch(path):
    """Pure decode: every sequence has one new token (q_len 1), G = 8, two kv heads."""
    gen = torch.Generator().manual_seed(31)
    seqs = [(1, int(L)) for L in torch.randint(1, 3000, (40,), generator=gen)]
    spec = wl.CaseSpec("decode", seqs, 16, 2, 16)
    case = wl.make_case(spec, device="cuda", seed=31, poison=True)
    gu.check_full(case, gu.run_library(case), "decode batch")


def test_longer_mtp_q5_to_q8(path):
    """q_len 5-8 with G = 16: 80-128 rows per kv head, past the 64-row verify blocks."""
    gen = torch.Generator().manual_seed(32)
    seqs = [(int(q), int(L)) for q, L in zip(torch.randint(5, 9, (24,), generator=gen),
                                                torch.randint(8, 2500, (24,), generator=gen))]
    spec = wl.CaseSpec("mtp q5-8", seqs, 16, 1, 16)
    case = wl.make_case(spec, device="cuda", seed=32, poison=True)
    gu.check_full(case, gu.run_library(case), "mtp q5-8")


@pytest.mark.parametrize("q_dtype", ["bf16", "e4m3"])
def test_group_of_32(path, q_dtype):
    """G = 32 (32 q heads on one kv head): 32-128 rows for q_len 1-4, both block classes."""
    spec = wl.CaseSpec("g32", [(1, 700), (2, 900), (3, 1300), (4, 400)], 32, 1, 64, q_dtype=q_dtype)
    case = wl.make_case(spec, device="cuda", seed=33, poison=True)
    gu.check_full(case, gu.run_library(case), f"G=32 {q_dtype}")


def test_long_single_sequence_is_split(path):
    """One sequence, one kv head: its keys are cut across all CTAs and merged."""
    spec = wl.CaseSpec("long", [(4, 40000)], 16, 1, 16)
    case = wl.make_case(spec, device="cuda", seed=13, poison=True)
    gu.check_full(case, gu.run_library(case), "long split")


def test_output_does_not_depend_on_untouched_rows():
    """Rows of zero-length queries are not written; everything else is."""
    spec = wl.CaseSpec("zeroq", [(0, 50), (3, 40), (0, 1), (2, 2)], 8, 1, 16)
    case = wl.make_case(spec, device="cuda", seed=21, poison=True)
    got = gu.run_library(case)
    gu.check_full(case, got, "zero-length queries")


def test_strided_views():
    """Non-packed q/out/cache/block-table strides (views into larger buffers)."""
    gen = torch.Generator().manual_seed(31)
    spec = wl.random_small_spec(gen, group=8, num_kv_heads=2, page_size=16, q_lens=[3, 4, 70], max_ctx=500)
    base = wl.make_case(spec, device="cuda", seed=31, poison=True)
    T, Hq, D = base.q.shape
    qbig = torch.zeros(T, Hq + 3, D + 64, dtype=base.q.dtype, device="cuda")
    qbig[:, :Hq, :D] = base.q
    NB, P, Hkv, _ = base.k_cache.shape
    kbig = torch.zeros(NB, P + 1, Hkv + 1, D + 32, dtype=base.k_cache.dtype, device="cuda")
    kbig[:, :P, :Hkv, :D] = base.k_cache
    vbig = torch.zeros(NB + 2, P, Hkv, D + 16, dtype=base.v_cache.dtype, device="cuda")
    vbig[:NB, :, :, :D] = base.v_cache
    btbig = torch.full((base.block_table.shape[0], base.block_table.shape[1] + 7), -1, dtype=torch.int32, device="cuda")
    btbig[:, :base.block_table.shape[1]] = base.block_table
    case = wl.Case(spec, qbig[:, :Hq, :D], kbig[:, :P, :Hkv, :D], vbig[:NB, :, :, :D],
                   btbig[:, :base.block_table.shape[1]], base.seq_lens, base.query_start_loc,
                   base.q_descale, base.k_descale, base.v_descale, base.softmax_scale)
    outbig = torch.full((T, Hq + 1, D + 8), float("nan"), dtype=torch.bfloat16, device="cuda")
    got = gu.run_library(case, out=outbig[:, :Hq, :D])
    gu.check_full(base, got.contiguous(), "strided")
    assert torch.isnan(outbig[:, Hq:, :].float()).all() and torch.isnan(outbig[:, :, D:].float()).all()


def test_device_errors_are_flagged_without_trapping():
    import paged_gqa_gb300 as pg
    spec = wl.CaseSpec("bad", [(2, 40), (3, 30)], 4, 1, 16)
    case = wl.make_case(spec, device="cuda", seed=41)
    # a page id outside [0, NB) for sequence 0
    bt = case.block_table.clone()
    bt[0, 1] = case.k_cache.shape[0] + 5
    bad = wl.Case(spec, case.q, case.k_cache, case.v_cache, bt, case.seq_lens, case.query_start_loc,
                  case.q_descale, case.k_descale, case.v_descale, case.softmax_scale)
    gu.run_library(bad, check_errors=False)
    assert pg.paged_gqa_check_device_errors() == -5
    # q_len > L for sequence 1: its rows are zeroed, the error is reported
    sl = case.seq_lens.clone()
    sl[1] = 2
    bad = wl.Case(spec, case.q, case.k_cache, case.v_cache, case.block_table, sl, case.query_start_loc,
                  case.q_descale, case.k_descale, case.v_descale, case.softmax_scale)
    out = gu.run_library(bad, check_errors=False)
    assert pg.paged_gqa_check_device_errors() == -5
    assert (out[2:5].float() == 0).all()
    # the error word was cleared; a good call reports nothing
    gu.run_library(case)
    assert pg.paged_gqa_check_device_errors() == 0


def test_caller_workspace_matches_library_workspace():
    import paged_gqa_gb300 as pg
    case = _small(77, group=16, num_kv_heads=1, page_size=16, q_lens=[4, 4, 2], max_ctx=5000)
    ref = gu.run_library(case)
    spec = case.spec
    nbytes = pg.paged_gqa_workspace_size(spec.num_seqs, spec.total_q, spec.num_q_heads, spec.num_kv_heads,
                                         spec.page_size, case.block_table.shape[1], 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(ref)
    pg.paged_gqa_attn_ex(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                         case.query_start_loc, 1.0, case.k_descale, case.v_descale, case.softmax_scale, out, ws)
    assert pg.paged_gqa_check_device_errors() == 0
    assert torch.equal(out, ref)
    with pytest.raises(pg.PagedGQAError, match="WORKSPACE"):
        pg.paged_gqa_attn_ex(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                             case.query_start_loc, 1.0, case.k_descale, case.v_descale, case.softmax_scale,
                             out, ws[: nbytes // 2])


@pytest.mark.parametrize("fill", ["zeros", "ones", "random", "left_by_another_shape"])
def test_caller_workspace_needs_no_initialisation(fill):
    """The split counters carry a per-call tag: a caller workspace filled with any bytes,
    or left by a call of another shape, gives the library workspace's result exactly, on
    both planning paths and over repeated calls."""
    import paged_gqa_gb300 as pg
    case = _small(78, group=16, num_kv_heads=1, page_size=16, q_lens=[4, 4, 2, 3], max_ctx=20000)
    other = _small(79, group=8, num_kv_heads=2, page_size=64, q_lens=[70, 4, 4, 1, 2], max_ctx=9000)
    ref = gu.run_library(case)
    nbytes = max(pg.paged_gqa_workspace_size(c.spec.num_seqs, c.spec.total_q, c.spec.num_q_heads,
                                             c.spec.num_kv_heads, c.spec.page_size, c.block_table.shape[1], 0)
                 for c in (case, other))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if fill == "zeros":
        ws.zero_()
    elif fill == "ones":
        ws.fill_(255)
    elif fill == "random":
        ws.copy_(torch.randint(0, 256, (nbytes,), generator=torch.Generator().manual_seed(5), dtype=torch.uint8))
    else:
        o = torch.empty(other.q.shape, dtype=torch.bfloat16, device="cuda")
        pg.paged_gqa_attn_ex(other.q, other.k_cache, other.v_cache, other.block_table, other.seq_lens,
                             other.query_start_loc, 1.0, other.k_descale, other.v_descale, other.softmax_scale,
                             o, ws)
    for path in (0, 3, 0):
        prev = pg.paged_gqa_set_path(path)
        try:
            out = torch.full_like(ref, float("nan"))
            pg.paged_gqa_attn_ex(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                 case.query_start_loc, 1.0, case.k_descale, case.v_descale, case.softmax_scale,
                                 out, ws)
            assert pg.paged_gqa_check_device_errors() == 0
        finally:
            pg.paged_gqa_set_path(prev)
        assert torch.equal(out, ref), f"fill {fill}, path {path}"


def test_deterministic_across_calls():
    case = _small(88, group=16, num_kv_heads=2, page_size=16, q_lens=[4, 3, 2, 4], max_ctx=9000)
    a = gu.run_library(case)
    b = gu.run_library(case)
    assert torch.equal(a, b)
