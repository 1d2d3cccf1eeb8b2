"""paged_gqa_attn_noalloc against paged_gqa_attn (GPU).

The no-allocation entry point is for callers that cannot allocate device memory when
they run attention (allocator callbacks, runtimes with a fixed device footprint). It
must give the results of the regular entry point. It shares one scratch array across
calls, so the test calls it several times in a row, on different problems and back
again, and checks every call.
"""
import ctypes

import pytest
import torch

import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import paged_gqa_gb300 as pg
    from paged_gqa_gb300 import _binding as B
    fn = pg.load().paged_gqa_attn_noalloc
    P = ctypes.POINTER(B.PgTensor)
    fn.argtypes = [P, P, P, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_float, P, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn, B


def _call_noalloc(case, out) -> int:
    fn, B = _noalloc_fn()
    d = [B._desc(t) for t in (case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                              case.query_start_loc)]
    o = B._desc(out)
    return fn(*[ctypes.byref(x) for x in d], case.k_descale, case.v_descale, case.softmax_scale,
              ctypes.byref(o), torch.cuda.current_stream().cuda_stream)


def _cases():
    gen = torch.Generator().manual_seed(4242)
    specs = [
        # verify blocks, one long sequence split across CTAs (partials + merge in the scratch)
        wl.CaseSpec("noalloc_verify", [(4, 9000), (2, 700), (3, 129)], 16, 1, 16),
        # prefill blocks with an FP8 query
        wl.random_small_spec(gen, group=8, num_kv_heads=1, page_size=64, q_lens=[150, 4], max_ctx=900,
                             q_dtype="e4m3", name="noalloc_prefill"),
        # bf16 cache, two kv heads
        wl.random_small_spec(gen, group=12, num_kv_heads=2, page_size=16, q_lens=[4, 1, 3], max_ctx=2000,
                             kv_dtype="bf16", name="noalloc_bf16"),
    ]
    return [wl.make_case(s, device="cuda", seed=11 + i, poison=True) for i, s in enumerate(specs)]


def test_noalloc_matches_regular_entry_point_on_calls_in_a_row():
    import paged_gqa_gb300 as pg
    cases = _cases()
    refs = [gu.run_library(c) for c in cases]
    # every case, then the first again: the scratch a call leaves behind must not leak
    for i in [0, 1, 2, 0]:
        case, ref = cases[i], refs[i]
        out = torch.full_like(ref, float("nan"))
        st = _call_noalloc(case, out)
        assert st == 0, pg.paged_gqa_last_error()
        assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
        gu.compare(out, ref.float().cpu().numpy().astype("float64"), f"no-alloc vs regular, case {i}")


def test_noalloc_rejects_calls_beyond_its_scratch():
    import paged_gqa_gb300 as pg
    # a million sequences (one query token in all, the rest with q_len 0) on two kv heads:
    # their verify blocks alone need more than the 64 MiB scratch
    n = 1 << 20
    need = pg.paged_gqa_workspace_size(n, 1, 32, 2, 16, 1, torch.cuda.current_device())
    assert need > (64 << 20)
    q = torch.zeros(1, 32, 256, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(4, 16, 2, 256, dtype=torch.uint8, device="cuda")
    qsl = torch.ones(n + 1, dtype=torch.int32, device="cuda")
    qsl[0] = 0
    case = wl.Case(wl.CaseSpec("big", [(1, 1)], 32, 2, 16), q, kv, kv,
                   torch.zeros(n, 1, dtype=torch.int32, device="cuda"),
                   torch.ones(n, dtype=torch.int32, device="cuda"), qsl, 1.0, 1.0, 1.0, 1.0 / 16)
    out = torch.zeros(1, 32, 256, dtype=torch.bfloat16, device="cuda")
    st = _call_noalloc(case, out)
    assert st == -6
    assert "workspace too small" in pg.paged_gqa_last_error()
