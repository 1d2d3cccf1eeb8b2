"""Failure detection on the GPU without a fault: a bounded device wait that runs out.

The tcgen05 kernels bound every mbarrier wait. The library's failure-path hook makes every
CTA's softmax warps wait on a shared-memory barrier that nothing ever arrives on, with a
short limit; the wait runs out, the CTA records a timeout in the device error word and
takes its abort path (the other roles give up, drain their own TMA copies and MMAs, TMEM is
freed). The host must read PG_ERR_TIMEOUT, and the next call, with the hook off, must be
correct: the context stays usable.
"""
import pytest
import torch

import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

PG_ERR_TIMEOUT = -4

CASES = {
    # verify blocks (q_len x G <= 64 rows), one sequence long enough to be split
    "verify": wl.CaseSpec("stall_verify", [(4, 3000), (2, 700), (3, 129)], 16, 1, 16),
    # prefill blocks (128-row blocks), FP8 q
    "prefill": wl.CaseSpec("stall_prefill", [(150, 400), (40, 300)], 8, 1, 64, q_dtype="e4m3"),
}


@pytest.mark.parametrize("which", sorted(CASES))
def test_a_wait_that_runs_out_reports_timeout_and_the_next_call_is_correct(which):
    import paged_gqa_gb300 as pg
    case = wl.make_case(CASES[which], device="cuda", seed=77, poison=True)
    assert pg.paged_gqa_check_device_errors() == 0
    prev = pg.paged_gqa_set_stall_test(200_000)  # 200 us
    try:
        gu.run_library(case, check_errors=False)
        st = pg.paged_gqa_check_device_errors()
    finally:
        pg.paged_gqa_set_stall_test(prev)
    assert st == PG_ERR_TIMEOUT, pg.paged_gqa_last_error()
    assert "bounded wait" in pg.paged_gqa_last_error()
    # hook off: the same call on the same context matches the oracle, with no error
    bits = 2 if which == "verify" else 4
    got = gu.run_library(case)
    assert pg.paged_gqa_last_plan()["path_bits"] & bits
    gu.check_full(case, got, f"after a timeout ({which})")


def test_sparse_kernel_wait_that_runs_out_reports_timeout():
    import paged_gqa_gb300 as pg
    from tests.test_sparse_gpu import _oracle, _run
    gen = torch.Generator().manual_seed(78)
    spec = wl.random_small_spec(gen, group=12, num_kv_heads=2, page_size=64, q_lens=[6, 3], max_ctx=800,
                                kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=78, poison=True)
    idx = wl.sparse_indices(case.spec, 200, device="cuda", seed=78)
    prev_path = pg.paged_gqa_set_path(2)  # the tcgen05 sparse kernel
    prev = pg.paged_gqa_set_stall_test(200_000)
    try:
        _run(case, idx, check=False)
        st = pg.paged_gqa_check_device_errors()
    finally:
        pg.paged_gqa_set_stall_test(prev)
    try:
        assert st == PG_ERR_TIMEOUT, pg.paged_gqa_last_error()
        gu.compare(_run(case, idx), _oracle(case, idx), "sparse after a timeout")
    finally:
        pg.paged_gqa_set_path(prev_path)
