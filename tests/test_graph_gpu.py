"""The caller-workspace call captured in a CUDA graph and replayed with new inputs.

The plan runs on the device and the call allocates nothing, so one capture serves every
replay with the same shapes: replays with fresh q values (and a changed block table, the
same sizes) must match the oracle on each replay's inputs."""
import pytest
import torch

import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _fresh_q(case, gen):
    """New N(0,1) q values drawn on the host. A case draws K, V and Q from CUDA generators
    seeded seed + 1 .. seed + 3; a replay q drawn from one of those streams would repeat
    rows of K, each such row scoring |k|^2 / 16 against its twin, so the attention would be
    one-hot and the output as large as a V value (|out| ~ 4, where bf16 rounding alone is
    up to 0.016: above the absolute bar)."""
    return torch.randn(case.q.shape, generator=gen).to(device=case.q.device, dtype=torch.bfloat16)


def test_attn_ex_replays_inside_a_cuda_graph():
    import paged_gqa_gb300 as pg
    gen = torch.Generator().manual_seed(120)
    spec = wl.random_small_spec(gen, group=16, num_kv_heads=1, page_size=16, q_lens=[4, 3, 150, 1], max_ctx=900,
                                kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=120, poison=True)
    ws_bytes = pg.paged_gqa_workspace_size(spec.num_seqs, spec.total_q, spec.num_q_heads, spec.num_kv_heads,
                                           spec.page_size, case.block_table.shape[1], torch.cuda.current_device())
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")

    def call():
        pg.paged_gqa_attn_ex(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                             case.query_start_loc, 1.0, case.k_descale, case.v_descale, case.softmax_scale, out, ws)

    call()  # outside capture first: per-device state and kernel attributes are set up once
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(121)
    for trial in range(3):
        case.q.copy_(_fresh_q(case, g))
        if trial == 2:
            # same sizes, other physical pages: swap two sequences' first pages in the table
            bt = case.block_table
            a, b = bt[0, 0].item(), bt[2, 0].item()
            case.k_cache[[a, b]] = case.k_cache[[b, a]].clone()
            case.v_cache[[a, b]] = case.v_cache[[b, a]].clone()
            bt[0, 0], bt[2, 0] = b, a
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
        gu.check_full(case, out, f"graph replay {trial}")


@pytest.mark.parametrize("path", [0, 3])
def test_split_blocks_merge_on_every_replay(path):
    """Long contexts split every verify block across many CTAs, so each replay merges
    through the split counters; a counter left by the previous replay must not count (the
    workspace's epoch word gives every replay a new tag). Both planning paths."""
    import paged_gqa_gb300 as pg
    spec = wl.CaseSpec("long graph", [(4, 40000), (2, 17000), (3, 30000)], 16, 1, 16)
    case = wl.make_case(spec, device="cuda", seed=122, poison=True)
    ws_bytes = pg.paged_gqa_workspace_size(spec.num_seqs, spec.total_q, spec.num_q_heads, spec.num_kv_heads,
                                           spec.page_size, case.block_table.shape[1], torch.cuda.current_device())
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")
    prev = pg.paged_gqa_set_path(path)
    try:
        def call():
            pg.paged_gqa_attn_ex(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                 case.query_start_loc, 1.0, case.k_descale, case.v_descale, case.softmax_scale,
                                 out, ws)

        call()
        torch.cuda.synchronize()
        assert pg.paged_gqa_last_plan()["verify_self_planned"] == (1 if path == 0 else 0)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        torch.cuda.synchronize()
        g = torch.Generator().manual_seed(123)
        for trial in range(4):
            case.q.copy_(_fresh_q(case, g))
            out.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
            gu.check_full(case, out, f"long graph replay {trial}, path {path}")
    finally:
        pg.paged_gqa_set_path(prev)
