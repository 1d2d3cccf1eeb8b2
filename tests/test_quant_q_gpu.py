"""paged_gqa_attn_quant_q on the GPU against the oracle: a bf16 Q quantised per tensor to
e4m3 inside the call, then the attention, compared element by element."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from oracle import quant_q as qq
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _run(case, out=None):
    import paged_gqa_gb300 as pg
    T, Hq = case.q.shape[0], case.q.shape[1]
    if out is None:
        out = torch.full((T, Hq, wl.HEAD_DIM), float("nan"), dtype=torch.bfloat16, device=case.q.device)
    pg.paged_gqa_attn_quant_q(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                              case.query_start_loc, case.k_descale, case.v_descale, case.softmax_scale, out)
    assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
    return out


def _oracle(case, seq_ids=None, rows=None, scales=None):
    c = gu.to_device(case, "cpu") if seq_ids is None else gu.subcase(case, seq_ids)
    return qq.attention_quant_q(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens, c.query_start_loc,
                                kv_dtype="e4m3", k_descale=case.k_descale, v_descale=case.v_descale,
                                softmax_scale=case.spec.softmax_scale, rows=rows, scales=scales)


SMALL = [
    # (group, kv heads, page size, q_lens, max context)
    (16, 1, 16, [1, 2, 3, 4, 4, 1], 900),        # verify class only
    (8, 1, 64, [130, 17, 300, 1], 1500),         # prefill class and a decode row
    (12, 2, 32, [4, 9, 64, 2, 200], 700),        # both classes, two kv heads
    (24, 2, 64, [4, 3, 40, 4], 3000),            # the mixed workload's head layout
]


@pytest.mark.parametrize("i", range(len(SMALL)))
def test_small_cases_match_the_oracle(i):
    G, hkv, page, q_lens, ctx = SMALL[i]
    gen = torch.Generator().manual_seed(70 + i)
    spec = wl.random_small_spec(gen, group=G, num_kv_heads=hkv, page_size=page, q_lens=q_lens, max_ctx=ctx,
                                kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=70 + i, poison=True)
    gu.compare(_run(case), _oracle(case), f"quant-q case {i}")


def test_scaled_q_and_an_all_zero_q():
    gen = torch.Generator().manual_seed(80)
    spec = wl.random_small_spec(gen, group=8, num_kv_heads=1, page_size=16, q_lens=[4, 150, 1], max_ctx=600,
                                kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=80, poison=True)
    q0 = case.q.clone()
    case.q = (q0.float() * 1e-4).to(torch.bfloat16)
    gu.compare(_run(case), _oracle(case), "q x 1e-4")
    # x 3 and x 37: peaked rows whose outputs approach single V rows (|out| up to ~4), where
    # rounding the exact output to bf16 alone moves it by up to 2^-8 of its size (7.8e-3 at
    # |out| = 4, measured on the oracle); the bar adds that term to the max-abs bound
    for scale in (3.0, 37.0):
        case.q = (q0.float() * scale).to(torch.bfloat16)
        got = _run(case).float().cpu().numpy().astype(np.float64)
        ref = _oracle(case)
        diff = np.abs(got - ref)
        assert (diff <= gu.MAX_ABS + 2.0 ** -8 * np.abs(ref)).all(), (scale, float(diff.max()))
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= gu.REL_L2, scale
    case.q = torch.zeros_like(q0)  # descale 1, every code 0: the mean of the visible V rows
    gu.compare(_run(case), _oracle(case), "zero q")


def test_prefix_prefill_with_bf16_q():
    """The prefix-hit prefill shape (16384 new tokens on 32768, 8 q / 1 kv head, 64-token
    pages) with a bf16 Q that the call quantises: sampled rows and the end rows."""
    spec = wl.config_spec(4)
    spec.q_dtype = "bf16"
    case = wl.make_case(spec, device="cuda", seed=0, poison=True)
    got = _run(case).reshape(-1, wl.HEAD_DIM)
    scales = qq.q_scales(case.q.float().cpu().numpy())
    gen = torch.Generator().manual_seed(4)
    rows = torch.cat([torch.arange(8), torch.randperm(16384 * 8, generator=gen)[:256],
                      torch.arange(16383 * 8, 16384 * 8)]).numpy().astype(np.int64)
    ref = _oracle(case, [0], rows=rows, scales=scales)
    gu.compare(got[torch.from_numpy(rows).cuda()], ref, "prefix prefill, quantised q")


def test_mixed_serving_step():
    """The mixed workload (8 prefill + 512 verify sequences, 24 q / 2 kv heads) through the
    quantising call: whole short sequences and sampled rows of the long ones."""
    case = wl.make_case(wl.config_spec(5), device="cuda", seed=0, poison=True)
    got = _run(case).reshape(-1, wl.HEAD_DIM)
    scales = qq.q_scales(case.q.float().cpu().numpy())
    qsl = case.query_start_loc.cpu().tolist()
    Hq = case.spec.num_q_heads
    # verify sequences 8.., whole
    picks = [8, 9, 300, 519]
    sub_rows, full_rows, base = [], [], 0
    for s in picks:
        n = (qsl[s + 1] - qsl[s]) * Hq
        sub_rows.append(np.arange(n) + base)
        full_rows.append(np.arange(n) + qsl[s] * Hq)
        base += n
    ref = _oracle(case, picks, rows=np.concatenate(sub_rows).astype(np.int64), scales=scales)
    gu.compare(got[torch.from_numpy(np.concatenate(full_rows)).cuda()], ref, "mixed: verify sequences")
    # prefill sequences 0 and 7: 96 random rows each plus each one's last token (all heads)
    gen = torch.Generator().manual_seed(5)
    for s in (0, 7):
        n = (qsl[s + 1] - qsl[s]) * Hq
        local = np.unique(np.concatenate([torch.randperm(n, generator=gen)[:96].numpy(), np.arange(n - Hq, n)]))
        ref = _oracle(case, [s], rows=local.astype(np.int64), scales=scales)
        gu.compare(got[torch.from_numpy(local + qsl[s] * Hq).cuda()], ref, f"mixed: prefill sequence {s}")


def test_the_warp_mma_path_refuses_to_quantise():
    import paged_gqa_gb300 as pg
    gen = torch.Generator().manual_seed(81)
    spec = wl.random_small_spec(gen, group=8, num_kv_heads=1, page_size=16, q_lens=[4], max_ctx=100,
                                kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, device="cuda", seed=81)
    out = torch.zeros(case.q.shape, dtype=torch.bfloat16, device="cuda")
    pg.paged_gqa_set_path(1)
    try:
        with pytest.raises(pg.PagedGQAError) as ei:
            pg.paged_gqa_attn_quant_q(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                      case.query_start_loc, case.k_descale, case.v_descale, case.softmax_scale,
                                      out)
        assert ei.value.status == -2
    finally:
        pg.paged_gqa_set_path(0)
    torch.cuda.synchronize()
    assert (out == 0).all()
