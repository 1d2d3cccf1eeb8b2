"""Pins of the per-tensor FP8 Q quantisation oracle (CPU only)."""
import numpy as np
import torch

import oracle
import workloads as wl
from oracle import quant_q as qq


def _bf16_values(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).float().numpy()


def test_largest_element_takes_the_largest_code():
    q = _bf16_values((40, 8, 256), 1, 3.0)
    codes, d = qq.quantize_q(q)
    i = np.unravel_index(np.argmax(np.abs(q)), q.shape)
    assert codes[i] & 0x7F == 0x7E  # +-448
    assert (codes & 0x7F).max() == 0x7E
    assert d == np.float32(np.abs(q).max() / np.float32(448))


def test_dequantised_values_lie_within_half_a_step():
    q = np.concatenate([_bf16_values((30, 4, 256), 2), _bf16_values((30, 4, 256), 3, 1e-3)])
    codes, d = qq.quantize_q(q)
    deq = oracle.e4m3_table()[codes] * np.float64(d)
    y = np.abs(q.astype(np.float64)) / np.float64(d)   # the value in code units
    # e4m3 step: 2^(e-3) for y in [2^e, 2^(e+1)), e >= -6; 2^-9 below 2^-6 (subnormals)
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    step = 2.0 ** (e - 3)
    # half a step, plus the float32 rounding of q * inv (relative 2^-24, twice)
    bound = (0.5 * step + y * 2.0 ** -22) * np.float64(d)
    assert (np.abs(deq - q) <= bound).all()


def test_codes_agree_with_the_torch_cast():
    q = _bf16_values((64, 16, 256), 4, 7.0)
    codes, d = qq.quantize_q(q)
    d2, inv = qq.q_scales(q)
    assert d2 == d
    ref = (torch.from_numpy(q) * torch.tensor(inv)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (codes == ref).all()


def test_power_of_two_scaling_keeps_the_codes():
    q = _bf16_values((20, 8, 256), 5)
    c0, d0 = qq.quantize_q(q)
    for k in (-7, 1, 5):
        c, d = qq.quantize_q(q * np.float32(2.0 ** k))
        assert (c == c0).all() and d == d0 * np.float32(2.0 ** k)


def test_degenerate_scales():
    codes, d = qq.quantize_q(np.zeros((3, 2, 256), np.float32))
    assert d == 1.0 and (codes == 0).all()
    q = _bf16_values((3, 2, 256), 6)
    q[0, 0, 0] = np.inf
    assert qq.q_scales(q) == (1.0, 1.0)
    q = _bf16_values((3, 2, 256), 7)
    amax = np.abs(q).max()
    q[1, 1, 7] = np.nan
    d, _ = qq.q_scales(q)
    assert d == np.float32(np.float32(amax) / np.float32(448))  # NaNs do not enter amax


def test_attention_stays_within_fp8_error_of_the_bf16_q_attention():
    gen = torch.Generator().manual_seed(8)
    spec = wl.random_small_spec(gen, group=8, num_kv_heads=1, page_size=16, q_lens=[1, 4, 37],
                                max_ctx=300, kv_dtype="e4m3", q_dtype="bf16")
    case = wl.make_case(spec, seed=8)
    kw = dict(kv_dtype="e4m3", k_descale=case.k_descale, v_descale=case.v_descale,
              softmax_scale=spec.softmax_scale)
    got = qq.attention_quant_q(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                               case.query_start_loc, **kw)
    ref = oracle.attention(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                           case.query_start_loc, q_dtype="bf16", q_descale=1.0, **kw)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    # e4m3 keeps 3 mantissa bits: scores move by a few percent of their spread, not more
    assert 1e-4 < rel < 0.08, rel
    # a descale applied the wrong way round (or not at all) moves every output
    codes, d = qq.quantize_q(case.q.float().numpy())
    wrong = oracle.attention(torch.from_numpy(codes), case.k_cache, case.v_cache, case.block_table,
                             case.seq_lens, case.query_start_loc, q_dtype="e4m3", q_descale=1.0, **kw)
    assert np.linalg.norm(wrong - ref) / np.linalg.norm(ref) > 0.3
