"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: a dense,
unpaged brute force written with numpy matrices, torch's SDPA in fp64, closed
forms, invariants the definition implies, and torch's own e4m3 decode. A
plausible mistake in the oracle (a dropped term, an off-by-one causal bound, a
wrong head group, a wrong page walk, a transposed operand) fails at least one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

D = wl.HEAD_DIM


# ---------------------------------------------------------------- helpers --

def _dequant(t: torch.Tensor, dtype: str) -> torch.Tensor:
    """Independent decode through torch's own dtypes (not the oracle's)."""
    t = t.detach().cpu()
    if dtype == "e4m3":
        return t.view(torch.float8_e4m3fn).to(torch.float64)
    return t.to(torch.float64)


def _logical_kv(case, s):
    """K/V of sequence s in logical order [L, Hkv, D], gathered page by page."""
    spec = case.spec
    L = int(case.seq_lens[s])
    P = spec.page_size
    k = _dequant(case.k_cache, spec.kv_dtype) * case.k_descale
    v = _dequant(case.v_cache, spec.kv_dtype) * case.v_descale
    pages = [int(b) for b in case.block_table[s, : (L + P - 1) // P]]
    kk = torch.cat([k[b] for b in pages], 0)[:L]
    vv = torch.cat([v[b] for b in pages], 0)[:L]
    return kk.numpy(), vv.numpy()


def brute_force(case):
    """Dense attention per (sequence, kv head): full score matrix, explicit mask."""
    spec = case.spec
    qd = case.q_descale if spec.q_dtype == "e4m3" else 1.0
    q = _dequant(case.q, spec.q_dtype).numpy() * qd
    T, Hq, _ = q.shape
    G = spec.group
    out = np.zeros((T, Hq, D))
    qsl = case.query_start_loc.cpu().numpy()
    for s in range(spec.num_seqs):
        q0, q1 = int(qsl[s]), int(qsl[s + 1])
        qn, L = q1 - q0, int(case.seq_lens[s])
        if qn == 0:
            continue
        kk, vv = _logical_kv(case, s)
        # mask[t, j] = key j visible to query token t (bottom-right aligned)
        mask = np.arange(L)[None, :] <= (L - qn + np.arange(qn))[:, None]
        for h in range(Hq):
            kvh = h // G
            S = spec.softmax_scale * (q[q0:q1, h, :] @ kk[:, kvh, :].T)   # [qn, L]
            S = np.where(mask, S, -np.inf)
            S = S - S.max(axis=1, keepdims=True)
            Pm = np.exp(S)
            Pm /= Pm.sum(axis=1, keepdims=True)
            out[q0:q1, h, :] = Pm @ vv[:, kvh, :]
    return out


def _case(seed, *, group, hkv, page, q_lens, max_ctx, kv="e4m3", qd="bf16", poison=False, spare=3):
    gen = torch.Generator().manual_seed(seed)
    spec = wl.random_small_spec(gen, group=group, num_kv_heads=hkv, page_size=page, q_lens=q_lens,
                                max_ctx=max_ctx, kv_dtype=kv, q_dtype=qd, spare_pages=spare)
    return wl.make_case(spec, seed=seed, poison=poison)


SMALL = [
    dict(group=16, hkv=1, page=16, q_lens=[2, 4, 1], max_ctx=70, kv="e4m3", qd="bf16"),
    dict(group=8, hkv=1, page=64, q_lens=[5, 0, 3], max_ctx=150, kv="e4m3", qd="e4m3"),
    dict(group=3, hkv=2, page=16, q_lens=[4, 4], max_ctx=40, kv="bf16", qd="bf16"),
    dict(group=12, hkv=2, page=16, q_lens=[1, 7, 2], max_ctx=50, kv="e4m3", qd="bf16"),
    dict(group=1, hkv=3, page=32, q_lens=[6, 2], max_ctx=33, kv="bf16", qd="bf16"),
]


# ---------------------------------------------------------------- pins --

def test_e4m3_table_matches_torch():
    table = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.isnan(table[nan]).all()
    np.testing.assert_array_equal(table[~nan], ref[~nan])
    assert table[0x7E] == 448.0 and table[0x01] == 2.0 ** -9 and table[0x08] == 2.0 ** -6


@pytest.mark.parametrize("i", range(len(SMALL)))
def test_oracle_matches_dense_brute_force(i):
    case = _case(100 + i, **SMALL[i])
    got = oracle.attention_case(case)
    ref = brute_force(case)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_oracle_matches_torch_sdpa_fp64():
    case = _case(7, group=4, hkv=2, page=16, q_lens=[3, 5], max_ctx=60, kv="bf16", qd="bf16")
    spec = case.spec
    got = oracle.attention_case(case)
    q = case.q.to(torch.float64)
    qsl = case.query_start_loc.tolist()
    for s in range(spec.num_seqs):
        q0, q1 = qsl[s], qsl[s + 1]
        qn, L = q1 - q0, int(case.seq_lens[s])
        kk, vv = (torch.from_numpy(x) for x in _logical_kv(case, s))
        mask = torch.arange(L)[None, :] <= (L - qn + torch.arange(qn))[:, None]
        qq = q[q0:q1].transpose(0, 1)                                      # [Hq, qn, D]
        kr = kk.transpose(0, 1).repeat_interleave(spec.group, 0)           # [Hq, L, D]
        vr = vv.transpose(0, 1).repeat_interleave(spec.group, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, kr, vr, attn_mask=mask, scale=spec.softmax_scale).transpose(0, 1)
        np.testing.assert_allclose(got[q0:q1], ref.numpy(), rtol=1e-11, atol=1e-12)


def test_full_prefill_equals_top_left_causal():
    """q_len == L (nothing cached): ordinary causal attention."""
    spec = wl.CaseSpec("nocache", [(37, 37)], 2, 1, 16, q_dtype="bf16", kv_dtype="bf16")
    case = wl.make_case(spec, seed=3)
    got = oracle.attention_case(case)
    kk, vv = (torch.from_numpy(x) for x in _logical_kv(case, 0))
    qq = case.q.to(torch.float64).transpose(0, 1)
    kr = kk.transpose(0, 1).repeat_interleave(2, 0)
    vr = vv.transpose(0, 1).repeat_interleave(2, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(qq, kr, vr, is_causal=True,
                                                           scale=spec.softmax_scale).transpose(0, 1)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_page_permutation_invariance():
    case = _case(11, group=16, hkv=1, page=16, q_lens=[3, 2], max_ctx=90)
    base = oracle.attention_case(case)
    NB = case.k_cache.shape[0]
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(NB)
    case.k_cache = case.k_cache[perm].clone()      # new physical page i holds old page perm[i]
    case.v_cache = case.v_cache[perm].clone()
    bt = case.block_table.clone()
    valid = bt >= 0
    bt[valid] = inv[bt[valid].long()].to(torch.int32)
    case.block_table = bt
    np.testing.assert_array_equal(oracle.attention_case(case), base)


def test_single_token_is_decode_and_last_row_is_decode():
    """q_len=1 is decode over all L keys; the last row of a query block sees all L keys too."""
    case = _case(13, group=8, hkv=1, page=16, q_lens=[4], max_ctx=80)
    L = int(case.seq_lens[0])
    got = oracle.attention_case(case)
    kk, vv = _logical_kv(case, 0)
    q = case.q.to(torch.float64).numpy()
    for h in range(8):
        s = case.spec.softmax_scale * (kk[:, 0, :] @ q[3, h])
        w = np.exp(s - s.max())
        np.testing.assert_allclose(got[3, h], (w @ vv[:, 0, :]) / w.sum(), rtol=1e-11, atol=1e-12)
    # q_len = 1 on the same cache: a decode call at L equals the block's last row
    dec = wl.Case(case.spec, case.q[3:4].clone(), case.k_cache, case.v_cache, case.block_table,
                  case.seq_lens, torch.tensor([0, 1], dtype=torch.int32), 1.0,
                  case.k_descale, case.v_descale, case.softmax_scale)
    dec.spec = wl.CaseSpec("dec", [(1, L)], 8, 1, 16, kv_dtype="e4m3")
    np.testing.assert_allclose(oracle.attention_case(dec)[0], got[3], rtol=0, atol=0)


def test_two_kv_heads_equal_two_independent_problems():
    """32q/2kv equals two 16q/1kv problems on the per-head slices."""
    case = _case(17, group=16, hkv=2, page=16, q_lens=[4, 2, 3], max_ctx=64)
    got = oracle.attention_case(case)
    for kvh in range(2):
        sub = wl.Case(case.spec, case.q[:, kvh * 16:(kvh + 1) * 16].contiguous(),
                      case.k_cache[:, :, kvh:kvh + 1].contiguous(),
                      case.v_cache[:, :, kvh:kvh + 1].contiguous(),
                      case.block_table, case.seq_lens, case.query_start_loc, 1.0,
                      case.k_descale, case.v_descale, case.softmax_scale)
        sub.spec = wl.CaseSpec("half", case.spec.seqs, 16, 1, 16, kv_dtype="e4m3")
        np.testing.assert_array_equal(oracle.attention_case(sub), got[:, kvh * 16:(kvh + 1) * 16])


def test_poisoned_tails_and_spare_pages_do_not_matter():
    for kv in ("e4m3", "bf16"):
        clean = _case(19, group=4, hkv=1, page=16, q_lens=[2, 3], max_ctx=45, kv=kv)
        dirty = _case(19, group=4, hkv=1, page=16, q_lens=[2, 3], max_ctx=45, kv=kv, poison=True)
        a, b = oracle.attention_case(clean), oracle.attention_case(dirty)
        assert np.isfinite(b).all()
        np.testing.assert_array_equal(a, b)


def test_lse_split_merge_reproduces_unsplit():
    """Split keys into segments, softmax each, merge by log-sum-exp: same result."""
    case = _case(23, group=2, hkv=1, page=16, q_lens=[1], max_ctx=300)
    out, lse = oracle.attention_case(case, with_lse=True)
    kk, vv = _logical_kv(case, 0)
    q = case.q.to(torch.float64).numpy()[0, 0]
    s = case.spec.softmax_scale * (kk[:, 0, :] @ q)
    cuts = [0, 37, 128, 129, len(s)]
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        m = s[a:b].max()
        w = np.exp(s[a:b] - m)
        parts.append(((w @ vv[a:b, 0, :]) / w.sum(), m + math.log(w.sum())))
    M = max(p[1] for p in parts)
    ws = [math.exp(p[1] - M) for p in parts]
    merged = sum(w * p[0] for w, p in zip(ws, parts)) / sum(ws)
    np.testing.assert_allclose(merged, out[0, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(M + math.log(sum(ws)), lse[0, 0], rtol=1e-12)


def test_closed_forms_constant_v_and_zero_q():
    case = _case(29, group=4, hkv=1, page=16, q_lens=[3, 4], max_ctx=50, kv="bf16")
    # V = c everywhere: output is exactly c
    v = case.v_cache.clone()
    v[:] = 0.75
    c2 = wl.Case(case.spec, case.q, case.k_cache, v, case.block_table, case.seq_lens,
                 case.query_start_loc, 1.0, 1.0, 1.0, case.softmax_scale)
    np.testing.assert_allclose(oracle.attention_case(c2), 0.75, rtol=0, atol=1e-15)
    # Q = 0: uniform weights, so each row is the mean of V over keys 0..pos
    q0 = torch.zeros_like(case.q)
    c3 = wl.Case(case.spec, q0, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                 case.query_start_loc, 1.0, 1.0, 1.0, case.softmax_scale)
    got = oracle.attention_case(c3)
    qsl = case.query_start_loc.tolist()
    for s in range(case.spec.num_seqs):
        qn, L = qsl[s + 1] - qsl[s], int(case.seq_lens[s])
        _, vv = _logical_kv(c3, s)
        for t in range(qn):
            pos = L - qn + t
            np.testing.assert_allclose(got[qsl[s] + t, 0], vv[: pos + 1, 0].mean(0), rtol=1e-13, atol=1e-14)


def test_closed_form_dominant_key():
    case = _case(31, group=2, hkv=1, page=16, q_lens=[2], max_ctx=40, kv="bf16")
    L = int(case.seq_lens[0])
    q = torch.zeros_like(case.q)
    q[:, :, 0] = 16.0
    k = case.k_cache.clone() * 0.01
    j = L // 2                                         # a key both rows can see
    b = int(case.block_table[0, j // 16])
    k[b, j % 16, 0, 0] = 32.0                          # score 16*32/16 = 32 >> others
    c = wl.Case(case.spec, q, k, case.v_cache, case.block_table, case.seq_lens,
                case.query_start_loc, 1.0, 1.0, 1.0, case.softmax_scale)
    got = oracle.attention_case(c)
    vj = case.v_cache[b, j % 16, 0].to(torch.float64).numpy()
    np.testing.assert_allclose(got[0, 0], vj, atol=1e-9)
    np.testing.assert_allclose(got[1, 1], vj, atol=1e-9)


def test_rows_subset_matches_full():
    case = _case(37, group=8, hkv=2, page=16, q_lens=[3, 1, 4], max_ctx=70)
    full = oracle.attention_case(case)
    rows = np.array([0, 5, 17, 40, 7 * 16 + 15], dtype=np.int64)
    sub = oracle.attention_case(case, rows=rows)
    np.testing.assert_array_equal(sub, full.reshape(-1, D)[rows])


def test_errors_are_reported():
    case = _case(41, group=2, hkv=1, page=16, q_lens=[2], max_ctx=40)
    bad = case.block_table.clone()
    bad[0, 0] = case.k_cache.shape[0]
    c = wl.Case(case.spec, case.q, case.k_cache, case.v_cache, bad, case.seq_lens,
                case.query_start_loc, 1.0, case.k_descale, case.v_descale, case.softmax_scale)
    with pytest.raises(ValueError, match="block-table"):
        oracle.attention_case(c)
    c = wl.Case(case.spec, case.q, case.k_cache, case.v_cache, case.block_table,
                torch.tensor([1], dtype=torch.int32), case.query_start_loc, 1.0,
                case.k_descale, case.v_descale, case.softmax_scale)
    with pytest.raises(ValueError, match="bad argument"):
        oracle.attention_case(c)


def test_config_specs_match_their_descriptions():
    s1 = wl.config_spec(1)
    assert s1.seqs == [(2, 600)] and s1.used_pages == 38 and s1.used_pages + s1.spare_pages == 64
    s2 = wl.config_spec(2)
    assert len(s2.seqs) == 64 and all(q == 4 and 1024 <= L <= 32768 for q, L in s2.seqs)
    s3 = wl.config_spec(3)
    assert len(s3.seqs) == 256 and {q for q, _ in s3.seqs} == {2, 3, 4} and s3.kv_bytes == 2147483648
    s4 = wl.config_spec(4)
    assert s4.flops == 4 * 256 * 8 * 402661376
    s5 = wl.config_spec(5)
    assert len(s5.seqs) == 520 and s5.group == 12 and s5.page_size == 64
