"""Pins of the sparse paged GQA oracle (CPU only).

The sparse oracle is checked against the dense oracle (pinned in test_oracle.py) and
against invariants of the definition: a full ascending list is the dense attention; a
list's order does not matter; a list equals the dense attention over a cache that holds
exactly the listed keys; entries that are negative or past the row's causal limit are not
used; a key listed twice counts twice; a row with nothing to attend is zero.
"""
import numpy as np
import torch

import oracle
import workloads as wl

KW = dict(q_dtype="bf16", kv_dtype="e4m3", q_descale=1.0)


def _case(seed=0, seqs=((5, 40), (1, 17), (3, 3)), G=4, Hkv=2, P=16):
    spec = wl.CaseSpec("sparse_pin", list(seqs), G * Hkv, Hkv, P, spare_pages=2)
    return wl.make_case(spec, seed=seed)


def _sparse(case, idx, **kw):
    return oracle.sparse_attention(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                   case.query_start_loc, torch.as_tensor(idx, dtype=torch.int32), **KW,
                                   k_descale=case.k_descale, v_descale=case.v_descale,
                                   softmax_scale=case.spec.softmax_scale, **kw)


def _dense(case, **kw):
    return oracle.attention_case(case, **kw)


def _limits(case):
    qsl, sl = case.query_start_loc.tolist(), case.seq_lens.tolist()
    lim = []
    for s in range(len(sl)):
        qn = qsl[s + 1] - qsl[s]
        lim += [sl[s] - qn + t for t in range(qn)]
    return np.array(lim)


def test_full_ascending_list_is_the_dense_attention():
    case = _case(1)
    T, Hkv = case.q.shape[0], case.spec.num_kv_heads
    Lmax = int(case.seq_lens.max())
    idx = np.broadcast_to(np.arange(Lmax, dtype=np.int32), (T, Hkv, Lmax)).copy()
    got, lse = _sparse(case, idx, with_lse=True)
    ref, rlse = _dense(case, with_lse=True)
    assert np.allclose(got, ref, rtol=0, atol=1e-12) and np.allclose(lse, rlse, rtol=0, atol=1e-12)


def test_order_of_the_list_does_not_matter():
    case = _case(2)
    T, Hkv = case.q.shape[0], case.spec.num_kv_heads
    rng = np.random.default_rng(2)
    idx = rng.integers(-3, 45, size=(T, Hkv, 23)).astype(np.int32)
    perm = np.argsort(rng.random(idx.shape), axis=2)
    shuffled = np.take_along_axis(idx, perm, axis=2)
    assert np.allclose(_sparse(case, idx), _sparse(case, shuffled), rtol=0, atol=1e-12)


def test_a_list_equals_dense_attention_over_a_cache_of_exactly_those_keys():
    """Gather each row's used keys (duplicates included) into a fresh paged cache whose
    single query token sees all of them; the dense oracle there must give the same row."""
    case = _case(3)
    T, Hkv, G = case.q.shape[0], case.spec.num_kv_heads, case.spec.group
    P = case.spec.page_size
    rng = np.random.default_rng(3)
    K = 19
    idx = rng.integers(-2, 42, size=(T, Hkv, K)).astype(np.int32)
    idx[0, 0, :4] = [7, 7, 7, 2]  # duplicates
    got = _sparse(case, idx)
    lim = _limits(case)
    qsl = case.query_start_loc.tolist()
    bt = case.block_table.numpy()
    for t in range(T):
        s = max(i for i in range(len(qsl) - 1) if qsl[i] <= t)
        for h in range(Hkv):
            used = [int(p) for p in idx[t, h] if 0 <= p <= lim[t]]
            if not used:
                assert (got[t, h * G:(h + 1) * G] == 0).all()
                continue
            n = len(used)
            pages = (n + P - 1) // P
            k = torch.zeros(pages, P, Hkv, 256, dtype=torch.uint8)
            v = torch.zeros_like(k)
            for i, p in enumerate(used):
                b = bt[s, p // P]
                k[i // P, i % P] = case.k_cache[b, p % P]
                v[i // P, i % P] = case.v_cache[b, p % P]
            sub = wl.Case(wl.CaseSpec("one", [(1, n)], case.spec.num_q_heads, Hkv, P), case.q[t:t + 1], k, v,
                          torch.arange(pages, dtype=torch.int32).view(1, -1), torch.tensor([n], dtype=torch.int32),
                          torch.tensor([0, 1], dtype=torch.int32), 1.0, case.k_descale, case.v_descale,
                          case.spec.softmax_scale)
            ref = _dense(sub)[0, h * G:(h + 1) * G]
            assert np.allclose(got[t, h * G:(h + 1) * G], ref, rtol=0, atol=1e-12), (t, h)


def test_entries_outside_the_causal_range_are_not_used():
    case = _case(4)
    T, Hkv = case.q.shape[0], case.spec.num_kv_heads
    lim = _limits(case)
    rng = np.random.default_rng(4)
    base = np.stack([np.stack([rng.choice(lim[t] + 1, size=min(6, lim[t] + 1), replace=False)
                               for _ in range(Hkv)]) if lim[t] >= 5 else np.zeros((Hkv, 6), int)
                     for t in range(T)]).astype(np.int32)
    junk = np.concatenate([base, np.full((T, Hkv, 2), -1, np.int32),
                           (lim[:, None, None] + 1 + rng.integers(0, 5, size=(T, Hkv, 3))).astype(np.int32)], axis=2)
    assert np.allclose(_sparse(case, base), _sparse(case, junk), rtol=0, atol=1e-12)


def test_single_key_and_empty_rows():
    case = _case(5)
    T, Hkv, G = case.q.shape[0], case.spec.num_kv_heads, case.spec.group
    idx = np.full((T, Hkv, 3), -1, np.int32)
    idx[:, 0, 0] = 0  # kv head 0 attends key 0 alone; kv head 1 attends nothing
    got, lse = _sparse(case, idx, with_lse=True)
    qsl, bt = case.query_start_loc.tolist(), case.block_table.numpy()
    vals = oracle.e4m3_table()
    for t in range(T):
        s = max(i for i in range(len(qsl) - 1) if qsl[i] <= t)
        v0 = vals[case.v_cache[bt[s, 0], 0, 0].numpy()] * case.v_descale  # softmax of one score is 1
        assert np.allclose(got[t, :G], v0[None, :], rtol=0, atol=1e-15)
        assert (got[t, G:] == 0).all() and np.isneginf(lse[t, G:]).all()


def test_a_key_listed_twice_counts_twice():
    """Two keys a, b: listing a twice gives weights 2e^sa : e^sb (closed form)."""
    case = _case(6, seqs=((1, 30),), G=2, Hkv=1)
    a, b = 3, 17
    once = _sparse(case, np.array([[[a, b]]], np.int32))
    twice = _sparse(case, np.array([[[a, a, b]]], np.int32))
    va = _sparse(case, np.array([[[a]]], np.int32))
    vb = _sparse(case, np.array([[[b]]], np.int32))
    # w = weight of a in the 2-key mix, recovered per row from the one-listing result
    w1 = ((once - vb) * (va - vb)).sum(-1) / ((va - vb) ** 2).sum(-1)
    r = w1 / (1 - w1)                       # e^sa / e^sb
    w2 = 2 * r / (2 * r + 1)
    assert np.allclose(twice, w2[..., None] * va + (1 - w2[..., None]) * vb, rtol=0, atol=1e-12)
    assert not np.allclose(twice, once, atol=1e-6)


def test_generated_lists_are_distinct_ascending_and_visible():
    spec = wl.CaseSpec("gen", [(7, 50), (2, 2), (40, 300)], 4, 2, 16)
    idx = wl.sparse_indices(spec, 21, seed=9).numpy()
    lim = np.concatenate([np.arange(L - q, L) for q, L in spec.seqs])
    for t in range(idx.shape[0]):
        for h in range(2):
            v = idx[t, h][idx[t, h] >= 0]
            assert len(v) == min(21, lim[t] + 1)
            assert (np.diff(v) > 0).all() and v.min() >= 0 and v.max() <= lim[t]
