"""The benchmark's unit counts (CPU only): the figures the reported throughputs divide by.

Each is recomputed here from its definition, one item at a time, on small specs."""
import importlib.util
import os

import torch

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_units_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_sparse_used_pairs_count_each_used_entry_once_per_query_head():
    b = _bench()
    spec = wl.CaseSpec("u", [(3, 10), (2, 40)], 6, 2, 16)
    idx = wl.sparse_indices(spec, 8, seed=4)
    idx[0, 0, 0] = 99      # past every limit: not used
    idx[1, 1, 2] = idx[1, 1, 1]  # a duplicate: used twice
    want = 0
    t = 0
    for q, L in spec.seqs:
        for i in range(q):
            lim = L - q + i
            for h in range(spec.num_kv_heads):
                want += sum(1 for p in idx[t, h].tolist() if 0 <= p <= lim) * spec.group
            t += 1
    assert b.sp_used_pairs(spec, idx) == want


def test_sparse_lists_fill_short_rows_and_pad():
    spec = wl.CaseSpec("p", [(4, 5)], 2, 1, 16)
    idx = wl.sparse_indices(spec, 3, seed=1)
    # rows see 2, 3, 4, 5 positions: the first lists both then -1, the others pick 3
    assert idx[0, 0].tolist() == [0, 1, -1]
    for t in range(1, 4):
        v = idx[t, 0].tolist()
        assert -1 not in v and v == sorted(set(v)) and max(v) <= t + 1


def test_cache_write_bytes_per_row_and_config():
    b = _bench()
    assert b.CW_ROW_BYTES == 2 * 256 * 2 + 2 * 256
    spec = wl.CaseSpec("w", [(3, 10), (5, 5)], 4, 2, 16)
    cfg = b.cw_config(spec, 0, 1, "n/a")
    assert cfg["rows"] == 8 * 2 and cfg["bytes"] == 16 * b.CW_ROW_BYTES


def test_dense_units_match_their_definitions():
    spec = wl.CaseSpec("d", [(4, 20), (1, 7), (130, 300)], 8, 2, 64)
    pairs = sum(L - q + t + 1 for q, L in spec.seqs for t in range(q))
    assert spec.flops == 4 * 256 * spec.num_q_heads * pairs
    assert spec.kv_bytes == sum(L for _, L in spec.seqs) * spec.num_kv_heads * 256 * 2
    # 16384 new tokens on 32768: 16384 * 16385 + 16383 * 16384 / 2 = 402,661,376 pairs per head
    assert wl.config_spec(4).flops == 402_661_376 * 8 * 4 * 256
