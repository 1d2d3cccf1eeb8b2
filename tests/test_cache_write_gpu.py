"""Paged KV-cache write on the GPU against the oracle, byte for byte."""
import numpy as np
import pytest
import torch

import paged_gqa_gb300 as pg
import workloads as wl
from oracle import cache_write as cw

pytestmark = pytest.mark.gpu

CASES = [
    # (name, seqs (q_len, L), Hkv, page size, value scale)
    ("decode", [(1, 37), (1, 1), (1, 300), (1, 64), (1, 65)], 2, 16, 1.0),
    ("mtp", [(4, 100), (2, 17), (3, 3), (4, 4000)], 1, 16, 1.0),
    ("prefill chunk", [(300, 1200), (17, 17), (129, 500)], 8, 64, 1.0),
    ("saturating", [(6, 200), (1, 9)], 2, 32, 600.0),
    ("tiny values", [(5, 80)], 1, 128, 1e-3),
]


def _new_tokens(spec, scale, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    shape = (spec.total_q, spec.num_kv_heads, wl.HEAD_DIM)
    kn = (torch.randn(shape, generator=g, device="cuda") * scale).to(torch.bfloat16)
    vn = (torch.randn(shape, generator=g, device="cuda") * scale).to(torch.bfloat16)
    return kn, vn


def _oracle(case, kn, vn, kc0, vc0, kd, vd):
    return cw.cache_write(kn.float().cpu().numpy(), vn.float().cpu().numpy(), kc0.cpu().numpy(),
                          vc0.cpu().numpy(), case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(),
                          case.query_start_loc.cpu().numpy(), kd, vd)


@pytest.mark.parametrize("i", range(len(CASES)))
def test_cache_write_matches_oracle(i):
    name, seqs, hkv, page, scale = CASES[i]
    spec = wl.CaseSpec(name, seqs, 4 * hkv, hkv, page, spare_pages=3, extra_table_cols=1)
    case = wl.make_case(spec, device="cuda", seed=50 + i, poison=True)
    kn, vn = _new_tokens(spec, scale, 50 + i)
    kc0, vc0 = case.k_cache.clone(), case.v_cache.clone()
    kd, vd = 0.75, 1.5
    pg.paged_gqa_cache_write(kn, vn, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                             case.query_start_loc, kd, vd)
    assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
    ref_k, ref_v = _oracle(case, kn, vn, kc0, vc0, kd, vd)
    got_k, got_v = case.k_cache.cpu().numpy(), case.v_cache.cpu().numpy()
    assert (got_k == ref_k).all(), f"{name}: {(got_k != ref_k).sum()} K bytes differ"
    assert (got_v == ref_v).all(), f"{name}: {(got_v != ref_v).sum()} V bytes differ"


def test_two_writes_in_a_row_and_strided_inputs():
    """New tokens given as a view with a head stride wider than 256, written twice."""
    spec = wl.CaseSpec("strided", [(3, 50), (2, 40)], 8, 2, 16)
    case = wl.make_case(spec, device="cuda", seed=61)
    big = torch.randn(spec.total_q, 2, 384, device="cuda").to(torch.bfloat16)
    kn = big[:, :, :256]
    vn = torch.randn(spec.total_q, 2, 256, device="cuda").to(torch.bfloat16)
    for _ in range(2):
        kc0, vc0 = case.k_cache.clone(), case.v_cache.clone()
        pg.paged_gqa_cache_write(kn, vn, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                 case.query_start_loc, 1.0, 1.0)
        ref_k, ref_v = _oracle(case, kn, vn, kc0, vc0, 1.0, 1.0)
        assert (case.k_cache.cpu().numpy() == ref_k).all() and (case.v_cache.cpu().numpy() == ref_v).all()
    assert pg.paged_gqa_check_device_errors() == 0


def test_bad_page_is_flagged_and_skipped_without_trapping():
    spec = wl.CaseSpec("bad page", [(2, 30), (1, 20)], 4, 1, 16)
    case = wl.make_case(spec, device="cuda", seed=62)
    kn, vn = _new_tokens(spec, 1.0, 62)
    bt = case.block_table.clone()
    bt[0, 1] = spec.num_seqs + 10_000  # the page of sequence 0's new tokens: out of range
    kc0 = case.k_cache.clone()
    pg.paged_gqa_cache_write(kn, vn, case.k_cache, case.v_cache, bt, case.seq_lens, case.query_start_loc, 1.0, 1.0)
    assert pg.paged_gqa_check_device_errors() == -5  # PG_ERR_DEVICE_BOUNDS
    # sequence 1's token is still written; nothing else changed
    ref_k, _ = cw.cache_write(kn[2:].float().cpu().numpy(), vn[2:].float().cpu().numpy(), kc0.cpu().numpy(),
                              kc0.cpu().numpy(), case.block_table[1:].cpu().numpy(), case.seq_lens[1:].cpu().numpy(),
                              (case.query_start_loc[1:] - 2).cpu().numpy(), 1.0, 1.0)
    assert (case.k_cache.cpu().numpy() == ref_k).all()


def test_tie_input_takes_the_code_of_the_product():
    """descale 1.7: every positive bf16 value up to 380 written once (and its negation); the inputs where
    value / descale and value * fl32(1 / descale) round to different e4m3 codes must take
    the product's code (the oracle's reading), as every other input must match byte for byte."""
    bits = (torch.arange(1, 0x43BF, dtype=torch.int32) << 16).view(torch.float32)  # 2^-133 .. 380
    vals = bits.to(torch.bfloat16)
    n = (vals.numel() + 255) // 256
    flat = torch.zeros(n * 256, dtype=torch.bfloat16)
    flat[: vals.numel()] = vals
    spec = wl.CaseSpec("ties", [(n, n + 5)], 4, 1, 16)
    case = wl.make_case(spec, device="cuda", seed=63)
    kn = flat.view(n, 1, 256).cuda()
    vn = (-flat).view(n, 1, 256).cuda()
    kc0, vc0 = case.k_cache.clone(), case.v_cache.clone()
    pg.paged_gqa_cache_write(kn, vn, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                             case.query_start_loc, 1.7, 1.7)
    assert pg.paged_gqa_check_device_errors() == 0, pg.paged_gqa_last_error()
    ref_k, ref_v = _oracle(case, kn, vn, kc0, vc0, 1.7, 1.7)
    assert (case.k_cache.cpu().numpy() == ref_k).all() and (case.v_cache.cpu().numpy() == ref_v).all()
