"""Helpers for the GPU parity tests: run the library, run the oracle, compare."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads as wl
from workloads import subcase, to_device  # noqa: F401

# Pass criterion for bf16 output against the fp64 oracle (max |diff| and rel-L2).
MAX_ABS = 1e-2
REL_L2 = 5e-3


def run_library(case: wl.Case, out=None, check_errors=True) -> torch.Tensor:
    import paged_gqa_gb300 as pg
    T, Hq = case.q.shape[0], case.q.shape[1]
    if out is None:
        out = torch.full((T, Hq, wl.HEAD_DIM), float("nan"), dtype=torch.bfloat16, device=case.q.device)
    pg.paged_gqa_attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                      case.query_start_loc, case.k_descale, case.v_descale, case.softmax_scale, out)
    if check_errors:
        st = pg.paged_gqa_check_device_errors()
        assert st == 0, pg.paged_gqa_last_error()
    return out


def compare(got: torch.Tensor, ref: np.ndarray, what: str = ""):
    """bf16 output vs fp64 oracle: finite, max-abs and rel-L2 within the bar."""
    g = got.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output ({(~np.isfinite(g)).sum()} values)"
    diff = g - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    denom = float(np.linalg.norm(ref)) or 1.0
    rel = float(np.linalg.norm(diff)) / denom
    assert max_abs <= MAX_ABS, f"{what}: max|diff| {max_abs:.3e} > {MAX_ABS}"
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    return max_abs, rel


def check_full(case_dev: wl.Case, got: torch.Tensor, what: str = ""):
    ref = oracle.attention_case(to_device(case_dev, "cpu"))
    return compare(got, ref, what)


def check_sampled(case_dev: wl.Case, got: torch.Tensor, seq_ids, rows_per_seq: int = 0, seed: int = 0,
                  what: str = ""):
    """Oracle on the listed sequences; all their rows, or a sample of rows_per_seq each."""
    sub = subcase(case_dev, seq_ids)
    qsl = case_dev.query_start_loc.cpu().tolist()
    Hq = case_dev.spec.num_q_heads
    gen = torch.Generator().manual_seed(seed)
    sub_rows, full_rows = [], []
    base = 0
    for s in seq_ids:
        n = (qsl[s + 1] - qsl[s]) * Hq
        local = torch.arange(n) if rows_per_seq <= 0 or rows_per_seq >= n else torch.randperm(n, generator=gen)[:rows_per_seq].sort().values
        sub_rows.append(local + base)
        full_rows.append(local + qsl[s] * Hq)
        base += n
    sub_rows = torch.cat(sub_rows).numpy()
    full_rows = torch.cat(full_rows)
    ref = oracle.attention_case(sub, rows=sub_rows)
    g = got.reshape(-1, wl.HEAD_DIM)[full_rows.to(got.device)]
    return compare(g, ref, what)
