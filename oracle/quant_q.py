"""Oracle of attention on a Q quantised per tensor to FP8 (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this module; the CUDA library never does, and this module never imports it.

What it computes ("asm FP8 FMHA for prefix-hit prefill", summary: the FP8 prefill
attention runs on Q, K and V cast to e4m3 with per-tensor scales, the casts counted in the
attention's time): a bf16 Q becomes e4m3 codes under one scale for the whole tensor, and
the attention is the ordinary one on those codes with that descale.

  amax      = max |q| over all elements (NaNs skipped; 0 if there are none)
  q_descale = amax / 448, inv = 1 / q_descale, each rounded to nearest in float32;
              both are 1 when amax is 0 or infinite (the pages are silent on these cases)
  code      = e4m3 of the float32 product q * inv (clamp to +-448, round half to even)
  out       = paged GQA attention (the fp64 oracle) with e4m3 Q = code and q_descale

The steps that decide a code (the scale, the product, the rounding) are taken in float32,
the precision the kernel takes them in; the attention itself is in fp64.

Parity status: pinned (tests/test_quant_q_oracle.py: the largest element maps to the
largest code, every dequantised value lies within half an e4m3 step of the input, codes
agree with torch.float8_e4m3fn, scaling Q by a power of two keeps the codes and scales
the descale, the degenerate scales, and the attention lies within the FP8 error of the
bf16-Q attention).
"""
from __future__ import annotations

import numpy as np

from . import attention
from .cache_write import e4m3_encode

E4M3_MAX = np.float32(448.0)


def q_scales(q: np.ndarray):
    """(q_descale, inv) in float32 for a Q given as float32 values."""
    a = np.abs(np.asarray(q, dtype=np.float32))
    a = a[~np.isnan(a)]
    amax = np.float32(a.max()) if a.size else np.float32(0.0)
    if not (amax > 0) or not np.isfinite(amax):
        return np.float32(1.0), np.float32(1.0)
    d = np.float32(amax / E4M3_MAX)
    return d, np.float32(np.float32(1.0) / d)


def quantize_q(q: np.ndarray):
    """float32 Q (any shape) -> (e4m3 codes as uint8, q_descale as float32)."""
    q = np.asarray(q, dtype=np.float32)
    d, inv = q_scales(q)
    return e4m3_encode((q * inv).astype(np.float32)), d


def attention_quant_q(q_bf16, k_cache, v_cache, block_table, seq_lens, query_start_loc, *, kv_dtype: str,
                      k_descale: float, v_descale: float, softmax_scale: float, rows=None, threads: int = 0,
                      scales=None):
    """fp64 attention with Q quantised per tensor; q_bf16 is a torch bf16 tensor [T, Hq, 256].

    ``scales``: the (q_descale, inv) pair of the whole Q when q_bf16 holds only some of its
    sequences (q_scales of the full tensor); by default they come from q_bf16 itself."""
    import torch
    q = q_bf16.detach().float().cpu().numpy()
    d, inv = scales if scales is not None else q_scales(q)
    codes = e4m3_encode((q * np.float32(inv)).astype(np.float32))
    q8 = torch.from_numpy(codes)
    return attention(q8, k_cache, v_cache, block_table, seq_lens, query_start_loc, q_dtype="e4m3",
                     kv_dtype=kv_dtype, q_descale=float(d), k_descale=k_descale, v_descale=v_descale,
                     softmax_scale=softmax_scale, rows=rows, threads=threads)
