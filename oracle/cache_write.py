"""Oracle of the paged KV-cache write (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this module; the CUDA library never does, and this module never imports it.

What it computes (the step before the attention path: new tokens' K and V go into the
cache the attention reads; "Optimize Qwen3.5 MTP unified attention on gfx950" and "asm FP8
FMHA for prefix-hit prefill" read a cache that this step fills): for sequence s with
q_len new tokens and total length L (seq_lens, which already counts the new tokens), new
token t sits at position L - q_len + t, i.e. in page block_table[s][pos // P], slot
pos % P, and every head's 256 values are stored as e4m3 codes of value * inv, with inv =
1 / descale rounded to float32 first (the per-tensor descale the attention path
multiplies back).

e4m3 (OCP E4M3FN) from its definition: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
exponent field 0 holds subnormals m * 2^-9; the code 0x7F/0xFF is NaN; the largest finite
value is 448. Encoding clamps to +-448 first, then rounds to the nearest representable
value, ties to the even mantissa. The product value * inv is taken in float32, as the
kernel takes it (the rounding that decides a code is taken in the kernel's precision); it
is not the division value / descale, which can round to the other code at an e4m3 tie.

Parity status: pinned (tests/test_cache_write_oracle.py: every finite code round-trips,
agreement with torch.float8_e4m3fn wherever that cast does not overflow, explicit ties and
saturation, and the scatter's positions against a direct reading of the definition).
"""
from __future__ import annotations

import numpy as np


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """float32 values -> e4m3 codes (uint8), clamp to +-448 then round half to even."""
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y.astype(np.float64))
    sign = np.signbit(y).astype(np.uint8) << 7
    nan = np.isnan(y)
    a = np.where(nan, 0.0, np.minimum(a, 448.0))
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # subnormal range: multiples of 2^-9; q = 8 is 2^-6, whose code 0x08 is the first normal
    code = np.where(sub, np.rint(a * 2.0 ** 9).astype(np.int64), code)
    # normal range: a = (1 + m/8) 2^E, E in [-6, 8]
    mant, exp = np.frexp(np.where(sub, 1.0, a))          # a = mant * 2^exp, mant in [0.5, 1)
    E = exp - 1
    mq = np.rint((mant * 2.0 - 1.0) * 8.0).astype(np.int64)  # 0 .. 8
    E = np.where(mq == 8, E + 1, E)
    mq = np.where(mq == 8, 0, mq)
    normal_code = (E + 7) * 8 + mq
    code = np.where(sub, code, normal_code)
    code = np.minimum(code, 0x7E)
    out = (code.astype(np.uint8) | sign).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), out)


def cache_write(k_new: np.ndarray, v_new: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                block_table: np.ndarray, seq_lens: np.ndarray, query_start_loc: np.ndarray,
                k_descale: float, v_descale: float):
    """Returns copies of the e4m3 caches ([NB, P, Hkv, 256] uint8) with the new tokens written.

    k_new, v_new: [T, Hkv, 256] float32 (the bf16 inputs' exact values)."""
    kc, vc = k_cache.copy(), v_cache.copy()
    P = kc.shape[1]
    inv_k = np.float32(1.0) / np.float32(k_descale)
    inv_v = np.float32(1.0) / np.float32(v_descale)
    for s in range(len(seq_lens)):
        q0, q1 = int(query_start_loc[s]), int(query_start_loc[s + 1])
        qn, L = q1 - q0, int(seq_lens[s])
        for t in range(qn):
            pos = L - qn + t
            page = int(block_table[s, pos // P])
            kc[page, pos % P] = e4m3_encode(k_new[q0 + t].astype(np.float32) * inv_k)
            vc[page, pos % P] = e4m3_encode(v_new[q0 + t].astype(np.float32) * inv_v)
    return kc, vc
