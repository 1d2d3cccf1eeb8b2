"""fp64 CPU oracle for paged GQA attention (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The CUDA library never does, and this package
never imports it: the two share no code.

``paged_gqa_oracle.c`` is the definition written out in fp64 (see its header
for the formula and the pages it follows). This module compiles it with gcc
(OpenMP) on first use and calls it through ctypes.

Parity status of every function here: pinned. The pins live in
``tests/test_oracle.py`` (brute-force dense attention, torch SDPA in fp64,
closed forms, invariants, the FP8 table against torch.float8_e4m3fn) and, for
``sparse_attention``, ``tests/test_sparse_oracle.py`` (the dense oracle on full
and compacted lists, order invariance, masking, duplicates, closed forms).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_gqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libpaged_gqa_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODE = {"bf16": 1, "e4m3": 3}
STATUS = {0: "ok", 1: "bad argument", 2: "block-table entry out of range", 3: "out of memory"}


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library next to its source."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c99",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_paged_gqa_attn.restype = ctypes.c_int
            P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_paged_gqa_attn.argtypes = [
                P, I, L, L,            # q, q_dtype, q strides
                P, P, I, L, L, L,      # k, v, kv_dtype, kv strides
                P, L, P, P,            # block_table, stride, seq_lens, qsl
                I, I, I, I, I, I,      # num_seqs, Hq, Hkv, D, P, NB
                D, D, D, D,            # descales, softmax_scale
                P, L, P, P, I]         # rows, nrows, out, lse, nthreads
            lib.oracle_paged_gqa_sparse_attn.restype = ctypes.c_int
            lib.oracle_paged_gqa_sparse_attn.argtypes = [
                P, I, L, L,            # q, q_dtype, q strides
                P, P, I, L, L, L,      # k, v, kv_dtype, kv strides
                P, L, P, P,            # block_table, stride, seq_lens, qsl
                P, L, L, I,            # indices, strides, K
                I, I, I, I, I, I,      # num_seqs, Hq, Hkv, D, P, NB
                D, D, D, D,            # descales, softmax_scale
                P, L, P, P, I]         # rows, nrows, out, lse, nthreads
            lib.oracle_e4m3_table.argtypes = [P]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def e4m3_table() -> np.ndarray:
    """fp64 value of every e4m3fn code, decoded from the format definition."""
    out = np.zeros(256, dtype=np.float64)
    _load().oracle_e4m3_table(out.ctypes.data)
    return out


def _np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.contiguous().numpy()


def attention(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, *,
              q_dtype: str, kv_dtype: str, q_descale: float, k_descale: float,
              v_descale: float, softmax_scale: float, rows: Optional[np.ndarray] = None,
              threads: int = 0, with_lse: bool = False):
    """fp64 paged GQA attention on host copies of the inputs.

    q: [T, Hq, D] (bf16 or uint8 e4m3 bits); caches: [NB, P, Hkv, D];
    block_table: [num_seqs, W] int32; seq_lens: [num_seqs]; query_start_loc:
    [num_seqs+1]. ``softmax_scale`` multiplies the dequantised dot product
    (q_descale is applied separately here, so pass 1.0 if the caller folded it).
    Returns out [T, Hq, D] (or [len(rows), D]) and optionally lse.
    """
    lib = _load()
    qn, kn, vn = _np(q), _np(k_cache), _np(v_cache)
    bt = _np(block_table).astype(np.int32)
    sl = _np(seq_lens).astype(np.int32)
    qsl = _np(query_start_loc).astype(np.int32)
    T, Hq, D = q.shape
    NB, P, Hkv, _ = k_cache.shape
    num_seqs = sl.shape[0]
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows.shape[0]
        out = np.zeros((n, D), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64) if with_lse else None
    else:
        out = np.zeros((T, Hq, D), dtype=np.float64)
        lse = np.zeros((T, Hq), dtype=np.float64) if with_lse else None
    bt_stride = bt.shape[1] if bt.ndim == 2 and bt.shape[1] > 0 else 1
    st = lib.oracle_paged_gqa_attn(
        qn.ctypes.data, DTYPE_CODE[q_dtype], Hq * D, D,
        kn.ctypes.data, vn.ctypes.data, DTYPE_CODE[kv_dtype], P * Hkv * D, Hkv * D, D,
        bt.ctypes.data, bt_stride, sl.ctypes.data, qsl.ctypes.data,
        num_seqs, Hq, Hkv, D, P, NB,
        q_descale, k_descale, v_descale, softmax_scale,
        rows.ctypes.data if rows is not None else None, rows.shape[0] if rows is not None else 0,
        out.ctypes.data, lse.ctypes.data if lse is not None else None, int(threads))
    if st != 0:
        raise ValueError(f"oracle: {STATUS.get(st, st)}")
    return (out, lse) if with_lse else out


def sparse_attention(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, indices, *,
                     q_dtype: str, kv_dtype: str, q_descale: float, k_descale: float,
                     v_descale: float, softmax_scale: float, rows: Optional[np.ndarray] = None,
                     threads: int = 0, with_lse: bool = False):
    """fp64 sparse paged GQA attention: row (t, h) attends the entries of indices[t, h // G]
    that lie in [0, its causal limit]; indices is [T, Hkv, K] int32 (see the C source)."""
    lib = _load()
    qn, kn, vn = _np(q), _np(k_cache), _np(v_cache)
    bt = _np(block_table).astype(np.int32)
    sl = _np(seq_lens).astype(np.int32)
    qsl = _np(query_start_loc).astype(np.int32)
    idx = np.ascontiguousarray(_np(indices).astype(np.int32))
    T, Hq, D = q.shape
    NB, P, Hkv, _ = k_cache.shape
    K = idx.shape[2] if idx.ndim == 3 else 0
    num_seqs = sl.shape[0]
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.zeros((rows.shape[0], D), dtype=np.float64)
        lse = np.zeros(rows.shape[0], dtype=np.float64) if with_lse else None
    else:
        out = np.zeros((T, Hq, D), dtype=np.float64)
        lse = np.zeros((T, Hq), dtype=np.float64) if with_lse else None
    bt_stride = bt.shape[1] if bt.ndim == 2 and bt.shape[1] > 0 else 1
    st = lib.oracle_paged_gqa_sparse_attn(
        qn.ctypes.data, DTYPE_CODE[q_dtype], Hq * D, D,
        kn.ctypes.data, vn.ctypes.data, DTYPE_CODE[kv_dtype], P * Hkv * D, Hkv * D, D,
        bt.ctypes.data, bt_stride, sl.ctypes.data, qsl.ctypes.data,
        idx.ctypes.data, Hkv * K, K, K,
        num_seqs, Hq, Hkv, D, P, NB,
        q_descale, k_descale, v_descale, softmax_scale,
        rows.ctypes.data if rows is not None else None, rows.shape[0] if rows is not None else 0,
        out.ctypes.data, lse.ctypes.data if lse is not None else None, int(threads))
    if st != 0:
        raise ValueError(f"oracle: {STATUS.get(st, st)}")
    return (out, lse) if with_lse else out


def attention_case(case, rows: Optional[np.ndarray] = None, threads: int = 0, with_lse: bool = False):
    """Run the oracle on a ``workloads.Case`` (q_descale applied here, not folded)."""
    spec = case.spec
    return attention(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                     case.query_start_loc, q_dtype=spec.q_dtype, kv_dtype=spec.kv_dtype,
                     q_descale=case.q_descale if spec.q_dtype == "e4m3" else 1.0,
                     k_descale=case.k_descale, v_descale=case.v_descale,
                     softmax_scale=spec.softmax_scale, rows=rows, threads=threads, with_lse=with_lse)
