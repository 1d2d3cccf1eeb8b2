"""ctypes binding of libpaged_gqa.so: argument marshalling only."""
from __future__ import annotations

import ctypes
import os
import struct
import threading
from typing import Optional

import torch

from . import build as _build

PG_BF16, PG_F16, PG_E4M3, PG_I32, PG_F32 = 1, 2, 3, 4, 5
STATUS_NAMES = {0: "PG_OK", -1: "PG_ERR_INVALID_ARG", -2: "PG_ERR_UNSUPPORTED", -3: "PG_ERR_CUDA",
                -4: "PG_ERR_TIMEOUT", -5: "PG_ERR_DEVICE_BOUNDS", -6: "PG_ERR_WORKSPACE"}

# Every symbol include/paged_gqa.h declares.
EXPORTED = ("paged_gqa_attn", "paged_gqa_attn_ex", "paged_gqa_attn_noalloc", "paged_gqa_attn_quant_q",
            "paged_gqa_sparse_attn", "paged_gqa_cache_write",
            "paged_gqa_workspace_size",
            "paged_gqa_last_error",
            "paged_gqa_check_device_errors", "paged_gqa_set_path", "paged_gqa_set_stall_test", "paged_gqa_last_plan",
            "paged_gqa_set_kernel_events", "paged_gqa_version")


class PagedGQAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class PgTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


_lock = threading.Lock()
_lib = None

# Descriptors are packed into a per-thread array of pg_tensor and passed by address: one
# struct.pack_into per tensor instead of a ctypes Structure built field by field.
_DESC_FMT = struct.Struct("=Qii4q4q")
assert ctypes.sizeof(PgTensor) == _DESC_FMT.size == 80
_tls = threading.local()


def _desc_buf():
    b = getattr(_tls, "buf", None)
    if b is None:
        arr = (PgTensor * 10)()
        b = _tls.buf = (arr, ctypes.addressof(arr), memoryview(arr).cast("B"))
    return b


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load the library (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if build_if_missing:
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libpaged_gqa.so not found at {_build.LIB}; run paged_gqa_gb300.build")
            lib = ctypes.CDLL(_build.LIB)
            P = ctypes.c_void_p  # descriptors are passed as addresses (see _pack)
            f, c_vp = ctypes.c_float, ctypes.c_void_p
            lib.paged_gqa_attn.argtypes = [P, P, P, P, P, P, f, f, f, P, c_vp]
            lib.paged_gqa_attn.restype = ctypes.c_int
            lib.paged_gqa_attn_ex.argtypes = [P, P, P, P, P, P, f, f, f, f, P, c_vp, ctypes.c_size_t, c_vp]
            lib.paged_gqa_attn_ex.restype = ctypes.c_int
            lib.paged_gqa_cache_write.argtypes = [P, P, P, P, P, P, P, f, f, c_vp]
            lib.paged_gqa_attn_quant_q.restype = ctypes.c_int
            lib.paged_gqa_attn_quant_q.argtypes = [P, P, P, P, P, P, f, f, f, P, c_vp]
            lib.paged_gqa_sparse_attn.restype = ctypes.c_int
            lib.paged_gqa_sparse_attn.argtypes = [P, P, P, P, P, P, P, f, f, f, P, c_vp]
            lib.paged_gqa_cache_write.restype = ctypes.c_int
            lib.paged_gqa_workspace_size.argtypes = [ctypes.c_int] * 7
            lib.paged_gqa_workspace_size.restype = ctypes.c_size_t
            lib.paged_gqa_last_error.restype = ctypes.c_char_p
            lib.paged_gqa_check_device_errors.argtypes = [c_vp]
            lib.paged_gqa_check_device_errors.restype = ctypes.c_int
            lib.paged_gqa_set_path.argtypes = [ctypes.c_int]
            lib.paged_gqa_set_path.restype = ctypes.c_int
            lib.paged_gqa_set_stall_test.argtypes = [ctypes.c_uint32]
            lib.paged_gqa_set_stall_test.restype = ctypes.c_int
            lib.paged_gqa_last_plan.argtypes = [ctypes.POINTER(ctypes.c_int64)]
            lib.paged_gqa_last_plan.restype = ctypes.c_int
            lib.paged_gqa_version.restype = ctypes.c_int
            lib.paged_gqa_set_kernel_events.argtypes = [ctypes.c_int, c_vp, c_vp]
            lib.paged_gqa_set_kernel_events.restype = ctypes.c_int
            _lib = lib
    return _lib


def exported_symbols():
    lib = load()
    return {name: hasattr(lib, name) for name in EXPORTED}


_DTYPES = {torch.bfloat16: PG_BF16, torch.float16: PG_F16, torch.int32: PG_I32, torch.float32: PG_F32,
           torch.uint8: PG_E4M3}
if hasattr(torch, "float8_e4m3fn"):
    _DTYPES[torch.float8_e4m3fn] = PG_E4M3


def _desc(t: Optional[torch.Tensor], dtype: Optional[int] = None) -> PgTensor:
    """pg_tensor view of a torch tensor (uint8 is read as e4m3 bit patterns)."""
    d = PgTensor()
    if t is None:
        return d
    if t.dim() > 4:
        raise ValueError("at most 4 dims")
    d.data = t.data_ptr() if t.numel() > 0 else 0
    d.dtype = dtype if dtype is not None else _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _pack(*tensors):
    """Addresses of pg_tensor descriptors of the given tensors, valid until the next call
    from this thread (the library copies what it needs before it returns)."""
    arr, base, mv = _desc_buf()
    pack, dt = _DESC_FMT.pack_into, _DTYPES
    out = []
    for i, t in enumerate(tensors):
        off = 80 * i
        n = t.dim()
        if n > 4:
            raise ValueError("at most 4 dims")
        sh, st = tuple(t.shape), t.stride()
        if n < 4:
            sh = sh + (0,) * (4 - n)
            st = st + (0,) * (4 - n)
        pack(mv, off, t.data_ptr() if t.numel() > 0 else 0, dt[t.dtype], n, *sh, *st)
        out.append(base + off)
    return out


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int):
    if status != 0:
        msg = load().paged_gqa_last_error().decode(errors="replace")
        raise PagedGQAError(status, msg)


def paged_gqa_attn(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, k_descale: float,
                   v_descale: float, softmax_scale: float, out, stream=None) -> None:
    """out[T, Hq, 256] (bf16) = paged GQA attention; see include/paged_gqa.h."""
    lib = load()
    d = _pack(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, out)
    _check(lib.paged_gqa_attn(*d[:6], float(k_descale), float(v_descale), float(softmax_scale), d[6],
                              _stream(stream)))


def paged_gqa_attn_ex(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, q_descale: float,
                      k_descale: float, v_descale: float, softmax_scale: float, out, workspace,
                      stream=None) -> None:
    """Same as paged_gqa_attn with q_descale and a caller-owned workspace tensor."""
    lib = load()
    d = _pack(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, out)
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    ptr = workspace.data_ptr() if workspace is not None else None
    _check(lib.paged_gqa_attn_ex(*d[:6], float(q_descale), float(k_descale), float(v_descale),
                                 float(softmax_scale), d[6], ptr, nbytes, _stream(stream)))


def paged_gqa_attn_quant_q(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, k_descale: float,
                           v_descale: float, softmax_scale: float, out, stream=None) -> None:
    """paged_gqa_attn on a bf16 q quantised inside the call to e4m3 with one per-tensor scale."""
    lib = load()
    d = _pack(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, out)
    _check(lib.paged_gqa_attn_quant_q(*d[:6], float(k_descale), float(v_descale), float(softmax_scale), d[6],
                                      _stream(stream)))


def paged_gqa_sparse_attn(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, indices,
                          k_descale: float, v_descale: float, softmax_scale: float, out, stream=None) -> None:
    """Sparse paged GQA attention: row (t, h) attends the listed positions indices[t, h // G]."""
    lib = load()
    d = _pack(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, indices, out)
    _check(lib.paged_gqa_sparse_attn(*d[:7], float(k_descale), float(v_descale), float(softmax_scale), d[7],
                                     _stream(stream)))


def paged_gqa_cache_write(k_new, v_new, k_cache, v_cache, block_table, seq_lens, query_start_loc,
                          k_descale: float, v_descale: float, stream=None) -> None:
    """Write the new tokens' K and V (bf16 [T, Hkv, 256]) into the e4m3 paged caches."""
    lib = load()
    d = _pack(k_new, v_new, k_cache, v_cache, block_table, seq_lens, query_start_loc)
    _check(lib.paged_gqa_cache_write(*d, float(k_descale), float(v_descale), _stream(stream)))


def paged_gqa_workspace_size(num_seqs: int, total_q: int, num_q_heads: int, num_kv_heads: int,
                             page_size: int, max_blocks_per_seq: int, device: int = 0) -> int:
    return int(load().paged_gqa_workspace_size(num_seqs, total_q, num_q_heads, num_kv_heads, page_size,
                                               max_blocks_per_seq, device))


def paged_gqa_last_error() -> str:
    return load().paged_gqa_last_error().decode(errors="replace")


def paged_gqa_check_device_errors(stream=None) -> int:
    """Synchronise, read and clear the device error word; returns the status code."""
    return int(load().paged_gqa_check_device_errors(_stream(stream)))


def paged_gqa_set_path(path: int) -> int:
    r = int(load().paged_gqa_set_path(path))
    if r < 0:
        _check(r)
    return r


def paged_gqa_set_stall_test(wait_ns: int) -> int:
    """Failure-path test hook: tcgen05 CTAs first wait wait_ns on a barrier nothing
    arrives on (0 turns it off). Returns the previous value."""
    return int(load().paged_gqa_set_stall_test(int(wait_ns)))


def paged_gqa_last_plan() -> dict:
    buf = (ctypes.c_int64 * 8)()
    _check(load().paged_gqa_last_plan(buf))
    keys = ("verify_ctas", "prefill_ctas", "kernels_launched", "path_bits", "max_verify_blocks",
            "max_prefill_blocks", "workspace_bytes", "verify_self_planned")
    return dict(zip(keys, list(buf)))


def paged_gqa_set_kernel_events(cls: int, start=None, stop=None) -> None:
    """Record torch.cuda.Event pairs around the class-`cls` attention kernel (None clears)."""
    for e in (start, stop):
        if e is not None and not e.cuda_event:
            e.record()  # torch creates the CUDA event lazily, on first record
    h0 = start.cuda_event if start is not None else None
    h1 = stop.cuda_event if stop is not None else None
    _check(load().paged_gqa_set_kernel_events(int(cls), h0, h1))


def paged_gqa_version() -> int:
    return int(load().paged_gqa_version())
