"""C-ABI boundary tests that need no GPU: the library builds, loads, exports every
symbol include/paged_gqa.h declares, and rejects invalid descriptors on the host
before anything is launched."""
import ctypes
import os
import re

import pytest
import torch

import paged_gqa_gb300 as pg
from paged_gqa_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_declarations_are_exported():
    header = open(os.path.join(ROOT, "include", "paged_gqa.h")).read()
    declared = set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(paged_gqa_\w+)\s*\(", header, re.M))
    assert declared == set(B.EXPORTED)
    lib = pg.load()
    for name in declared:
        assert hasattr(lib, name), name
    assert pg.paged_gqa_version() == 100


class FakeTensor:
    """Just enough of a tensor for descriptor marshalling (never dereferenced)."""

    def __init__(self, shape, dtype, ptr=1 << 20, stride=None):
        self.shape = shape
        self.dtype = dtype
        self._ptr = ptr
        if stride is None:
            stride, acc = [], 1
            for s in reversed(shape):
                stride.insert(0, acc)
                acc *= s
        self._stride = stride

    def dim(self):
        return len(self.shape)

    def numel(self):
        n = 1
        for s in self.shape:
            n *= s
        return n

    def data_ptr(self):
        return self._ptr

    def stride(self, i):
        return self._stride[i]


def _args(**over):
    a = dict(
        q=FakeTensor((8, 16, 256), torch.bfloat16),
        k=FakeTensor((10, 16, 1, 256), torch.uint8),
        v=FakeTensor((10, 16, 1, 256), torch.uint8),
        bt=FakeTensor((2, 5), torch.int32),
        sl=FakeTensor((2,), torch.int32),
        qsl=FakeTensor((3,), torch.int32),
        out=FakeTensor((8, 16, 256), torch.bfloat16),
    )
    a.update(over)
    return a


def _call(a, scale=1 / 16):
    d = [B._desc(a[n]) for n in ("q", "k", "v", "bt", "sl", "qsl")]
    o = B._desc(a["out"])
    return pg.load().paged_gqa_attn(*[ctypes.byref(x) for x in d], 1.0, 1.0, scale, ctypes.byref(o), None)


@pytest.mark.parametrize("over,code,msg", [
    (dict(q=FakeTensor((8, 16, 128), torch.bfloat16)), -2, "head_dim"),
    (dict(k=FakeTensor((10, 16, 3, 256), torch.uint8), v=FakeTensor((10, 16, 3, 256), torch.uint8)), -1, "multiple"),
    (dict(k=FakeTensor((10, 24, 1, 256), torch.uint8), v=FakeTensor((10, 24, 1, 256), torch.uint8)), -2, "page size"),
    (dict(out=FakeTensor((8, 16, 256), torch.float32)), -2, "out must be bf16"),
    (dict(q=FakeTensor((8, 16, 256), torch.uint8), k=FakeTensor((10, 16, 1, 256), torch.bfloat16),
          v=FakeTensor((10, 16, 1, 256), torch.bfloat16)), -2, "e4m3 q"),
    (dict(v=FakeTensor((10, 16, 1, 256), torch.bfloat16)), -1, "dtypes differ"),
    (dict(bt=FakeTensor((3, 5), torch.int32)), -1, "block_table rows"),
    (dict(qsl=FakeTensor((2,), torch.int32)), -1, "query_start_loc"),
    (dict(q=FakeTensor((8, 16, 256), torch.bfloat16, ptr=(1 << 20) + 2)), -1, "aligned"),
    (dict(q=FakeTensor((8, 16, 256), torch.bfloat16, stride=[4096, 256, 2])), -1, "contiguous"),
    (dict(k=FakeTensor((10, 16, 1, 256), torch.uint8, stride=[4104, 264, 264, 1]),
          v=FakeTensor((10, 16, 1, 256), torch.uint8)), -1, "16 bytes"),
    (dict(sl=FakeTensor((2,), torch.float32)), -1, "int32"),
    (dict(out=FakeTensor((9, 16, 256), torch.bfloat16)), -1, "out shape"),
    # out rows that overlap: a broadcast token axis, heads 128 elements apart, a head axis
    # stepping inside the token axis' span
    (dict(out=FakeTensor((8, 16, 256), torch.bfloat16, stride=[0, 256, 1])), -1, "overlap"),
    (dict(out=FakeTensor((8, 16, 256), torch.bfloat16, stride=[4096, 128, 1])), -1, "overlap"),
    (dict(out=FakeTensor((8, 16, 256), torch.bfloat16, stride=[256, 1024, 1])), -1, "overlap"),
])
def test_invalid_arguments_are_rejected_on_host(over, code, msg):
    st = _call(_args(**over))
    assert st == code
    assert msg in pg.paged_gqa_last_error()


def test_non_finite_scale_rejected():
    assert _call(_args(), scale=float("inf")) == -1
    assert "finite" in pg.paged_gqa_last_error()


def test_null_descriptor_rejected():
    d = [B._desc(x) for x in (_args()["q"],)]
    st = pg.load().paged_gqa_attn(None, None, None, None, None, None, 1.0, 1.0, 1.0, None, None)
    assert st == -1 and "null descriptor" in pg.paged_gqa_last_error()


def test_empty_batch_is_a_no_op():
    # zero sequences: validated, nothing launched, no device touched
    a = _args(bt=FakeTensor((0, 5), torch.int32), sl=FakeTensor((0,), torch.int32),
              qsl=FakeTensor((1,), torch.int32), q=FakeTensor((0, 16, 256), torch.bfloat16),
              out=FakeTensor((0, 16, 256), torch.bfloat16))
    assert _call(a) == 0


def test_set_stall_test_roundtrip():
    prev = pg.paged_gqa_set_stall_test(1000)
    assert pg.paged_gqa_set_stall_test(prev) == 1000


def test_set_path_roundtrip():
    prev = pg.paged_gqa_set_path(1)
    assert pg.paged_gqa_set_path(prev) == 1
    assert pg.paged_gqa_set_path(2) == prev
    assert pg.paged_gqa_set_path(prev) == 2
    with pytest.raises(pg.PagedGQAError):
        pg.paged_gqa_set_path(7)


def _cw_args(**over):
    a = dict(
        kn=FakeTensor((8, 2, 256), torch.bfloat16),
        vn=FakeTensor((8, 2, 256), torch.bfloat16),
        kc=FakeTensor((10, 16, 2, 256), torch.uint8),
        vc=FakeTensor((10, 16, 2, 256), torch.uint8),
        bt=FakeTensor((2, 5), torch.int32),
        sl=FakeTensor((2,), torch.int32),
        qsl=FakeTensor((3,), torch.int32),
    )
    a.update(over)
    return a


def _cw_call(a, kd=1.0, vd=1.0):
    d = [B._desc(a[n]) for n in ("kn", "vn", "kc", "vc", "bt", "sl", "qsl")]
    return pg.load().paged_gqa_cache_write(*[ctypes.byref(x) for x in d], kd, vd, None)


@pytest.mark.parametrize("over,scales,code,msg", [
    (dict(kn=FakeTensor((8, 2, 256), torch.uint8)), (1.0, 1.0), -2, "bf16"),
    (dict(kc=FakeTensor((10, 16, 2, 256), torch.bfloat16), vc=FakeTensor((10, 16, 2, 256), torch.bfloat16)),
     (1.0, 1.0), -2, "e4m3"),
    (dict(kc=FakeTensor((10, 16, 4, 256), torch.uint8), vc=FakeTensor((10, 16, 4, 256), torch.uint8)),
     (1.0, 1.0), -1, "num_kv_heads"),
    (dict(kn=FakeTensor((8, 2, 128), torch.bfloat16), vn=FakeTensor((8, 2, 128), torch.bfloat16)), (1.0, 1.0), -2,
     "head_dim"),
    (dict(kn=FakeTensor((8, 2, 256), torch.bfloat16, stride=[516, 258, 1])), (1.0, 1.0), -1, "16 bytes"),
    (dict(qsl=FakeTensor((2,), torch.int32)), (1.0, 1.0), -1, "query_start_loc"),
    (dict(kc=FakeTensor((10, 16, 2, 256), torch.uint8, stride=[8192, 0, 256, 1])), (1.0, 1.0), -1, "overlap"),
    (dict(vc=FakeTensor((10, 16, 2, 256), torch.uint8, stride=[4096, 512, 128, 1])), (1.0, 1.0), -1, "overlap"),
    ({}, (0.0, 1.0), -1, "positive"),
    ({}, (1.0, float("nan")), -1, "positive"),
])
def test_cache_write_rejects_bad_arguments_before_any_launch(over, scales, code, msg):
    assert _cw_call(_cw_args(**over), *scales) == code
    assert msg in B.paged_gqa_last_error()


def _qq_call(a, scale=1 / 16):
    d = [B._desc(a[n]) for n in ("q", "k", "v", "bt", "sl", "qsl")]
    o = B._desc(a["out"])
    return pg.load().paged_gqa_attn_quant_q(*[ctypes.byref(x) for x in d], 1.0, 1.0, scale, ctypes.byref(o), None)


@pytest.mark.parametrize("over,code,msg", [
    (dict(q=FakeTensor((8, 16, 256), torch.uint8)), -2, "bf16 q"),
    (dict(k=FakeTensor((10, 16, 1, 256), torch.bfloat16), v=FakeTensor((10, 16, 1, 256), torch.bfloat16)), -2,
     "e4m3 caches"),
    (dict(q=FakeTensor((8, 16, 128), torch.bfloat16)), -2, "head_dim"),
    (dict(q=FakeTensor((8, 16, 256), torch.bfloat16, ptr=(1 << 20) + 2)), -1, "aligned"),
])
def test_quant_q_rejects_bad_arguments_before_any_launch(over, code, msg):
    assert _qq_call(_args(**over)) == code
    assert msg in pg.paged_gqa_last_error()


def test_quant_q_empty_batch_is_a_no_op():
    a = _args(bt=FakeTensor((0, 5), torch.int32), sl=FakeTensor((0,), torch.int32),
              qsl=FakeTensor((1,), torch.int32), q=FakeTensor((0, 16, 256), torch.bfloat16),
              out=FakeTensor((0, 16, 256), torch.bfloat16))
    assert _qq_call(a) == 0


def _sp_call(a, idx):
    d = [B._desc(a[n]) for n in ("q", "k", "v", "bt", "sl", "qsl")] + [B._desc(idx)]
    o = B._desc(a["out"])
    return pg.load().paged_gqa_sparse_attn(*[ctypes.byref(x) for x in d], 1.0, 1.0, 1 / 16, ctypes.byref(o), None)


@pytest.mark.parametrize("over,idx,code,msg", [
    (dict(q=FakeTensor((8, 16, 256), torch.uint8)), FakeTensor((8, 1, 64), torch.int32), -2, "bf16 q"),
    (dict(k=FakeTensor((10, 16, 1, 256), torch.bfloat16), v=FakeTensor((10, 16, 1, 256), torch.bfloat16)),
     FakeTensor((8, 1, 64), torch.int32), -2, "e4m3 caches"),
    (dict(v=FakeTensor((10, 16, 1, 256), torch.uint8, stride=[8192, 512, 512, 1])),
     FakeTensor((8, 1, 64), torch.int32), -1, "same strides"),
    ({}, FakeTensor((8, 2, 64), torch.int32), -1, "[T, num_kv_heads, K]"),
    ({}, FakeTensor((8, 1, 64), torch.float32), -1, "int32"),
    ({}, FakeTensor((8, 1, 64), torch.int32, stride=[128, 128, 2]), -1, "contiguous"),
    ({}, FakeTensor((8, 1, 64), torch.int32, ptr=(1 << 20) + 2), -1, "aligned"),
])
def test_sparse_rejects_bad_arguments_before_any_launch(over, idx, code, msg):
    assert _sp_call(_args(**over), idx) == code
    assert msg in pg.paged_gqa_last_error()


def test_sparse_empty_batch_is_a_no_op():
    a = _args(bt=FakeTensor((0, 5), torch.int32), sl=FakeTensor((0,), torch.int32),
              qsl=FakeTensor((1,), torch.int32), q=FakeTensor((0, 16, 256), torch.bfloat16),
              out=FakeTensor((0, 16, 256), torch.bfloat16))
    assert _sp_call(a, FakeTensor((0, 1, 64), torch.int32)) == 0


def test_cache_write_without_new_tokens_is_a_no_op():
    a = _cw_args(kn=FakeTensor((0, 2, 256), torch.bfloat16), vn=FakeTensor((0, 2, 256), torch.bfloat16))
    assert _cw_call(a) == 0
