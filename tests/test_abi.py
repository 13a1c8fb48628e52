"""The C-ABI library loads, exports every declared entry point, and validates
arguments on the host (CPU only: no call here reaches a kernel)."""
import ctypes as C
import os
import re

import pytest

import allreduce_ddp_assign_gb300 as D

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ddp_bucket.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    from allreduce_ddp_assign_gb300 import _build

    _build.build()


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:ddp_status|void|const char\s*\*|int32_t)\s+\*?\s*(ddp_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported():
    names = declared()
    assert len(names) >= 15, names
    lib = C.CDLL(D.library_path())
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding wraps each of them under the same name
    assert all(hasattr(D, n) for n in names)


def test_version_and_status_strings():
    assert D.ddp_version() == 100
    assert D.ddp_status_str(D.DDP_E_TIMEOUT) == "DDP_E_TIMEOUT"
    assert D.ddp_status_str(99) == "DDP_E_UNKNOWN"


def _err(fn, *a):
    with pytest.raises(D.DdpError) as e:
        fn(*a)
    return e.value


def test_allreduce_validation():
    e = _err(D.ddp_bucket_allreduce, 0x1000, 16, 16, 0, D.DDP_ALLREDUCE, 0)
    assert e.status == D.DDP_E_INVAL and "W = 0" in str(e)
    assert _err(D.ddp_bucket_allreduce, 0x1000, 16, 16, 65, 0, 0).status == D.DDP_E_INVAL
    assert _err(D.ddp_bucket_allreduce, None, 16, 16, 2, 0, 0).status == D.DDP_E_INVAL
    assert _err(D.ddp_bucket_allreduce, 0x1000, 8, 16, 2, 0, 0).status == D.DDP_E_INVAL      # stride < n
    e = _err(D.ddp_bucket_allreduce, 0x1000, 16, 15, 2, D.DDP_REDUCE_SCATTER, 0)
    assert e.status == D.DDP_E_INVAL and "numel % W" in str(e)
    assert _err(D.ddp_bucket_allreduce, 0x1000, 16, 16, 2, 7, 0).status == D.DDP_E_INVAL
    # n == 0 and W == 1 are no-ops that never touch the device
    D.ddp_bucket_allreduce(0x1000, 16, 0, 4, 0, 0)
    D.ddp_bucket_allreduce(0x1000, 16, 16, 1, 0, 0)


def test_bucket_call_validation():
    d = D.BucketDesc(16, 2, D.DDP_F32, None, None)
    assert _err(D.ddp_pack, d, 0x1000, None, 2, 2, 0x2000, 16, 0, 0).status == D.DDP_E_INVAL   # no tables
    d = D.BucketDesc(16, 2, 9, 0x10, 0x20)
    assert "dtype" in str(_err(D.ddp_pack, d, 0x1000, None, 2, 2, 0x2000, 16, 0, 0))
    d = D.BucketDesc(16, 2, D.DDP_F32, 0x10, 0x20)
    assert _err(D.ddp_fused_bucket, d, 0x1000, None, 2, 2, 0, 0, None, 16, None, None, 0).status == D.DDP_E_INVAL
    assert _err(D.ddp_fused_bucket, d, 0x1000, None, 2, 2, 0, 1, None, 16, 0x3000, None, 0).status == D.DDP_E_INVAL
    assert _err(D.ddp_unpack, d, 0x2000, 16, 2, 0, None, 2, None, 0).status == D.DDP_E_INVAL
    assert _err(D.ddp_pack, d, 0x1000, None, 0, 2, 0x2000, 16, 0, 0).status == D.DDP_E_INVAL    # ld < 1
    # empty bucket: a no-op
    D.ddp_pack(D.BucketDesc(0, 0, 0, None, None), None, None, 1, 2, 0x2000, 16, 0, 0)


def test_assign_validation():
    assert _err(D.ddp_assign_buckets, [1, -2]).status == D.DDP_E_INVAL
    assert _err(D.ddp_assign_buckets, [1, 2], [0, 5]).status == D.DDP_E_INVAL
    assert _err(D.ddp_assign_buckets, [1, 2], None, 0).status == D.DDP_E_INVAL
    assert _err(D.ddp_assign_buckets, [1, 2], None, 4, 4, 3).status == D.DDP_E_INVAL
    assert _err(D.ddp_assign_buckets, [1, 2], None, 4, 4, 0, 0).status == D.DDP_E_INVAL
    assert D.ddp_assign_buckets([])["nbuckets"] == 0


def test_assign_capacity():
    import numpy as np

    n = np.full(5, 10, np.int64)
    d = np.zeros(5, np.int32)
    P = 5
    outs = [np.zeros(P, np.int32), np.zeros(P, np.int64), np.zeros(P, np.int32)]
    small = [np.zeros(2, np.int64), np.zeros(2, np.int64), np.zeros(2, np.int32), np.zeros(2, np.int32)]
    nb = C.c_int32(0)
    i64, i32 = C.POINTER(C.c_int64), C.POINTER(C.c_int32)
    st = D.lib().ddp_assign_buckets(n.ctypes.data_as(i64), d.ctypes.data_as(i32), P, 4, 4, 0, 1, 1,
                                    outs[0].ctypes.data_as(i32), outs[1].ctypes.data_as(i64),
                                    outs[2].ctypes.data_as(i32), small[0].ctypes.data_as(i64),
                                    small[1].ctypes.data_as(i64), small[2].ctypes.data_as(i32),
                                    small[3].ctypes.data_as(i32), 2, C.byref(nb))
    assert st == D.DDP_E_CAPACITY and nb.value == 5


def test_wait_selftest_validation():
    with pytest.raises(D.DdpError, match="limit_ns"):
        D.ddp_wait_selftest(0, 10, stream=0)
    with pytest.raises(D.DdpError, match="limit_ns"):
        D.ddp_wait_selftest(0, 3_000_000_000, stream=0)


def test_copy_rows_validation():
    """Refused on the host before any copy is issued; empty copies are no-ops."""
    with pytest.raises(D.DdpError, match="negative size"):
        D.ddp_copy_rows(0x1000, 64, 0x2000, 64, -1, 2, stream=0)
    with pytest.raises(D.DdpError, match="NULL pointer"):
        D.ddp_copy_rows(None, 64, 0x2000, 64, 64, 2, stream=0)
    with pytest.raises(D.DdpError, match="pitch below the row"):
        D.ddp_copy_rows(0x1000, 32, 0x2000, 64, 64, 2, stream=0)
    D.ddp_copy_rows(None, 0, None, 0, 0, 5, stream=0)
    D.ddp_copy_rows(None, 0, None, 0, 64, 0, stream=0)


def header_constants():
    """Every NAME = value inside an enum of the header, comments removed."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    consts = {}
    for body in re.findall(r"enum\s*\{(.*?)\}", text, flags=re.S):
        for name, value in re.findall(r"(DDP_\w+)\s*=\s*(\d+)", body):
            consts[name] = int(value)
    return consts


def test_binding_constants_match_the_header():
    consts = header_constants()
    assert len(consts) >= 25, consts
    missing = [n for n in consts if not hasattr(D, n)]
    assert not missing, missing
    wrong = {n: (getattr(D, n), v) for n, v in consts.items() if getattr(D, n) != v}
    assert not wrong, wrong
