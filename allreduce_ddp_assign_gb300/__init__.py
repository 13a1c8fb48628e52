"""Python binding of libddpbucket (the C ABI in include/ddp_bucket.h).

Argument marshalling only: every step of the path -- bucket assignment, pack,
ring-ordered reduction, unpack, scheduling -- runs in the library (host C++ and
sm_103a kernels).  PyTorch supplies device memory and streams.  The library is
loaded on first use; if it has not been built, every call raises.

Functions keep the C names.  Device arguments accept a torch tensor (its
data_ptr is passed), an integer address, or None (NULL).  A non-OK status
raises DdpError carrying the status and the library's message.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import _build

# status codes, dtypes, orders, modes, reducer flags (mirror the header)
DDP_OK, DDP_E_INVAL, DDP_E_ALIGN, DDP_E_CUDA, DDP_E_STATE, DDP_E_INCOMPLETE, DDP_E_TIMEOUT, DDP_E_CAPACITY = range(8)
DDP_F32, DDP_BF16, DDP_F16 = 0, 1, 2
DDP_ORDER_REVERSE, DDP_ORDER_FWD_THEN_REVERSE, DDP_ORDER_MEGATRON = 0, 1, 2
DDP_ALLREDUCE, DDP_REDUCE_SCATTER = 0, 1
DDP_R_FUSED, DDP_R_COPY_BACK, DDP_R_TIMING, DDP_R_DRY_RUN, DDP_R_COALESCE = 1, 2, 4, 8, 16
DDP_R_WIRE_BF16, DDP_R_WIRE_F16, DDP_R_BUCKET_DONE = 32, 64, 128
DDP_KERNEL_AUTO, DDP_KERNEL_PLAIN, DDP_KERNEL_STREAM, DDP_KERNEL_STREAM_DYNAMIC = 0, 1, 2, 3


class DdpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


class BucketDesc(C.Structure):
    """ddp_bucket_desc: host struct holding device table pointers."""
    _fields_ = [("numel", C.c_int64), ("nseg", C.c_int32), ("dtype", C.c_int32),
                ("seg_offset", C.c_void_p), ("seg_param", C.c_void_p)]


_i64p = C.POINTER(C.c_int64)
_i32p = C.POINTER(C.c_int32)
_vp = C.c_void_p
_LIB = None

_SIGS = {
    "ddp_assign_buckets": (C.c_int32, [_i64p, _i32p, C.c_int32, C.c_int64, C.c_int64, C.c_int32, C.c_int32,
                                       C.c_int32, _i32p, _i64p, _i32p, _i64p, _i64p, _i32p, _i32p, C.c_int32,
                                       _i32p]),
    "ddp_assign_buckets_ordered": (C.c_int32, [_i64p, _i32p, C.c_int32, _i32p, C.c_int64, C.c_int64, C.c_int32,
                                               C.c_int32, _i32p, _i64p, _i32p, _i64p, _i64p, _i32p, _i32p,
                                               C.c_int32, _i32p]),
    "ddp_overlap_timeline": (C.c_int32, [C.c_int32, C.POINTER(C.c_double), C.c_int32, _i32p, _i32p, _i64p,
                                         C.c_double, C.c_double, C.POINTER(C.c_double), C.POINTER(C.c_double),
                                         C.POINTER(C.c_double), C.POINTER(C.c_double)]),
    "ddp_reducer_ready_order": (C.c_int32, [_vp, _i32p, C.c_int32, _i32p]),
    "ddp_pack": (C.c_int32, [C.POINTER(BucketDesc), _vp, _vp, C.c_int32, C.c_int32, _vp, C.c_int64, C.c_int32, _vp]),
    "ddp_bucket_allreduce": (C.c_int32, [_vp, C.c_int64, C.c_int64, C.c_int32, C.c_int32, _vp]),
    "ddp_bucket_allreduce_wire": (C.c_int32, [_vp, C.c_int64, C.c_int64, C.c_int32, C.c_int32, C.c_int32, _vp]),
    "ddp_fused_bucket_group_wire": (C.c_int32, [C.POINTER(BucketDesc), _i64p, C.c_int32, _vp, _vp, C.c_int32,
                                                C.c_int32, C.c_int32, C.c_int32, _vp, C.c_int64, _vp, _vp, C.c_int32,
                                                _vp]),
    "ddp_unpack": (C.c_int32, [C.POINTER(BucketDesc), _vp, C.c_int64, C.c_int32, C.c_int32, _vp, C.c_int32, _vp,
                               _vp]),
    "ddp_fused_bucket": (C.c_int32, [C.POINTER(BucketDesc), _vp, _vp, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                     _vp, C.c_int64, _vp, _vp, _vp]),
    "ddp_pack_group": (C.c_int32, [C.POINTER(BucketDesc), _i64p, C.c_int32, _vp, _vp, C.c_int32, C.c_int32, _vp,
                                   C.c_int64, C.c_int32, _vp]),
    "ddp_fused_bucket_group": (C.c_int32, [C.POINTER(BucketDesc), _i64p, C.c_int32, _vp, _vp, C.c_int32, C.c_int32,
                                           C.c_int32, C.c_int32, _vp, C.c_int64, _vp, _vp, _vp]),
    "ddp_reducer_create": (C.c_int32, [C.c_int32, C.c_int32, _i32p, _i32p, C.POINTER(BucketDesc), _i64p, C.c_int32,
                                       C.c_int32, C.c_int32, _vp, _vp, C.c_int32, _vp, C.c_int64, _vp, _vp, _vp,
                                       C.POINTER(_vp)]),
    "ddp_reducer_prepare": (C.c_int32, [_vp, C.c_int32]),
    "ddp_used_allreduce": (C.c_int32, [_vp, C.c_int32, C.c_int32, C.c_int32, _vp, _vp, _vp]),
    "ddp_reducer_find_unused": (C.c_int32, [_vp, _vp, _vp, _vp]),
    "ddp_reducer_register_powersgd": (C.c_int32, [_vp, C.c_int32, _vp]),
    "ddp_powersgd_create": (C.c_int32, [C.c_int32, C.c_int32, C.c_int32, _i64p, _i64p, _i64p, C.c_int64, C.c_int32,
                                        C.c_int32, C.POINTER(_vp)]),
    "ddp_powersgd_sizes": (C.c_int32, [_vp, _i64p, _i64p, _i32p]),
    "ddp_powersgd_matrix": (C.c_int32, [_vp, C.c_int32, _i64p, _i32p, _i32p, _i32p, _i32p]),
    "ddp_powersgd_bind": (C.c_int32, [_vp, _vp, C.c_int64, _vp, _vp, C.c_int64, _vp]),
    "ddp_powersgd_set_q": (C.c_int32, [_vp, C.c_int32, _vp, _vp]),
    "ddp_powersgd_reduce": (C.c_int32, [_vp, _vp, C.c_int64, _vp]),
    "ddp_powersgd_reduce_static": (C.c_int32, [_vp, _vp, C.c_int64, _vp]),
    "ddp_powersgd_iter": (C.c_int32, [_vp, _i32p]),
    "ddp_powersgd_destroy": (None, [_vp]),
    "ddp_reducer_set_local_used": (C.c_int32, [_vp, _vp, C.c_int32]),
    "ddp_reducer_mark_ready": (C.c_int32, [_vp, C.c_int32, _vp]),
    "ddp_reducer_mark_ready_many": (C.c_int32, [_vp, _i32p, C.c_int32, _vp]),
    "ddp_reducer_finalize": (C.c_int32, [_vp, _vp, C.c_int64]),
    "ddp_reducer_issue_log": (C.c_int32, [_vp, _i32p, C.c_int32, _i32p]),
    "ddp_reducer_wait_bucket": (C.c_int32, [_vp, C.c_int32, _vp]),
    "ddp_reducer_bucket_ms": (C.c_int32, [_vp, C.POINTER(C.c_float), C.c_int32]),
    "ddp_reducer_destroy": (None, [_vp]),
    "ddp_set_kernel_variant": (C.c_int32, [C.c_int32]),
    "ddp_device_status": (C.c_int32, [_vp, _i32p, C.c_int32]),
    "ddp_wait_selftest": (C.c_int32, [C.c_int32, C.c_int64, _vp]),
    "ddp_copy_rows": (C.c_int32, [_vp, C.c_int64, _vp, C.c_int64, C.c_int64, C.c_int64, _vp]),
    "ddp_host_front_create": (C.c_int32, [_vp, _vp, C.c_int64, _i64p, C.c_int32, C.POINTER(_vp)]),
    "ddp_host_front_step": (C.c_int32, [_vp, _vp, C.c_int64, _vp, _vp]),
    "ddp_host_front_destroy": (None, [_vp]),
    "ddp_plan_create": (C.c_int32, [_i64p, _i32p, C.c_int32, C.c_int64, C.c_int64, C.c_int32, C.c_int32, C.c_int32,
                                    C.c_int64, C.POINTER(_vp)]),
    "ddp_plan_describe": (C.c_int32, [_vp, _vp, _i64p, _i64p, _i32p, _i32p, _i64p, _i32p, _i32p, _i32p, _i64p]),
    "ddp_plan_tables": (C.c_int32, [_vp, _i64p, _i32p]),
    "ddp_plan_bucket_descs": (C.c_int32, [_vp, _vp, _vp, C.POINTER(BucketDesc)]),
    "ddp_plan_rebuilt": (C.c_int32, [_vp, _i32p, _i64p, _i64p, C.c_int32, _i32p]),
    "ddp_reducer_create_from_plan": (C.c_int32, [_vp, C.POINTER(BucketDesc), C.c_int32, C.c_int32, C.c_int32, _vp, _vp,
                                                 C.c_int32, _vp, _vp, _vp, _vp, C.POINTER(_vp)]),
    "ddp_plan_destroy": (None, [_vp]),
    "ddp_status_str": (C.c_char_p, [C.c_int32]),
    "ddp_last_error_message": (C.c_char_p, []),
    "ddp_version": (C.c_int32, []),
}


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libddpbucket; raises if it was never built (no fallback exists)."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libddpbucket is not built ({path} missing): run __graft_entry__.build() "
                               "or python -m allreduce_ddp_assign_gb300._build")
        h = C.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _LIB = h
    return _LIB


def _status_name(s: int) -> str:
    try:
        return lib().ddp_status_str(s).decode()
    except Exception:  # pragma: no cover - library missing
        return f"status {s}"


def _check(status: int) -> None:
    if status != DDP_OK:
        raise DdpError(status, lib().ddp_last_error_message().decode())


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr() or None
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s) -> int | None:
    if s is None:
        try:
            import torch

            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream or None
        except Exception:
            pass
        return None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


def _a(x, dt):
    return np.ascontiguousarray(x, dtype=dt)


def _cp(a: np.ndarray, t):
    return a.ctypes.data_as(t)


# ---------------------------------------------------------------------------
# step 1
# ---------------------------------------------------------------------------
def ddp_assign_buckets(numels, dtypes=None, cap_bytes=25 << 20, first_cap_bytes=1 << 20, order=DDP_ORDER_REVERSE,
                       pad_multiple=1, grad_reduce_in_fp32=1) -> dict:
    numels = _a(numels, np.int64)
    P = len(numels)
    dtypes = np.zeros(P, np.int32) if dtypes is None else _a(dtypes, np.int32)
    cap = P + 2
    out = dict(bucket_of=np.zeros(P, np.int32), offset_of=np.zeros(P, np.int64), members=np.zeros(max(P, 1), np.int32),
               bucket_numel=np.zeros(cap, np.int64), bucket_bytes=np.zeros(cap, np.int64),
               bucket_dtype=np.zeros(cap, np.int32), bucket_order=np.zeros(cap, np.int32))
    nb = C.c_int32(0)
    _check(lib().ddp_assign_buckets(_cp(numels, _i64p), _cp(dtypes, _i32p), P, int(cap_bytes), int(first_cap_bytes),
                                    int(order), int(pad_multiple), int(grad_reduce_in_fp32),
                                    _cp(out["bucket_of"], _i32p), _cp(out["offset_of"], _i64p),
                                    _cp(out["members"], _i32p), _cp(out["bucket_numel"], _i64p),
                                    _cp(out["bucket_bytes"], _i64p), _cp(out["bucket_dtype"], _i32p),
                                    _cp(out["bucket_order"], _i32p), cap, C.byref(nb)))
    B = nb.value
    for k in ("bucket_numel", "bucket_bytes", "bucket_dtype", "bucket_order"):
        out[k] = out[k][:B].copy()
    out["members"] = out["members"][:P].copy()
    out["nbuckets"] = B
    return out


class PlanInfo(C.Structure):
    """ddp_plan_info."""
    _fields_ = [("nparams", C.c_int32), ("nbuckets", C.c_int32), ("order", C.c_int32), ("pad_multiple", C.c_int32),
                ("grad_reduce_in_fp32", C.c_int32), ("reserved_", C.c_int32), ("cap_bytes", C.c_int64),
                ("first_cap_bytes", C.c_int64), ("align_elems", C.c_int64), ("replica_stride", C.c_int64),
                ("seg_offset_len", C.c_int64), ("seg_param_len", C.c_int64)]


def ddp_plan_create(numels, dtypes=None, cap_bytes=25 << 20, first_cap_bytes=1 << 20, order=DDP_ORDER_REVERSE,
                    pad_multiple=1, grad_reduce_in_fp32=1, align_elems=64) -> int:
    numels = _a(numels, np.int64)
    dt = None if dtypes is None else _a(dtypes, np.int32)
    h = _vp()
    _check(lib().ddp_plan_create(_cp(numels, _i64p), None if dt is None else _cp(dt, _i32p), len(numels),
                                 int(cap_bytes), int(first_cap_bytes), int(order), int(pad_multiple),
                                 int(grad_reduce_in_fp32), int(align_elems), C.byref(h)))
    return h.value


def ddp_plan_describe(h) -> dict:
    """Every table of the plan as numpy arrays, plus the ddp_plan_info fields."""
    info = PlanInfo()
    _check(lib().ddp_plan_describe(h, C.byref(info), None, None, None, None, None, None, None, None, None))
    B, P = info.nbuckets, info.nparams
    out = {name: getattr(info, name) for name, _ in PlanInfo._fields_ if name != "reserved_"}
    arrs = dict(bucket_numel=np.zeros(max(B, 1), np.int64), bucket_bytes=np.zeros(max(B, 1), np.int64),
                bucket_dtype=np.zeros(max(B, 1), np.int32), bucket_order=np.zeros(max(B, 1), np.int32),
                bucket_start=np.zeros(max(B, 1), np.int64), member_start=np.zeros(B + 1, np.int32),
                members=np.zeros(max(P, 1), np.int32), bucket_of=np.zeros(max(P, 1), np.int32),
                offset_of=np.zeros(max(P, 1), np.int64))
    _check(lib().ddp_plan_describe(h, None, *(_cp(arrs[k], _i64p if arrs[k].dtype == np.int64 else _i32p) for k in
                                             ("bucket_numel", "bucket_bytes", "bucket_dtype", "bucket_order",
                                              "bucket_start", "member_start", "members", "bucket_of", "offset_of"))))
    for k in ("bucket_numel", "bucket_bytes", "bucket_dtype", "bucket_order", "bucket_start"):
        arrs[k] = arrs[k][:B].copy()
    for k in ("members", "bucket_of", "offset_of"):
        arrs[k] = arrs[k][:P].copy()
    out.update(arrs)
    return out


def ddp_plan_tables(h, seg_offset_len: int, seg_param_len: int):
    so = np.zeros(max(seg_offset_len, 1), np.int64)
    sp = np.zeros(max(seg_param_len, 1), np.int32)
    _check(lib().ddp_plan_tables(h, _cp(so, _i64p), _cp(sp, _i32p)))
    return so[:seg_offset_len].copy(), sp[:seg_param_len].copy()


def ddp_plan_bucket_descs(h, nbuckets: int, seg_offset_dev, seg_param_dev) -> list:
    arr = (BucketDesc * max(nbuckets, 1))()
    _check(lib().ddp_plan_bucket_descs(h, _ptr(seg_offset_dev), _ptr(seg_param_dev), arr))
    return [arr[b] for b in range(nbuckets)]


def ddp_plan_rebuilt(h, sequence, nparams: int) -> dict:
    seq = _a(sequence, np.int32)
    cap = nparams + 2
    by, nm = np.zeros(cap, np.int64), np.zeros(cap, np.int64)
    nb = C.c_int32(0)
    _check(lib().ddp_plan_rebuilt(h, _cp(seq, _i32p), _cp(by, _i64p), _cp(nm, _i64p), cap, C.byref(nb)))
    return dict(nbuckets=nb.value, bucket_bytes=by[:nb.value].copy(), bucket_numel=nm[:nb.value].copy())


def ddp_plan_destroy(h):
    if h:
        lib().ddp_plan_destroy(h)


def ddp_assign_buckets_ordered(numels, sequence, dtypes=None, cap_bytes=25 << 20, first_cap_bytes=1 << 20,
                               pad_multiple=1, grad_reduce_in_fp32=1) -> dict:
    numels = _a(numels, np.int64)
    P = len(numels)
    seq = _a(sequence, np.int32)
    dtypes = np.zeros(P, np.int32) if dtypes is None else _a(dtypes, np.int32)
    cap = P + 2
    out = dict(bucket_of=np.zeros(P, np.int32), offset_of=np.zeros(P, np.int64), members=np.zeros(max(P, 1), np.int32),
               bucket_numel=np.zeros(cap, np.int64), bucket_bytes=np.zeros(cap, np.int64),
               bucket_dtype=np.zeros(cap, np.int32), bucket_order=np.zeros(cap, np.int32))
    nb = C.c_int32(0)
    _check(lib().ddp_assign_buckets_ordered(_cp(numels, _i64p), _cp(dtypes, _i32p), P, _cp(seq, _i32p),
                                            int(cap_bytes), int(first_cap_bytes), int(pad_multiple),
                                            int(grad_reduce_in_fp32), _cp(out["bucket_of"], _i32p),
                                            _cp(out["offset_of"], _i64p), _cp(out["members"], _i32p),
                                            _cp(out["bucket_numel"], _i64p), _cp(out["bucket_bytes"], _i64p),
                                            _cp(out["bucket_dtype"], _i32p), _cp(out["bucket_order"], _i32p), cap,
                                            C.byref(nb)))
    B = nb.value
    for k in ("bucket_numel", "bucket_bytes", "bucket_dtype", "bucket_order"):
        out[k] = out[k][:B].copy()
    out["members"] = out["members"][:P].copy()
    out["nbuckets"] = B
    return out


def ddp_overlap_timeline(ready_ms, bucket_of, bucket_order, bucket_bytes, alpha_ms, ms_per_byte) -> dict:
    ready = _a(ready_ms, np.float64)
    bof = _a(bucket_of, np.int32)
    bord = _a(bucket_order, np.int32)
    bb = _a(bucket_bytes, np.int64)
    B = len(bord)
    start, end = np.zeros(max(B, 1)), np.zeros(max(B, 1))
    step, serial = C.c_double(0), C.c_double(0)
    dp = C.POINTER(C.c_double)
    _check(lib().ddp_overlap_timeline(len(ready), _cp(ready, dp), B, _cp(bof, _i32p), _cp(bord, _i32p),
                                      _cp(bb, _i64p), float(alpha_ms), float(ms_per_byte), _cp(start, dp),
                                      _cp(end, dp), C.byref(step), C.byref(serial)))
    return dict(start_ms=start[:B], end_ms=end[:B], step_ms=step.value, serial_ms=serial.value)


# ---------------------------------------------------------------------------
# steps 2-4
# ---------------------------------------------------------------------------
def ddp_pack(desc: BucketDesc, grads, used, ld, W, main_grad, replica_stride, accumulate=0, stream=None) -> None:
    _check(lib().ddp_pack(C.byref(desc), _ptr(grads), _ptr(used), int(ld), int(W), _ptr(main_grad),
                          int(replica_stride), int(accumulate), _stream(stream)))


def ddp_bucket_allreduce(replicas, replica_stride, numel, W, mode=DDP_ALLREDUCE, stream=None) -> None:
    _check(lib().ddp_bucket_allreduce(_ptr(replicas), int(replica_stride), int(numel), int(W), int(mode),
                                      _stream(stream)))


def ddp_bucket_allreduce_wire(replicas, replica_stride, numel, W, mode=DDP_ALLREDUCE, wire_dtype=DDP_BF16,
                              stream=None) -> None:
    _check(lib().ddp_bucket_allreduce_wire(_ptr(replicas), int(replica_stride), int(numel), int(W), int(mode),
                                           int(wire_dtype), _stream(stream)))


def ddp_unpack(desc: BucketDesc, main_grad, replica_stride, W, mode, grads_out, ld, global_used=None,
               stream=None) -> None:
    _check(lib().ddp_unpack(C.byref(desc), _ptr(main_grad), int(replica_stride), int(W), int(mode),
                            _ptr(grads_out), int(ld), _ptr(global_used), _stream(stream)))


def ddp_fused_bucket(desc: BucketDesc, grads, used, ld, W, mode, accumulate, main_grad, replica_stride,
                     grads_out=None, global_used=None, stream=None) -> None:
    _check(lib().ddp_fused_bucket(C.byref(desc), _ptr(grads), _ptr(used), int(ld), int(W), int(mode),
                                  int(accumulate), _ptr(main_grad), int(replica_stride), _ptr(grads_out),
                                  _ptr(global_used), _stream(stream)))


def ddp_pack_group(descs, bucket_start, grads, used, ld, W, main_grad, replica_stride, accumulate=0,
                   stream=None) -> None:
    B = len(descs)
    arr = (BucketDesc * max(B, 1))(*descs)
    starts = _a(bucket_start, np.int64)
    _check(lib().ddp_pack_group(arr, _cp(starts, _i64p), B, _ptr(grads), _ptr(used), int(ld), int(W),
                                _ptr(main_grad), int(replica_stride), int(accumulate), _stream(stream)))


def ddp_fused_bucket_group(descs, bucket_start, grads, used, ld, W, mode, accumulate, main_grad, replica_stride,
                           grads_out=None, global_used=None, stream=None) -> None:
    B = len(descs)
    arr = (BucketDesc * max(B, 1))(*descs)
    starts = _a(bucket_start, np.int64)
    _check(lib().ddp_fused_bucket_group(arr, _cp(starts, _i64p), B, _ptr(grads), _ptr(used), int(ld), int(W),
                                        int(mode), int(accumulate), _ptr(main_grad), int(replica_stride),
                                        _ptr(grads_out), _ptr(global_used), _stream(stream)))


def ddp_fused_bucket_group_wire(descs, bucket_start, grads, used, ld, W, mode, accumulate, main_grad,
                                replica_stride, grads_out=None, global_used=None, wire_dtype=DDP_BF16,
                                stream=None) -> None:
    B = len(descs)
    arr = (BucketDesc * max(B, 1))(*descs)
    starts = _a(bucket_start, np.int64)
    _check(lib().ddp_fused_bucket_group_wire(arr, _cp(starts, _i64p), B, _ptr(grads), _ptr(used), int(ld), int(W),
                                             int(mode), int(accumulate), _ptr(main_grad), int(replica_stride),
                                             _ptr(grads_out), _ptr(global_used), int(wire_dtype), _stream(stream)))


# ---------------------------------------------------------------------------
# step 5
# ---------------------------------------------------------------------------
def ddp_reducer_create(nparams, bucket_of, bucket_order, descs, bucket_start, W, mode, flags, grads=None, used=None,
                       ld=0, main_grad=None, replica_stride=0, grads_out=None, global_used=None, side_stream=None):
    bucket_of = _a(bucket_of, np.int32)
    bucket_order = _a(bucket_order, np.int32)
    bucket_start = _a(bucket_start, np.int64)
    B = len(bucket_order)
    arr = (BucketDesc * max(B, 1))(*descs)
    h = _vp()
    side = None if flags & DDP_R_DRY_RUN else _stream(side_stream)
    _check(lib().ddp_reducer_create(int(nparams), B, _cp(bucket_of, _i32p), _cp(bucket_order, _i32p), arr,
                                    _cp(bucket_start, _i64p), int(W), int(mode), int(flags), _ptr(grads), _ptr(used),
                                    int(ld), _ptr(main_grad), int(replica_stride), _ptr(grads_out), _ptr(global_used),
                                    side, C.byref(h)))
    return h.value


def ddp_reducer_create_from_plan(plan, descs, W, mode, flags, grads=None, used=None, ld=0, main_grad=None,
                                 grads_out=None, global_used=None, side_stream=None):
    arr = (BucketDesc * max(len(descs), 1))(*descs)
    h = _vp()
    side = None if flags & DDP_R_DRY_RUN else _stream(side_stream)
    _check(lib().ddp_reducer_create_from_plan(plan, arr, int(W), int(mode), int(flags), _ptr(grads), _ptr(used),
                                              int(ld), _ptr(main_grad), _ptr(grads_out), _ptr(global_used), side,
                                              C.byref(h)))
    return h.value


def ddp_used_allreduce(local_used, ld, W, nparams, global_count=None, global_used=None, stream=None) -> None:
    _check(lib().ddp_used_allreduce(_ptr(local_used), int(ld), int(W), int(nparams), _ptr(global_count),
                                    _ptr(global_used), _stream(stream)))


def ddp_reducer_find_unused(r, local_used, global_used, global_count=None) -> None:
    _check(lib().ddp_reducer_find_unused(r, _ptr(local_used), _ptr(global_used), _ptr(global_count)))


def ddp_reducer_set_local_used(r, flags, ld=None) -> None:
    """flags: host uint8 array [W, >= nparams] (nonzero = replica w used parameter p)."""
    f = np.ascontiguousarray(np.asarray(flags), dtype=np.uint8)
    if f.ndim != 2:
        raise ValueError("flags must be [W, nparams]")
    _check(lib().ddp_reducer_set_local_used(r, f.ctypes.data_as(_vp), int(f.shape[1] if ld is None else ld)))


# ---------------------------------------------------------------------------
# the PowerSGD hook
# ---------------------------------------------------------------------------
def ddp_powersgd_create(W, rank, seg_offset, seg_numel, seg_rows, bucket_numel, error_feedback=1, start_iter=0):
    off = _a(seg_offset, np.int64)
    num = _a(seg_numel, np.int64)
    rows = _a(seg_rows, np.int64)
    h = _vp()
    _check(lib().ddp_powersgd_create(int(W), int(rank), len(off), _cp(off, _i64p), _cp(num, _i64p), _cp(rows, _i64p),
                                     int(bucket_numel), int(error_feedback), int(start_iter), C.byref(h)))
    return h.value


def ddp_powersgd_sizes(h) -> dict:
    ws, q, nm = C.c_int64(0), C.c_int64(0), C.c_int32(0)
    _check(lib().ddp_powersgd_sizes(h, C.byref(ws), C.byref(q), C.byref(nm)))
    return dict(workspace_bytes=ws.value, q_elems=q.value, nmatrices=nm.value)


def ddp_powersgd_matrix(h, seg) -> dict:
    off, rows, cols, re, rp = C.c_int64(0), C.c_int32(0), C.c_int32(0), C.c_int32(0), C.c_int32(0)
    _check(lib().ddp_powersgd_matrix(h, int(seg), C.byref(off), C.byref(rows), C.byref(cols), C.byref(re),
                                     C.byref(rp)))
    return dict(q_offset=off.value, rows=rows.value, cols=cols.value, rank_eff=re.value, rank_pad=rp.value)


def ddp_powersgd_bind(h, workspace, workspace_bytes, q_state, error=None, error_stride=0, stream=None) -> None:
    _check(lib().ddp_powersgd_bind(h, _ptr(workspace), int(workspace_bytes), _ptr(q_state), _ptr(error),
                                   int(error_stride), _stream(stream)))


def ddp_powersgd_set_q(h, seg, q, stream=None) -> None:
    qa = np.ascontiguousarray(q, dtype=np.float32)
    _check(lib().ddp_powersgd_set_q(h, int(seg), qa.ctypes.data, _stream(stream)))


def ddp_powersgd_reduce(h, main_grad, replica_stride, stream=None) -> None:
    _check(lib().ddp_powersgd_reduce(h, _ptr(main_grad), int(replica_stride), _stream(stream)))


def ddp_powersgd_reduce_static(h, main_grad, replica_stride, stream=None) -> None:
    _check(lib().ddp_powersgd_reduce_static(h, _ptr(main_grad), int(replica_stride), _stream(stream)))


def ddp_powersgd_iter(h) -> int:
    it = C.c_int32(0)
    _check(lib().ddp_powersgd_iter(h, C.byref(it)))
    return it.value


def ddp_powersgd_destroy(h) -> None:
    if h:
        lib().ddp_powersgd_destroy(h)


def ddp_reducer_register_powersgd(r, bucket, h) -> None:
    _check(lib().ddp_reducer_register_powersgd(r, int(bucket), h))


def ddp_reducer_prepare(r, accumulate=0) -> None:
    _check(lib().ddp_reducer_prepare(r, int(accumulate)))


def ddp_reducer_mark_ready(r, param, producer_stream=None) -> None:
    _check(lib().ddp_reducer_mark_ready(r, int(param), _stream(producer_stream)))


def ddp_reducer_mark_ready_many(r, params, producer_stream=None) -> None:
    params = _a(params, np.int32)
    _check(lib().ddp_reducer_mark_ready_many(r, _cp(params, _i32p), len(params), _stream(producer_stream)))


def ddp_reducer_finalize(r, consumer_stream=None, timeout_us=0) -> None:
    _check(lib().ddp_reducer_finalize(r, _stream(consumer_stream), int(timeout_us)))


def ddp_reducer_wait_bucket(r, bucket, consumer_stream=None) -> None:
    _check(lib().ddp_reducer_wait_bucket(r, int(bucket), _stream(consumer_stream)))


def ddp_reducer_issue_log(r, cap=4096) -> list:
    out = np.zeros(cap, np.int32)
    n = C.c_int32(0)
    _check(lib().ddp_reducer_issue_log(r, _cp(out, _i32p), cap, C.byref(n)))
    return [int(v) for v in out[:n.value]]


def ddp_reducer_ready_order(r, cap=1 << 20) -> list:
    out = np.zeros(cap, np.int32)
    n = C.c_int32(0)
    _check(lib().ddp_reducer_ready_order(r, _cp(out, _i32p), cap, C.byref(n)))
    return [int(v) for v in out[:n.value]]


def ddp_reducer_bucket_ms(r, nbuckets) -> np.ndarray:
    out = np.zeros(max(nbuckets, 1), np.float32)
    _check(lib().ddp_reducer_bucket_ms(r, out.ctypes.data_as(C.POINTER(C.c_float)), len(out)))
    return out[:nbuckets]


def ddp_reducer_destroy(r) -> None:
    if r:
        lib().ddp_reducer_destroy(r)


def ddp_set_kernel_variant(variant: int) -> None:
    _check(lib().ddp_set_kernel_variant(int(variant)))


def ddp_device_status(stream=None, reset=False) -> int:
    v = C.c_int32(0)
    _check(lib().ddp_device_status(_stream(stream), C.byref(v), int(bool(reset))))
    return v.value


def ddp_wait_selftest(arrive, limit_ns, stream=None) -> None:
    _check(lib().ddp_wait_selftest(int(arrive), int(limit_ns), _stream(stream)))


def ddp_copy_rows(dst, dst_pitch, src, src_pitch, row_bytes, rows, stream=None) -> None:
    """Pointers (tensors or integer addresses) and pitches in bytes."""
    _check(lib().ddp_copy_rows(_ptr(dst), int(dst_pitch), _ptr(src), int(src_pitch), int(row_bytes), int(rows),
                               _stream(stream)))


def ddp_host_front_create(r, dev_in, dev_pitch, param_offset, elem_bytes):
    """The host-buffer front end of reducer r; dev_in a pointer (or tensor), pitch in bytes."""
    off = np.ascontiguousarray(param_offset, np.int64)
    h = _vp()
    _check(lib().ddp_host_front_create(r, _ptr(dev_in), int(dev_pitch), _cp(off, _i64p), int(elem_bytes), C.byref(h)))
    return h


def ddp_host_front_step(h, host_in, host_pitch, host_out, stream=None) -> None:
    _check(lib().ddp_host_front_step(h, _ptr(host_in), int(host_pitch), _ptr(host_out), _stream(stream)))


def ddp_host_front_destroy(h) -> None:
    lib().ddp_host_front_destroy(h)


def ddp_status_str(s: int) -> str:
    return lib().ddp_status_str(int(s)).decode()


def ddp_last_error_message() -> str:
    return lib().ddp_last_error_message().decode()


def ddp_version() -> int:
    return int(lib().ddp_version())


from .plan import Plan  # noqa: E402  (plumbing over the calls above)

__all__ = [n for n in _SIGS] + ["Plan", "BucketDesc", "DdpError", "lib", "library_path"]

