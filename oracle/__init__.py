"""ctypes wrapper of the plain-C oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use this module; the library never does.  It shares no code
with the CUDA path.

``build()`` compiles ``oracle.c`` with ``-ffp-contract=off`` into
``oracle/_lib/liboracle.so``; ``load()`` returns a handle.  The helpers below
only marshal numpy arrays; every step of the method is in the C file.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "liboracle.so")

REVERSE, FWD_THEN_REVERSE, MEGATRON = 0, 1, 2
ALLREDUCE, REDUCE_SCATTER = 0, 1
F32, BF16, F16 = 0, 1, 2

_i64p = C.POINTER(C.c_int64)
_i32p = C.POINTER(C.c_int32)
_u8p = C.POINTER(C.c_uint8)
_u64p = C.POINTER(C.c_uint64)
_vpp = C.POINTER(C.c_void_p)


def build(src: str = SRC, out: str = LIB, extra: tuple = ()) -> str:
    """Compile the oracle (plain C99, no FMA contraction). Rebuilds when the source is newer."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src) and not extra:
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["cc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", *extra, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """One loaded copy of the oracle library (tests may load mutated copies)."""

    def __init__(self, path: str):
        lib = C.CDLL(path)
        lib.oracle_assign.restype = C.c_int
        lib.oracle_assign.argtypes = [_i64p, _i32p, C.c_int32, C.c_int64, C.c_int64, C.c_int32,
                                      C.c_int32, C.c_int32, _i32p, _i64p, _i64p, _i64p, _i32p,
                                      _i32p, _i32p, C.c_int32, _i32p]
        lib.oracle_assign_sequence.restype = C.c_int
        lib.oracle_assign_sequence.argtypes = [_i64p, _i32p, C.c_int32, _i32p, C.c_int64, C.c_int64, C.c_int32,
                                               C.c_int32, _i32p, _i64p, _i64p, _i64p, _i32p, _i32p, _i32p,
                                               C.c_int32, _i32p]
        _dp = C.POINTER(C.c_double)
        lib.oracle_overlap_timeline.restype = C.c_int
        lib.oracle_overlap_timeline.argtypes = [C.c_int32, _dp, C.c_int32, _i32p, _i32p, _i64p, C.c_double,
                                                C.c_double, _dp, _dp, _dp, _dp]
        lib.oracle_pack.restype = None
        lib.oracle_pack.argtypes = [C.c_int32, C.c_int32, _i64p, _i64p, _i32p, _vpp, _u8p, C.c_int32,
                                    _vpp, C.c_int64]
        lib.oracle_ring_allreduce.restype = C.c_int
        lib.oracle_ring_allreduce.argtypes = [_vpp, C.c_int32, C.c_int64, C.c_int32, _u64p]
        lib.oracle_ring_allreduce_wire.restype = C.c_int
        lib.oracle_ring_allreduce_wire.argtypes = [_vpp, C.c_int32, C.c_int64, C.c_int32, C.c_int32, _u64p]
        lib.oracle_round_wire.restype = C.c_uint16
        lib.oracle_round_wire.argtypes = [C.c_double, C.c_int32]
        lib.oracle_wire_value.restype = C.c_double
        lib.oracle_wire_value.argtypes = [C.c_uint16, C.c_int32]
        lib.oracle_used_allreduce.restype = C.c_int
        lib.oracle_used_allreduce.argtypes = [C.c_int32, C.c_int32, _u8p, _i32p, _u8p]
        lib.oracle_unpack.restype = None
        lib.oracle_unpack.argtypes = [C.c_int32, C.c_int32, _i64p, _i64p, _vpp, C.c_int64, C.c_int32,
                                      _u8p, _vpp]
        self.lib = lib

    # -- assignment --------------------------------------------------------
    def assign(self, numels, dtypes=None, cap_bytes=25 << 20, first_cap_bytes=1 << 20,
               order=REVERSE, pad_multiple=1, grad_reduce_in_fp32=1) -> dict:
        numels = np.ascontiguousarray(numels, dtype=np.int64)
        P = len(numels)
        dtypes = np.zeros(P, np.int32) if dtypes is None else np.ascontiguousarray(dtypes, dtype=np.int32)
        bucket_of = np.full(P, -1, np.int32)
        offset_of = np.full(P, -1, np.int64)
        cap = P + 3
        bn = np.zeros(cap, np.int64)
        bb = np.zeros(cap, np.int64)
        bd = np.zeros(cap, np.int32)
        bo = np.zeros(cap, np.int32)
        mem = np.zeros(max(P, 1), np.int32)
        nb = C.c_int32(0)
        rc = self.lib.oracle_assign(_p(numels, _i64p), _p(dtypes, _i32p), P, int(cap_bytes),
                                    int(first_cap_bytes), int(order), int(pad_multiple),
                                    int(grad_reduce_in_fp32), _p(bucket_of, _i32p), _p(offset_of, _i64p),
                                    _p(bn, _i64p), _p(bb, _i64p), _p(bd, _i32p), _p(bo, _i32p), _p(mem, _i32p), cap,
                                    C.byref(nb))
        if rc != 0:
            raise ValueError(f"oracle_assign returned {rc}")
        B = nb.value
        members = [[] for _ in range(B)]
        for p in mem[:P]:
            members[bucket_of[p]].append(int(p))
        return dict(bucket_of=bucket_of, offset_of=offset_of, bucket_numel=bn[:B].copy(),
                    bucket_bytes=bb[:B].copy(), bucket_dtype=bd[:B].copy(), bucket_order=bo[:B].copy(),
                    members=members, nbuckets=B)

    def assign_sequence(self, numels, sequence, dtypes=None, cap_bytes=25 << 20, first_cap_bytes=1 << 20,
                        pad_multiple=1, grad_reduce_in_fp32=1) -> dict:
        """Rebuilt buckets over an observed gradient-ready order."""
        numels = np.ascontiguousarray(numels, dtype=np.int64)
        P = len(numels)
        seq = np.ascontiguousarray(sequence, dtype=np.int32)
        dtypes = np.zeros(P, np.int32) if dtypes is None else np.ascontiguousarray(dtypes, dtype=np.int32)
        out = self._assign_out(P)
        nb = C.c_int32(0)
        rc = self.lib.oracle_assign_sequence(_p(numels, _i64p), _p(dtypes, _i32p), P, _p(seq, _i32p),
                                             int(cap_bytes), int(first_cap_bytes), int(pad_multiple),
                                             int(grad_reduce_in_fp32), *out["ptrs"], out["cap"], C.byref(nb))
        if rc != 0:
            raise ValueError(f"oracle_assign_sequence returned {rc}")
        return self._assign_result(out, nb.value, P)

    def _assign_out(self, P):
        cap = P + 3
        arrs = dict(bucket_of=np.full(P, -1, np.int32), offset_of=np.full(P, -1, np.int64),
                    bucket_numel=np.zeros(cap, np.int64), bucket_bytes=np.zeros(cap, np.int64),
                    bucket_dtype=np.zeros(cap, np.int32), bucket_order=np.zeros(cap, np.int32),
                    mem=np.zeros(max(P, 1), np.int32))
        ptrs = [_p(arrs["bucket_of"], _i32p), _p(arrs["offset_of"], _i64p), _p(arrs["bucket_numel"], _i64p),
                _p(arrs["bucket_bytes"], _i64p), _p(arrs["bucket_dtype"], _i32p), _p(arrs["bucket_order"], _i32p),
                _p(arrs["mem"], _i32p)]
        return dict(arrs=arrs, ptrs=ptrs, cap=cap)

    def _assign_result(self, out, B, P):
        a = out["arrs"]
        members = [[] for _ in range(B)]
        for p in a["mem"][:P]:
            members[a["bucket_of"][p]].append(int(p))
        return dict(bucket_of=a["bucket_of"], offset_of=a["offset_of"], bucket_numel=a["bucket_numel"][:B].copy(),
                    bucket_bytes=a["bucket_bytes"][:B].copy(), bucket_dtype=a["bucket_dtype"][:B].copy(),
                    bucket_order=a["bucket_order"][:B].copy(), members=members, nbuckets=B)

    def overlap_timeline(self, ready_ms, bucket_of, bucket_order, bucket_bytes, alpha_ms, ms_per_byte) -> dict:
        ready = np.ascontiguousarray(ready_ms, dtype=np.float64)
        bof = np.ascontiguousarray(bucket_of, dtype=np.int32)
        bord = np.ascontiguousarray(bucket_order, dtype=np.int32)
        bb = np.ascontiguousarray(bucket_bytes, dtype=np.int64)
        B = len(bord)
        start, end = np.zeros(max(B, 1)), np.zeros(max(B, 1))
        step, serial = C.c_double(0), C.c_double(0)
        _dp = C.POINTER(C.c_double)
        rc = self.lib.oracle_overlap_timeline(len(ready), _p(ready, _dp), B, _p(bof, _i32p), _p(bord, _i32p),
                                              _p(bb, _i64p), float(alpha_ms), float(ms_per_byte), _p(start, _dp),
                                              _p(end, _dp), C.byref(step), C.byref(serial))
        if rc != 0:
            raise ValueError(f"oracle_overlap_timeline returned {rc}")
        return dict(start_ms=start[:B], end_ms=end[:B], step_ms=step.value, serial_ms=serial.value)

    # -- pack ---------------------------------------------------------------
    def pack(self, grads, seg_offset, bucket_numel, seg_dtype=None, used=None, accumulate=False,
             out=None) -> np.ndarray:
        """grads: list over replicas of lists over segments (np arrays: float32 or uint16 bit patterns).
        Returns the [W, bucket_numel] fp32 bucket (``out`` updated in place when given)."""
        W, S = len(grads), len(seg_offset)
        seg_offset = np.ascontiguousarray(seg_offset, dtype=np.int64)
        seg_numel = np.array([len(grads[0][s]) if grads[0][s] is not None else 0 for s in range(S)],
                             dtype=np.int64)
        if used is not None:
            # unused segments may carry None; take the length from any replica that has it
            for s in range(S):
                for w in range(W):
                    if grads[w][s] is not None:
                        seg_numel[s] = len(grads[w][s])
                        break
        seg_dtype = np.zeros(S, np.int32) if seg_dtype is None else np.ascontiguousarray(seg_dtype, np.int32)
        keep = []
        ptrs = (C.c_void_p * max(W * S, 1))()
        for w in range(W):
            for s in range(S):
                g = grads[w][s]
                if g is None:
                    ptrs[w * S + s] = None
                else:
                    g = np.ascontiguousarray(g)
                    keep.append(g)
                    ptrs[w * S + s] = g.ctypes.data
        if out is None:
            out = np.zeros((W, bucket_numel), np.float32)
        assert out.dtype == np.float32 and out.flags.c_contiguous
        rows = (C.c_void_p * W)(*[out[w].ctypes.data for w in range(W)])
        used_arr = None if used is None else np.ascontiguousarray(used, dtype=np.uint8).reshape(-1)
        self.lib.oracle_pack(W, S, _p(seg_offset, _i64p), _p(seg_numel, _i64p), _p(seg_dtype, _i32p),
                             ptrs, None if used_arr is None else _p(used_arr, _u8p), int(bool(accumulate)),
                             rows, int(bucket_numel))
        return out

    # -- ring ---------------------------------------------------------------
    def ring(self, bufs: np.ndarray, mode=ALLREDUCE):
        """bufs: [W, n] float32, replaced in place. Returns (bufs, bytes_sent[W])."""
        assert bufs.dtype == np.float32 and bufs.flags.c_contiguous and bufs.ndim == 2
        W, n = bufs.shape
        rows = (C.c_void_p * W)(*[bufs[w].ctypes.data for w in range(W)])
        sent = np.zeros(W, np.uint64)
        rc = self.lib.oracle_ring_allreduce(rows, W, n, int(mode), _p(sent, _u64p))
        if rc != 0:
            raise ValueError(f"oracle_ring_allreduce returned {rc}")
        return bufs, sent

    def ring_wire(self, bufs: np.ndarray, mode=ALLREDUCE, wire=BF16):
        """The compression hook's ring: messages and partial sums in the wire type
        (bf16 or fp16).  bufs: [W, n] float32, replaced in place."""
        assert bufs.dtype == np.float32 and bufs.flags.c_contiguous and bufs.ndim == 2
        W, n = bufs.shape
        rows = (C.c_void_p * W)(*[bufs[w].ctypes.data for w in range(W)])
        sent = np.zeros(W, np.uint64)
        rc = self.lib.oracle_ring_allreduce_wire(rows, W, n, int(mode), int(wire), _p(sent, _u64p))
        if rc != 0:
            raise ValueError(f"oracle_ring_allreduce_wire returned {rc}")
        return bufs, sent

    def round_wire(self, x: float, wire=BF16) -> int:
        return int(self.lib.oracle_round_wire(float(x), int(wire)))

    def wire_value(self, h: int, wire=BF16) -> float:
        return float(self.lib.oracle_wire_value(int(h), int(wire)))

    # -- local-used bitmap ---------------------------------------------------
    def used_allreduce(self, local_used) -> tuple:
        """local_used [W, P] (nonzero = used) -> (global_count int32[P], global_used uint8[P])."""
        lu = np.ascontiguousarray(np.asarray(local_used, np.uint8))
        if lu.ndim != 2:
            raise ValueError("local_used must be [W, P]")
        W, P = lu.shape
        count = np.zeros(max(P, 1), np.int32)
        glob = np.zeros(max(P, 1), np.uint8)
        rc = self.lib.oracle_used_allreduce(W, P, _p(lu, _u8p), _p(count, _i32p), _p(glob, _u8p))
        if rc != 0:
            raise ValueError("oracle_used_allreduce rejected its arguments")
        return count[:P], glob[:P]

    # -- unpack -------------------------------------------------------------
    def unpack(self, bucket: np.ndarray, seg_offset, seg_numel, mode=ALLREDUCE, global_used=None, outs=None):
        """bucket: [W, n] fp32. outs: list over replicas of lists over segments (fp32 arrays,
        updated in place); fresh zero arrays when not given."""
        W, n = bucket.shape
        S = len(seg_offset)
        seg_offset = np.ascontiguousarray(seg_offset, dtype=np.int64)
        seg_numel = np.ascontiguousarray(seg_numel, dtype=np.int64)
        if outs is None:
            outs = [[np.zeros(int(seg_numel[s]), np.float32) for s in range(S)] for _ in range(W)]
        ptrs = (C.c_void_p * max(W * S, 1))()
        for w in range(W):
            for s in range(S):
                assert outs[w][s].dtype == np.float32 and outs[w][s].flags.c_contiguous
                ptrs[w * S + s] = outs[w][s].ctypes.data
        rows = (C.c_void_p * W)(*[bucket[w].ctypes.data for w in range(W)])
        gu = None if global_used is None else np.ascontiguousarray(global_used, dtype=np.uint8)
        self.lib.oracle_unpack(W, S, _p(seg_offset, _i64p), _p(seg_numel, _i64p), rows, n, int(mode),
                               None if gu is None else _p(gu, _u8p), ptrs)
        return outs


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


_DEFAULT: Oracle | None = None


def load() -> Oracle:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle(build())
    return _DEFAULT


# ---------------------------------------------------------------------------
# the whole path over one workload (composition of the four steps above)
# ---------------------------------------------------------------------------
def run_workload(wl, orc: Oracle | None = None, grads=None, copy_back: bool = True, wire=None):
    """Assign, then for every bucket: pack (accumulating over the workload's
    micro-steps), ring-reduce, unpack.  ``grads[m][w][p]`` may be given (raw
    storage arrays); otherwise they are generated.  Returns a dict with the plan,
    the reduced buckets ``bucket[b]`` ([W, numel]) and, when ``copy_back``, the
    per-parameter outputs ``out[w][p]`` (None for globally unused parameters).
    ``wire`` (BF16 / F16) reduces through the compression hook's ring instead."""
    import workloads as W_

    orc = orc or load()
    P = wl.nparams
    plan = orc.assign(wl.numels, [wl.dtype] * P, wl.cap_bytes, wl.first_cap_bytes, wl.order,
                      wl.pad_multiple, wl.grad_reduce_in_fp32)
    if grads is None:
        grads = [[[W_.grad_raw_np(wl, p, w, m) for p in range(P)] for w in range(wl.W)]
                 for m in range(wl.micro_steps)]
    used = W_.local_used_np(wl)
    global_used = orc.used_allreduce(used)[1]
    buckets, sent = [], []
    out = [[None] * P for _ in range(wl.W)]
    for b in range(plan["nbuckets"]):
        mem = plan["members"][b]
        offs = [int(plan["offset_of"][p]) for p in mem]
        nb = int(plan["bucket_numel"][b])
        buf = None
        for m in range(wl.micro_steps):
            gl = [[grads[m][w][p] for p in mem] for w in range(wl.W)]
            buf = orc.pack(gl, offs, nb, [wl.dtype] * len(mem), used[:, mem], accumulate=m > 0, out=buf)
        buf, s = orc.ring(buf, wl.mode) if wire is None else orc.ring_wire(buf, wl.mode, wire)
        buckets.append(buf)
        sent.append(s)
        if copy_back:
            outs = orc.unpack(buf, offs, [wl.numels[p] for p in mem], wl.mode, global_used[mem])
            for w in range(wl.W):
                for j, p in enumerate(mem):
                    out[w][p] = outs[w][j] if global_used[p] else None
    return dict(plan=plan, bucket=buckets, bytes_sent=sent, out=out, global_used=global_used)
