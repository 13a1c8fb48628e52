"""Plumbing around ddp_assign_buckets: the caller-owned tables the kernels read.

A Plan runs the library's bucket assignment once, lays the buckets out in one
fp32 main_grad buffer per replica (each bucket starting on a 64-element,
256-byte boundary so every replica's copy is vector-aligned), and uploads the
per-bucket segment tables (ddp_bucket_desc.seg_offset / seg_param) to the
device.  Nothing here computes any part of the path.
"""
from __future__ import annotations

import numpy as np

from . import BucketDesc, ddp_assign_buckets, ddp_assign_buckets_ordered

ALIGN_ELEMS = 64


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


class Plan:
    def __init__(self, numels, dtypes=None, cap_bytes=25 << 20, first_cap_bytes=1 << 20, order=0, pad_multiple=1,
                 grad_reduce_in_fp32=1, device="cuda"):
        import torch

        self.numels = [int(v) for v in numels]
        P = self.nparams = len(self.numels)
        self.dtypes = [0] * P if dtypes is None else [int(v) for v in dtypes]
        a = ddp_assign_buckets(self.numels, self.dtypes, cap_bytes, first_cap_bytes, order, pad_multiple,
                               grad_reduce_in_fp32)
        self.assignment = a
        self.caps = dict(cap_bytes=int(cap_bytes), first_cap_bytes=int(first_cap_bytes), order=int(order),
                         pad_multiple=int(pad_multiple), grad_reduce_in_fp32=int(grad_reduce_in_fp32))
        self.nbuckets = B = a["nbuckets"]
        self.bucket_of = a["bucket_of"]
        self.offset_of = a["offset_of"]
        self.bucket_numel = a["bucket_numel"]
        self.bucket_bytes = a["bucket_bytes"]
        self.bucket_dtype = a["bucket_dtype"]
        self.bucket_order = a["bucket_order"]
        self.members = [[] for _ in range(B)]
        for p in a["members"]:
            self.members[self.bucket_of[p]].append(int(p))
        starts, pos = [], 0
        for b in range(B):
            starts.append(pos)
            pos = _round_up(pos + int(self.bucket_numel[b]), ALIGN_ELEMS)
        self.bucket_start = np.array(starts, dtype=np.int64)
        self.replica_stride = max(pos, ALIGN_ELEMS)
        self.device = torch.device(device)

        # segment tables, all buckets in one tensor each
        seg_off, seg_par, self._seg_base = [], [], []
        for b in range(B):
            self._seg_base.append((len(seg_off), len(seg_par)))
            for p in self.members[b]:
                seg_off.append(int(self.offset_of[p]))
                seg_par.append(p)
            end = int(self.offset_of[self.members[b][-1]]) + self.numels[self.members[b][-1]] if self.members[b] else 0
            seg_off.append(end)
        self.seg_offset_dev = torch.tensor(seg_off or [0], dtype=torch.int64, device=self.device)
        self.seg_param_dev = torch.tensor(seg_par or [0], dtype=torch.int32, device=self.device)
        self.descs = []
        for b in range(B):
            o, q = self._seg_base[b]
            self.descs.append(BucketDesc(int(self.bucket_numel[b]), len(self.members[b]), int(self.bucket_dtype[b]),
                                         self.seg_offset_dev.data_ptr() + 8 * o,
                                         self.seg_param_dev.data_ptr() + 4 * q))

    # -- description ----------------------------------------------------------
    def describe(self) -> dict:
        """The plan as DDP's logging data reports it ("DDP: ring AllReduce and
        gradient buckets" 17.13: bucket_sizes): per bucket its bytes, padded
        elements, dtype and parameter indices, and the issue order."""
        B = self.nbuckets
        return dict(num_buckets=B, bucket_sizes=[int(self.bucket_bytes[b]) for b in range(B)],
                    bucket_numel=[int(self.bucket_numel[b]) for b in range(B)],
                    bucket_dtype=[int(self.bucket_dtype[b]) for b in range(B)],
                    bucket_params=[list(self.members[b]) for b in range(B)],
                    bucket_order=[int(v) for v in self.bucket_order], **self.caps)

    def rebuilt(self, sequence) -> dict:
        """The buckets a rebuild would form over the observed gradient-ready
        sequence (ddp_assign_buckets_ordered), as plain lists."""
        a = ddp_assign_buckets_ordered(self.numels, sequence, self.dtypes, self.caps["cap_bytes"],
                                       self.caps["first_cap_bytes"], self.caps["pad_multiple"],
                                       self.caps["grad_reduce_in_fp32"])
        return dict(num_buckets=int(a["nbuckets"]), bucket_sizes=[int(v) for v in a["bucket_bytes"]])

    # -- buffers and tables -------------------------------------------------
    def alloc_main_grad(self, W: int, fill: float = 0.0):
        import torch

        return torch.full((W * self.replica_stride,), fill, dtype=torch.float32, device=self.device)

    def main_grad_at(self, main_grad, b: int, w: int = 0) -> int:
        """Device address of replica w's copy of bucket b."""
        return main_grad.data_ptr() + 4 * (w * self.replica_stride + int(self.bucket_start[b]))

    def pointer_table(self, tensors):
        """tensors[w][p] (torch tensors or None) -> device int64 [W * P] of addresses."""
        import torch

        W = len(tensors)
        t = np.zeros(W * self.nparams, dtype=np.int64)
        for w in range(W):
            for p in range(self.nparams):
                x = tensors[w][p]
                t[w * self.nparams + p] = 0 if x is None else x.data_ptr()
        return torch.from_numpy(t).to(self.device)

    def flag_table(self, flags):
        import torch

        return torch.from_numpy(np.ascontiguousarray(flags, dtype=np.uint8).reshape(-1)).to(self.device)

    def view(self, main_grad, p: int, w: int = 0):
        """gradient_as_bucket_view: parameter p's gradient on replica w as a view of main_grad."""
        b = int(self.bucket_of[p])
        s = w * self.replica_stride + int(self.bucket_start[b]) + int(self.offset_of[p])
        return main_grad[s:s + self.numels[p]]

    def bucket_view(self, main_grad, b: int):
        """[W, numel] view of bucket b across replicas."""
        W = main_grad.numel() // self.replica_stride
        m = main_grad.view(W, self.replica_stride)
        s = int(self.bucket_start[b])
        return m[:, s:s + int(self.bucket_numel[b])]
