"""Plumbing around the library's plan object (ddp_plan_create): the caller-owned
tables the kernels read.

A Plan asks the library for the bucket assignment and its layout (each bucket
starting on a 64-element, 256-byte boundary of the per-replica fp32 main_grad
buffer, so every replica's copy is vector-aligned), copies the plan's segment
tables to the device and gets the bucket descriptors over those copies.
Nothing here computes any part of the path.
"""
from __future__ import annotations

import numpy as np

from . import (ddp_plan_bucket_descs, ddp_plan_create, ddp_plan_describe, ddp_plan_destroy, ddp_plan_rebuilt,
               ddp_plan_tables)

ALIGN_ELEMS = 64


class Plan:
    def __init__(self, numels, dtypes=None, cap_bytes=25 << 20, first_cap_bytes=1 << 20, order=0, pad_multiple=1,
                 grad_reduce_in_fp32=1, device="cuda"):
        import torch

        self.numels = [int(v) for v in numels]
        P = self.nparams = len(self.numels)
        self.dtypes = [0] * P if dtypes is None else [int(v) for v in dtypes]
        self.handle = ddp_plan_create(self.numels, self.dtypes, cap_bytes, first_cap_bytes, order, pad_multiple,
                                      grad_reduce_in_fp32, ALIGN_ELEMS)
        a = self.assignment = ddp_plan_describe(self.handle)
        self.caps = dict(cap_bytes=int(cap_bytes), first_cap_bytes=int(first_cap_bytes), order=int(order),
                         pad_multiple=int(pad_multiple), grad_reduce_in_fp32=int(grad_reduce_in_fp32))
        self.nbuckets = B = a["nbuckets"]
        self.bucket_of = a["bucket_of"]
        self.offset_of = a["offset_of"]
        self.bucket_numel = a["bucket_numel"]
        self.bucket_bytes = a["bucket_bytes"]
        self.bucket_dtype = a["bucket_dtype"]
        self.bucket_order = a["bucket_order"]
        self.bucket_start = a["bucket_start"]
        self.replica_stride = int(a["replica_stride"])
        ms = a["member_start"]
        self.members = [[int(p) for p in a["members"][ms[b]:ms[b + 1]]] for b in range(B)]
        self.device = torch.device(device)

        # the kernels' segment tables, all buckets in one device tensor each
        so, sp = ddp_plan_tables(self.handle, a["seg_offset_len"], a["seg_param_len"])
        self.seg_offset_dev = torch.from_numpy(so if len(so) else np.zeros(1, np.int64)).to(self.device)
        self.seg_param_dev = torch.from_numpy(sp if len(sp) else np.zeros(1, np.int32)).to(self.device)
        self.descs = ddp_plan_bucket_descs(self.handle, B, self.seg_offset_dev, self.seg_param_dev)

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
        sequence (ddp_plan_rebuilt), as plain lists."""
        a = ddp_plan_rebuilt(self.handle, sequence, self.nparams)
        return dict(num_buckets=int(a["nbuckets"]), bucket_sizes=[int(v) for v in a["bucket_bytes"]])

    def close(self):
        if getattr(self, "handle", None):
            ddp_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

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
