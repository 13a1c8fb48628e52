"""The PowerSGD hook's buffers for one bucket: plumbing over ddp_powersgd_*.

Owns the caller-side memory the C ABI asks for (workspace, Q state, error
buffers) as torch tensors, writes each matrix's initial Q, and forwards
``reduce`` to ``ddp_powersgd_reduce``; every step of the hook runs in
libddpbucket ("DDP: ring AllReduce and gradient buckets", section 17.27).
"""
from __future__ import annotations

import numpy as np

from . import (ddp_powersgd_bind, ddp_powersgd_create, ddp_powersgd_destroy, ddp_powersgd_iter,
               ddp_powersgd_matrix, ddp_powersgd_reduce, ddp_powersgd_set_q, ddp_powersgd_sizes)


def matrix_rows(shape) -> int:
    """Rows of the hook's matrix view (shape[0]) for tensors of two or more
    dimensions, 0 for 1-D ones (they take the plain all-reduce)."""
    return int(shape[0]) if len(shape) >= 2 else 0


class PowerSGDBucket:
    """seg_offset / seg_numel / shapes: the bucket's tensors; q0(k, n, r) returns
    tensor k's initial Q (n x r floats) -- the hook's random draw."""

    def __init__(self, W, rank, seg_offset, seg_numel, shapes, bucket_numel, q0, error_feedback=True,
                 start_iter=0, device="cuda", stream=None):
        import torch

        self.W, self.numel = int(W), int(bucket_numel)
        rows = [matrix_rows(s) for s in shapes]
        self.handle = ddp_powersgd_create(W, rank, seg_offset, seg_numel, rows, bucket_numel, int(error_feedback),
                                          start_iter)
        sz = ddp_powersgd_sizes(self.handle)
        self.workspace = torch.empty(sz["workspace_bytes"] + 256, dtype=torch.uint8, device=device)
        ws_ptr = (self.workspace.data_ptr() + 255) // 256 * 256
        self.q_state = torch.zeros(max(sz["q_elems"], 4), dtype=torch.float32, device=device)
        self.error = (torch.zeros(self.W * max(self.numel, 1), dtype=torch.float32, device=device)
                      if error_feedback else None)
        ddp_powersgd_bind(self.handle, ws_ptr, sz["workspace_bytes"], self.q_state, self.error,
                          max(self.numel, 1), stream)
        self.matrices = {}
        for k, r in enumerate(rows):
            if r > 0:
                info = ddp_powersgd_matrix(self.handle, k)
                self.matrices[k] = info
                ddp_powersgd_set_q(self.handle, k, np.asarray(q0(k, info["cols"], info["rank_eff"]), np.float32),
                                   stream)

    def reduce(self, main_grad, replica_stride, stream=None):
        ddp_powersgd_reduce(self.handle, main_grad, replica_stride, stream)

    @property
    def iteration(self) -> int:
        return ddp_powersgd_iter(self.handle)

    def q(self, k):
        """Segment k's current Q as an (N, rank_eff) tensor view."""
        i = self.matrices[k]
        v = self.q_state[i["q_offset"]:i["q_offset"] + i["cols"] * i["rank_pad"]].view(i["cols"], i["rank_pad"])
        return v[:, :i["rank_eff"]]

    def error_of(self, w, off, n):
        return self.error[w * self.numel + off:w * self.numel + off + n]

    def close(self):
        if self.handle:
            ddp_powersgd_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
