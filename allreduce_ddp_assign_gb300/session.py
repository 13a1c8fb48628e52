"""User-level API: one object that owns a bucket plan, the replicas' buffers'
pointer tables and a reducer, and runs DDP's synchronised backward over them.

Plumbing over the C ABI: the assignment, every kernel and the schedule run in
libddpbucket.  Gradients are marked ready in reverse parameter order, the order
backward produces them ("DDP: ring AllReduce and gradient buckets", 17.3.1).
"""
from __future__ import annotations

import numpy as np

from . import (DDP_BF16, DDP_F16, DDP_R_COALESCE, DDP_R_COPY_BACK, DDP_R_FUSED, DDP_R_TIMING, DDP_R_WIRE_BF16,
               DDP_R_WIRE_F16, DDP_R_BUCKET_DONE, Plan, ddp_pack, ddp_pack_group,
               ddp_reducer_bucket_ms, ddp_reducer_create,
               ddp_reducer_destroy, ddp_reducer_finalize, ddp_reducer_issue_log, ddp_reducer_mark_ready,
               ddp_host_front_create, ddp_host_front_destroy, ddp_host_front_step,
               ddp_reducer_find_unused, ddp_reducer_mark_ready_many, ddp_reducer_prepare,
               ddp_reducer_ready_order, ddp_reducer_register_powersgd, ddp_reducer_set_local_used, DdpError)


class BucketReducer:
    """W data-parallel replicas of one model's gradients on this GPU.

    grads[w][p]   replica w's gradient tensor of parameter p (fp32/bf16/fp16,
                  contiguous, on the device), or None if never produced.
    used[w][p]    optional 0/1 array: replica w produced p this iteration.
    grads_out     optional [w][p] fp32 tensors receiving the reduced gradients
                  (copy-back); otherwise read them through ``view``.
    """

    def __init__(self, numels, dtypes, W, mode, order, cap_bytes, first_cap_bytes, pad_multiple, grads, used=None,
                 grads_out=None, fused=True, timing=False, side_stream=None, main_grad=True, grad_reduce_in_fp32=1,
                 coalesce=False, wire=None, powersgd=None, bucket_done=False):
        """powersgd: dict(rank, shapes, q0, error_feedback=True, start_iter=0) registers the
        PowerSGD hook on every bucket; shapes[p] is parameter p's shape and q0(p, n, r)
        its initial Q (n x r), the hook's random draw."""
        import torch

        self.W, self.mode = int(W), int(mode)
        self.coalesce = bool(coalesce)
        self.plan = Plan(numels, dtypes, cap_bytes, first_cap_bytes, order, pad_multiple, grad_reduce_in_fp32)
        P = self.plan.nparams
        self.side = side_stream if side_stream is not None else torch.cuda.Stream()
        self.main_grad = self.plan.alloc_main_grad(self.W) if main_grad else None
        self._tensors = (grads, grads_out)   # the pointer tables below point into these
        self.grads_tab = self.plan.pointer_table(grads)
        self.used_np = None if used is None else np.ascontiguousarray(used, dtype=np.uint8).reshape(self.W, P)
        self.used_tab = None if used is None else self.plan.flag_table(self.used_np)   # no_sync packs
        self.out_tab = None if grads_out is None else self.plan.pointer_table(grads_out)
        flags = (DDP_R_FUSED if fused else 0) | (DDP_R_COPY_BACK if grads_out is not None else 0) | \
                (DDP_R_TIMING if timing else 0) | (DDP_R_COALESCE if coalesce and fused else 0) | \
                {None: 0, DDP_BF16: DDP_R_WIRE_BF16, DDP_F16: DDP_R_WIRE_F16}[wire] | \
                (DDP_R_BUCKET_DONE if bucket_done else 0)
        self.handle = ddp_reducer_create(P, self.plan.bucket_of, self.plan.bucket_order, self.plan.descs,
                                         self.plan.bucket_start, self.W, self.mode, flags, self.grads_tab,
                                         None, P, self.main_grad, self.plan.replica_stride, self.out_tab,
                                         None, self.side)
        self.ready_order = np.arange(P - 1, -1, -1, dtype=np.int32)
        self.hooks = []
        if powersgd is not None:
            from .powersgd import PowerSGDBucket

            cfg = dict(error_feedback=True, start_iter=0)
            cfg.update(powersgd)
            for b in range(self.plan.nbuckets):
                mem = self.plan.members[b]
                hook = PowerSGDBucket(self.W, cfg["rank"], [int(self.plan.offset_of[p]) for p in mem],
                                      [int(self.plan.numels[p]) for p in mem], [cfg["shapes"][p] for p in mem],
                                      int(self.plan.bucket_numel[b]),
                                      lambda k, n, r, mem=mem: cfg["q0"](mem[k], n, r),
                                      error_feedback=cfg["error_feedback"], start_iter=cfg["start_iter"],
                                      device=self.plan.device, stream=self.side)
                ddp_reducer_register_powersgd(self.handle, b, hook.handle)
                self.hooks.append(hook)
        if used is not None:
            # find_unused_parameters: the reducer uploads the host bitmap at every prepare,
            # all-reduces it on the side stream and marks the parameters nobody used
            dev = self.plan.device
            self.local_used_dev = torch.zeros(max(self.W * P, 1), dtype=torch.uint8, device=dev)
            self.global_used_dev = torch.zeros(max(P, 1), dtype=torch.uint8, device=dev)
            self.global_count_dev = torch.zeros(max(P, 1), dtype=torch.int32, device=dev)
            ddp_reducer_find_unused(self.handle, self.local_used_dev, self.global_used_dev, self.global_count_dev)
            self.set_local_used(self.used_np)

    def set_local_used(self, used):
        """This iteration's local-used bitmap [W, P] (find_unused_parameters)."""
        self.used_np = np.ascontiguousarray(used, dtype=np.uint8).reshape(self.W, self.plan.nparams)
        ddp_reducer_set_local_used(self.handle, self.used_np)
        # parameters nobody used are marked by prepare; the backward produces the rest
        produced = self.used_np.any(axis=0)
        self.ready_order = np.array([p for p in range(self.plan.nparams - 1, -1, -1) if produced[p]], np.int32)

    # -- one iteration ----------------------------------------------------
    def accumulate_local(self, grads_tab, first: bool, stream=None):
        """A no_sync micro-step: add (or, for the first, copy) this micro-step's
        gradients into main_grad without reducing (ddp_pack).  The tensors behind
        grads_tab must stay alive until the stream has run the kernels."""
        if self.coalesce:
            ddp_pack_group(self.plan.descs, self.plan.bucket_start, grads_tab, self.used_tab, self.plan.nparams, self.W,
                           self.main_grad, self.plan.replica_stride, 0 if first else 1, stream)
            return
        for b in range(self.plan.nbuckets):
            ddp_pack(self.plan.descs[b], grads_tab, self.used_tab, self.plan.nparams, self.W,
                     self.plan.main_grad_at(self.main_grad, b), self.plan.replica_stride, 0 if first else 1, stream)

    def backward(self, producer_stream=None, accumulate=False, order=None, one_by_one=False):
        """Mark every parameter ready in gradient-ready order; buckets go out on
        the side stream as they complete, in issue order."""
        ddp_reducer_prepare(self.handle, int(accumulate))
        order = self.ready_order if order is None else order
        if one_by_one:
            for p in order:
                ddp_reducer_mark_ready(self.handle, int(p), producer_stream)
        else:
            ddp_reducer_mark_ready_many(self.handle, order, producer_stream)

    def finalize(self, consumer_stream=None, timeout_us=0):
        ddp_reducer_finalize(self.handle, consumer_stream, timeout_us)

    def step(self, producer_stream=None, consumer_stream=None, accumulate=False):
        self.backward(producer_stream, accumulate)
        self.finalize(consumer_stream)

    # -- results ------------------------------------------------------------
    def view(self, p: int, w: int = 0):
        return self.plan.view(self.main_grad, p, w)

    def issue_log(self):
        return ddp_reducer_issue_log(self.handle)

    def logging_data(self) -> dict:
        """DDP's logging data ("DDP: ring AllReduce and gradient buckets" 17.13):
        the plan's bucket sizes and parameters, and once an iteration has been
        finalized the order its gradients arrived in and the rebuilt bucket sizes
        that order gives (rebuilt_bucket_sizes)."""
        d = self.plan.describe()
        try:
            seq = ddp_reducer_ready_order(self.handle)
        except DdpError:
            return d
        d["ready_order"] = [int(p) for p in seq]
        if len(seq) == self.plan.nparams:
            d["rebuilt_bucket_sizes"] = self.plan.rebuilt(seq)["bucket_sizes"]
        return d

    def bucket_ms(self):
        return ddp_reducer_bucket_ms(self.handle, self.plan.nbuckets)

    def close(self):
        if self.handle:
            ddp_reducer_destroy(self.handle)
            self.handle = None
        for h in getattr(self, "hooks", []):
            h.close()
        self.hooks = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostBucketReducer:
    """Host-buffer front end of BucketReducer over ddp_host_front_*: each step
    copies every replica's gradients from pinned host memory to the device, runs
    the synchronised backward's bucket reduction, and copies the reduced buckets
    back, as a pipeline over the buckets in issue order that also overlaps
    consecutive steps bucket by bucket (the library's two copy streams and the
    reducer's side stream; see ddp_host_front_step in the header).

    host_in   pinned [W, total] tensor (gradient dtype): replica w's gradients of
              all parameters back to back in parameter order.
    host_out  pinned [W * replica_stride] fp32 tensor in main_grad layout.  After an
              allreduce every bucket's elements are written (the alignment gaps
              between buckets are not); after a reduce_scatter replica w's copy
              receives only its own shard w of each bucket, the part a rank
              keeps (Megatron's start_grad_sync).
    """

    def __init__(self, numels, dtypes, W, mode, order, cap_bytes, first_cap_bytes, pad_multiple, torch_dtype,
                 used=None, fused=True, timing=False, coalesce=False):
        import torch

        numels = [int(v) for v in numels]
        self.W = int(W)
        self.offs = np.concatenate([[0], np.cumsum(numels)]).astype(np.int64)
        self.dev_in = torch.empty((W, int(self.offs[-1])), dtype=torch_dtype, device="cuda")
        grads = [[self.dev_in[w, self.offs[p]:self.offs[p + 1]] for p in range(len(numels))] for w in range(W)]
        self.reducer = BucketReducer(numels, dtypes, W, mode, order, cap_bytes, first_cap_bytes, pad_multiple, grads,
                                     used=used, fused=fused, timing=timing, coalesce=coalesce, bucket_done=True)
        es = self.dev_in.element_size()
        self.handle = ddp_host_front_create(self.reducer.handle, self.dev_in, self.dev_in.stride(0) * es, self.offs, es)
        plan = self.reducer.plan
        self.h2d_bytes = int(self.offs[-1]) * W * es
        if int(mode) == 1:
            self.d2h_bytes = sum(int(plan.bucket_numel[b]) for b in range(plan.nbuckets)) * 4
        else:
            self.d2h_bytes = sum(int(plan.bucket_numel[b]) for b in range(plan.nbuckets)) * W * 4

    @property
    def replica_stride(self) -> int:
        return self.reducer.plan.replica_stride

    def step(self, host_in, host_out, stream=None):
        import torch

        stream = torch.cuda.current_stream() if stream is None else stream
        if host_in.shape != self.dev_in.shape or host_in.dtype != self.dev_in.dtype or host_in.stride(1) != 1:
            raise ValueError(f"host_in must be a [W, total] {self.dev_in.dtype} tensor with contiguous rows")
        if host_out.dtype != torch.float32 or not host_out.is_contiguous() or \
                host_out.numel() < self.W * self.reducer.plan.replica_stride:
            raise ValueError("host_out must be a contiguous fp32 tensor of W * replica_stride elements")
        ddp_host_front_step(self.handle, host_in, host_in.stride(0) * host_in.element_size(), host_out, stream)

    def close(self):
        if self.handle is not None:
            ddp_host_front_destroy(self.handle)   # before the reducer it gates
            self.handle = None
        self.reducer.close()
