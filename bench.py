#!/usr/bin/env python
"""Benchmark of the gradient-bucket path: bucket-allreduce HBM GB/s.

One step = one synchronised backward's bucket reduction over the whole
workload: the reducer is prepared, every parameter is marked ready in
gradient-ready order (reverse parameter order) on the compute stream, each
bucket is issued in order on a side stream as soon as it and every bucket
before it are complete (fused pack + ring-ordered reduce + 1/W kernel), and
finalize makes the compute stream wait.  Inputs are resident in HBM when the
timed region starts.  GB/s counts the path's algorithmic bytes: every gradient
byte read once (plus main_grad when accumulating) and every result byte
written once.

Default workload: W = 8 replicas of ResNet-50's 161 gradient tensors (25.6M
fp32 parameters), reverse-order buckets capped at 25 MiB with a 1 MiB first
bucket (5 buckets), allreduce mean.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Under torchrun (N > 1) every rank runs the whole workload on its own GPU
(replicas only, no collective on the data path); the barrier and the maximum
over ranks of the elapsed time give the whole-job number.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

METRIC = "bucket-allreduce HBM GB/s (and % of 8 TB/s roofline) per bucket size and W"
NOMINAL_HBM_GBS = 8000.0
WORKLOADS = {
    "mlp3_w4_allreduce": WL.c1_mlp,
    "resnet50_w8_allreduce": WL.c2_resnet50,
    "gpt2_small_w8_reduce_scatter": WL.c3_gpt2,
    "bert_large_w4_nosync4_allreduce": WL.c4_bert_large,
    "bert_large_w4_find_unused_allreduce": WL.c6_bert_find_unused,
}
DEFAULT = "resnet50_w8_allreduce"
ELEM = {WL.F32: 4, WL.BF16: 2}


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------
def bucket_bytes(wl, numel: int, param_elems: int, used_elems: int, kind: str) -> int:
    """Bytes one launch must move for one bucket.  used_elems: gradient elements the
    replicas used, summed over the replicas.
    fused:  every used gradient read, main_grad read when accumulating, result written
            (allreduce: W replicas; reduce_scatter: one shard per replica = one bucket);
    pack0:  gradients read, bucket written (copy); packN: gradients + bucket read, bucket written
            (only used segments are touched when accumulating)."""
    W, b_in = wl.W, ELEM[wl.dtype]
    if kind == "fused":
        rd = used_elems * b_in
        wr = W * numel * 4 if wl.mode == WL.ALLREDUCE else numel * 4
        return rd + wr
    if kind == "fused_acc":
        rd = used_elems * b_in + W * numel * 4
        wr = W * numel * 4 if wl.mode == WL.ALLREDUCE else numel * 4
        return rd + wr
    if kind == "pack0":
        return used_elems * b_in + W * numel * 4
    if kind == "packN":
        return used_elems * (b_in + 8)
    raise ValueError(kind)


def step_launches(wl, plan):
    """[(kind, bucket, bytes)] of one step, in launch order."""
    used = WL.local_used_np(wl)
    out = []
    per_bucket = []
    for b in range(plan.nbuckets):
        mem = plan.members[b]
        pe = sum(wl.numels[p] for p in mem)
        ue = sum(wl.numels[p] * int(np.count_nonzero(used[:, p])) for p in mem)
        per_bucket.append((int(plan.bucket_numel[b]), pe, ue))
    for m in range(wl.micro_steps - 1):
        for b in range(plan.nbuckets):
            out.append(("pack0" if m == 0 else "packN", b, bucket_bytes(wl, *per_bucket[b], "pack0" if m == 0 else "packN")))
    kind = "fused_acc" if wl.micro_steps > 1 else "fused"
    for b in plan.bucket_order:
        out.append((kind, int(b), bucket_bytes(wl, *per_bucket[int(b)], kind)))
    return out


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
        self.gpu = vis[local_rank].strip() if len(vis) > local_rank and vis[local_rank].strip() else str(local_rank)
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def mark(self, which):
        setattr(self, which, time.time())

    def __exit__(self, *exc):
        if self.proc is None:
            return False
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.rows = []
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + float("0." + f[0].split(".")[1])
                self.rows.append((ts, float(f[2]), float(f[3]), f[5], f[6], f[7], f[8], f[9]))
            except (ValueError, IndexError):
                continue
        return False

    def summary(self):
        if self.proc is None or not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for r in self.rows if self.t0 is not None and self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        use = inside or sorted(self.rows, key=lambda r: abs(r[0] - (self.t0 or 0)))[:3]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in use for n, v in zip(names, r[4:]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in use])), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------
# the oracle: CPU baseline and reference arm
# ---------------------------------------------------------------------------
_SAMPLE_CACHE: dict = {}
ORACLE_SAMPLE_BYTES = 4 << 30   # a workload moving more than this per step is sampled by buckets


def _oracle_inputs(wl):
    """The oracle's plan of the workload and the raw gradients of the buckets one
    oracle step covers: every bucket, in issue order, while the step's
    algorithmic bytes stay within ORACLE_SAMPLE_BYTES (the whole workload for
    ResNet-50, GPT-2 and the MLP).  Generated once and kept."""
    import oracle

    orc = oracle.load()
    if wl.name not in _SAMPLE_CACHE:
        plan = orc.assign(wl.numels, [wl.dtype] * wl.nparams, wl.cap_bytes, wl.first_cap_bytes, wl.order,
                          wl.pad_multiple, wl.grad_reduce_in_fp32)
        used = WL.local_used_np(wl)
        chosen, total = [], 0
        for b in plan["bucket_order"]:
            b = int(b)
            mem = plan["members"][b]
            numel = int(plan["bucket_numel"][b])
            ue = sum(wl.numels[p] * int(np.count_nonzero(used[:, p])) for p in mem)
            pe = sum(wl.numels[p] for p in mem)
            nbytes = sum(bucket_bytes(wl, numel, pe, ue, "pack0" if m == 0 else "packN")
                         for m in range(wl.micro_steps - 1))
            nbytes += bucket_bytes(wl, numel, pe, ue, "fused_acc" if wl.micro_steps > 1 else "fused")
            if chosen and total + nbytes > ORACLE_SAMPLE_BYTES:
                break
            grads = [[[WL.grad_raw_np(wl, p, w, m) for p in mem] for w in range(wl.W)]
                     for m in range(wl.micro_steps)]
            chosen.append(dict(bucket=b, offs=[int(plan["offset_of"][p]) for p in mem], numel=numel,
                               used=used[:, mem], grads=grads, nparams=len(mem), bytes=nbytes))
            total += nbytes
        _SAMPLE_CACHE[wl.name] = (plan, chosen, total)
    return orc, _SAMPLE_CACHE[wl.name]


def _oracle_bucket(orc, wl, c):
    """One bucket through the oracle as it is: the no_sync packs, then pack and ring."""
    buf = None
    for m in range(wl.micro_steps):
        buf = orc.pack(c["grads"][m], c["offs"], c["numel"], [wl.dtype] * c["nparams"], c["used"],
                       accumulate=m > 0, out=buf)
    orc.ring(buf, wl.mode)


def oracle_step(wl, threads: int = 1) -> tuple:
    """One step of the oracle over the sampled buckets (single-threaded C, pack then
    ring, bucket after bucket; with threads > 1 the buckets run side by side in a
    thread pool, each in the oracle's own order -- ctypes releases the GIL in the
    C calls).  Returns (bytes, seconds)."""
    orc, (plan, chosen, total) = _oracle_inputs(wl)
    t = time.perf_counter()
    if threads <= 1:
        for c in chosen:
            _oracle_bucket(orc, wl, c)
    else:
        import concurrent.futures as cf

        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda c: _oracle_bucket(orc, wl, c), sorted(chosen, key=lambda c: -c["bytes"])))
    return total, time.perf_counter() - t


def oracle_sample_desc(wl) -> str:
    _, (plan, chosen, total) = _oracle_inputs(wl)
    whole = len(chosen) == plan["nbuckets"]
    what = (f"the whole workload: all {plan['nbuckets']} buckets" if whole else
            f"buckets {[c['bucket'] for c in chosen]} of {plan['nbuckets']} in issue order (bounded at "
            f"{ORACLE_SAMPLE_BYTES >> 30} GiB a step)")
    return (f"{what} ({sum(c['nparams'] for c in chosen)} tensors, {sum(c['numel'] for c in chosen)} elements x "
            f"W={wl.W}, {total} algorithmic bytes a step), "
            f"{'no_sync packs + ' if wl.micro_steps > 1 else ''}pack + ring per bucket, inputs pre-generated")


def oracle_sample(wl, seconds: float, min_reps: int = 1, threads: int = 1):
    """Time oracle steps for about `seconds` (at least min_reps).  Returns
    (GB/s, description, reps, seconds)."""
    reps, t_total, nbytes = 0, 0.0, 0
    while reps < min_reps or t_total < seconds:
        b, t = oracle_step(wl, threads)
        nbytes += b
        t_total += t
        reps += 1
    return nbytes / t_total / 1e9, oracle_sample_desc(wl), reps, t_total


def oracle_threads(wl) -> int:
    _, (plan, chosen, total) = _oracle_inputs(wl)
    return max(1, min(len(chosen), len(os.sched_getaffinity(0))))


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    t_gen = time.perf_counter()
    _oracle_inputs(wl)
    t_gen = time.perf_counter() - t_gen
    for _ in range(args.warmup):
        oracle_step(wl)
    t0 = time.perf_counter()
    nbytes, tt = 0, 0.0
    for _ in range(args.steps):
        b, t = oracle_step(wl)
        nbytes += b
        tt += t
    elapsed = time.perf_counter() - t0
    value = nbytes / tt / 1e9
    desc = oracle_sample_desc(wl)
    cpu = {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc,
           "cpu_model": _cpu_model(), "host_cores": len(os.sched_getaffinity(0))}
    if not args.no_threaded:
        th = oracle_threads(wl)
        tv, _, treps, _ = oracle_sample(wl, 0.0, min_reps=max(3, args.steps // 4), threads=th)
        cpu["threaded"] = {"value": round(tv, 4), "unit": "GB/s", "threads": th, "reps": treps,
                           "kind": "oracle, buckets side by side in a thread pool"}
    _, (plan, chosen, total) = _oracle_inputs(wl)
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * tt / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32" if wl.dtype == WL.F32 else "bf16->f32",
            "data": "synthetic (seeded splitmix64 gradients of the model's parameter shapes)",
            "impl": "reference",
            "config": {"workload": wl.name, "W": wl.W, "mode": "allreduce" if wl.mode == 0 else "reduce_scatter",
                       "buckets": plan["nbuckets"], "params": wl.nparams, "elements": sum(wl.numels),
                       "bytes_per_step": int(total), "sample": desc},
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "input_generation_s": round(t_gen, 2), "wall_s": round(elapsed, 2)}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
KERNEL_SOURCES = ("kernels.cu", "stream_impl.cuh", "stream_ring.cu", "stream_fused.cu", "stream_pack.cu",
                  "device_common.cuh", "common.h")


def kernel_source_hash() -> str:
    """sha256 over the device sources, to tell whether a committed ncu figure is current."""
    import hashlib

    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "allreduce_ddp_assign_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


def profile_traffic(kernel_tag: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary
    (profiles/traffic.json), or None if it was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path)).get(kernel_tag)
        if rec and rec.get("kernel_sources_sha256") == kernel_source_hash():
            return rec.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        return None
    return None


def rotation_copies(step_bytes: int, l2_bytes: int, micro_steps: int = 1) -> int:
    """Copies of a workload's inputs the timed steps rotate over so that each step
    reads from HBM: 1 when a step moves at least twice the L2, else enough copies
    that together they exceed twice the L2 (at most 64; no_sync workloads are large
    and keep one)."""
    if micro_steps != 1 or step_bytes >= 2 * l2_bytes or step_bytes <= 0:
        return 1
    return min(64, -(-2 * l2_bytes // step_bytes) + 1)


def run_ours(args, wl):
    import torch

    import allreduce_ddp_assign_gb300 as D
    from allreduce_ddp_assign_gb300.session import BucketReducer, HostBucketReducer

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    D.lib()
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    # inputs resident in HBM
    used = WL.local_used_np(wl) if (wl.unused or wl.partial_unused) else None
    micro = [[[None if p in wl.unused else WL.grad_torch(wl, p, w, m, dev) for p in range(wl.nparams)]
              for w in range(wl.W)] for m in range(wl.micro_steps)]
    coalesce = not args.no_coalesce
    sess = BucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                         wl.first_cap_bytes, wl.pad_multiple, micro[-1], used=used, fused=True,
                         timing=not coalesce, coalesce=coalesce)
    tabs = [sess.plan.pointer_table(micro[m]) for m in range(wl.micro_steps - 1)]
    compute = torch.cuda.current_stream()
    launches = step_launches(wl, sess.plan)
    step_bytes = sum(x[2] for x in launches)

    # A step that moves less than twice the L2 would find its inputs in L2 on the next
    # step: such workloads rotate over R copies of their gradients and main_grad (R
    # sessions sharing one side stream), R x the step's bytes above twice the L2, so
    # every step reads from HBM.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = rotation_copies(step_bytes, l2, wl.micro_steps)
    sessions = [sess]
    for _ in range(R - 1):
        copy = [[None if t is None else t.clone() for t in row] for row in micro[-1]]
        sessions.append(BucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                                      wl.first_cap_bytes, wl.pad_multiple, copy, used=used, fused=True,
                                      timing=not coalesce, coalesce=coalesce, side_stream=sess.side))
    l2_note = (f"inputs rotated over {R} copies ({R} x {step_bytes} B > 2 x L2 of {l2} B)" if R > 1
               else "inputs larger than L2 (no flush)")

    pack_ev = []

    def step(k, timed=False):
        s_ = sessions[k % R]
        if wl.micro_steps > 1:
            if timed:
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ev[0].record(compute)
            for m in range(wl.micro_steps - 1):   # no_sync micro-steps: local accumulation on the compute stream
                s_.accumulate_local(tabs[m], first=m == 0, stream=compute)
            if timed:
                ev[1].record(compute)
                pack_ev.append(ev)
        s_.backward(compute, accumulate=wl.micro_steps > 1)
        s_.finalize(compute)

    for k in range(max(args.warmup, 3) * R):
        step(k)
    torch.cuda.synchronize()

    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        clocks.mark("t0")
        ev0.record(compute)
        for k in range(K):
            step(k)
        ev1.record(compute)
        torch.cuda.synchronize()
        clocks.mark("t1")
        if dist:
            dist.barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    value = job_value(world, step_bytes, K, elapsed_ms)

    # the dominant kernel's time inside the step: the same K steps again with CUDA
    # events around each step's launches on the side stream (kept out of the run
    # above, whose per-step event records would add host time to small steps)
    side_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for k in range(K):
        side_ev[k][0].record(sess.side)
        step(k, timed=True)
        side_ev[k][1].record(sess.side)
    torch.cuda.synchronize()
    side_ms = sum(a.elapsed_time(b) for a, b in side_ev)

    # the same step with one launch per bucket (no coalescing): per-bucket figures.
    # Workloads rotated over copies are single-bucket steps: there the coalesced
    # figure is the per-bucket one and this part is skipped.
    pb_value, per_bucket_ms, Kp = None, None, max(3, min(K, 50))
    if R == 1:
        pb_sess = sess
        if coalesce:
            pb_sess = BucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                                    wl.first_cap_bytes, wl.pad_multiple, micro[-1], used=used, fused=True,
                                    timing=True, main_grad=True)

        def pb_step():
            for m in range(wl.micro_steps - 1):
                pb_sess.accumulate_local(tabs[m], first=m == 0, stream=compute)
            pb_sess.backward(compute, accumulate=wl.micro_steps > 1)
            pb_sess.finalize(compute)
        for _ in range(3):
            pb_step()
        torch.cuda.synchronize()
        pa, pb_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pa.record(compute)
        for _ in range(Kp):
            pb_step()
        pb_ev.record(compute)
        torch.cuda.synchronize()
        pb_value = job_value(1, step_bytes, Kp, pa.elapsed_time(pb_ev))
        # each bucket's launch time (events around it on the side stream): the median
        # over Kp more steps, read back after each step
        samples = []
        for _ in range(Kp):
            pb_step()
            samples.append([float(x) for x in pb_sess.bucket_ms()])
        per_bucket_ms = [float(np.median([smp[b] for smp in samples])) for b in range(len(samples[0]))]
        if pb_sess is not sess:
            pb_sess.close()

    # the dominant kernel: the fused pack+reduce launch(es) on the side stream (the
    # no_sync packs of an accumulating workload run on the compute stream)
    fused = [x for x in launches if x[0].startswith("fused")]
    fused_bytes = sum(x[2] for x in fused)
    packs = [x for x in launches if x[0].startswith("pack")]
    pack_bytes = sum(x[2] for x in packs)
    if packs:
        # the side stream's span also holds the wait for the packs: split the step
        pack_ms = sum(a.elapsed_time(b) for a, b in pack_ev) / K
        fused_ms = max(side_ms / K - pack_ms, 1e-6)
    else:
        pack_ms, fused_ms = 0.0, side_ms / K
    if pack_ms > fused_ms:   # no_sync workloads: the local accumulation dominates
        dominant, dom_bytes, kern_ms = "pack", pack_bytes, pack_ms
        timing_src = "CUDA events on the compute stream around each timed step's no_sync pack launches"
    else:
        dominant, dom_bytes, kern_ms = "fused", fused_bytes, fused_ms
        timing_src = ("CUDA events on the side stream around each timed step's fused launches"
                      + (" (minus the packs it waits for)" if packs else ""))
    achieved = dom_bytes / (kern_ms * 1e-3) / 1e9
    tag = f"{dominant}_{wl.name}"
    if not coalesce and sess.plan.nbuckets > 1:
        tag += "_per_bucket"   # other launches than the recorded coalesced one: no traffic record
    traffic = profile_traffic(tag)

    # context: the same fused launches back to back on the side stream, without
    # the reducer's cross-stream hand-offs (kernel time alone)
    kernel_only = None
    if wl.micro_steps == 1:
        import allreduce_ddp_assign_gb300 as D2

        plan = sess.plan
        order = [int(b) for b in plan.bucket_order]
        descs = [plan.descs[b] for b in order]
        starts = [int(plan.bucket_start[b]) for b in order]
        ka, kb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def launch(r, stream):
            s_ = sessions[r % R]
            D2.ddp_fused_bucket_group(descs, starts, s_.grads_tab, s_.used_tab, wl.nparams, wl.W, wl.mode, 0,
                                      s_.main_grad, plan.replica_stride, None, None, stream)
        if R > 1:
            # small launches: replayed from a CUDA graph of one launch per input copy, so
            # the figure is the GPU's time per launch (from HBM), not the host's rate of
            # issuing them
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=sess.side):
                for r in range(R):
                    launch(r, torch.cuda.current_stream())
            reps = max(3, -(-Kp // R))
            g.replay()
            torch.cuda.synchronize()
            ka.record(sess.side)
            with torch.cuda.stream(sess.side):
                for _ in range(reps):
                    g.replay()
            kb.record(sess.side)
            torch.cuda.synchronize()
            kms = ka.elapsed_time(kb) / (reps * R)
            del g
        else:
            with torch.cuda.stream(sess.side):
                for r in range(Kp + 3):
                    if r == 3:
                        ka.record(sess.side)
                    launch(r, sess.side)
                kb.record(sess.side)
            torch.cuda.synchronize()
            kms = ka.elapsed_time(kb) / Kp
        kernel_only = {"value": round(fused_bytes / (kms * 1e-3) / 1e9, 1), "unit": "GB/s", "us_per_step": round(kms * 1e3, 1),
                       "frac_of_measured_peak": round(fused_bytes / (kms * 1e-3) / 1e9 / peak, 4),
                       "timing": (f"CUDA graph of {R} launches (one per input copy) replayed, GPU time per launch"
                                  if R > 1 else "launches back to back on the side stream")}

    # end to end: pinned host buffers in, reduced main_grad out, through the public API
    e2e = None
    if not args.no_e2e and wl.micro_steps == 1:
        tdt = torch.float32 if wl.dtype == WL.F32 else torch.bfloat16
        host = HostBucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                                 wl.first_cap_bytes, wl.pad_multiple, tdt, used=used, coalesce=coalesce)
        total = sum(wl.numels)
        h_in = torch.empty((wl.W, total), dtype=tdt, pin_memory=True)
        for w in range(wl.W):
            h_in[w] = torch.cat([micro[-1][w][p].reshape(-1) if micro[-1][w][p] is not None else
                                 torch.zeros(wl.numels[p], dtype=tdt, device=dev)
                                 for p in range(wl.nparams)]).cpu()
        h_out = torch.empty((wl.W * host.replica_stride,), dtype=torch.float32, pin_memory=True)
        for _ in range(max(args.warmup, 3)):
            host.step(h_in, h_out)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        Ke = max(3, min(K, 50))
        a.record()
        for _ in range(Ke):
            host.step(h_in, h_out)
        b.record()
        torch.cuda.synchronize()
        e_ms = max_over_ranks(a.elapsed_time(b), dist, dev)
        e2e = {"value": round(job_value(world, step_bytes, Ke, e_ms), 3), "unit": "GB/s",
               "h2d_bytes_per_step": int(h_in.numel() * h_in.element_size()),
               "d2h_bytes_per_step": int(host.d2h_bytes), "steps": Ke}
        host.close()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, desc, reps, t = oracle_sample(wl, args.cpu_seconds)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc, "reps": reps,
               "seconds": round(t, 2), "cpu_model": _cpu_model(), "host_cores": len(os.sched_getaffinity(0))}

    clk = clocks.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": max(args.warmup, 3), "ms_per_step": round(elapsed_ms / K, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32" if wl.dtype == WL.F32 else "bf16->f32",
            "data": "synthetic (seeded splitmix64 gradients of the model's parameter shapes)",
            "config": {"workload": wl.name, "W": wl.W, "mode": "allreduce" if wl.mode == 0 else "reduce_scatter",
                       "buckets": sess.plan.nbuckets, "params": wl.nparams, "elements": sum(wl.numels),
                       "bytes_per_step": step_bytes, "l2": l2_note,
                       "parallelism": f"replicas x{world}", "pct_of_nominal_8TBs": round(100 * value / NOMINAL_HBM_GBS, 2),
                       "buckets_per_s": round(world * K * sess.plan.nbuckets / (elapsed_ms * 1e-3), 1),
                       "issue": "coalesced (ready buckets in one launch)" if coalesce else "one launch per bucket",
                       "per_bucket_issue": None if pb_value is None else {
                           "value": round(pb_value, 1), "unit": "GB/s", "steps": Kp,
                           "per_bucket_timing": f"events around each launch, median of {Kp} steps",
                           "per_bucket_gbs": [round(x[2] / (per_bucket_ms[x[1]] * 1e-3) / 1e9, 1)
                                              if per_bucket_ms[x[1]] > 0 else None for x in fused],
                           "bucket_bytes": [int(x[2]) for x in fused]}},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_src,
                         "kernel": tag, "timing": timing_src, "kernel_only": kernel_only,
                         "step_split_ms": {"pack": round(pack_ms, 4), "fused": round(fused_ms, 4)} if packs else None},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": ((((wl.micro_steps - 1) * -(-sess.plan.nbuckets // 32) + -(-len(fused) // 32)) if coalesce
                              else len(launches)) + (1 if used is not None else 0)) * K,   # + the used-bitmap kernel
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    for s_ in sessions:
        s_.close()
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def max_over_ranks(x: float, dist, device) -> float:
    """Maximum of x over the ranks of the default process group (x itself alone)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, bytes_per_step: int, steps: int, max_elapsed_ms: float) -> float:
    """Whole-job GB/s: every rank moved bytes_per_step per step; the slowest rank sets the time."""
    return world * bytes_per_step * steps / (max_elapsed_ms * 1e-3) / 1e9


def _cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.processor() or platform.machine()


def run_sweep(args):
    """Bandwidth sweep (one fp32 bucket, S = 1 KiB * 4^k up to 1 GiB, W in {2, 4, 8, 16},
    allreduce mean): ddp_bucket_allreduce timed alone with CUDA events, L2 flushed
    before every rep by writing a buffer twice the L2 size; median of the reps.
    Prints one JSON line per point."""
    import torch

    import allreduce_ddp_assign_gb300 as D

    dev = torch.device("cuda", 0)
    D.lib()
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(peaks.get("hbm_gbs", 6800.0))
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    points = WL.c5_sweep_points()
    if args.sweep_max_bytes:
        points = [(b, w) for b, w in points if b <= args.sweep_max_bytes]
    for nbytes, W in points:
        n = nbytes // 4
        x = WL.bucket_torch(nbytes, W, dev)
        moved = 2 * W * nbytes
        if moved < (256 << 20):
            # launch-latency regime: replay 20 launches from a CUDA graph and take
            # the GPU time per launch (the data then sit in L2: labelled so)
            s = torch.cuda.Stream()
            D.ddp_bucket_allreduce(x, n, n, W, D.DDP_ALLREDUCE, s)   # first call outside capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(20):
                    D.ddp_bucket_allreduce(x, n, n, W, D.DDP_ALLREDUCE, torch.cuda.current_stream())
            g.replay()
            torch.cuda.synchronize()
            times = []
            for r in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                b.synchronize()
                times.append(a.elapsed_time(b) / 20)
            reps, timing = 100, "graph replay, 20 launches x 5, L2-resident"
            del g
        else:
            reps = 5 if nbytes >= (256 << 20) else 20
            times = []
            for r in range(reps + 3):
                flush.fill_(float(r))
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                D.ddp_bucket_allreduce(x, n, n, W, D.DDP_ALLREDUCE)
                b.record()
                b.synchronize()
                if r >= 3:
                    times.append(a.elapsed_time(b))
            timing = "one launch per rep, L2 flushed before each"
        ms = float(np.median(times))
        gbs = moved / (ms * 1e-3) / 1e9
        print(json.dumps({"sweep": True, "bucket_bytes": nbytes, "W": W, "us": round(ms * 1e3, 2),
                          "GBps": round(gbs, 1), "frac_measured": round(gbs / peak, 4),
                          "pct_of_8TBs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
                          "buckets_per_s": round(1e3 / ms, 1), "bytes_moved": moved,
                          "l2_resident": moved < l2, "reps": reps, "timing": timing}), flush=True)
        del x
        torch.cuda.empty_cache()


def run_bitmap(args):
    """find_unused_parameters' bitmap all-reduce ("Lecture 15: PyTorch DDP" 4.2).
    (1) ddp_used_allreduce alone on 16M parameters x 8 replicas (HBM-bound: W*P bytes
    read, 5*P written), L2 flushed before each rep; (2) at BERT-large's 391 parameters,
    W = 4, back-to-back launches (launch-bound); (3) the reducer's step on BERT-large
    with the bitmap path (upload, all-reduce, host marking) against the same step
    without it, all parameters used -- the cost the lecture says find_unused adds to
    every iteration.  One JSON line."""
    import torch

    import allreduce_ddp_assign_gb300 as D
    from allreduce_ddp_assign_gb300.session import BucketReducer

    dev = torch.device("cuda", 0)
    D.lib()
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(peaks.get("hbm_gbs", 6800.0))
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    W, P = 8, 1 << 24
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    local = (torch.rand((W, P), generator=g, device=dev) < 0.02).to(torch.uint8)
    cnt = torch.empty(P, dtype=torch.int32, device=dev)
    flg = torch.empty(P, dtype=torch.uint8, device=dev)
    times = []
    for r in range(13):
        flush.fill_(float(r))
        a, b = ev(), ev()
        a.record()
        D.ddp_used_allreduce(local, P, W, P, cnt, flg)
        b.record()
        b.synchronize()
        if r >= 3:
            times.append(a.elapsed_time(b))
    ms_single = float(np.median(times))
    # back to back over four input sets (each 134 MB map is read again only after the
    # other three, 0.5 GB of traffic later: larger than L2), so the per-launch figure
    # carries no idle gap between the flush and the launch
    sets = [local] + [(torch.rand((W, P), generator=g, device=dev) < 0.02).to(torch.uint8) for _ in range(3)]
    outs = [(torch.empty(P, dtype=torch.int32, device=dev), torch.empty(P, dtype=torch.uint8, device=dev))
            for _ in range(4)]
    for k in range(8):
        D.ddp_used_allreduce(sets[k % 4], P, W, P, outs[k % 4][0], outs[k % 4][1])
    reps = []
    for r in range(5):
        a, b = ev(), ev()
        a.record()
        for k in range(40):
            D.ddp_used_allreduce(sets[k % 4], P, W, P, outs[k % 4][0], outs[k % 4][1])
        b.record()
        b.synchronize()
        reps.append(a.elapsed_time(b) / 40)
    ms = float(np.median(reps))
    moved = W * P + 5 * P
    large = {"W": W, "params": P, "bytes": moved, "us": round(ms * 1e3, 2),
             "GBps": round(moved / (ms * 1e-3) / 1e9, 1),
             "frac_measured": round(moved / (ms * 1e-3) / 1e9 / peak, 4),
             "timing": "40 launches back to back over 4 input sets (0.5 GB apart, larger than L2), median of 5",
             "single_launch_us": round(ms_single * 1e3, 2),
             "single_launch_timing": "one launch between CUDA events after an L2 flush, median of 10"}
    del local, cnt, flg, sets, outs

    wl = WL.c6_bert_find_unused()
    Wm, Pm = wl.W, wl.nparams
    lu = torch.ones(Wm * Pm, dtype=torch.uint8, device=dev)
    c2 = torch.empty(Pm, dtype=torch.int32, device=dev)
    f2 = torch.empty(Pm, dtype=torch.uint8, device=dev)
    for _ in range(10):
        D.ddp_used_allreduce(lu, Pm, Wm, Pm, c2, f2)
    torch.cuda.synchronize()
    a, b = ev(), ev()
    a.record()
    for _ in range(1000):
        D.ddp_used_allreduce(lu, Pm, Wm, Pm, c2, f2)
    b.record()
    b.synchronize()
    model = {"W": Wm, "params": Pm, "us_per_call": round(a.elapsed_time(b), 3),
             "timing": "1000 back-to-back launches, GPU time per launch (includes launch gaps)"}

    grads = [[WL.grad_torch(wl, p, w, 0, dev) for p in range(Pm)] for w in range(Wm)]

    def step_ms(used):
        sess = BucketReducer(wl.numels, None, Wm, wl.mode, wl.order, wl.cap_bytes, wl.first_cap_bytes,
                             wl.pad_multiple, grads, used=used, coalesce=True)
        comp = torch.cuda.current_stream()
        for _ in range(5):
            sess.step(comp, comp)
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record(comp)
        for _ in range(args.steps):
            if used is not None:
                sess.set_local_used(used)
            sess.step(comp, comp)
        b.record(comp)
        b.synchronize()
        sess.close()
        return a.elapsed_time(b) / args.steps

    t_plain = step_ms(None)
    t_fu_all = step_ms(np.ones((Wm, Pm), np.uint8))
    t_fu = step_ms(WL.local_used_np(wl))
    line = {"bitmap": True, "kernel_large": large, "kernel_model_size": model,
            "reducer_step_ms": {"workload": wl.name, "without_bitmap": round(t_plain, 4),
                                "find_unused_all_used": round(t_fu_all, 4),
                                "find_unused_workload_bitmap": round(t_fu, 4),
                                "overhead_ms": round(t_fu_all - t_plain, 4), "steps": args.steps}}
    print(json.dumps(line), flush=True)
    return line


def powersgd_bytes(wl, plan, b, rank, ef=True):
    """Algorithmic HBM bytes of one compressed hook call on bucket b, and the elements
    a rank would all-reduce (P and Q of every matrix, the 1-D tensors whole).
    Per matrix element and replica: P pass reads G (and E, writing M back to E),
    the Q pass reads M, the output pass writes the result (and reads M, writes E):
    12 + 4 + 12 bytes with error feedback, 4 + 4 + 4 without.  1-D tensors: W
    reads and W writes of 4 bytes."""
    W = wl.W
    nbytes, comm, elems = 0, 0, 0
    for p in plan.members[b]:
        shape, n = wl.shapes[p], wl.numels[p]
        elems += n
        if len(shape) >= 2:
            m, k = shape[0], n // shape[0]
            nbytes += W * n * (28 if ef else 12)
            comm += (m + k) * min(rank, m, k)
        else:
            nbytes += 2 * W * n * 4
            comm += n
    return nbytes, comm, elems


def run_powersgd(args):
    """The PowerSGD hook (DDP chapter 17.27) on ResNet-50's buckets, W = 8, error
    feedback, rank --psgd-rank: (1) ddp_powersgd_reduce alone per bucket against
    ddp_bucket_allreduce on the same packed bucket; (2) the reducer's step with every
    bucket hooked against the plain fused step.  CUDA events on the launching
    stream, inputs resident and larger than L2.  One JSON line."""
    import torch

    import allreduce_ddp_assign_gb300 as D
    from allreduce_ddp_assign_gb300.session import BucketReducer

    dev = torch.device("cuda", 0)
    D.lib()
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(peaks.get("hbm_gbs", 6800.0))
    rank = args.psgd_rank
    wl = WL.c7_resnet50_powersgd(rank)
    grads = [[WL.grad_torch(wl, p, w, 0, dev) for p in range(wl.nparams)] for w in range(wl.W)]
    cfg = dict(rank=rank, shapes=wl.shapes, q0=lambda p, n, r: WL.powersgd_q0_np(wl.seed, p, n, r))
    sess = BucketReducer(wl.numels, None, wl.W, wl.mode, wl.order, wl.cap_bytes, wl.first_cap_bytes,
                         wl.pad_multiple, grads, powersgd=cfg)
    plain = BucketReducer(wl.numels, None, wl.W, wl.mode, wl.order, wl.cap_bytes, wl.first_cap_bytes,
                          wl.pad_multiple, grads, coalesce=True)
    plan = sess.plan
    comp = torch.cuda.current_stream()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record(comp)
        for _ in range(reps):
            fn()
        b.record(comp)
        b.synchronize()
        return a.elapsed_time(b) / reps

    sess.step(comp, comp)   # packs the buckets once
    torch.cuda.synchronize()
    per_bucket = []
    tot_bytes = tot_comm = tot_elems = 0
    t_hook = t_ring = 0.0
    for b in range(plan.nbuckets):
        mg = plan.main_grad_at(sess.main_grad, b)
        nb, cm, el = powersgd_bytes(wl, plan, b, rank)
        th = timed(lambda: sess.hooks[b].reduce(mg, plan.replica_stride, comp), args.steps)
        tr = timed(lambda: D.ddp_bucket_allreduce(mg, plan.replica_stride, int(plan.bucket_numel[b]), wl.W,
                                                  D.DDP_ALLREDUCE, comp), args.steps)
        per_bucket.append({"bucket": b, "elements": el, "hook_us": round(th * 1e3, 2), "ring_us": round(tr * 1e3, 2),
                           "hook_GBps": round(nb / (th * 1e-3) / 1e9, 1), "compression": round(el / cm, 1)})
        tot_bytes += nb
        tot_comm += cm
        tot_elems += el
        t_hook += th
        t_ring += tr
    step_hook = timed(lambda: sess.step(comp, comp), max(args.steps // 4, 10))
    step_plain = timed(lambda: plain.step(comp, comp), max(args.steps // 4, 10))
    achieved = tot_bytes / (t_hook * 1e-3) / 1e9
    line = {"powersgd": True, "workload": wl.name, "rank": rank, "W": wl.W, "error_feedback": True,
            "hook_ms_per_step": round(t_hook, 4), "ring_allreduce_ms_per_step": round(t_ring, 4),
            "reducer_step_ms": {"powersgd": round(step_hook, 4), "plain_fused_coalesced": round(step_plain, 4)},
            "compression_ratio": round(tot_elems / tot_comm, 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "bytes_per_step": tot_bytes,
                         "kernel": "the hook's four launches per bucket (P, orthonormalisation, Q, output), summed"},
            "per_bucket": per_bucket, "steps": args.steps}
    print(json.dumps(line), flush=True)
    sess.close()
    plain.close()
    return line


def run_overlap(args, wl=None):
    """The reducer's overlap with a synthetic backward ("Lecture 15: PyTorch DDP" 3.1):
    the compute stream runs one bounded spin kernel per parameter, in reverse order,
    with a length proportional to the parameter, and marks it ready; buckets go out on
    the side stream as they fill.  Measured: backward alone, reduction alone, the
    overlapped step, the serial step.  Predicted: ddp_overlap_timeline from the
    recorded ready times and per-bucket times.  One JSON line."""
    import torch

    import allreduce_ddp_assign_gb300 as D
    from allreduce_ddp_assign_gb300.session import BucketReducer

    wl = wl or WL.c2_resnet50()
    dev = torch.device("cuda", 0)
    D.lib()
    grads = [[WL.grad_torch(wl, p, w, 0, dev) for p in range(wl.nparams)] for w in range(wl.W)]
    sess = BucketReducer(wl.numels, None, wl.W, wl.mode, wl.order, wl.cap_bytes, wl.first_cap_bytes,
                         wl.pad_multiple, grads, timing=True)
    comp = torch.cuda.current_stream()
    # calibrate the spin kernel: cycles per millisecond at the clock it actually runs at
    probe = 2_000_000
    for _ in range(3):
        torch.cuda._sleep(probe)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(torch.cuda.current_stream())
    torch.cuda._sleep(probe)
    e1.record(torch.cuda.current_stream())
    torch.cuda.synchronize()
    clock_hz = probe / (e0.elapsed_time(e1) * 1e-3)
    total = sum(wl.numels)
    bwd_ms = args.backward_ms
    cycles = [max(1000, int(bwd_ms * 1e-3 * clock_hz * n / total)) for n in wl.numels]
    order = list(range(wl.nparams - 1, -1, -1))

    def backward(mark: bool, evs=None):
        for i, p in enumerate(order):
            torch.cuda._sleep(cycles[p])
            if evs is not None:
                evs[i].record(comp)
            if mark:
                D.ddp_reducer_mark_ready(sess.handle, p, comp)

    def timed(fn, reps=5):
        out = []
        for r in range(reps + 2):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(comp)
            fn()
            b.record(comp)
            torch.cuda.synchronize()
            if r >= 2:
                out.append(a.elapsed_time(b))
        return float(np.median(out))

    t_bwd = timed(lambda: backward(False))

    def reduce_only():
        D.ddp_reducer_prepare(sess.handle, 0)
        D.ddp_reducer_mark_ready_many(sess.handle, order, comp)
        D.ddp_reducer_finalize(sess.handle, comp, 0)

    t_red = timed(reduce_only)
    per_bucket_ms = [float(x) for x in sess.bucket_ms()]

    def overlapped():
        D.ddp_reducer_prepare(sess.handle, 0)
        backward(True)
        D.ddp_reducer_finalize(sess.handle, comp, 0)

    t_ovl = timed(overlapped)

    def serial():
        backward(False)
        reduce_only()

    t_ser = timed(serial)
    # ready times of one overlapped step, for the model
    evs = [torch.cuda.Event(enable_timing=True) for _ in order]
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    a.record(comp)
    D.ddp_reducer_prepare(sess.handle, 0)
    backward(True, evs)
    D.ddp_reducer_finalize(sess.handle, comp, 0)
    torch.cuda.synchronize()
    ready = np.zeros(wl.nparams)
    for i, p in enumerate(order):
        ready[p] = a.elapsed_time(evs[i])
    plan = sess.plan
    nbytes = np.array([2 * wl.W * 4 * int(plan.bucket_numel[b]) for b in range(plan.nbuckets)], np.float64)
    slope, icpt = np.polyfit(nbytes, np.array(per_bucket_ms), 1)
    model = D.ddp_overlap_timeline(ready, plan.bucket_of, plan.bucket_order, nbytes.astype(np.int64),
                                   max(float(icpt), 0.0), max(float(slope), 0.0))
    line = {"overlap": True, "workload": wl.name, "backward_ms": round(t_bwd, 4), "reduce_ms": round(t_red, 4),
            "overlapped_step_ms": round(t_ovl, 4), "serial_step_ms": round(t_ser, 4),
            "exposed_ms": round(t_ovl - t_bwd, 4), "hidden_fraction": round(1 - (t_ovl - t_bwd) / t_red, 4),
            "model": {"alpha_ms": round(max(float(icpt), 0.0), 5), "ms_per_GB": round(max(float(slope), 0.0) * 1e9, 5),
                      "step_ms": round(model["step_ms"], 4), "serial_ms": round(model["serial_ms"], 4)},
            "per_bucket_ms": [round(x, 4) for x in per_bucket_ms],
            "bucket_ready_ms": [round(float(max(ready[p] for p in plan.members[b])), 4) for b in range(plan.nbuckets)]}
    print(json.dumps(line), flush=True)
    sess.close()
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-coalesce", action="store_true", help="one launch per bucket in the timed steps")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-threaded", action="store_true", help="reference arm: skip the threaded oracle run")
    ap.add_argument("--sweep", action="store_true", help="bandwidth sweep of ddp_bucket_allreduce (JSON per point)")
    ap.add_argument("--sweep-max-bytes", type=int, default=0)
    ap.add_argument("--overlap", action="store_true", help="overlap with a synthetic backward (JSON line)")
    ap.add_argument("--bitmap", action="store_true", help="find_unused bitmap all-reduce (JSON line)")
    ap.add_argument("--powersgd", action="store_true", help="PowerSGD hook on ResNet-50 (JSON line)")
    ap.add_argument("--psgd-rank", type=int, default=4)
    ap.add_argument("--backward-ms", type=float, default=3.0)
    args = ap.parse_args(argv)
    if args.sweep:
        return run_sweep(args)
    if args.overlap:
        return run_overlap(args)
    if args.bitmap:
        return run_bitmap(args)
    if args.powersgd:
        return run_powersgd(args)
    wl = WORKLOADS[args.workload]()
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
