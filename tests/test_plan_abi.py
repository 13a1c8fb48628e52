"""The plan object of the C ABI (ddp_plan_*) against the oracle's assignment (CPU only).

ddp_plan_describe must report the oracle's buckets bit for bit (bytes, padded
elements, dtype, members in layout order, issue order, per-parameter bucket and
offset: "DDP: ring AllReduce and gradient buckets" 17.13, bucket_sizes), the
layout must place every bucket on the stated alignment without overlap, the
segment tables must describe exactly each bucket's parameters, and
ddp_plan_rebuilt must equal the oracle's assignment over the same ready order
(rebuilt_bucket_sizes).
"""
import ctypes as C

import numpy as np
import pytest

import allreduce_ddp_assign_gb300 as D
import workloads as WL


def check_plan(orc, numels, dtypes, cap, first, order, pad, fp32, align):
    h = D.ddp_plan_create(numels, dtypes, cap, first, order, pad, fp32, align)
    try:
        d = D.ddp_plan_describe(h)
        r = orc.assign(numels, dtypes, cap, first, order, pad, fp32)
        P, B = len(numels), r["nbuckets"]
        assert (d["nparams"], d["nbuckets"]) == (P, B)
        assert (d["cap_bytes"], d["first_cap_bytes"], d["order"], d["pad_multiple"]) == (cap, first, order, pad)
        for k in ("bucket_of", "offset_of", "bucket_numel", "bucket_bytes", "bucket_dtype", "bucket_order"):
            assert np.array_equal(d[k], r[k]), k
        ms = d["member_start"]
        assert ms[0] == 0 and ms[-1] == P
        assert [[int(p) for p in d["members"][ms[b]:ms[b + 1]]] for b in range(B)] == [list(m) for m in r["members"]]
        # layout: aligned starts, buckets in index order without overlap, the stride holds them all
        st = d["bucket_start"]
        for b in range(B):
            assert st[b] % align == 0
            if b:
                assert st[b] >= st[b - 1] + d["bucket_numel"][b - 1]
                assert st[b] - (st[b - 1] + d["bucket_numel"][b - 1]) < align
        assert d["replica_stride"] >= (st[-1] + d["bucket_numel"][-1] if B else 0)
        assert d["replica_stride"] % align == 0 and d["replica_stride"] >= align
        # segment tables: per bucket its members' offsets, then the end of its gradients
        assert (d["seg_offset_len"], d["seg_param_len"]) == (P + B, P)
        so, sp = D.ddp_plan_tables(h, d["seg_offset_len"], d["seg_param_len"])
        descs = D.ddp_plan_bucket_descs(h, B, 0x10000, 0x20000)
        for b in range(B):
            mem = r["members"][b]
            o = (descs[b].seg_offset - 0x10000) // 8
            q = (descs[b].seg_param - 0x20000) // 4
            assert (descs[b].numel, descs[b].nseg, descs[b].dtype) == (r["bucket_numel"][b], len(mem),
                                                                      r["bucket_dtype"][b])
            assert list(sp[q:q + len(mem)]) == list(mem)
            assert list(so[o:o + len(mem)]) == [int(r["offset_of"][p]) for p in mem]
            end = int(r["offset_of"][mem[-1]]) + int(numels[mem[-1]]) if mem else 0
            assert so[o + len(mem)] == end <= r["bucket_numel"][b]
        return d
    finally:
        D.ddp_plan_destroy(h)


@pytest.mark.parametrize("name", sorted(WL.ALL))
def test_plan_matches_oracle_on_configs(orc, name):
    wl = WL.ALL[name]()
    check_plan(orc, wl.numels, [wl.dtype] * wl.nparams, wl.cap_bytes, wl.first_cap_bytes, wl.order,
               wl.pad_multiple, 1, 64)


def test_plan_random_lists(orc):
    rng = np.random.default_rng(12)
    for trial in range(300):
        P = int(rng.integers(0, 25))
        n = rng.integers(0, 3000, size=P)
        dt = rng.integers(0, 3, size=P) if trial % 2 else np.zeros(P, np.int64)
        args = (n, dt, int(rng.integers(1, 15000)), int(rng.integers(1, 15000)), int(rng.integers(0, 3)),
                int(rng.integers(1, 9)), int(rng.integers(0, 2)), int(rng.choice([1, 4, 64, 100])))
        check_plan(orc, *args)


def test_plan_rebuilt_matches_oracle(orc):
    """The twelve-Linear model's rebuilt byte list from its reverse ready order
    (DDP chapter 17.13), and random orders against the oracle."""
    wl = WL.c2_resnet50()
    rng = np.random.default_rng(5)
    for trial in range(40):
        seq = np.arange(wl.nparams - 1, -1, -1) if trial == 0 else rng.permutation(wl.nparams)
        h = D.ddp_plan_create(wl.numels, None, wl.cap_bytes, wl.first_cap_bytes, wl.order)
        try:
            got = D.ddp_plan_rebuilt(h, seq, wl.nparams)
        finally:
            D.ddp_plan_destroy(h)
        want = orc.assign_sequence(wl.numels, seq, None, wl.cap_bytes, wl.first_cap_bytes)
        assert got["nbuckets"] == want["nbuckets"]
        assert np.array_equal(got["bucket_bytes"], want["bucket_bytes"])
        assert np.array_equal(got["bucket_numel"], want["bucket_numel"])


def test_plan_errors():
    with pytest.raises(D.DdpError) as e:
        D.ddp_plan_create([10, 20], None, 0, 1 << 20)
    assert e.value.status == D.DDP_E_INVAL
    with pytest.raises(D.DdpError):
        D.ddp_plan_create([10], None, 1 << 20, 1 << 20, 0, 1, 1, 0)   # align_elems 0
    h = D.ddp_plan_create([10, 20, 30], None, 40, 40)
    try:
        with pytest.raises(D.DdpError):
            D.ddp_plan_rebuilt(h, [0, 0, 1], 3)    # not a permutation
        with pytest.raises(D.DdpError) as e:
            cap = 0
            nb = C.c_int32(0)
            seq = np.array([2, 1, 0], np.int32)
            D._check(D.lib().ddp_plan_rebuilt(h, seq.ctypes.data_as(D._i32p), None, None, cap, C.byref(nb)))
        assert e.value.status == D.DDP_E_CAPACITY
    finally:
        D.ddp_plan_destroy(h)


def test_reducer_from_plan_dry_run():
    """A reducer made from a plan issues the plan's buckets in its issue order."""
    wl = WL.c3_gpt2()
    h = D.ddp_plan_create(wl.numels, None, wl.cap_bytes, wl.first_cap_bytes, wl.order, wl.pad_multiple)
    d = D.ddp_plan_describe(h)
    descs = D.ddp_plan_bucket_descs(h, d["nbuckets"], 0x10000, 0x20000)
    r = D.ddp_reducer_create_from_plan(h, descs, wl.W, wl.mode, D.DDP_R_DRY_RUN | D.DDP_R_FUSED)
    D.ddp_plan_destroy(h)   # the reducer keeps its own copy
    try:
        D.ddp_reducer_prepare(r, 0)
        D.ddp_reducer_mark_ready_many(r, np.arange(wl.nparams - 1, -1, -1, dtype=np.int32), None)
        D.ddp_reducer_finalize(r, None, 0)
        assert D.ddp_reducer_issue_log(r) == [int(b) for b in d["bucket_order"]]
    finally:
        D.ddp_reducer_destroy(r)


def test_host_front_rejects_bad_arguments():
    """ddp_host_front_create checks its arguments before touching CUDA: a dry-run
    reducer, NULL arguments."""
    wl = WL.c1_mlp()
    h = D.ddp_plan_create(wl.numels, None, wl.cap_bytes, wl.first_cap_bytes, wl.order, wl.pad_multiple)
    d = D.ddp_plan_describe(h)
    descs = D.ddp_plan_bucket_descs(h, d["nbuckets"], 0x10000, 0x20000)
    r = D.ddp_reducer_create_from_plan(h, descs, wl.W, wl.mode, D.DDP_R_DRY_RUN | D.DDP_R_FUSED | D.DDP_R_BUCKET_DONE)
    D.ddp_plan_destroy(h)
    offs = np.concatenate([[0], np.cumsum(wl.numels)]).astype(np.int64)
    try:
        with pytest.raises(D.DdpError) as e:
            D.ddp_host_front_create(r, 0x1000, int(offs[-1]) * 4, offs, 4)   # dry run
        assert e.value.status == D.DDP_E_INVAL
        out = D._vp()
        st = D.lib().ddp_host_front_create(r, D._vp(0x1000), int(offs[-1]) * 4, None, 4, C.byref(out))
        assert st == D.DDP_E_INVAL and not out.value
        st = D.lib().ddp_host_front_create(None, D._vp(0x1000), 4, D._cp(offs, D._i64p), 4, C.byref(out))
        assert st == D.DDP_E_INVAL
        assert D.lib().ddp_host_front_create(r, None, 0, D._cp(offs, D._i64p), 4, None) == D.DDP_E_INVAL
    finally:
        D.ddp_reducer_destroy(r)
    D.ddp_host_front_destroy(None)   # a NULL handle is ignored
