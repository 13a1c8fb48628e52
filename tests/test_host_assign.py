"""The library's bucket assignment equals the oracle's, bit for bit (CPU only)."""
import numpy as np
import pytest

import allreduce_ddp_assign_gb300 as D
import workloads as WL

KEYS = ("bucket_of", "offset_of", "bucket_numel", "bucket_bytes", "bucket_dtype", "bucket_order")


def same(a, r):
    assert a["nbuckets"] == r["nbuckets"]
    for k in KEYS:
        assert np.array_equal(a[k], r[k]), k
    assert [int(p) for p in a["members"]] == [p for m in r["members"] for p in m]


@pytest.mark.parametrize("name", sorted(WL.ALL))
def test_configs(orc, name):
    wl = WL.ALL[name]()
    args = (wl.numels, [wl.dtype] * wl.nparams, wl.cap_bytes, wl.first_cap_bytes, wl.order, wl.pad_multiple, 1)
    same(D.ddp_assign_buckets(*args), orc.assign(*args))


@pytest.mark.parametrize("order", [0, 1, 2])
def test_page_examples(orc, order):
    for n, cap, first in ((WL.numels(WL.linear12()), 25 << 20, 1 << 20),
                          ([2_500_000, 500_000, 2_000_000, 5_000_000, 1_000_000], 12_000_000, 12_000_000),
                          (WL.numels(WL.resnet50()), 25_000_000, 25_000_000),
                          (WL.numels(WL.bert_large()), 25_000_000, 25_000_000)):
        same(D.ddp_assign_buckets(n, None, cap, first, order), orc.assign(n, None, cap, first, order))


def test_random(orc):
    rng = np.random.default_rng(3)
    for trial in range(400):
        P = int(rng.integers(0, 30))
        n = rng.integers(0, 5000, size=P)
        dt = rng.integers(0, 3, size=P) if trial % 3 else np.zeros(P, np.int64)
        cap = int(rng.integers(1, 20000))
        first = int(rng.integers(1, 20000))
        order = int(rng.integers(0, 3))
        pad = int(rng.integers(1, 9))
        fp32 = int(rng.integers(0, 2))
        same(D.ddp_assign_buckets(n, dt, cap, first, order, pad, fp32), orc.assign(n, dt, cap, first, order, pad, fp32))


def test_ordered_assignment_vs_oracle(orc):
    rng = np.random.default_rng(4)
    for trial in range(300):
        P = int(rng.integers(0, 30))
        n = rng.integers(0, 5000, size=P)
        dt = rng.integers(0, 3, size=P) if trial % 3 else np.zeros(P, np.int64)
        seq = rng.permutation(P)
        cap, first = int(rng.integers(1, 20000)), int(rng.integers(1, 20000))
        pad, fp32 = int(rng.integers(1, 9)), int(rng.integers(0, 2))
        same(D.ddp_assign_buckets_ordered(n, seq, dt, cap, first, pad, fp32),
             orc.assign_sequence(n, seq, dt, cap, first, pad, fp32))


def test_ordered_assignment_rejects_non_permutation():
    with pytest.raises(D.DdpError):
        D.ddp_assign_buckets_ordered([1, 2, 3], [0, 0, 1])
    with pytest.raises(D.DdpError):
        D.ddp_assign_buckets_ordered([1, 2, 3], [0, 1, 3])


def test_overlap_timeline_vs_oracle(orc):
    rng = np.random.default_rng(6)
    for trial in range(200):
        P = int(rng.integers(1, 40))
        n = rng.integers(1, 10 ** 6, P)
        r = D.ddp_assign_buckets(n, None, int(rng.integers(10 ** 5, 10 ** 7)), int(rng.integers(10 ** 4, 10 ** 6)),
                                 int(rng.integers(0, 3)))
        ready = rng.random(P) * 20
        a, b = float(rng.random()), float(rng.random()) * 1e-6
        got = D.ddp_overlap_timeline(ready, r["bucket_of"], r["bucket_order"], r["bucket_bytes"], a, b)
        want = orc.overlap_timeline(ready, r["bucket_of"], r["bucket_order"], r["bucket_bytes"], a, b)
        assert np.array_equal(got["start_ms"], want["start_ms"]) and np.array_equal(got["end_ms"], want["end_ms"])
        assert got["step_ms"] == want["step_ms"] and got["serial_ms"] == want["serial_ms"]


def test_plan_describe_and_rebuild_twelve_linear():
    """The plan's logging data: the twelve Linear(1024, 1024) layers give the DDP
    chapter's rebuilt byte list (17.13) when rebuilt over the reverse order, and the
    description lists every parameter once."""
    from allreduce_ddp_assign_gb300.plan import Plan

    numels = [n for _ in range(12) for n in (1024 * 1024, 1024)]
    plan = Plan(numels, device="cpu")
    d = plan.describe()
    assert sorted(p for b in d["bucket_params"] for p in b) == list(range(24))
    assert d["num_buckets"] == len(d["bucket_sizes"]) == plan.nbuckets
    assert plan.rebuilt(list(range(23, -1, -1)))["bucket_sizes"] == [4198400, 29388800, 16793600]
