"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bit-exact comparisons throughout: the kernels reproduce the ring's summation
order, the fp32 1/W pre-scale and the exact bf16/fp16 widening, so every result
must match the oracle's bits (the 1e-6 relative bound is never needed).
"""
import numpy as np
import pytest

import allreduce_ddp_assign_gb300 as D
import oracle as O
import workloads as WL
from gpu_util import GUARD, SENTINEL, assert_bits_equal, bits, chunk_of, oracle_at, packed_at

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")


@pytest.fixture(params=[D.DDP_KERNEL_AUTO, D.DDP_KERNEL_PLAIN, D.DDP_KERNEL_STREAM, D.DDP_KERNEL_STREAM_DYNAMIC],
                ids=["auto", "plain", "stream", "stream_pool"])
def variant(request):
    """Both implementations (the TMA-pipelined streaming kernel wherever it applies,
    with its static split and with the claimed pool of units, and the plain
    16-byte-load kernel) and the default mix (small single-bucket launches plain,
    a pool on large launches) must match the oracle."""
    D.ddp_set_kernel_variant(request.param)
    yield request.param
    D.ddp_set_kernel_variant(D.DDP_KERNEL_AUTO)
    assert D.ddp_device_status(reset=True) == 0


def guarded(n_elems: int, offset: int = 0):
    """A device fp32 buffer of n_elems (+offset) elements with sentinel guard bands."""
    buf = torch.full((GUARD + offset + n_elems + GUARD,), float(SENTINEL), dtype=torch.float32, device=DEV)
    return buf, GUARD + offset


def check_guards(buf, start, n_elems):
    h = buf.cpu().numpy()
    assert np.all(bits(h[:start]) == bits(np.array([SENTINEL]))), "write before the buffer"
    assert np.all(bits(h[start + n_elems:]) == bits(np.array([SENTINEL]))), "write after the buffer"


# ---------------------------------------------------------------------------
# step 3 alone: ddp_bucket_allreduce
# ---------------------------------------------------------------------------
ALLREDUCE_CASES = [(W, n) for W in (1, 2, 3, 4, 5, 8, 16, 64) for n in (0, 1, 3, 4, 7, 64, 1000, 4099, 65549)]


@pytest.mark.parametrize("layout", ["tight", "stride_pad", "misaligned"])
@pytest.mark.parametrize("W,n", ALLREDUCE_CASES)
def test_allreduce_vs_oracle(orc, W, n, layout, variant):
    rng = np.random.default_rng(1000 * W + n)
    for mode in (D.DDP_ALLREDUCE, D.DDP_REDUCE_SCATTER):
        nn = n - n % W if mode == D.DDP_REDUCE_SCATTER else n
        stride = nn + (5 if layout == "stride_pad" else 0)
        stride = max(stride, 1)
        off = 1 if layout == "misaligned" else 0
        x = rng.standard_normal((W, nn)).astype(np.float32)
        buf, start = guarded(W * stride, off)
        view = buf[start:start + W * stride].view(W, stride)
        view[:, :nn] = torch.from_numpy(x).to(DEV)
        D.ddp_bucket_allreduce(buf.data_ptr() + 4 * start, stride, nn, W, mode)
        torch.cuda.synchronize()
        want, sent = orc.ring(x.copy(), mode)
        got = view.cpu().numpy()
        assert_bits_equal(got[:, :nn], want, f"W={W} n={nn} {layout} mode={mode}")
        if stride > nn:
            assert np.all(bits(got[:, nn:]) == bits(np.array([SENTINEL])))
        check_guards(buf, start, W * stride)


def test_allreduce_nonfinite_propagates(orc):
    """An inf in one replica reaches every replica; +inf and -inf give NaN
    (DDP chapter, 17.18: one rank's overflow is seen by all)."""
    W, n = 4, 4096
    x = np.ones((W, n), np.float32)
    x[2, 10] = np.inf
    x[1, 20], x[3, 20] = np.inf, -np.inf
    x[0, 3000] = np.nan            # a poisoned gradient on one rank reaches every rank
    t = torch.from_numpy(x).to(DEV)
    D.ddp_bucket_allreduce(t, n, n, W, D.DDP_ALLREDUCE)
    got = t.cpu().numpy()
    want, _ = orc.ring(x.copy())
    assert np.all(np.isposinf(got[:, 10])) and np.all(np.isnan(got[:, 20])) and np.all(np.isnan(got[:, 3000]))
    assert np.all(np.isnan(want[:, 3000]))
    mask = np.ones(n, bool)
    mask[[20, 3000]] = False
    assert_bits_equal(got[:, mask], want[:, mask])


# ---------------------------------------------------------------------------
# steps 2-4: pack, unpack, fused over random segment lists
# ---------------------------------------------------------------------------
def random_bucket(rng, W, dtype, nseg, misalign):
    sizes = [int(s) for s in rng.choice([0, 1, 2, 3, 5, 17, 64, 255, 1024, 4097, 20000], size=nseg)]
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    pad = int(rng.integers(0, 8))
    numel = int(offs[-1]) + pad
    grads_np = []
    for w in range(W):
        row = []
        for s in range(nseg):
            v = rng.standard_normal(sizes[s]).astype(np.float32)
            if dtype == D.DDP_BF16:
                v = WL.f32_to_bf16_bits_np(v)
            elif dtype == D.DDP_F16:
                v = v.astype(np.float16).view(np.uint16)
            row.append(v)
        grads_np.append(row)
    used = (rng.random((W, nseg)) > 0.2).astype(np.uint8) if nseg else np.zeros((W, 0), np.uint8)
    # device copies: each replica's segments carved out of one flat allocation at
    # offsets that are odd when `misalign` (exercising the scalar path)
    tdt = {D.DDP_F32: torch.float32, D.DDP_BF16: torch.int16, D.DDP_F16: torch.int16}[dtype]
    keep, ptrs = [], np.zeros(W * max(nseg, 1), np.int64)
    for w in range(W):
        total = sum(sizes) + 3 * nseg + 8
        flat = torch.zeros(total, dtype=tdt, device=DEV)
        keep.append(flat)
        pos = 1 if misalign else 0
        for s in range(nseg):
            a = grads_np[w][s]
            t = torch.from_numpy(a.view(np.int16) if dtype != D.DDP_F32 else a)
            flat[pos:pos + sizes[s]] = t.to(DEV)
            ptrs[w * nseg + s] = flat.data_ptr() + pos * flat.element_size()
            pos += sizes[s] + (int(rng.integers(0, 3)) if misalign else (-sizes[s]) % 4)
    seg_off = torch.from_numpy(offs).to(DEV)
    seg_par = torch.arange(max(nseg, 1), dtype=torch.int32, device=DEV)
    desc = D.BucketDesc(numel, nseg, dtype, seg_off.data_ptr(), seg_par.data_ptr())
    tab = torch.from_numpy(ptrs).to(DEV)
    return dict(sizes=sizes, offs=offs, numel=numel, grads_np=grads_np, used=used, desc=desc, tab=tab,
                keep=keep + [seg_off, seg_par], nseg=nseg)


def oracle_pack(orc, bk, W, dtype, accumulate, init):
    segs = [[bk["grads_np"][w][s] if bk["used"][w, s] else None for s in range(bk["nseg"])] for w in range(W)]
    out = init.copy()
    return orc.pack(segs, bk["offs"][:-1], bk["numel"], [dtype] * bk["nseg"], used=bk["used"],
                    accumulate=accumulate, out=out)


def alloc_outs(bk, W, fill):
    outs = [[torch.full((max(s, 1),), fill, dtype=torch.float32, device=DEV) for s in bk["sizes"]] for _ in range(W)]
    ptrs = np.array([outs[w][s].data_ptr() for w in range(W) for s in range(bk["nseg"])] or [0], np.int64)
    return outs, torch.from_numpy(ptrs).to(DEV)


SEG_CASES = [(W, dt, mis) for W in (1, 2, 3, 4, 8, 16) for dt in (D.DDP_F32, D.DDP_BF16, D.DDP_F16)
             for mis in (False, True)]


@pytest.mark.parametrize("W,dtype,misalign", SEG_CASES)
def test_staged_pack_reduce_unpack(orc, W, dtype, misalign, variant):
    rng = np.random.default_rng(W * 31 + dtype * 7 + misalign)
    for trial in range(3):
        bk = random_bucket(rng, W, dtype, int(rng.integers(0, 9)), misalign)
        n, nseg = bk["numel"], bk["nseg"]
        mode = D.DDP_REDUCE_SCATTER if (trial == 2 and n % W == 0) else D.DDP_ALLREDUCE
        stride = n + 3
        init = rng.standard_normal((W, n)).astype(np.float32)
        buf, start = guarded(W * stride)
        mg = buf[start:start + W * stride].view(W, stride)
        mg[:, :n] = torch.from_numpy(init).to(DEV)
        used_t = torch.from_numpy(bk["used"].reshape(-1).copy()).to(DEV) if nseg else None
        mgp = buf.data_ptr() + 4 * start
        for accumulate in (0, 1):
            D.ddp_pack(bk["desc"], bk["tab"], used_t, max(nseg, 1), W, mgp, stride, accumulate)
            init = oracle_pack(orc, bk, W, dtype, accumulate, init)
            assert_bits_equal(mg[:, :n].cpu().numpy(), init, f"pack acc={accumulate}")
        D.ddp_bucket_allreduce(mgp, stride, n, W, mode)
        want, _ = orc.ring(init.copy(), mode)
        assert_bits_equal(mg[:, :n].cpu().numpy(), want, "reduce")
        gu = bk["used"].max(axis=0) if nseg else np.zeros(0, np.uint8)
        outs, out_tab = alloc_outs(bk, W, -3.0)
        gu_t = torch.from_numpy(gu.copy()).to(DEV) if nseg else None
        D.ddp_unpack(bk["desc"], mgp, stride, W, mode, out_tab, max(nseg, 1), gu_t)
        exp = orc.unpack(want.copy(), bk["offs"][:-1], bk["sizes"], mode, gu,
                         outs=[[np.full(s, -3.0, np.float32) for s in bk["sizes"]] for _ in range(W)])
        for w in range(W):
            for s in range(nseg):
                assert_bits_equal(outs[w][s][:bk["sizes"][s]].cpu().numpy(), exp[w][s], f"unpack w={w} s={s}")
        check_guards(buf, start, W * stride)


@pytest.mark.parametrize("W,dtype,misalign", SEG_CASES)
def test_fused_matches_staged_oracle(orc, W, dtype, misalign, variant):
    rng = np.random.default_rng(W * 131 + dtype * 17 + misalign)
    for trial in range(4):
        bk = random_bucket(rng, W, dtype, int(rng.integers(0, 9)), misalign)
        n, nseg = bk["numel"], bk["nseg"]
        mode = D.DDP_REDUCE_SCATTER if (trial % 2 and n % W == 0) else D.DDP_ALLREDUCE
        accumulate = trial >= 2
        copy_back = trial in (1, 2)
        stride = n + (0 if misalign else 4)
        init = rng.standard_normal((W, n)).astype(np.float32)
        buf, start = guarded(W * stride)
        mg = buf[start:start + W * stride].view(W, stride)
        mg[:, :n] = torch.from_numpy(init).to(DEV)
        used_t = torch.from_numpy(bk["used"].reshape(-1).copy()).to(DEV) if nseg else None
        gu = bk["used"].max(axis=0) if nseg else np.zeros(0, np.uint8)
        gu_t = torch.from_numpy(gu.copy()).to(DEV) if nseg else None
        outs, out_tab = alloc_outs(bk, W, 5.0) if copy_back else (None, None)
        D.ddp_fused_bucket(bk["desc"], bk["tab"], used_t, max(nseg, 1), W, mode, int(accumulate),
                           buf.data_ptr() + 4 * start, stride, out_tab, gu_t)
        packed = oracle_pack(orc, bk, W, dtype, accumulate, init)
        want, _ = orc.ring(packed.copy(), mode)
        got = mg[:, :n].cpu().numpy()
        if mode == D.DDP_ALLREDUCE:
            assert_bits_equal(got, want, "fused main_grad")
        else:
            k = n // W
            for w in range(W):  # shard w of replica w reduced; the rest untouched
                assert_bits_equal(got[w, w * k:(w + 1) * k], want[w, w * k:(w + 1) * k], f"shard {w}")
                rest = np.ones(n, bool)
                rest[w * k:(w + 1) * k] = False
                assert_bits_equal(got[w, rest], init[w, rest], f"outside shard {w}")
        if copy_back:
            exp = orc.unpack(want.copy(), bk["offs"][:-1], bk["sizes"], mode, gu,
                             outs=[[np.full(s, 5.0, np.float32) for s in bk["sizes"]] for _ in range(W)])
            for w in range(W):
                for s in range(nseg):
                    assert_bits_equal(outs[w][s][:bk["sizes"][s]].cpu().numpy(), exp[w][s], f"copy-back {w},{s}")
        check_guards(buf, start, W * stride)


def test_fused_in_place_without_main_grad(orc, variant):
    """grads_out aliasing fp32 grads, no bucket buffer: DDP without
    gradient_as_bucket_view, reduced straight back into .grad."""
    rng = np.random.default_rng(5)
    W = 8
    bk = random_bucket(rng, W, D.DDP_F32, 7, False)
    D.ddp_fused_bucket(bk["desc"], bk["tab"], None, bk["nseg"], W, D.DDP_ALLREDUCE, 0, None, 0, bk["tab"], None)
    bk["used"][:] = 1
    packed = oracle_pack(orc, bk, W, D.DDP_F32, False, np.zeros((W, bk["numel"]), np.float32))
    want, _ = orc.ring(packed, D.DDP_ALLREDUCE)
    flat = bk["keep"]
    for w in range(W):
        pos = 0
        for s, sz in enumerate(bk["sizes"]):
            got = flat[w][pos:pos + sz].cpu().numpy()
            assert_bits_equal(got, want[w, bk["offs"][s]:bk["offs"][s] + sz], f"in place w={w} s={s}")
            pos += sz + (-sz) % 4


# ---------------------------------------------------------------------------
# the workloads, through the same reducer path the benchmark times
# ---------------------------------------------------------------------------
def device_grads(wl, m=0, skip_unused=True):
    return [[None if (skip_unused and p in wl.unused) else WL.grad_torch(wl, p, w, m, DEV)
             for p in range(wl.nparams)] for w in range(wl.W)]


def used_flags(wl):
    u = np.ones((wl.W, wl.nparams), np.uint8)
    u[:, wl.unused] = 0
    return u


def make_session(wl, grads, fused=True, grads_out=None, timing=False):
    from allreduce_ddp_assign_gb300.session import BucketReducer

    return BucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                         wl.first_cap_bytes, wl.pad_multiple, grads, used=used_flags(wl) if wl.unused else None,
                         grads_out=grads_out, fused=fused, timing=timing)


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("name", ["c1", "c2"])
def test_workload_full_vs_oracle(orc, name, fused, variant):
    wl = WL.ALL[name]()
    sess = make_session(wl, device_grads(wl), fused=fused)
    sess.step()
    torch.cuda.synchronize()
    ref = O.run_workload(wl, orc, copy_back=False)
    assert sess.plan.nbuckets == ref["plan"]["nbuckets"]
    for b in range(sess.plan.nbuckets):
        got = sess.plan.bucket_view(sess.main_grad, b).cpu().numpy()
        assert_bits_equal(got, ref["bucket"][b], f"{name} bucket {b}")
    if name == "c1":  # dyadic inputs: the mean is exact
        x = [[WL.grad_np(wl, p, w) for p in range(wl.nparams)] for w in range(wl.W)]
        for p in range(wl.nparams):
            mean = sum(x[w][p].astype(np.float64) for w in range(wl.W)) / wl.W
            assert np.array_equal(sess.view(p, 3).cpu().numpy().astype(np.float64), mean)
    sess.close()


def test_mlp_copy_back_partial_use(orc):
    """C1 with copy-back, parameter 2 unused on replica 1 only and parameter 4 on no
    replica: partial use averages in a zero, global non-use leaves .grad alone."""
    wl = WL.c1_mlp()
    grads = device_grads(wl)
    used = np.ones((wl.W, wl.nparams), np.uint8)
    used[1, 2] = 0
    used[:, 4] = 0
    outs = [[torch.full((n,), 9.0, device=DEV) for n in wl.numels] for _ in range(wl.W)]
    from allreduce_ddp_assign_gb300.session import BucketReducer

    for fused in (True, False):
        for w in range(wl.W):
            for p in range(wl.nparams):
                outs[w][p].fill_(9.0)
        sess = BucketReducer(wl.numels, None, wl.W, wl.mode, wl.order, wl.cap_bytes, wl.first_cap_bytes, 1, grads,
                             used=used, grads_out=outs, fused=fused)
        sess.step()
        torch.cuda.synchronize()
        raw = [[[None if not used[w, p] else WL.grad_raw_np(wl, p, w) for p in range(wl.nparams)]
                for w in range(wl.W)]]
        plan = orc.assign(wl.numels, None, wl.cap_bytes, wl.first_cap_bytes, wl.order)
        mem = plan["members"][0]
        offs = [int(plan["offset_of"][p]) for p in mem]
        buf = orc.pack([[raw[0][w][p] for p in mem] for w in range(wl.W)], offs, int(plan["bucket_numel"][0]),
                       used=used[:, mem])
        buf, _ = orc.ring(buf)
        exp = orc.unpack(buf, offs, [wl.numels[p] for p in mem], 0, orc.used_allreduce(used)[1][mem],
                         outs=[[np.full(wl.numels[p], 9.0, np.float32) for p in mem] for _ in range(wl.W)])
        for w in range(wl.W):
            for j, p in enumerate(mem):
                assert_bits_equal(outs[w][p].cpu().numpy(), exp[w][j], f"fused={fused} w={w} p={p}")
        assert np.all(outs[0][4].cpu().numpy() == 9.0)
        sess.close()


def boundary_sample(rng, n, W, seg_offsets=(), k=1500):
    """Sampled element indices of an n-element bucket: k random ones plus the
    elements on both sides of every place where the kernels' work changes hands --
    every ring chunk's first and last element, every parameter segment's first and
    last, the first and last element of each CTA's slice for one and two CTAs per
    SM (152 and 304 slices, cut on 16-element multiples) and of the streaming
    tiles that follow each slice start (1024, 2048 and 4096 elements), and every
    multiple of 1024 within the first and last 64 Ki elements of each chunk."""
    pts = [0, n - 1]
    L = max(1, -(-n // W))
    for c in range(W + 1):
        pts += [c * L - 1, c * L, c * L + 1]
        for t in range(0, 65536, 1024):
            pts += [c * L + t, c * L + t - 1, c * L - t, c * L - t - 1]
    for o in seg_offsets:
        pts += [o - 1, o, o + 1]
    for G in (152, 304):
        for b in range(G + 1):
            lo = (b * n // G) & ~15
            for tile in (0, 1024, 2048, 4096, 8192):
                pts += [lo + tile - 1, lo + tile]
    pts = np.array(pts, np.int64)
    pts = pts[(pts >= 0) & (pts < n)]
    return np.unique(np.concatenate([pts, rng.integers(0, n, k)]))


@pytest.mark.slow
def test_gpt2_reduce_scatter_full_size(orc):
    """GPT-2 small, bf16 -> fp32, Megatron buckets, W = 8 reduce_scatter: every
    element of every shard of all nine buckets against the oracle (pack, then the
    ring's reduce-scatter), and nothing outside the shards written.  The oracle's
    inputs are the seeded generator's gradients (its torch form, checked bit for
    bit against its numpy form by the workload tests), copied to the host."""
    wl = WL.c3_gpt2()
    grads = device_grads(wl)
    sess = make_session(wl, grads)
    sess.main_grad.fill_(float(SENTINEL))
    sess.step()
    torch.cuda.synchronize()
    plan = sess.plan
    assert plan.nbuckets == 9
    for b in range(plan.nbuckets):
        n = int(plan.bucket_numel[b])
        got = plan.bucket_view(sess.main_grad, b).cpu().numpy()
        k = n // wl.W
        for w in range(wl.W):  # outside shard w, replica w keeps the sentinel
            assert np.all(bits(got[w, :w * k]) == bits(np.array([SENTINEL])))
            assert np.all(bits(got[w, (w + 1) * k:]) == bits(np.array([SENTINEL])))
        mem = plan.members[b]
        raw = [[grads[w][p].view(torch.int16).cpu().numpy().view(np.uint16) for p in mem] for w in range(wl.W)]
        packed = orc.pack(raw, [int(plan.offset_of[p]) for p in mem], n, [wl.dtype] * len(mem))
        del raw
        want, _ = orc.ring(packed, D.DDP_REDUCE_SCATTER)
        for w in range(wl.W):
            assert_bits_equal(got[w, w * k:(w + 1) * k], want[w, w * k:(w + 1) * k], f"bucket {b} shard {w}")
        del packed, want, got
    sess.close()


@pytest.mark.slow
def test_bert_nosync_full_size_sampled(orc):
    """BERT-large, W = 4: three no_sync micro-steps accumulated locally, the fourth
    reduced with the accumulated sum; one encoder layer unused (zero).  Sampled at
    every place where the kernels' work changes hands (boundary_sample) plus 500
    random elements per bucket."""
    wl = WL.c4_bert_large()
    sess = make_session(wl, device_grads(wl, 3))
    for m in range(3):
        g = device_grads(wl, m)
        tab = sess.plan.pointer_table(g)
        sess.accumulate_local(tab, first=m == 0)
        torch.cuda.synchronize()
        del tab, g
    sess.step(accumulate=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(44)
    plan = sess.plan
    used = used_flags(wl)
    for b in range(plan.nbuckets):
        n = int(plan.bucket_numel[b])
        got = plan.bucket_view(sess.main_grad, b).cpu().numpy()
        for w in range(1, wl.W):
            assert np.array_equal(bits(got[0]), bits(got[w]))
        segs = [int(plan.offset_of[p]) for p in plan.members[b]]
        e = boundary_sample(rng, n, wl.W, segs + [segs[-1] + wl.numels[plan.members[b][-1]]], 500)
        t = np.zeros((wl.W, len(e)), np.float32)
        for p in plan.members[b]:
            lo, hi = int(plan.offset_of[p]), int(plan.offset_of[p]) + wl.numels[p]
            sel = np.nonzero((e >= lo) & (e < hi))[0]
            if len(sel):
                t[:, sel] = packed_at(orc, wl, p, e[sel] - lo, 4, used[:, p])
        want = oracle_at(orc, t, chunk_of(e, n, wl.W))
        assert_bits_equal(got[0, e], want, f"bucket {b}")
    for p in wl.unused:
        assert not torch.any(sess.view(p, 2))
    sess.close()


@pytest.mark.slow
@pytest.mark.parametrize("nbytes,W", [(1 << 30, 16), (1 << 28, 2), ((1 << 20) + 4 * 13, 8)])
def test_sweep_bucket_sampled(orc, nbytes, W):
    n = nbytes // 4
    x = WL.bucket_torch(nbytes, W, DEV)
    D.ddp_bucket_allreduce(x, n, n, W, D.DDP_ALLREDUCE)
    torch.cuda.synchronize()
    for w in range(1, W):
        assert torch.equal(x[0], x[w])
    rng = np.random.default_rng(55)
    e = boundary_sample(rng, n, W, (), 4000)
    t = np.stack([WL.values_np(WL.bits_at_np(WL.stream_key(1005, WL.stream_id(0, w)), e), "uniform")
                  for w in range(W)])
    want = oracle_at(orc, t, chunk_of(e, n, W))
    assert_bits_equal(x[W - 1, torch.from_numpy(e).to(DEV)].cpu().numpy(), want)


# ---------------------------------------------------------------------------
# the reducer on real streams
# ---------------------------------------------------------------------------
def test_reducer_waits_for_producer_stream(orc):
    """Gradients are written on a delayed producer stream just before each
    mark_ready; the side stream must see them (event-gated issue)."""
    wl = WL.Workload("linear12", WL.linear12(), 4, 0, 0, 25 << 20, 1 << 20, 1, 0, "dyadic12", 1.0, 77)
    final = device_grads(wl)
    grads = [[torch.zeros_like(final[w][p]) for p in range(wl.nparams)] for w in range(wl.W)]
    sess = make_session(wl, grads, timing=True)
    prod = torch.cuda.Stream()
    torch.cuda.synchronize()
    D.ddp_reducer_prepare(sess.handle, 0)
    with torch.cuda.stream(prod):
        for p in sess.ready_order:
            torch.cuda._sleep(200_000)
            for w in range(wl.W):
                grads[w][p].copy_(final[w][p])
            D.ddp_reducer_mark_ready(sess.handle, p, prod)
    sess.finalize(torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert sess.issue_log() == [0, 1, 2]
    ref = O.run_workload(wl, orc, copy_back=False)
    for b in range(3):
        assert_bits_equal(sess.plan.bucket_view(sess.main_grad, b).cpu().numpy(), ref["bucket"][b], f"bucket {b}")
    ms = sess.bucket_ms()
    assert np.all(ms > 0)
    sess.close()


def test_reducer_finalize_timeout_then_recovers(orc):
    wl = WL.c1_mlp()
    sess = make_session(wl, device_grads(wl))
    sess.step()                # loads the library's kernels first (a lazy module load can wait for the GPU)
    torch.cuda.synchronize()
    with torch.cuda.stream(sess.side):
        torch.cuda._sleep(400_000_000)   # ~0.2 s of spinning on the side stream (bounded)
    sess.backward()
    with pytest.raises(D.DdpError) as e:
        sess.finalize(None, timeout_us=2000)
    assert e.value.status == D.DDP_E_TIMEOUT
    sess.finalize(None, timeout_us=30_000_000)    # same iteration: now it completes
    torch.cuda.synchronize()
    ref = O.run_workload(wl, orc, copy_back=False)
    assert_bits_equal(sess.plan.bucket_view(sess.main_grad, 0).cpu().numpy(), ref["bucket"][0])
    sess.close()


def test_finalize_orders_the_default_stream(orc):
    """finalize(consumer = the legacy default stream) must make that stream wait
    for the side stream: a copy taken on it right after finalize sees the result
    even though the side stream was held back first."""
    wl = WL.c1_mlp()
    sess = make_session(wl, device_grads(wl))
    sess.step()                # loads the library's kernels first (a lazy module load can wait for the GPU)
    sess.main_grad.zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(sess.side):
        torch.cuda._sleep(100_000_000)   # bounded spin, ~50 ms
    assert torch.cuda.current_stream().cuda_stream == 0   # the legacy default stream
    sess.step()                                          # producer and consumer: the current stream
    snap = sess.main_grad.clone()                        # queued on the default stream
    torch.cuda.synchronize()
    ref = O.run_workload(wl, orc, copy_back=False)
    got = sess.plan.bucket_view(snap, 0).cpu().numpy()
    assert_bits_equal(got, ref["bucket"][0], "default-stream snapshot")
    sess.close()


def test_device_status_clean():
    assert D.ddp_device_status(reset=True) == 0


@pytest.mark.parametrize("W", [2, 3, 4, 8, 16])
def test_fused_bucket_group_vs_oracle(orc, W, variant):
    """Several buckets (mixed dtypes, so the group splits into runs) in one call:
    every bucket equals the oracle's pack + ring (+ unpack)."""
    rng = np.random.default_rng(900 + W)
    for trial in range(3):
        mode = D.DDP_REDUCE_SCATTER if trial == 1 else D.DDP_ALLREDUCE
        accumulate = trial == 2
        dts = [int(d) for d in rng.choice([D.DDP_F32, D.DDP_F32, D.DDP_BF16, D.DDP_F16], size=5)]
        bks = [random_bucket(rng, W, dt, int(rng.integers(1, 7)), bool(rng.integers(0, 2))) for dt in dts]
        for bk in bks:   # reduce_scatter needs numel % W == 0: pad the buckets
            bk["numel"] += (-bk["numel"]) % W
            bk["desc"].numel = bk["numel"]
        starts, pos = [], 0
        for bk in bks:
            starts.append(pos)
            pos += (bk["numel"] + 63) // 64 * 64
        stride = max(pos, 64)
        # one table for all buckets: bucket i's segment s is parameter cols[i] + s
        cols = np.cumsum([0] + [bk["nseg"] for bk in bks])
        ld = int(cols[-1])
        ptrs = np.zeros(W * ld, np.int64)
        usedf = np.zeros((W, ld), np.uint8)
        for i, bk in enumerate(bks):
            t = bk["tab"].cpu().numpy().reshape(W, bk["nseg"])
            ptrs.reshape(W, ld)[:, cols[i]:cols[i + 1]] = t
            usedf[:, cols[i]:cols[i + 1]] = bk["used"]
            par = torch.arange(cols[i], cols[i + 1], dtype=torch.int32, device=DEV)
            bk["keep"].append(par)
            bk["desc"].seg_param = par.data_ptr()
        tab = torch.from_numpy(ptrs).to(DEV)
        used_t = torch.from_numpy(usedf.reshape(-1).copy()).to(DEV)
        gu = usedf.max(axis=0)
        gu_t = torch.from_numpy(gu.copy()).to(DEV)
        init = rng.standard_normal((W, stride)).astype(np.float32)
        mg = torch.from_numpy(init.copy()).to(DEV)
        outs = [[torch.full((max(n, 1),), 2.0, device=DEV) for bk in bks for n in bk["sizes"]] for _ in range(W)]
        out_tab = torch.from_numpy(np.array([o.data_ptr() for w in range(W) for o in outs[w]], np.int64)).to(DEV)
        D.ddp_fused_bucket_group([bk["desc"] for bk in bks], starts, tab, used_t, ld, W, mode, int(accumulate), mg,
                                 stride, out_tab, gu_t)
        got = mg.cpu().numpy()
        for i, bk in enumerate(bks):
            n, s0 = bk["numel"], starts[i]
            packed = oracle_pack(orc, bk, W, dts[i], accumulate, init[:, s0:s0 + n].copy())
            want, _ = orc.ring(packed.copy(), mode)
            g = got[:, s0:s0 + n]
            if mode == D.DDP_ALLREDUCE:
                assert_bits_equal(g, want, f"bucket {i}")
            else:
                k = n // W
                for w in range(W):
                    assert_bits_equal(g[w, w * k:(w + 1) * k], want[w, w * k:(w + 1) * k], f"bucket {i} shard {w}")
            exp = orc.unpack(want.copy(), bk["offs"][:-1], bk["sizes"], mode, gu[cols[i]:cols[i + 1]],
                             outs=[[np.full(s, 2.0, np.float32) for s in bk["sizes"]] for _ in range(W)])
            for w in range(W):
                for s in range(bk["nseg"]):
                    o = outs[w][cols[i] + s][:bk["sizes"][s]].cpu().numpy()
                    assert_bits_equal(o, exp[w][s], f"copy-back bucket {i} w={w} s={s}")


@pytest.mark.parametrize("name", ["c1", "c2", "c3"])
def test_coalesced_reducer_vs_oracle(orc, name):
    """The reducer issuing every ready bucket in one launch gives the same bits."""
    from allreduce_ddp_assign_gb300.session import BucketReducer

    wl = WL.ALL[name]()
    sess = BucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                         wl.first_cap_bytes, wl.pad_multiple, device_grads(wl), coalesce=True, timing=True)
    if wl.mode == D.DDP_REDUCE_SCATTER:
        sess.main_grad.fill_(float(SENTINEL))
    sess.step()
    torch.cuda.synchronize()
    assert sess.issue_log() == [int(b) for b in sess.plan.bucket_order]
    assert np.all(sess.bucket_ms() > 0)
    rng = np.random.default_rng(5)
    for b in range(sess.plan.nbuckets):
        got = sess.plan.bucket_view(sess.main_grad, b).cpu().numpy()
        n = int(sess.plan.bucket_numel[b])
        if name != "c3":
            ref = O.run_workload(wl, orc, copy_back=False) if b == 0 else ref
            assert_bits_equal(got, ref["bucket"][b], f"{name} bucket {b}")
        else:
            segs = [int(sess.plan.offset_of[p]) for p in sess.plan.members[b]]
            e = boundary_sample(rng, n, wl.W, segs, 400)
            owner = chunk_of(e, n, wl.W)
            t = np.zeros((wl.W, len(e)), np.float32)
            for p in sess.plan.members[b]:
                lo, hi = int(sess.plan.offset_of[p]), int(sess.plan.offset_of[p]) + wl.numels[p]
                sel = np.nonzero((e >= lo) & (e < hi))[0]
                if len(sel):
                    t[:, sel] = packed_at(orc, wl, p, e[sel] - lo, 1)
            assert_bits_equal(got[owner, e], oracle_at(orc, t, owner), f"c3 bucket {b}")
    sess.close()


@pytest.mark.parametrize("W", [2, 3, 4, 8, 16])
def test_pack_group_vs_oracle(orc, W, variant):
    """A no_sync micro-step over several buckets in one call (copy, then accumulate):
    every bucket equals the oracle's pack."""
    rng = np.random.default_rng(700 + W)
    dts = [int(d) for d in rng.choice([D.DDP_F32, D.DDP_F32, D.DDP_BF16, D.DDP_F16], size=5)]
    bks = [random_bucket(rng, W, dt, int(rng.integers(1, 7)), bool(rng.integers(0, 2))) for dt in dts]
    starts, pos = [], 0
    for bk in bks:
        starts.append(pos)
        pos += (bk["numel"] + 63) // 64 * 64
    stride = max(pos, 64)
    cols = np.cumsum([0] + [bk["nseg"] for bk in bks])
    ld = int(cols[-1])
    ptrs = np.zeros(W * ld, np.int64)
    usedf = np.zeros((W, ld), np.uint8)
    for i, bk in enumerate(bks):
        ptrs.reshape(W, ld)[:, cols[i]:cols[i + 1]] = bk["tab"].cpu().numpy().reshape(W, bk["nseg"])
        usedf[:, cols[i]:cols[i + 1]] = bk["used"]
        par = torch.arange(cols[i], cols[i + 1], dtype=torch.int32, device=DEV)
        bk["keep"].append(par)
        bk["desc"].seg_param = par.data_ptr()
    tab = torch.from_numpy(ptrs).to(DEV)
    used_t = torch.from_numpy(usedf.reshape(-1).copy()).to(DEV)
    init = rng.standard_normal((W, stride)).astype(np.float32)
    mg = torch.from_numpy(init.copy()).to(DEV)
    want = init.copy()
    for accumulate in (0, 1):
        D.ddp_pack_group([bk["desc"] for bk in bks], starts, tab, used_t, ld, W, mg, stride, accumulate)
        for i, bk in enumerate(bks):
            n, s0 = bk["numel"], starts[i]
            want[:, s0:s0 + n] = oracle_pack(orc, bk, W, dts[i], accumulate, want[:, s0:s0 + n].copy())
        got = mg.cpu().numpy()
        for i, bk in enumerate(bks):
            n, s0 = bk["numel"], starts[i]
            assert_bits_equal(got[:, s0:s0 + n], want[:, s0:s0 + n], f"bucket {i} accumulate={accumulate}")
        # nothing outside the buckets was written
        mask = np.ones(stride, bool)
        for i, bk in enumerate(bks):
            mask[starts[i]:starts[i] + bk["numel"]] = False
        assert_bits_equal(got[:, mask], init[:, mask], "outside the buckets")


@pytest.mark.slow
def test_bert_nosync_coalesced_sampled(orc):
    """The benchmark's configuration for BERT-large: pack groups for the no_sync
    micro-steps, coalesced fused issue for the synchronised one."""
    from allreduce_ddp_assign_gb300.session import BucketReducer

    wl = WL.c4_bert_large()
    sess = BucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                         wl.first_cap_bytes, wl.pad_multiple, device_grads(wl, 3), used=used_flags(wl), coalesce=True)
    for m in range(3):
        g = device_grads(wl, m)
        tab = sess.plan.pointer_table(g)
        sess.accumulate_local(tab, first=m == 0)
        torch.cuda.synchronize()
        del tab, g
    sess.step(accumulate=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(45)
    plan = sess.plan
    used = used_flags(wl)
    for b in range(0, plan.nbuckets, 3):
        n = int(plan.bucket_numel[b])
        got = plan.bucket_view(sess.main_grad, b).cpu().numpy()
        e = boundary_sample(rng, n, wl.W, [int(plan.offset_of[p]) for p in plan.members[b]], 300)
        t = np.zeros((wl.W, len(e)), np.float32)
        for p in plan.members[b]:
            lo, hi = int(plan.offset_of[p]), int(plan.offset_of[p]) + wl.numels[p]
            sel = np.nonzero((e >= lo) & (e < hi))[0]
            if len(sel):
                t[:, sel] = packed_at(orc, wl, p, e[sel] - lo, 4, used[:, p])
        assert_bits_equal(got[wl.W - 1, e], oracle_at(orc, t, chunk_of(e, n, wl.W)), f"bucket {b}")
    sess.close()


# ---------------------------------------------------------------------------
# the compression hook (bf16 / fp16 wire)
# ---------------------------------------------------------------------------
def assert_wire_equal(got, want, what):
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan), what
    assert_bits_equal(np.where(nan, 0, got), np.where(nan, 0, want), what)


@pytest.mark.parametrize("wire", [D.DDP_BF16, D.DDP_F16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("W,n", [(W, n) for W in (1, 2, 3, 4, 5, 8, 16) for n in (0, 7, 1000, 4099, 65549)])
def test_allreduce_wire_vs_oracle(orc, W, n, wire, variant):
    rng = np.random.default_rng(500 * W + n + wire)
    for mode in (D.DDP_ALLREDUCE, D.DDP_REDUCE_SCATTER):
        nn = n - n % W if mode == D.DDP_REDUCE_SCATTER else n
        for misaligned in (False, True):
            x = (rng.standard_normal((W, nn)) * 10.0 ** rng.integers(-6, 5, (W, nn))).astype(np.float32)
            if wire == D.DDP_F16 and nn:
                x[0, 0] = 1e5          # beyond fp16: the hook saturates to infinity
            stride = max(nn, 1)
            buf, start = guarded(W * stride, 1 if misaligned else 0)
            view = buf[start:start + W * stride].view(W, stride)
            view[:, :nn] = torch.from_numpy(x).to(DEV)
            D.ddp_bucket_allreduce_wire(buf.data_ptr() + 4 * start, stride, nn, W, mode, wire)
            want, _ = orc.ring_wire(x.copy(), mode, wire)
            assert_wire_equal(view[:, :nn].cpu().numpy(), want, f"W={W} n={nn} wire={wire} mode={mode}")
            check_guards(buf, start, W * stride)


@pytest.mark.parametrize("wire", [D.DDP_BF16, D.DDP_F16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("W", [2, 3, 4, 8])
def test_fused_group_wire_vs_oracle(orc, W, wire, variant):
    rng = np.random.default_rng(800 + W + 10 * wire)
    dt = D.DDP_F32
    bks = [random_bucket(rng, W, dt, int(rng.integers(1, 6)), bool(rng.integers(0, 2))) for _ in range(3)]
    for mode in (D.DDP_ALLREDUCE, D.DDP_REDUCE_SCATTER):
        for accumulate in (0, 1):
            for bk in bks:
                bk["numel"] += (-bk["numel"]) % W
                bk["desc"].numel = bk["numel"]
            starts, pos = [], 0
            for bk in bks:
                starts.append(pos)
                pos += (bk["numel"] + 63) // 64 * 64
            stride = max(pos, 64)
            cols = np.cumsum([0] + [bk["nseg"] for bk in bks])
            ld = int(cols[-1])
            ptrs = np.zeros(W * ld, np.int64)
            usedf = np.zeros((W, ld), np.uint8)
            for i, bk in enumerate(bks):
                ptrs.reshape(W, ld)[:, cols[i]:cols[i + 1]] = bk["tab"].cpu().numpy().reshape(W, bk["nseg"])
                usedf[:, cols[i]:cols[i + 1]] = bk["used"]
                par = torch.arange(cols[i], cols[i + 1], dtype=torch.int32, device=DEV)
                bk["keep"].append(par)
                bk["desc"].seg_param = par.data_ptr()
            tab = torch.from_numpy(ptrs).to(DEV)
            used_t = torch.from_numpy(usedf.reshape(-1).copy()).to(DEV)
            init = rng.standard_normal((W, stride)).astype(np.float32)
            mg = torch.from_numpy(init.copy()).to(DEV)
            D.ddp_fused_bucket_group_wire([bk["desc"] for bk in bks], starts, tab, used_t, ld, W, mode, accumulate,
                                          mg, stride, None, None, wire)
            got = mg.cpu().numpy()
            for i, bk in enumerate(bks):
                n, s0 = bk["numel"], starts[i]
                packed = oracle_pack(orc, bk, W, dt, accumulate, init[:, s0:s0 + n].copy())
                want, _ = orc.ring_wire(packed.copy(), mode, wire)
                if mode == D.DDP_ALLREDUCE:
                    assert_wire_equal(got[:, s0:s0 + n], want, f"bucket {i}")
                else:
                    k = n // W
                    for w in range(W):
                        assert_wire_equal(got[w, s0 + w * k:s0 + (w + 1) * k], want[w, w * k:(w + 1) * k],
                                          f"bucket {i} shard {w}")


@pytest.mark.parametrize("coalesce", [False, True])
def test_reducer_bf16_hook_resnet50(orc, coalesce):
    """ResNet-50 W=8 through the reducer with the bf16 compression hook."""
    from allreduce_ddp_assign_gb300.session import BucketReducer

    wl = WL.c2_resnet50()
    sess = BucketReducer(wl.numels, None, wl.W, wl.mode, wl.order, wl.cap_bytes, wl.first_cap_bytes, 1,
                         device_grads(wl), coalesce=coalesce, wire=D.DDP_BF16)
    sess.step()
    torch.cuda.synchronize()
    ref = O.run_workload(wl, orc, copy_back=False, wire=O.BF16)
    for b in range(sess.plan.nbuckets):
        assert_bits_equal(sess.plan.bucket_view(sess.main_grad, b).cpu().numpy(), ref["bucket"][b], f"bucket {b}")
    sess.close()


def test_overlap_hides_reduction():
    """With a synthetic backward of about 3 ms, the reductions run on the side stream while
    it proceeds: the overlapped step is shorter than the serial one, and the model's
    prediction from the recorded ready times lands near the measured step."""
    import argparse

    import bench

    line = bench.run_overlap(argparse.Namespace(backward_ms=3.0))
    assert line["overlapped_step_ms"] < line["serial_step_ms"]
    assert line["overlapped_step_ms"] >= line["backward_ms"] * 0.98
    assert abs(line["model"]["step_ms"] - line["overlapped_step_ms"]) < 0.25 * line["overlapped_step_ms"]


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_host_front_end_pipeline_vs_oracle(orc, name):
    """HostBucketReducer: pinned host gradients in, reduced buckets out, with the
    copies in both directions pipelined against the reductions bucket by bucket.
    Two steps in a row with different inputs, every bucket bit for bit."""
    from allreduce_ddp_assign_gb300.session import HostBucketReducer

    wl = WL.ALL[name]()
    host = HostBucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                             wl.first_cap_bytes, wl.pad_multiple, torch.float32)
    plan = host.reducer.plan
    total = int(host.offs[-1])
    h_out = torch.full((wl.W * host.replica_stride,), -1.0, dtype=torch.float32, pin_memory=True)
    for m in range(2):
        h_in = torch.empty((wl.W, total), dtype=torch.float32, pin_memory=True)
        for w in range(wl.W):
            h_in[w] = torch.from_numpy(np.concatenate([WL.grad_np(wl, p, w, m) for p in range(wl.nparams)]))
        host.step(h_in, h_out)
        torch.cuda.synchronize()
        raw = [[[WL.grad_raw_np(wl, p, w, m) for p in range(wl.nparams)] for w in range(wl.W)]]
        ref = O.run_workload(wl, orc, grads=raw, copy_back=False)
        out = h_out.numpy().reshape(wl.W, host.replica_stride)
        for b in range(plan.nbuckets):
            lo, n = int(plan.bucket_start[b]), int(plan.bucket_numel[b])
            assert_bits_equal(out[:, lo:lo + n], ref["bucket"][b], f"step {m} bucket {b}")
    host.close()


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_host_front_end_steps_back_to_back(orc, name):
    """Three steps issued without a host synchronisation between them, each with its
    own inputs and output buffer: step k + 1's uploads and reductions overlap step k's
    downloads bucket by bucket, and every step's output must still be its own inputs'
    reduction, bit for bit."""
    from allreduce_ddp_assign_gb300.session import HostBucketReducer

    wl = WL.ALL[name]()
    host = HostBucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                             wl.first_cap_bytes, wl.pad_multiple, torch.float32)
    plan = host.reducer.plan
    total = int(host.offs[-1])
    h_in, h_out = [], []
    for m in range(3):
        x = torch.empty((wl.W, total), dtype=torch.float32, pin_memory=True)
        for w in range(wl.W):
            x[w] = torch.from_numpy(np.concatenate([WL.grad_np(wl, p, w, m) for p in range(wl.nparams)]))
        h_in.append(x)
        h_out.append(torch.full((wl.W * host.replica_stride,), -1.0, dtype=torch.float32, pin_memory=True))
    host.step(h_in[0], h_out[0])   # first step (and lazy module loading) outside the race
    torch.cuda.synchronize()
    for m in range(3):
        host.step(h_in[m], h_out[m])
    torch.cuda.synchronize()
    for m in range(3):
        raw = [[[WL.grad_raw_np(wl, p, w, m) for p in range(wl.nparams)] for w in range(wl.W)]]
        ref = O.run_workload(wl, orc, grads=raw, copy_back=False)
        out = h_out[m].numpy().reshape(wl.W, host.replica_stride)
        for b in range(plan.nbuckets):
            lo, n = int(plan.bucket_start[b]), int(plan.bucket_numel[b])
            assert_bits_equal(out[:, lo:lo + n], ref["bucket"][b], f"step {m} bucket {b}")
    host.close()


def test_host_front_end_reduce_scatter_shards(orc):
    """Reduce_scatter through the host front end: replica w's host copy receives
    exactly shard w of every bucket (bit for bit), and nothing outside it."""
    from allreduce_ddp_assign_gb300.session import HostBucketReducer

    wl = WL.Workload("linear12_rs", WL.linear12(), 4, 1, 2, 8 << 20, 8 << 20, 4, 0, "dyadic12", 1.0, 91)
    host = HostBucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                             wl.first_cap_bytes, wl.pad_multiple, torch.float32)
    plan = host.reducer.plan
    total = int(host.offs[-1])
    h_in = torch.empty((wl.W, total), dtype=torch.float32, pin_memory=True)
    for w in range(wl.W):
        h_in[w] = torch.from_numpy(np.concatenate([WL.grad_np(wl, p, w) for p in range(wl.nparams)]))
    h_out = torch.full((wl.W * host.replica_stride,), -5.0, dtype=torch.float32, pin_memory=True)
    host.step(h_in, h_out)
    torch.cuda.synchronize()
    ref = O.run_workload(wl, orc, copy_back=False)
    out = h_out.numpy().reshape(wl.W, host.replica_stride)
    for b in range(plan.nbuckets):
        lo, n = int(plan.bucket_start[b]), int(plan.bucket_numel[b])
        k = n // wl.W
        for w in range(wl.W):
            assert_bits_equal(out[w, lo + w * k:lo + (w + 1) * k], ref["bucket"][b][w, w * k:(w + 1) * k],
                              f"bucket {b} shard {w}")
            assert np.all(out[w, lo:lo + w * k] == -5.0) and np.all(out[w, lo + (w + 1) * k:lo + n] == -5.0)
    host.close()


def test_wait_failure_path_reports_and_recovers(orc):
    """Failure detection without a fault: a bounded wait on a barrier nothing
    completes gives up after its limit and sets the device status word; with the
    arrival it completes cleanly; afterwards the context still reduces correctly."""
    assert D.ddp_device_status(reset=True) in (0, 1)
    D.ddp_wait_selftest(1, 1_000_000)
    assert D.ddp_device_status() == 0
    D.ddp_wait_selftest(0, 1_000_000)        # nothing arrives: gives up after ~1 ms
    assert D.ddp_device_status(reset=True) == 1
    assert D.ddp_device_status() == 0
    x = WL.bucket_np(4096 * 4 * 8, 8)
    t = torch.from_numpy(x).to(DEV)
    D.ddp_bucket_allreduce(t, t.shape[1], t.shape[1], 8, D.DDP_ALLREDUCE)
    want, _ = orc.ring(x.copy())
    assert_bits_equal(t.cpu().numpy(), want, "allreduce after the timed-out wait")
    assert D.ddp_device_status() == 0


def test_reducer_logging_data_after_iteration():
    """After one iteration the reducer reports the plan, the gradient-ready order it
    saw and the rebuilt bucket sizes of that order (twelve Linear layers: the DDP
    chapter's 4198400 / 29388800 / 16793600)."""
    wl = WL.Workload("linear12", WL.linear12(), 2, 0, 1, 25 << 20, 1 << 20, 1, 0, "dyadic12", 1.0, 78)
    sess = make_session(wl, device_grads(wl))
    assert "ready_order" not in sess.logging_data()
    sess.step()
    torch.cuda.synchronize()
    d = sess.logging_data()
    assert d["ready_order"] == list(range(wl.nparams - 1, -1, -1))
    assert d["rebuilt_bucket_sizes"] == [4198400, 29388800, 16793600]
    sess.close()


def test_host_front_end_bf16_megatron_reduce_scatter(orc):
    """bf16 gradients from pinned host memory, Megatron buckets (padded to W),
    reduce_scatter: each replica's shard of every bucket, bit for bit."""
    from allreduce_ddp_assign_gb300.session import HostBucketReducer

    wl = WL.Workload("linear12_bf16_rs", WL.linear12(), 4, 1, 2, 6 << 20, 6 << 20, 4, WL.BF16, "normal", 1e-2, 92)
    host = HostBucketReducer(wl.numels, [wl.dtype] * wl.nparams, wl.W, wl.mode, wl.order, wl.cap_bytes,
                             wl.first_cap_bytes, wl.pad_multiple, torch.bfloat16)
    plan = host.reducer.plan
    total = int(host.offs[-1])
    h_in = torch.empty((wl.W, total), dtype=torch.bfloat16, pin_memory=True)
    for w in range(wl.W):
        raw = np.concatenate([WL.grad_raw_np(wl, p, w) for p in range(wl.nparams)]).astype(np.uint16)
        h_in[w] = torch.from_numpy(raw.view(np.int16)).view(torch.bfloat16)
    h_out = torch.full((wl.W * host.replica_stride,), -5.0, dtype=torch.float32, pin_memory=True)
    host.step(h_in, h_out)
    torch.cuda.synchronize()
    ref = O.run_workload(wl, orc, copy_back=False)
    out = h_out.numpy().reshape(wl.W, host.replica_stride)
    assert plan.nbuckets > 1
    for b in range(plan.nbuckets):
        lo, n = int(plan.bucket_start[b]), int(plan.bucket_numel[b])
        k = n // wl.W
        for w in range(wl.W):
            assert_bits_equal(out[w, lo + w * k:lo + (w + 1) * k], ref["bucket"][b][w, w * k:(w + 1) * k],
                              f"bucket {b} shard {w}")
    host.close()


@pytest.mark.parametrize("coalesce", [False, True])
def test_reducer_mixed_dtypes_vs_oracle(orc, coalesce):
    """fp32, bf16 and fp16 gradients in one model: each dtype gets its own buckets and
    cap sequence (reading U6), every bucket is fp32 main_grad.  The reducer's plan
    equals the oracle's assignment and every bucket its ring result, bit for bit."""
    from allreduce_ddp_assign_gb300.session import BucketReducer

    numels = [3000, 64, 5000, 128, 7000, 257, 4097, 33, 6000, 90, 2500, 1]
    dtypes = [[D.DDP_F32, D.DDP_BF16, D.DDP_F16][p % 3] for p in range(len(numels))]
    W, cap, first = 4, 16 << 10, 8 << 10
    rng = np.random.default_rng(33)
    raw, dev = [], []
    for w in range(W):
        rr, dd = [], []
        for n, dt in zip(numels, dtypes):
            v = rng.standard_normal(n).astype(np.float32)
            if dt == D.DDP_BF16:
                bits = WL.f32_to_bf16_bits_np(v)
                rr.append(bits)
                dd.append(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV))
            elif dt == D.DDP_F16:
                h = v.astype(np.float16)
                rr.append(h.view(np.uint16))
                dd.append(torch.from_numpy(h).to(DEV))
            else:
                rr.append(v)
                dd.append(torch.from_numpy(v).to(DEV))
        raw.append(rr)
        dev.append(dd)
    sess = BucketReducer(numels, dtypes, W, D.DDP_ALLREDUCE, D.DDP_ORDER_REVERSE, cap, first, 1, dev,
                         coalesce=coalesce)
    sess.step()
    torch.cuda.synchronize()
    plan = orc.assign(numels, dtypes, cap, first, D.DDP_ORDER_REVERSE, 1, 1)
    assert sess.plan.nbuckets == plan["nbuckets"] > 3
    assert [int(x) for x in sess.plan.bucket_of] == [int(x) for x in plan["bucket_of"]]
    assert [int(x) for x in sess.plan.offset_of] == [int(x) for x in plan["offset_of"]]
    for b in range(plan["nbuckets"]):
        mem = plan["members"][b]
        assert len({dtypes[p] for p in mem}) == 1
        offs = [int(plan["offset_of"][p]) for p in mem]
        packed = orc.pack([[raw[w][p] for p in mem] for w in range(W)], offs, int(plan["bucket_numel"][b]),
                          [dtypes[p] for p in mem])
        want, _ = orc.ring(packed)
        assert_bits_equal(sess.plan.bucket_view(sess.main_grad, b).cpu().numpy(), want, f"bucket {b}")
    assert sess.issue_log() == [int(x) for x in plan["bucket_order"]]
    sess.close()
