"""The local-used bitmap all-reduce (find_unused_parameters) on the GPU against
the oracle, through the C ABI: counts and flags bit for bit, alone and inside the
reducer's schedule."""
import numpy as np
import pytest

import allreduce_ddp_assign_gb300 as D
import oracle as O
import workloads as WL
from gpu_util import assert_bits_equal

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")
GUARD = 32
SENT_COUNT, SENT_FLAG = -123456, 0xA5


def random_bitmap(rng, W, P, density=0.7):
    vals = np.array([1, 2, 0x80, 0xFF], np.uint8)
    keep = rng.random((W, P)) < density
    return np.where(keep, vals[rng.integers(0, 4, (W, P))], 0).astype(np.uint8)


def run_kernel(local, ld, off_in, off_out, want_count=True, want_flag=True):
    """Place local [W, P] in a device buffer with row stride ld at byte offset off_in,
    outputs at element offset off_out inside guarded buffers; run; return host copies."""
    W, P = local.shape
    host = np.zeros(off_in + W * ld + GUARD, np.uint8)
    for w in range(W):
        host[off_in + w * ld: off_in + w * ld + P] = local[w]
        host[off_in + w * ld + P: off_in + (w + 1) * ld] = 0xEE   # row padding must be ignored
    dev_in = torch.from_numpy(host).to(DEV)
    cnt = torch.full((GUARD + off_out + P + GUARD,), SENT_COUNT, dtype=torch.int32, device=DEV)
    flg = torch.full((GUARD + off_out + P + GUARD,), SENT_FLAG, dtype=torch.uint8, device=DEV)
    c_ptr = cnt.data_ptr() + 4 * (GUARD + off_out) if want_count else None
    f_ptr = flg.data_ptr() + (GUARD + off_out) if want_flag else None
    D.ddp_used_allreduce(dev_in.data_ptr() + off_in, ld, W, P, c_ptr, f_ptr)
    torch.cuda.synchronize()
    return cnt.cpu().numpy(), flg.cpu().numpy()


CASES = [(W, P) for W in (1, 2, 3, 4, 8, 16, 64) for P in (0, 1, 15, 16, 17, 161, 391, 4099)]


@pytest.mark.parametrize("layout", ["aligned", "ld_ragged", "base_misaligned", "out_misaligned"])
@pytest.mark.parametrize("W,P", CASES)
def test_used_allreduce_vs_oracle(orc, W, P, layout):
    rng = np.random.default_rng(97 * W + P)
    local = random_bitmap(rng, W, P)
    ld = {"aligned": -(-max(P, 1) // 16) * 16, "ld_ragged": P + 3, "base_misaligned": -(-max(P, 1) // 16) * 16,
          "out_misaligned": -(-max(P, 1) // 16) * 16}[layout]
    off_in = 5 if layout == "base_misaligned" else 0
    off_out = 3 if layout == "out_misaligned" else 0
    cnt, flg = run_kernel(local, ld, off_in, off_out)
    want_c, want_f = orc.used_allreduce(local)
    s = GUARD + off_out
    assert np.array_equal(cnt[s:s + P], want_c)
    assert np.array_equal(flg[s:s + P], want_f)
    assert np.all(cnt[:s] == SENT_COUNT) and np.all(cnt[s + P:] == SENT_COUNT)
    assert np.all(flg[:s] == SENT_FLAG) and np.all(flg[s + P:] == SENT_FLAG)


@pytest.mark.parametrize("which", ["count_only", "flag_only"])
def test_used_allreduce_single_output(orc, which):
    rng = np.random.default_rng(5)
    local = random_bitmap(rng, 8, 1000, 0.3)
    cnt, flg = run_kernel(local, 1008, 0, 0, want_count=which == "count_only", want_flag=which == "flag_only")
    want_c, want_f = orc.used_allreduce(local)
    if which == "count_only":
        assert np.array_equal(cnt[GUARD:GUARD + 1000], want_c) and np.all(flg == SENT_FLAG)
    else:
        assert np.array_equal(flg[GUARD:GUARD + 1000], want_f) and np.all(cnt == SENT_COUNT)


def test_used_allreduce_large_sampled(orc):
    """16M parameters x 8 replicas (the bandwidth measurement's size): sampled columns
    against the oracle (columns are independent), every flag against its count."""
    W, P = 8, 1 << 24
    g = torch.Generator(device=DEV)
    g.manual_seed(11)
    local = (torch.rand((W, P), generator=g, device=DEV) < 0.02).to(torch.uint8)
    cnt = torch.empty(P, dtype=torch.int32, device=DEV)
    flg = torch.empty(P, dtype=torch.uint8, device=DEV)
    D.ddp_used_allreduce(local, P, W, P, cnt, flg)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    cols = np.unique(np.concatenate([rng.integers(0, P, 4000), [0, P - 1]]))
    sub = local[:, torch.from_numpy(cols).to(DEV)].cpu().numpy()
    want_c, want_f = orc.used_allreduce(sub)
    assert np.array_equal(cnt[torch.from_numpy(cols).to(DEV)].cpu().numpy(), want_c)
    assert np.array_equal(flg[torch.from_numpy(cols).to(DEV)].cpu().numpy(), want_f)
    assert torch.equal(flg.to(torch.int32), (cnt > 0).to(torch.int32))
    assert int(cnt.max()) <= W


# ---------------------------------------------------------------------------
# inside the reducer: find_unused_parameters on BERT-large
# ---------------------------------------------------------------------------
def _outs(wl, fill):
    return [[torch.full((n,), fill, dtype=torch.float32, device=DEV) for n in wl.numels] for _ in range(wl.W)]


@pytest.mark.parametrize("fused,coalesce", [(True, False), (True, True), (False, False)])
def test_reducer_find_unused_bert_vs_oracle(orc, fused, coalesce):
    """BERT-large, W = 4, layer 11 unused everywhere and 5% of the other (replica,
    parameter) pairs unused locally: the reducer uploads the bitmap, all-reduces it
    on the side stream, marks the globally unused parameters itself; results match
    the oracle's path bit for bit, globally unused gradients stay untouched."""
    from allreduce_ddp_assign_gb300.session import BucketReducer

    wl = WL.c6_bert_find_unused()
    used = WL.local_used_np(wl)
    grads = [[WL.grad_torch(wl, p, w, 0, DEV) for p in range(wl.nparams)] for w in range(wl.W)]
    outs = _outs(wl, 7.0)
    sess = BucketReducer(wl.numels, None, wl.W, wl.mode, wl.order, wl.cap_bytes, wl.first_cap_bytes,
                         wl.pad_multiple, grads, used=used, grads_out=outs, fused=fused, coalesce=coalesce)
    sess.step()
    torch.cuda.synchronize()
    ref = O.run_workload(wl, orc)
    want_c, want_f = orc.used_allreduce(used)
    assert np.array_equal(sess.global_count_dev.cpu().numpy()[:wl.nparams], want_c)
    assert np.array_equal(sess.global_used_dev.cpu().numpy()[:wl.nparams], want_f)
    assert np.array_equal(sess.local_used_dev.cpu().numpy()[:wl.W * wl.nparams].reshape(wl.W, wl.nparams),
                          (used != 0).astype(np.uint8))
    assert sorted(sess.issue_log()) == list(range(sess.plan.nbuckets))
    for w in range(wl.W):
        for p in range(wl.nparams):
            got = outs[w][p].cpu().numpy()
            if ref["out"][w][p] is None:
                assert np.all(got == 7.0), f"globally unused parameter {p} was written"
            else:
                assert_bits_equal(got, ref["out"][w][p], f"w={w} p={p}")
    sess.close()


def test_reducer_find_unused_bitmap_changes_between_iterations(orc):
    """Two iterations with different bitmaps through one reducer: each matches the
    oracle for its own bitmap (the host copy is refreshed before each prepare)."""
    from allreduce_ddp_assign_gb300.session import BucketReducer

    wl = WL.c1_mlp()
    grads = [[WL.grad_torch(wl, p, w, 0, DEV) for p in range(wl.nparams)] for w in range(wl.W)]
    outs = _outs(wl, -3.0)
    u1 = np.ones((wl.W, wl.nparams), np.uint8)
    u1[:, 1] = 0
    u1[2, 4] = 0
    u2 = np.ones((wl.W, wl.nparams), np.uint8)
    u2[0, 1] = 0
    u2[:, 5] = 0
    sess = BucketReducer(wl.numels, None, wl.W, wl.mode, wl.order, wl.cap_bytes, wl.first_cap_bytes, 1, grads,
                         used=u1, grads_out=outs, fused=True)
    for used in (u1, u2):
        for w in range(wl.W):
            for p in range(wl.nparams):
                outs[w][p].fill_(-3.0)
        sess.set_local_used(used)
        sess.step()
        torch.cuda.synchronize()
        plan = orc.assign(wl.numels, None, wl.cap_bytes, wl.first_cap_bytes, wl.order)
        _, glob = orc.used_allreduce(used)
        for b in range(plan["nbuckets"]):
            mem = plan["members"][b]
            offs = [int(plan["offset_of"][p]) for p in mem]
            raw = [[WL.grad_raw_np(wl, p, w) for p in mem] for w in range(wl.W)]
            buf = orc.pack(raw, offs, int(plan["bucket_numel"][b]), used=used[:, mem])
            buf, _ = orc.ring(buf)
            exp = orc.unpack(buf, offs, [wl.numels[p] for p in mem], 0, glob[mem],
                             outs=[[np.full(wl.numels[p], -3.0, np.float32) for p in mem] for _ in range(wl.W)])
            for w in range(wl.W):
                for j, p in enumerate(mem):
                    assert_bits_equal(outs[w][p].cpu().numpy(), exp[w][j], f"w={w} p={p}")
    sess.close()
