"""The PowerSGD hook on the GPU against the oracle (``oracle/powersgd.py``).

1-D tensors and the plain warm-up iterations are compared bit for bit (the ring's
arithmetic).  Compressed tensors are compared with the fp64 oracle in the max
norm relative to max |output| (Q: max |Q|; error buffer: the larger of max
|output| and max |error|), within

    TOL_OUT_Q * k * u * kappa(P) * amp   for the output and Q,
    TOL_ERR   * k * u * kappa(P) * amp   for the error-feedback buffer,

u = 2^-24, k = compressed iterations so far (each one's error reaches the next
through the warm-started Q and the error buffer), kappa(P) = the condition
number of the summed P (the orthonormalisation amplifies the error of P by
about that much), amp = the larger product condition of P = sum_w M_w Q and
Q = sum_w M_w^T P (max |sum |A||B|| / max |sum A B|, at least 1), both from the
oracle.  A float product is off by at most gamma_n |A||B| entrywise, so amp
carries the cancellation inside the products: on short wide matrices
(5 x 4096 at rank 1) it reaches the tens and an fp32 emulation on the CPU
(numpy products and Gram-Schmidt) misses the fp64 result by as much as the
kernels do.  Measured over every case below and the ResNet-50 buckets, the
worst output error is 4.4 k u kappa amp, the worst Q error 6.1 and the worst
error-buffer error 2.9; the constants sit at least a factor 2.6 above them, so
a lost term or a half-precision intermediate, hundreds of these units, fails.
"""
import numpy as np
import pytest

import allreduce_ddp_assign_gb300 as D
from oracle import powersgd as OP
import workloads as WL
from gpu_util import assert_bits_equal

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")
U = 2.0 ** -24
TOL_OUT_Q = 16.0   # output and Q: k * u * kappa(P) * amp units (worst measured 4.4 and 6.1)
TOL_ERR = 8.0      # error-feedback buffer (worst measured 2.9)

SHAPES = [(64, 3, 7, 7), (8,), (256, 64), (3, 5), (1, 16), (10,), (40, 36), (2048,), (130, 2, 3)]


def layout(shapes, pad_to=1):
    offs, pos = [], 0
    for s in shapes:
        pos = -(-pos // pad_to) * pad_to
        offs.append(pos)
        pos += int(np.prod(s))
    return offs, pos + 3   # three elements of padding at the end


def make_bucket(rng, shapes, W, offs, numel, stride):
    host = np.zeros((W, stride), np.float32)
    for w in range(W):
        for s, o in zip(shapes, offs):
            k = int(np.prod(s))
            host[w, o:o + k] = rng.standard_normal(k).astype(np.float32)
        host[w, numel - 3:numel] = rng.standard_normal(3).astype(np.float32)
    return host


def q0_of(rng_seed, shapes, rank):
    out = []
    for t, s in enumerate(shapes):
        mv = OP.matrix_view(s)
        out.append(None if mv is None else WL.powersgd_q0_np(rng_seed, t, mv[1], OP.effective_rank(mv[0], mv[1], rank)))
    return out


def check_against(state, want, got, shapes, offs, it, what):
    """Vectors bit for bit, matrices within TOL_OUT_Q k u kappa(P) of max |output|."""
    W = want.shape[0]
    for t, s in enumerate(shapes):
        lo, k = offs[t], int(np.prod(s))
        mv = OP.matrix_view(s)
        if mv is None:
            assert_bits_equal(got[:, lo:lo + k], want[:, lo:lo + k].astype(np.float32), f"{what}: 1-D tensor {t}")
            continue
        tol = TOL_OUT_Q * it * U * max(state.cond.get(t, 1.0), 1.0) * state.amp.get(t, 1.0)
        ref = want[:, lo:lo + k]
        scale = max(np.abs(ref).max(), 1e-30)
        err = np.abs(got[:, lo:lo + k].astype(np.float64) - ref).max() / scale
        assert err <= tol, f"{what}: tensor {t} {s}: max error {err:.3e} of max |out|, tolerance {tol:.3e}"
        for w in range(1, W):
            assert np.array_equal(got[w, lo:lo + k], got[0, lo:lo + k]), f"{what}: replicas differ on tensor {t}"


CASES = [(W, rank, ef, aligned) for W in (1, 2, 3, 8) for rank in (1, 3, 4, 8) for ef in (0, 1)
         for aligned in (True, False)]


@pytest.mark.parametrize("W,rank,ef,aligned", CASES)
def test_powersgd_bucket_vs_oracle(orc, W, rank, ef, aligned):
    """Three iterations (the first one plain when W is odd) on a bucket mixing 1-D
    tensors, a conv weight with N = 147 (unaligned path), a 256 x 64 matrix (16-byte
    path), rank-clamped 3 x 5 and 1 x 16 matrices and a 130 x 6 matrix."""
    rng = np.random.default_rng(1000 * W + 10 * rank + ef)
    offs, numel = layout(SHAPES, pad_to=4 if aligned else 1)
    stride = numel + (4 - numel % 4) % 4 + (0 if aligned else 1)
    start_iter = W % 2
    q0 = q0_of(77, SHAPES, rank)
    st = OP.make_state(SHAPES, W, rank, q0, error_feedback=bool(ef), start_iter=start_iter)
    from allreduce_ddp_assign_gb300.powersgd import PowerSGDBucket

    hook = PowerSGDBucket(W, rank, offs, [int(np.prod(s)) for s in SHAPES], SHAPES, numel,
                          lambda k, n, r: q0[k], error_feedback=bool(ef), start_iter=start_iter)
    for it in range(1, 4):
        host = make_bucket(rng, SHAPES, W, offs, numel, stride)
        dev = torch.from_numpy(host).to(DEV)
        want = OP.step(st, host[:, :numel], offs, orc)
        hook.reduce(dev, stride)
        torch.cuda.synchronize()
        got = dev.cpu().numpy()
        if it <= start_iter:
            assert_bits_equal(got[:, :numel], want.astype(np.float32), f"plain iteration {it}")
            continue
        check_against(st, want, got[:, :numel], SHAPES, offs, it - start_iter, f"iteration {it}")
        # padding is left alone once compression starts
        assert_bits_equal(got[:, numel - 3:numel], host[:, numel - 3:numel], "padding")
        for t, s in enumerate(SHAPES):
            mv = OP.matrix_view(s)
            if mv is None:
                continue
            qg = hook.q(t).cpu().numpy().astype(np.float64)
            unit = (it - start_iter) * U * max(st.cond[t], 1.0) * st.amp[t]
            assert np.abs(qg - st.q[t]).max() <= TOL_OUT_Q * unit * max(np.abs(st.q[t]).max(), 1e-30), f"Q of tensor {t}"
            if ef:
                for w in range(W):
                    eg = hook.error_of(w, offs[t], mv[0] * mv[1]).cpu().numpy().astype(np.float64)
                    er = st.error[w][t].reshape(-1)
                    scale = max(np.abs(want[w, offs[t]:offs[t] + mv[0] * mv[1]]).max(), np.abs(er).max(), 1e-30)
                    assert np.abs(eg - er).max() <= TOL_ERR * unit * scale, f"error of tensor {t} replica {w}"
    assert hook.iteration == 3
    hook.close()


LONG_SHAPES = [(24, 256), (8,), (3, 512), (70, 128), (33, 1280), (5, 4096), (17, 384)]
LONG_CASES = [(W, rank, ef, aligned) for W in (1, 2, 4, 8) for rank in (1, 4, 8) for ef in (0, 1)
             for aligned in (True, False)]


@pytest.mark.parametrize("W,rank,ef,aligned", LONG_CASES)
def test_powersgd_long_rows_vs_oracle(orc, W, rank, ef, aligned):
    """Row-aligned matrices with long rows: 128-element multiples on 16-byte
    boundaries (or one element off, misaligned), from square-ish 24 x 256 to short
    wide 3 x 512 and 5 x 4096, whose P products cancel strongly (amp in the tens to
    the hundreds), with one-row, rank-clamped and odd row counts.  Three
    iterations, the same checks and tolerance as the other bucket cases."""
    rng = np.random.default_rng(7000 + 100 * W + 10 * rank + ef)
    shapes = LONG_SHAPES
    offs, numel = layout(shapes, pad_to=4)
    stride = numel + (4 - numel % 4) % 4 + (0 if aligned else 1)
    q0 = q0_of(91, shapes, rank)
    st = OP.make_state(shapes, W, rank, q0, error_feedback=bool(ef), start_iter=0)
    from allreduce_ddp_assign_gb300.powersgd import PowerSGDBucket

    hook = PowerSGDBucket(W, rank, offs, [int(np.prod(s)) for s in shapes], shapes, numel,
                          lambda k, n, r: q0[k], error_feedback=bool(ef), start_iter=0)
    for it in range(1, 4):
        host = make_bucket(rng, shapes, W, offs, numel, stride)
        dev = torch.from_numpy(host).to(DEV)
        want = OP.step(st, host[:, :numel], offs, orc)
        hook.reduce(dev, stride)
        torch.cuda.synchronize()
        got = dev.cpu().numpy()
        check_against(st, want, got[:, :numel], shapes, offs, it, f"iteration {it}")
        for t, s in enumerate(shapes):
            mv = OP.matrix_view(s)
            if mv is None:
                continue
            qg = hook.q(t).cpu().numpy().astype(np.float64)
            unit = it * U * max(st.cond[t], 1.0) * st.amp[t]
            assert np.abs(qg - st.q[t]).max() <= TOL_OUT_Q * unit * max(np.abs(st.q[t]).max(), 1e-30), f"Q of tensor {t}"
            if ef:
                for w in range(W):
                    eg = hook.error_of(w, offs[t], mv[0] * mv[1]).cpu().numpy().astype(np.float64)
                    er = st.error[w][t].reshape(-1)
                    scale = max(np.abs(want[w, offs[t]:offs[t] + mv[0] * mv[1]]).max(), np.abs(er).max(), 1e-30)
                    assert np.abs(eg - er).max() <= TOL_ERR * unit * scale, f"error of tensor {t} replica {w}"
    hook.close()
    assert D.ddp_device_status(reset=True) == 0


SPLIT_SHAPES = [(7, 1030), (3,), (2, 3001), (9, 2052), (4, 1025), (6, 4104)]
SPLIT_CASES = [(W, rank, ef, aligned) for W in (2, 5) for rank in (1, 3, 8) for ef in (0, 1)
               for aligned in (True, False)]


@pytest.mark.parametrize("W,rank,ef,aligned", SPLIT_CASES)
def test_powersgd_column_splits_vs_oracle(orc, W, rank, ef, aligned):
    """Rows longer than one P tile's column split: lengths that are not multiples of 4
    (the scalar path), of 128, or of the split count, so the splits end mid-block and
    the last one is short (2052 and 4104 columns take the 16-byte path when aligned);
    rank 8 doubles the split width.  Three iterations against the oracle with the same
    checks and tolerance as the other bucket cases."""
    rng = np.random.default_rng(9100 + 100 * W + 10 * rank + ef)
    shapes = SPLIT_SHAPES
    offs, numel = layout(shapes, pad_to=4 if aligned else 1)
    stride = numel + (4 - numel % 4) % 4 + (0 if aligned else 1)
    q0 = q0_of(93, shapes, rank)
    st = OP.make_state(shapes, W, rank, q0, error_feedback=bool(ef), start_iter=0)
    from allreduce_ddp_assign_gb300.powersgd import PowerSGDBucket

    hook = PowerSGDBucket(W, rank, offs, [int(np.prod(s)) for s in shapes], shapes, numel,
                          lambda k, n, r: q0[k], error_feedback=bool(ef), start_iter=0)
    for it in range(1, 4):
        host = make_bucket(rng, shapes, W, offs, numel, stride)
        dev = torch.from_numpy(host).to(DEV)
        want = OP.step(st, host[:, :numel], offs, orc)
        hook.reduce(dev, stride)
        torch.cuda.synchronize()
        got = dev.cpu().numpy()
        check_against(st, want, got[:, :numel], shapes, offs, it, f"iteration {it}")
        for t, s in enumerate(shapes):
            mv = OP.matrix_view(s)
            if mv is None:
                continue
            qg = hook.q(t).cpu().numpy().astype(np.float64)
            unit = it * U * max(st.cond[t], 1.0) * st.amp[t]
            assert np.abs(qg - st.q[t]).max() <= TOL_OUT_Q * unit * max(np.abs(st.q[t]).max(), 1e-30), f"Q of tensor {t}"
            if ef:
                for w in range(W):
                    eg = hook.error_of(w, offs[t], mv[0] * mv[1]).cpu().numpy().astype(np.float64)
                    er = st.error[w][t].reshape(-1)
                    scale = max(np.abs(want[w, offs[t]:offs[t] + mv[0] * mv[1]]).max(), np.abs(er).max(), 1e-30)
                    assert np.abs(eg - er).max() <= TOL_ERR * unit * scale, f"error of tensor {t} replica {w}"
    hook.close()


def test_powersgd_zero_gradients_stay_finite(orc):
    W, rank = 4, 2
    shapes = [(32, 32), (5,)]
    offs, numel = layout(shapes, 4)
    q0 = q0_of(5, shapes, rank)
    from allreduce_ddp_assign_gb300.powersgd import PowerSGDBucket

    hook = PowerSGDBucket(W, rank, offs, [int(np.prod(s)) for s in shapes], shapes, numel, lambda k, n, r: q0[k])
    dev = torch.zeros((W, numel), dtype=torch.float32, device=DEV)
    hook.reduce(dev, numel)
    torch.cuda.synchronize()
    assert torch.all(dev == 0)
    assert torch.all(torch.isfinite(hook.q_state))
    hook.close()


# ---------------------------------------------------------------------------
# through the reducer: ResNet-50, W = 8, rank 4, every bucket hooked
# ---------------------------------------------------------------------------
def _resnet_session(wl, rank, ef):
    from allreduce_ddp_assign_gb300.session import BucketReducer

    grads = [[WL.grad_torch(wl, p, w, 0, DEV) for p in range(wl.nparams)] for w in range(wl.W)]
    cfg = dict(rank=rank, shapes=wl.shapes, error_feedback=ef,
               q0=lambda p, n, r: WL.powersgd_q0_np(wl.seed, p, n, r))
    sess = BucketReducer(wl.numels, None, wl.W, wl.mode, wl.order, wl.cap_bytes, wl.first_cap_bytes,
                         wl.pad_multiple, grads, powersgd=cfg)
    return sess, grads


def _check_reducer_buckets(orc, buckets, iters=2, rank=4):
    wl = WL.c7_resnet50_powersgd(rank)
    sess, grads = _resnet_session(wl, rank, True)
    plan = sess.plan
    states = {}
    for b in buckets:
        mem = plan.members[b]
        q0 = []
        for p in mem:
            mv = OP.matrix_view(wl.shapes[p])
            q0.append(None if mv is None else WL.powersgd_q0_np(wl.seed, p, mv[1], OP.effective_rank(mv[0], mv[1], rank)))
        states[b] = OP.make_state([wl.shapes[p] for p in mem], wl.W, rank, q0)
    for it in range(iters):
        if it > 0:
            for w in range(wl.W):
                for p in range(wl.nparams):
                    grads[w][p].copy_(WL.grad_torch(wl, p, w, it, DEV))
        sess.step()
        torch.cuda.synchronize()
        for b in buckets:
            mem = plan.members[b]
            offs = [int(plan.offset_of[p]) for p in mem]
            numel = int(plan.bucket_numel[b])
            raw = [[WL.grad_raw_np(wl, p, w, it) for p in mem] for w in range(wl.W)]
            packed = orc.pack(raw, offs, numel)
            want = OP.step(states[b], packed, offs, orc)
            got = plan.bucket_view(sess.main_grad, b).cpu().numpy()
            check_against(states[b], want, got, [wl.shapes[p] for p in mem], offs, it + 1, f"bucket {b} iteration {it}")
    assert sess.issue_log() == list(range(plan.nbuckets))
    sess.close()


def test_reducer_powersgd_resnet50_first_bucket(orc):
    """Bucket 0 (the 1 MiB-cap bucket: fc weight and bias) over two iterations."""
    _check_reducer_buckets(orc, [0])


@pytest.mark.slow
def test_reducer_powersgd_resnet50_all_buckets(orc):
    """Every bucket of ResNet-50 at full size, two iterations, rank 4."""
    _check_reducer_buckets(orc, list(range(5)))
