"""Pins of the PowerSGD oracle (``oracle/powersgd.py``), each reached by another route.

Each ``pin_*`` takes the loaded C oracle and a PowerSGD oracle module and raises
AssertionError on a mismatch.  The routes: the page's printed compression ratio;
the projector onto span(sum_w M_w Q) from an SVD, and the positive-diagonal
orthonormal basis from a Cholesky factor (not a QR); exact reconstruction of
low-rank gradients; conservation under error feedback; two steps of the power
iteration written as one; exact rational means for the 1-D tensors and the
warm-up iterations; the clamped rank making the projector the identity.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def _dyadic(rng, shape, k=4096):
    return (rng.integers(-k, k + 1, shape) / 4096.0).astype(np.float32)


def _bucket(mats, W):
    """mats[w][t] arrays -> ([W, numel] fp32, offsets, shapes)."""
    shapes = [m.shape for m in mats[0]]
    offs, pos = [], 0
    for s in shapes:
        offs.append(pos)
        pos += int(np.prod(s))
    b = np.zeros((W, pos), np.float32)
    for w in range(W):
        for t, m in enumerate(mats[w]):
            b[w, offs[t]:offs[t] + m.size] = np.asarray(m, np.float32).reshape(-1)
    return b, offs, shapes


def _projector(a):
    """Orthogonal projector onto the column space of a (full column rank) via SVD."""
    u, s, _ = np.linalg.svd(a, full_matrices=False)
    return u @ u.T


def _chol_basis(p):
    """P R^{-1} with R^T R = P^T P (Cholesky): the orthonormal basis whose
    triangle has a positive diagonal, without a QR."""
    lo = np.linalg.cholesky(p.T @ p)
    return np.linalg.solve(lo, p.T).T


def pin_psgd_compression_ratio(orc, psgd):
    """DDP chapter 17.27: M = N = 4096 at rank 4 sends (M+N) R elements instead of
    M N, a ratio of 512."""
    assert psgd.comm_elements(4096, 4096, 4) == 2 * 4096 * 4
    assert 4096 * 4096 // psgd.comm_elements(4096, 4096, 4) == 512
    assert psgd.effective_rank(3, 100, 4) == 3 and psgd.effective_rank(100, 2, 4) == 2
    assert psgd.matrix_view((64, 3, 7, 7)) == (64, 147) and psgd.matrix_view((10,)) is None


def pin_psgd_projection_closed_form(orc, psgd):
    """One step without error feedback: every rank ends with Pi M_bar, Pi the
    projector onto span(sum_w G_w Q0) (SVD), and the kept Q equals M_bar^T B with
    B the positive-diagonal basis from a Cholesky factor."""
    rng = np.random.default_rng(51)
    W, m, n, r = 3, 7, 5, 2
    for trial in range(8):   # columns of either sign in P
        g = [[rng.standard_normal((m, n)).astype(np.float32)] for _ in range(W)]
        q0 = rng.standard_normal((n, r))
        b, offs, shapes = _bucket(g, W)
        st = psgd.make_state(shapes, W, r, [q0], error_feedback=False)
        out = psgd.step(st, b, offs, orc)
        gm = [x[0].astype(np.float64) for x in g]
        mbar = sum(gm) / W
        p = sum(x @ q0 for x in gm)
        want = _projector(p) @ mbar
        for w in range(W):
            assert np.allclose(out[w].reshape(m, n), want, rtol=0, atol=1e-12)
        assert np.allclose(st.q[0], mbar.T @ _chol_basis(p), rtol=0, atol=1e-12)


def pin_psgd_low_rank_exact(orc, psgd):
    """Identical gradients of rank <= R on every rank are reconstructed exactly and
    leave no error."""
    rng = np.random.default_rng(52)
    W, m, n, r = 4, 12, 9, 3
    a, c = _dyadic(rng, (m, 2)), _dyadic(rng, (n, 2))
    gm = (a.astype(np.float64) @ c.astype(np.float64).T).astype(np.float32)
    b, offs, shapes = _bucket([[gm] for _ in range(W)], W)
    st = psgd.make_state(shapes, W, r, [rng.standard_normal((n, r))])
    out = psgd.step(st, b, offs, orc)
    for w in range(W):
        assert np.allclose(out[w].reshape(m, n), gm, rtol=0, atol=1e-12)
        assert np.abs(st.error[w][0]).max() < 1e-12


def pin_psgd_error_feedback(orc, psgd):
    """Error feedback loses nothing: new error + output = gradient + old error on
    every rank; a following step with zero gradients transmits the projection of
    the mean error (the error is fed back)."""
    rng = np.random.default_rng(53)
    W, m, n, r = 2, 8, 6, 1
    g = [[rng.standard_normal((m, n)).astype(np.float32)] for _ in range(W)]
    b, offs, shapes = _bucket(g, W)
    st = psgd.make_state(shapes, W, r, [rng.standard_normal((n, r))])
    out = psgd.step(st, b, offs, orc)
    for w in range(W):
        assert np.allclose(st.error[w][0] + out[w].reshape(m, n), g[w][0], rtol=0, atol=1e-12)
    e = [st.error[w][0].copy() for w in range(W)]
    q1 = st.q[0].copy()
    out2 = psgd.step(st, np.zeros_like(b), offs, orc)
    want = _projector(sum(x @ q1 for x in e)) @ (sum(e) / W)
    assert np.abs(want).max() > 1e-3
    for w in range(W):
        assert np.allclose(out2[w].reshape(m, n), want, rtol=0, atol=1e-12)


def pin_psgd_warm_start_power_iteration(orc, psgd):
    """Without error feedback and with the same gradient G on every rank, two steps
    are two power iterations: the second output is the projection of G onto
    span(G G^T G Q0)."""
    rng = np.random.default_rng(54)
    W, m, n, r = 3, 10, 8, 2
    gm = rng.standard_normal((m, n)).astype(np.float32)
    b, offs, shapes = _bucket([[gm] for _ in range(W)], W)
    q0 = rng.standard_normal((n, r))
    st = psgd.make_state(shapes, W, r, [q0], error_feedback=False)
    psgd.step(st, b, offs, orc)
    out2 = psgd.step(st, b, offs, orc)
    g = gm.astype(np.float64)
    want = _projector(g @ g.T @ g @ q0) @ g
    for w in range(W):
        assert np.allclose(out2[w].reshape(m, n), want, rtol=0, atol=1e-10)


def pin_psgd_vectors_and_warmup(orc, psgd):
    """1-D tensors take the plain mean; the first start_iter iterations take the
    plain mean of the whole bucket and leave Q and the error alone (dyadic inputs:
    exact rational means)."""
    rng = np.random.default_rng(55)
    W = 4
    mats = [[_dyadic(rng, (6,)), _dyadic(rng, (5, 4)), _dyadic(rng, (3,))] for _ in range(W)]
    b, offs, shapes = _bucket(mats, W)
    q0 = rng.standard_normal((4, 2))
    st = psgd.make_state(shapes, W, 2, [None, q0, None], start_iter=1)
    out = psgd.step(st, b, offs, orc)
    exact = [sum(Fraction(float(b[w, e])) for w in range(W)) / W for e in range(b.shape[1])]
    for w in range(W):
        assert [Fraction(float(x)) for x in out[w]] == exact
    assert np.array_equal(st.q[1], q0) and not np.any(st.error[0][1])
    out2 = psgd.step(st, b, offs, orc)
    for t in (0, 2):
        lo, k = offs[t], int(np.prod(shapes[t]))
        for w in range(W):
            assert [Fraction(float(x)) for x in out2[w, lo:lo + k]] == exact[lo:lo + k]
    lo = offs[1]
    assert not np.allclose(out2[0, lo:lo + 20], np.array([float(x) for x in exact[lo:lo + 20]]))


def pin_psgd_rank_clamped_identity(orc, psgd):
    """With M <= R the basis spans everything: the output is the plain mean."""
    rng = np.random.default_rng(56)
    W, m, n, r = 3, 2, 6, 4
    g = [[_dyadic(rng, (m, n))] for _ in range(W)]
    b, offs, shapes = _bucket(g, W)
    st = psgd.make_state(shapes, W, r, [rng.standard_normal((n, 2))], error_feedback=False)
    out = psgd.step(st, b, offs, orc)
    mbar = sum(x[0].astype(np.float64) for x in g) / W
    for w in range(W):
        assert np.allclose(out[w].reshape(m, n), mbar, rtol=0, atol=1e-12)


def pin_psgd_zero_gradient(orc, psgd):
    """All-zero gradients give zero output and zero error, no NaN."""
    W, m, n, r = 2, 5, 4, 2
    b, offs, shapes = _bucket([[np.zeros((m, n), np.float32)] for _ in range(W)], W)
    st = psgd.make_state(shapes, W, r, [np.ones((n, r))])
    out = psgd.step(st, b, offs, orc)
    assert np.all(out == 0) and not np.any(st.error[0][0]) and not np.any(np.isnan(st.q[0]))


def pin_psgd_product_condition(orc, psgd):
    """The tolerance diagnostic: exactly 1 without cancellation (nonnegative
    factors), the hand-computed ratio on a 1 x 2 times 2 x 1 product with one
    cancelling pair, and the max over the P and Q products after a step."""
    rng = np.random.default_rng(57)
    a = [np.abs(rng.standard_normal((4, 6))) for _ in range(3)]
    b = np.abs(rng.standard_normal((6, 2)))
    assert psgd.product_condition(a, b) == 1.0
    # [1, -0.75] . [1, 1]: terms 1 and -0.75, sum 0.25 -> ratio 1.75 / 0.25 = 7
    assert psgd.product_condition([np.array([[1.0, -0.75]])], np.array([[1.0], [1.0]])) == 7.0
    assert psgd.product_condition([np.zeros((2, 2))], np.ones((2, 1))) == 1.0
    W, m, n, r = 2, 3, 5, 2
    g = [[_dyadic(rng, (m, n))] for _ in range(W)]
    bk, offs, shapes = _bucket(g, W)
    q0 = rng.standard_normal((n, r))
    st = psgd.make_state(shapes, W, r, [q0], error_feedback=False)
    psgd.step(st, bk, offs, orc)
    mw = [x[0].astype(np.float64) for x in g]
    p = sum(x @ q0 for x in mw)
    basis = _chol_basis(p)
    want = max(np.abs(sum(np.abs(x) @ np.abs(q0) for x in mw)).max() / np.abs(p).max(),
               np.abs(sum(np.abs(x.T) @ np.abs(basis) for x in mw)).max() / np.abs(sum(x.T @ basis for x in mw)).max(),
               1.0)
    assert abs(st.amp[0] - want) <= 1e-9 * want


POWERSGD_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_psgd_")]
