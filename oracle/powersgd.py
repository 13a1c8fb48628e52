"""PowerSGD compression of one gradient bucket, as the DDP communication hook does it.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use this module; the library never does.  It shares no code
with the CUDA path.  Plain numpy in float64; the 1-D tensors go through the
ring of ``oracle.c`` (fp32, bit-exact reference).

Source: "DDP: ring AllReduce and gradient buckets" (PyTorch internals book,
chapter 17), section 17.27 (the hook's steps: P = G Q, all-reduce P,
orthogonalise P by QR, Q = G^T P, all-reduce Q, reconstruct P Q^T; each tensor
of two or more dimensions is decomposed on its own, 1-D tensors take a plain
all-reduce; error feedback, a warm-started Q, plain all-reduce for the first
start_powerSGD_iter iterations and a division by the world size complete it)
and section 17.9 (the hook list and the compression ratios).

Per bucket and iteration, with W ranks, rank R:

* before ``start_iter`` iterations: the plain ring all-reduce (mean) of the
  whole bucket; error and Q untouched;
* afterwards, 1-D tensors: the ring mean of their concatenation (bucket order);
* every tensor of two or more dimensions, viewed as M x N (shape[0] x the
  product of the rest), with R' = min(R, M, N), in the page's order:
    0. error feedback: M_w = G_w + E_w   (E_w = 0 without error feedback)
    1. P_w = M_w Q                       (Q: N x R', shared by the ranks)
    2. P = sum_w P_w                     (all-reduce)
    3. P = orthonormal basis of P's columns: the QR factor whose triangle has
       a positive diagonal (the unique one for full-rank P); a column whose
       diagonal entry is exactly 0 becomes 0
    4. Q_w = M_w^T P
    5. Q = (sum_w Q_w) / W               (all-reduce, divided by the world size)
    6. every rank's tensor becomes P Q^T; E_w = M_w - P Q^T; Q is kept as the
       next iteration's start (warm start).

Readings taken where the page leaves a step open: the matrix view is
shape[0] x rest (the page's reshape(M, N) of one tensor); R is clamped to
min(M, N) so that the QR is defined; the initial Q (the page's torch.randn) is
an input, so that both sides see the same numbers; padding of the bucket is
left alone once compression starts.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def matrix_view(shape) -> tuple[int, int] | None:
    """(M, N) of a tensor of two or more dimensions, None for a 1-D (or 0-D) one."""
    shape = tuple(int(s) for s in shape)
    if len(shape) < 2:
        return None
    n = 1
    for s in shape[1:]:
        n *= s
    return shape[0], n


def effective_rank(m: int, n: int, rank: int) -> int:
    return min(rank, m, n)


def comm_elements(m: int, n: int, rank: int) -> int:
    """Elements one rank all-reduces for one M x N tensor: P (M x R') and Q (N x R')."""
    r = effective_rank(m, n, rank)
    return (m + n) * r


@dataclass
class State:
    """The hook's state for one bucket: per-tensor Q (warm start), per-rank error."""
    shapes: list
    W: int
    rank: int
    q: list                      # per tensor: N x R' float64 (None for 1-D tensors)
    error_feedback: bool = True
    start_iter: int = 0
    iter: int = 0
    error: list = field(default_factory=list)   # error[w][t]: M x N float64 (None for 1-D)
    cond: dict = field(default_factory=dict)    # per tensor: 2-norm condition number of the last P (for tolerances)
    amp: dict = field(default_factory=dict)     # per tensor: product condition of the last step (for tolerances)

    def __post_init__(self):
        if not self.error:
            self.error = [[None if matrix_view(s) is None else np.zeros(matrix_view(s), np.float64)
                           for s in self.shapes] for _ in range(self.W)]


def make_state(shapes, W: int, rank: int, q0, error_feedback: bool = True, start_iter: int = 0) -> State:
    """q0[t]: the initial Q of tensor t (N x R', any float type), None for 1-D tensors."""
    q = [None if q0[t] is None else np.array(q0[t], dtype=np.float64) for t in range(len(shapes))]
    for t, s in enumerate(shapes):
        mv = matrix_view(s)
        if mv is not None and q[t].shape != (mv[1], effective_rank(mv[0], mv[1], rank)):
            raise ValueError(f"q0[{t}] has shape {q[t].shape}")
    return State(list(shapes), W, rank, q, error_feedback, start_iter)


def _orthonormal(p: np.ndarray) -> np.ndarray:
    qm, rm = np.linalg.qr(p)
    d = np.diag(rm)
    qm = qm * np.where(d < 0, -1.0, 1.0)
    qm[:, d == 0] = 0.0
    return qm


def product_condition(a_list, b) -> float:
    """max |sum_w |A_w| |B|| / max |sum_w A_w B|, at least 1: how far the entries of
    the summed product sit below the sums of their terms' magnitudes.  A float
    product obeys |fl(A B) - A B| <= gamma_n |A| |B| entrywise (Higham, Accuracy and
    Stability of Numerical Algorithms, 2nd ed., section 3.5), so its error relative
    to max |A B| is this ratio times the summation's growth factor.  Diagnostic for
    tolerances only: it changes nothing the step computes."""
    num = np.abs(sum(np.abs(a) @ np.abs(b) for a in a_list)).max(initial=0.0)
    den = np.abs(sum(a @ b for a in a_list)).max(initial=0.0)
    if den == 0.0:
        return 1.0
    return max(1.0, float(num / den))


def step(state: State, bucket: np.ndarray, seg_offset, orc) -> np.ndarray:
    """One iteration of the hook on bucket [W, numel] (fp32 replicas, tensors at
    seg_offset[t]).  Returns the new bucket contents as float64 [W, numel] and
    advances the state."""
    W = state.W
    bucket = np.asarray(bucket, np.float32)
    assert bucket.shape[0] == W
    out = bucket.astype(np.float64)
    if state.iter < state.start_iter:
        mean, _ = orc.ring(bucket.copy())
        state.iter += 1
        return mean.astype(np.float64)

    vec = [t for t, s in enumerate(state.shapes) if matrix_view(s) is None]
    if vec:
        cat = np.concatenate([bucket[:, seg_offset[t]:seg_offset[t] + _numel(state.shapes[t])] for t in vec], axis=1)
        if cat.shape[1] > 0:
            mean, _ = orc.ring(np.ascontiguousarray(cat))
            pos = 0
            for t in vec:
                k = _numel(state.shapes[t])
                out[:, seg_offset[t]:seg_offset[t] + k] = mean[:, pos:pos + k]
                pos += k

    for t, s in enumerate(state.shapes):
        mv = matrix_view(s)
        if mv is None:
            continue
        m, n = mv
        lo = seg_offset[t]
        mw = []
        for w in range(W):
            g = bucket[w, lo:lo + m * n].astype(np.float64).reshape(m, n)
            mw.append(g + state.error[w][t] if state.error_feedback else g)
        q = state.q[t]
        p = sum(mw[w] @ q for w in range(W))
        sv = np.linalg.svd(p, compute_uv=False)
        state.cond[t] = float(sv[0] / sv[-1]) if sv[-1] > 0 else float("inf")
        amp_p = product_condition(mw, q)
        p = _orthonormal(p)
        qn = sum(mw[w].T @ p for w in range(W)) / W
        state.amp[t] = max(amp_p, product_condition([x.T for x in mw], p))
        approx = p @ qn.T
        for w in range(W):
            out[w, lo:lo + m * n] = approx.reshape(-1)
            if state.error_feedback:
                state.error[w][t] = mw[w] - approx
        state.q[t] = qn
    state.iter += 1
    return out


def _numel(shape) -> int:
    n = 1
    for s in shape:
        n *= int(s)
    return n
