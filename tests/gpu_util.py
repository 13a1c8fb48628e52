"""Helpers for the GPU parity tests: buffers with guard bands, and the oracle's
value for sampled elements of a full-size bucket."""
from __future__ import annotations

import numpy as np

import workloads as WL

GUARD = 64          # guard elements before and after every device buffer
SENTINEL = np.float32(-7.75e33)


def bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str = ""):
    g, w = bits(got), bits(want)
    if not np.array_equal(g, w):
        bad = np.argwhere(g != w)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} elements differ; first at {i}: got {got[i]!r} want {want[i]!r}")


def chunk_of(e: np.ndarray, n: int, W: int) -> np.ndarray:
    L = max(1, -(-n // W))
    return np.minimum(e // L, W - 1)


def oracle_at(orc, t: np.ndarray, chunks: np.ndarray, mode: int = 0) -> np.ndarray:
    """Oracle result of the ring reduction for k sampled elements.

    t[w, j] is replica w's packed fp32 value of element j and chunks[j] its ring
    chunk in the full bucket.  Elements are laid into a small [W, W*m] bucket at
    the same chunk (chunk length m), so the oracle sums each in the same order."""
    W, k = t.shape
    out = np.empty(k, np.float32)
    for c in range(W):
        js = np.nonzero(chunks == c)[0]
        if len(js) == 0:
            continue
        m = len(js)
        small = np.zeros((W, W * m), np.float32)
        small[:, c * m:(c + 1) * m] = t[:, js]
        small, _ = orc.ring(small, mode)
        out[js] = small[c, c * m:(c + 1) * m]
    return out


def packed_at(orc, wl, p: int, idx: np.ndarray, micro_steps: int, used_w=None) -> np.ndarray:
    """Oracle-packed fp32 values t[w, j] of parameter p at element indices idx, after
    `micro_steps` micro-steps of pack (copy, then accumulate)."""
    W, k = wl.W, len(idx)
    acc = None
    for m in range(micro_steps):
        segs = []
        for w in range(W):
            v = WL.grad_at_np(wl, p, w, m, idx)
            raw = WL.f32_to_bf16_bits_np(v) if wl.dtype == WL.BF16 else v
            segs.append([raw])
        used = None if used_w is None else np.asarray(used_w, np.uint8).reshape(W, 1)
        acc = orc.pack(segs, [0], k, [wl.dtype], used=used, accumulate=m > 0, out=acc)
    return acc
