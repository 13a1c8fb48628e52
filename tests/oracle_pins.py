"""Pins of the CPU oracle: facts the DDP pages and the mathematics fix.

Each ``pin_*`` takes a loaded oracle and raises AssertionError on a mismatch.
``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutants.py`` runs
them on copies of the oracle with a planted mistake and requires that some pin
fails for each.  No pin recomputes the oracle's own formula: they check printed
values (golden files), closed forms (exact rational means of dyadic inputs), a
characterisation of the bucket rule, invariants and library routines.
"""
from __future__ import annotations

import os
from fractions import Fraction
from itertools import permutations

import numpy as np

import workloads as WL

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
REVERSE, FWD_THEN_REVERSE, MEGATRON = 0, 1, 2
ALLREDUCE, REDUCE_SCATTER = 0, 1


def read_golden(name: str) -> dict:
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#") or "=" not in line:
            continue
        k, v = (s.strip() for s in line.split("=", 1))
        out[k] = [int(t) for t in v.split()]
    return out


def ring_fixture(name: str = "ring_order_w4.txt"):
    rows = [l.split() for l in open(os.path.join(GOLDEN, name)) if l.startswith("e")]
    x = np.array([[float.fromhex(r[2 + k]) for r in rows] for k in range(4)], np.float32)
    exp = np.array([float.fromhex(r[7]) for r in rows], np.float32)
    return x, exp


# ---------------------------------------------------------------------------
# assignment
# ---------------------------------------------------------------------------
def pin_linear12_rebuilt(orc):
    g = read_golden("linear12_bucket_bytes.txt")
    n = WL.numels(WL.linear12())
    r = orc.assign(n, cap_bytes=g["cap_bytes"][0], first_cap_bytes=g["first_cap_bytes"][0], order=REVERSE)
    assert list(r["bucket_bytes"]) == g["rebuilt_bucket_bytes"], r["bucket_bytes"]
    assert sorted(r["members"][0]) == g["rebuilt_bucket0_params"]


def pin_linear12_initial(orc):
    g = read_golden("linear12_bucket_bytes.txt")
    n = WL.numels(WL.linear12())
    r = orc.assign(n, cap_bytes=g["cap_bytes"][0], first_cap_bytes=g["first_cap_bytes"][0],
                   order=FWD_THEN_REVERSE)
    assert list(r["bucket_bytes"]) == g["initial_bucket_bytes"], r["bucket_bytes"]
    assert sorted(r["members"][-1]) == g["initial_last_bucket_params"]


def pin_exercise3(orc):
    g = read_golden("lecture15_exercise3.txt")
    MB = 10 ** 6
    n = [mb * MB // 4 for mb in g["param_mb"]]
    cap = g["cap_mb"][0] * MB
    r = orc.assign(n, cap_bytes=cap, first_cap_bytes=cap, order=REVERSE)
    assert r["members"] == [g["bucket0"], g["bucket1"]], r["members"]
    assert list(r["bucket_bytes"]) == [mb * MB for mb in g["bucket_mb"]]


def pin_bucket_counts(orc):
    g = read_golden("lecture15_bucket_counts.txt")
    cap = g["cap_bytes"][0]
    rn, bn = WL.numels(WL.resnet50()), WL.numels(WL.bert_large())
    assert len(rn) == g["resnet50_tensors"][0] and len(bn) == g["bert_large_tensors"][0]
    assert orc.assign(rn, cap_bytes=cap, first_cap_bytes=cap)["nbuckets"] == g["resnet50_buckets"][0]
    assert orc.assign(bn, cap_bytes=cap, first_cap_bytes=cap)["nbuckets"] == g["bert_large_buckets"][0]


def _characterise(r, numels, dtypes, cap, first_cap, order, esize):
    """The greedy close-on-reach rule, stated as properties of its result:
    within each dtype group, concatenating the buckets in closing order gives the
    iteration order; every bucket but the group's last has bytes >= its cap while
    bytes minus its last member < cap; the group's last bucket stays below its cap
    unless it closed exactly at the end."""
    P = len(numels)
    seq = list(range(P - 1, -1, -1)) if order == REVERSE else list(range(P))
    buckets = [list(m) for m in r["members"]]
    if order == FWD_THEN_REVERSE:
        buckets = buckets[::-1]
    # members of every bucket are in iteration order, one dtype per bucket
    pos = {p: k for k, p in enumerate(seq)}
    for m in buckets:
        assert [pos[p] for p in m] == sorted(pos[p] for p in m)
        assert len({dtypes[p] for p in m}) == 1
    for g in sorted(set(dtypes)):
        gb = [m for m in buckets if dtypes[m[0]] == g]
        gb.sort(key=lambda m: pos[m[0]])
        flat = [p for m in gb for p in m]
        assert flat == [p for p in seq if dtypes[p] == g]
        for k, m in enumerate(gb):
            c = first_cap if (k == 0 and order != MEGATRON) else cap
            by = sum(numels[p] * esize[dtypes[p]] for p in m)
            last = numels[m[-1]] * esize[dtypes[m[-1]]]
            if k < len(gb) - 1:
                assert by >= c and by - last < c, (k, by, last, c)
            else:
                assert by - last < c, (k, by, last, c)


def pin_assignment_characterised(orc):
    rng = np.random.default_rng(7)
    for trial in range(300):
        P = int(rng.integers(0, 12))
        numels = [int(v) for v in rng.integers(0, 40, size=P)]
        dtypes = [int(v) for v in rng.integers(0, 2, size=P)] if trial % 2 else [0] * P
        cap = int(rng.integers(1, 120))
        first = int(rng.integers(1, 120))
        for order in (REVERSE, FWD_THEN_REVERSE, MEGATRON):
            for fp32 in (0, 1):
                r = orc.assign(numels, dtypes, cap, first, order, 1, fp32)
                esize = {0: 4, 1: 4 if fp32 else 2}
                _characterise(r, numels, dtypes, cap, first, order, esize)
                # offsets: tight, in member order
                for m in r["members"]:
                    off = 0
                    for p in m:
                        assert r["offset_of"][p] == off
                        off += numels[p]


def pin_assignment_brute_force(orc):
    """Every permutation of five small sizes, every cap in 1..12: the bucket list equals
    the one found by trying all ways to cut the sequence and keeping the unique cut
    whose pieces satisfy the close-on-reach rule."""
    sizes = [1, 2, 3, 5, 8]
    for perm in permutations(sizes):
        for cap in range(1, 13):
            r = orc.assign(list(perm), cap_bytes=cap * 4, first_cap_bytes=cap * 4, order=REVERSE)
            seq = list(range(len(perm) - 1, -1, -1))
            valid = []
            for mask in range(1 << (len(seq) - 1)):
                cuts, cur = [], [seq[0]]
                for k in range(1, len(seq)):
                    if mask >> (k - 1) & 1:
                        cuts.append(cur)
                        cur = []
                    cur.append(seq[k])
                cuts.append(cur)
                ok = all(sum(perm[p] for p in m) >= cap and sum(perm[p] for p in m[:-1]) < cap for m in cuts[:-1])
                ok = ok and sum(perm[p] for p in cuts[-1][:-1]) < cap
                if ok:
                    valid.append(cuts)
            assert len(valid) == 1
            assert r["members"] == valid[0], (perm, cap, r["members"], valid[0])


def pin_first_cap_only_first(orc):
    """With the first cap at 1 byte every bucket after the first still uses the big cap."""
    n = [4] * 10
    r = orc.assign(n, cap_bytes=40, first_cap_bytes=1, order=REVERSE)
    assert [len(m) for m in r["members"]] == [1, 3, 3, 3]


def pin_megatron_padding(orc):
    wl = WL.c3_gpt2()
    r = orc.assign(wl.numels, [wl.dtype] * wl.nparams, wl.cap_bytes, wl.first_cap_bytes, wl.order,
                   wl.pad_multiple, 1)
    assert list(r["bucket_order"]) == list(range(r["nbuckets"] - 1, -1, -1))
    assert r["members"][0][0] == 0          # p0 at the front of bucket 0
    for b, m in enumerate(r["members"]):
        tot = sum(wl.numels[p] for p in m)
        assert r["bucket_numel"][b] % wl.pad_multiple == 0
        assert tot <= r["bucket_numel"][b] < tot + wl.pad_multiple
    # an odd layout really is padded
    r = orc.assign([3, 5, 7], cap_bytes=16, first_cap_bytes=16, order=MEGATRON, pad_multiple=8)
    assert list(r["bucket_numel"]) == [8, 8]
    assert r["members"] == [[0, 1], [2]]


def pin_mlp_single_bucket(orc):
    wl = WL.c1_mlp()
    r = orc.assign(wl.numels, cap_bytes=wl.cap_bytes, first_cap_bytes=wl.first_cap_bytes, order=wl.order)
    assert r["nbuckets"] == 1 and r["bucket_bytes"][0] == 4 * 199690 < (1 << 20)
    assert r["members"][0] == [5, 4, 3, 2, 1, 0]


# ---------------------------------------------------------------------------
# ring reduction
# ---------------------------------------------------------------------------
def _exact_mean(x: np.ndarray) -> list:
    W = x.shape[0]
    return [sum(Fraction(float(v)) for v in x[:, e]) / W for e in range(x.shape[1])]


def pin_ring_dyadic_exact(orc):
    """Sums of dyadic values k * 2^-12 are exact, so the result is the mean itself."""
    rng = np.random.default_rng(11)
    for W in (1, 2, 3, 4, 5, 8, 16):
        for n in (0, 1, 2, 7, 16, 33, 100):
            x = (rng.integers(-4096, 4097, size=(W, n)) * 2.0 ** -12).astype(np.float32)
            if W in (3, 5):   # 1/W is not dyadic; use multiples of W so the mean stays exact
                x = (rng.integers(-100, 101, size=(W, n)) * W * 2.0 ** -10).astype(np.float32)
            want = _exact_mean(x)
            y, _ = orc.ring(x.copy(), ALLREDUCE)
            for w in range(W):
                assert [Fraction(float(v)) for v in y[w]] == want, (W, n, w)


def pin_ring_bit_identical(orc):
    rng = np.random.default_rng(12)
    for W in (2, 3, 4, 7, 8, 16):
        x = rng.standard_normal((W, 257)).astype(np.float32)
        y, _ = orc.ring(x.copy(), ALLREDUCE)
        for w in range(1, W):
            assert np.array_equal(y[0].view(np.uint32), y[w].view(np.uint32))


def pin_ring_traffic(orc):
    """Each rank sends 2(W-1)/W of the bucket in allreduce, (W-1)/W in reduce-scatter."""
    for W in (1, 2, 3, 4, 8, 16):
        for n in (W * 5, W * 64):
            S = 4 * n
            _, s = orc.ring(np.ones((W, n), np.float32), ALLREDUCE)
            assert all(int(v) * W == 2 * (W - 1) * S for v in s), (W, n, s)
            _, s = orc.ring(np.ones((W, n), np.float32), REDUCE_SCATTER)
            assert all(int(v) * W == (W - 1) * S for v in s), (W, n, s)


def pin_ring_identity_w1(orc):
    rng = np.random.default_rng(13)
    x = rng.standard_normal((1, 1000)).astype(np.float32)
    y, s = orc.ring(x.copy(), ALLREDUCE)
    assert np.array_equal(x.view(np.uint32), y.view(np.uint32)) and int(s[0]) == 0


def pin_ring_error_bound(orc):
    """General inputs: |result - exact mean| <= (W + 2) * 2^-24 * sum|x| / W: W-1 additions
    plus the rounding of fp32(1/W) and of each product, each within a unit roundoff."""
    rng = np.random.default_rng(14)
    for W in (2, 3, 4, 6, 8):
        x = rng.standard_normal((W, 64)).astype(np.float32)
        want = _exact_mean(x)
        y, _ = orc.ring(x.copy(), ALLREDUCE)
        for e in range(64):
            bound = Fraction(W + 2) * Fraction(2) ** -24 * sum(abs(Fraction(float(v))) for v in x[:, e]) / W
            assert abs(Fraction(float(y[0, e])) - want[e]) <= bound


def pin_ring_order_golden(orc):
    x, exp = ring_fixture()
    y, _ = orc.ring(x.copy(), ALLREDUCE)
    for w in range(4):
        assert np.array_equal(y[w].view(np.uint32), exp.view(np.uint32)), (w, y[w], exp)
    y, _ = orc.ring(x.copy(), REDUCE_SCATTER)
    for r in range(4):
        assert np.array_equal(y[r, 2 * r:2 * r + 2].view(np.uint32), exp[2 * r:2 * r + 2].view(np.uint32))


def pin_ring_ragged_golden(orc):
    x, exp = ring_fixture("ring_ragged_w4.txt")
    y, _ = orc.ring(x.copy(), ALLREDUCE)
    for w in range(4):
        assert np.array_equal(y[w].view(np.uint32), exp.view(np.uint32)), (w, y[w], exp)


def pin_reduce_scatter_shards(orc):
    """Rank r's shard r equals slice r of the allreduce result; outside it nothing changes."""
    rng = np.random.default_rng(15)
    for W in (2, 4, 8):
        n = W * 37
        x = rng.standard_normal((W, n)).astype(np.float32)
        ar, _ = orc.ring(x.copy(), ALLREDUCE)
        rs, _ = orc.ring(x.copy(), REDUCE_SCATTER)
        k = n // W
        for r in range(W):
            assert np.array_equal(rs[r, r * k:(r + 1) * k], ar[r, r * k:(r + 1) * k])
            mask = np.ones(n, bool)
            mask[r * k:(r + 1) * k] = False
            assert np.array_equal(rs[r, mask], x[r, mask])


def pin_partial_use(orc):
    """A parameter used on rank 0 only: rank 1 contributes a zero segment, result (g0 + 0) / 2
    (Lecture 15 notes, section 4.2)."""
    g0 = np.array([0.5, -3.0, 1.25, 7.0], np.float32)
    bucket = orc.pack([[g0], [None]], [0], 4, used=[[1], [0]])
    assert np.array_equal(bucket[1], np.zeros(4, np.float32))
    y, _ = orc.ring(bucket, ALLREDUCE)
    assert np.array_equal(y[1], g0 / 2) and np.array_equal(y[0], g0 / 2)


def pin_accumulation_linear(orc):
    """no_sync: accumulating four micro-steps then reducing equals reducing each micro-step
    and adding the results (exact for dyadic inputs; Lecture 15 notes, section 4.1)."""
    rng = np.random.default_rng(16)
    W, n, M = 4, 50, 4
    g = (rng.integers(-4096, 4097, size=(M, W, n)) * 2.0 ** -12).astype(np.float32)
    acc = None
    for m in range(M):
        acc = orc.pack([[g[m, w]] for w in range(W)], [0], n, accumulate=m > 0, out=acc)
    y, _ = orc.ring(acc, ALLREDUCE)
    want = [sum(Fraction(float(v)) for v in g[:, :, e].reshape(-1)) / W for e in range(n)]
    assert [Fraction(float(v)) for v in y[0]] == want


# ---------------------------------------------------------------------------
# pack / unpack
# ---------------------------------------------------------------------------
def pin_pack_flatten(orc):
    """pack = concatenation of the segments at their offsets, zero padding after."""
    rng = np.random.default_rng(17)
    segs = [rng.standard_normal(k).astype(np.float32) for k in (3, 1, 10, 4)]
    offs = np.cumsum([0] + [len(s) for s in segs[:-1]])
    b = orc.pack([segs], offs, 24)
    assert np.array_equal(b[0], np.concatenate(segs + [np.zeros(6, np.float32)]))


def pin_pack_bf16_widening(orc):
    """bf16 -> fp32 widening is exact: every bf16 bit pattern widens to the fp32 with the
    same upper 16 bits (checked against numpy's float32 view)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = ((bits.astype(np.uint32) & 0x7F80) != 0x7F80)
    b = orc.pack([[bits[finite]]], [0], int(finite.sum()), seg_dtype=[WL.BF16])
    want = (bits[finite].astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(b[0].view(np.uint32), want.view(np.uint32))


def pin_pack_f16_widening(orc):
    """fp16 -> fp32 against numpy's float16 conversion, all finite bit patterns."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = np.isfinite(bits.view(np.float16))
    b = orc.pack([[bits[finite]]], [0], int(finite.sum()), seg_dtype=[2])
    want = bits[finite].view(np.float16).astype(np.float32)
    assert np.array_equal(b[0].view(np.uint32), want.view(np.uint32))


def pin_pack_unused_zero_and_accumulate(orc):
    a = np.array([1.0, 2.0], np.float32)
    b = orc.pack([[a, a]], [0, 2], 5, used=[[1, 0]], out=np.full((1, 5), 7.0, np.float32))
    assert list(b[0]) == [1.0, 2.0, 0.0, 0.0, 0.0]
    b[0, 2:4] = 9.0
    b = orc.pack([[a, a]], [0, 2], 5, used=[[0, 1]], accumulate=True, out=b)
    assert list(b[0]) == [1.0, 2.0, 10.0, 11.0, 0.0]


def pin_unpack_roundtrip(orc):
    """W = 1: pack, reduce (identity), unpack returns every segment unchanged."""
    rng = np.random.default_rng(18)
    segs = [rng.standard_normal(k).astype(np.float32) for k in (5, 9, 2)]
    offs = [0, 5, 14]
    b = orc.pack([segs], offs, 17)
    b, _ = orc.ring(b, ALLREDUCE)
    outs = orc.unpack(b, offs, [5, 9, 2])
    for s in range(3):
        assert np.array_equal(outs[0][s], segs[s])


def pin_unpack_skips_unused_and_shards(orc):
    b = np.arange(16, dtype=np.float32).reshape(2, 8)
    outs = [[np.full(3, -1, np.float32), np.full(5, -1, np.float32)] for _ in range(2)]
    orc.unpack(b, [0, 3], [3, 5], ALLREDUCE, global_used=[1, 0], outs=outs)
    assert list(outs[1][0]) == [8, 9, 10] and list(outs[1][1]) == [-1] * 5
    outs = [[np.full(3, -1, np.float32), np.full(5, -1, np.float32)] for _ in range(2)]
    orc.unpack(b, [0, 3], [3, 5], REDUCE_SCATTER, outs=outs)
    # shard 0 = elements 0..3 of rank 0, shard 1 = elements 4..7 of rank 1
    assert list(outs[0][0]) == [0, 1, 2] and list(outs[0][1]) == [3, -1, -1, -1, -1]
    assert list(outs[1][0]) == [-1, -1, -1] and list(outs[1][1]) == [-1, 12, 13, 14, 15]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


# ---------------------------------------------------------------------------
# compression hook (bf16 / fp16 wire)
# ---------------------------------------------------------------------------
BF16_W, F16_W = 1, 2


def _rne_fraction(q: Fraction, p: int, emin: int) -> Fraction:
    """Nearest value with a p-bit significand (exponent >= emin, subnormals below),
    ties to even, by exact rational arithmetic (no overflow handling)."""
    if q == 0:
        return Fraction(0)
    s = -1 if q < 0 else 1
    a = abs(q)
    e = 0
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    quantum = Fraction(2) ** (e - p + 1)
    k = a // quantum
    lo, hi = k * quantum, (k + 1) * quantum
    if a - lo < hi - a or (a - lo == hi - a and k % 2 == 0):
        return s * lo
    return s * hi


def pin_wire_rounding_f16(orc):
    """fp16 rounding of doubles: numpy's correctly rounded float64 -> float16."""
    rng = np.random.default_rng(21)
    xs = rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000)
    xs = np.concatenate([xs, [65504.0, 65519.99, 5.96e-8, 2.9802322387695312e-08, 1e-9, -0.0, 0.5 + 2 ** -12]])
    for x in xs:
        assert orc.round_wire(float(x), F16_W) == int(np.float64(x).astype(np.float16).view(np.uint16)), x


def pin_wire_rounding_bf16(orc):
    """bf16 rounding: of floats, against the upper-half rule with nearest-even carry;
    of doubles, against exact rational nearest-even."""
    rng = np.random.default_rng(22)
    f = (rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)).astype(np.float32)
    want = WL.f32_to_bf16_bits_np(f)
    for x, w in zip(f, want):
        assert orc.round_wire(float(x), BF16_W) == int(w), x
    for x in rng.standard_normal(300) * 10.0 ** rng.integers(-5, 5, 300):
        h = orc.round_wire(float(x), BF16_W)
        assert Fraction(orc.wire_value(h, BF16_W)) == _rne_fraction(Fraction(float(x)), 8, -126), x


def pin_wire_ring_golden(orc):
    x, exp = ring_fixture("ring_wire_bf16_w4.txt")
    y, sent = orc.ring_wire(x.copy(), ALLREDUCE, BF16_W)
    for w in range(4):
        assert np.array_equal(y[w].view(np.uint32), exp.view(np.uint32)), (w, y[w], exp)
    assert all(int(s) == 2 * 3 * 2 for s in sent)   # 2(W-1) chunks of one 2-byte element


def pin_wire_ring_brute_force(orc):
    """W = 3 (1/3 is not a power of two, so where the division sits matters) and W = 5:
    compress, divide, and every ring addition rounded to the wire type, redone with
    exact rationals in the ring order c+1, ..., c."""
    rng = np.random.default_rng(23)
    for wire, p, emin in ((BF16_W, 8, -126), (F16_W, 11, -14)):
        for W in (3, 5):
            n = 2 * W
            x = (rng.standard_normal((W, n)) * 3).astype(np.float32)
            y, _ = orc.ring_wire(x.copy(), ALLREDUCE, wire)
            L = -(-n // W)
            for e in range(n):
                c = min(e // L, W - 1)
                z = [_rne_fraction(_rne_fraction(Fraction(float(x[w, e])), p, emin) / W, p, emin) for w in range(W)]
                s = z[(c + 1) % W]
                for k in range(2, W + 1):
                    s = _rne_fraction(s + z[(c + k) % W], p, emin)
                assert Fraction(float(y[0, e])) == s, (wire, W, e)


def pin_wire_w1_rounds(orc):
    """One rank: the hook still converts to the wire type and back."""
    x = np.array([[1.0 + 2 ** -9, 3.0, 1e-3, -7.75]], np.float32)
    y, sent = orc.ring_wire(x.copy(), ALLREDUCE, BF16_W)
    bf = float(WL.bf16_bits_to_f32_np(WL.f32_to_bf16_bits_np(np.array([1e-3], np.float32)))[0])
    assert list(y[0]) == [1.0, 3.0, bf, -7.75]
    assert int(sent[0]) == 0


def pin_wire_reduce_scatter_shards(orc):
    rng = np.random.default_rng(24)
    W, n = 4, 4 * 9
    x = rng.standard_normal((W, n)).astype(np.float32)
    ar, _ = orc.ring_wire(x.copy(), ALLREDUCE, F16_W)
    rs, sent = orc.ring_wire(x.copy(), REDUCE_SCATTER, F16_W)
    k = n // W
    for r in range(W):
        assert np.array_equal(rs[r, r * k:(r + 1) * k], ar[r, r * k:(r + 1) * k])
        mask = np.ones(n, bool)
        mask[r * k:(r + 1) * k] = False
        assert np.array_equal(rs[r, mask], x[r, mask])
    assert all(int(s) * W == (W - 1) * 2 * n for s in sent)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


# ---------------------------------------------------------------------------
# rebuilt buckets and the overlap timeline
# ---------------------------------------------------------------------------
def _exercise3_plan(orc, single=False):
    g = read_golden("lecture15_exercise3.txt")
    MB = 10 ** 6
    n = [mb * MB // 4 for mb in g["param_mb"]]
    cap = (10 ** 12) if single else g["cap_mb"][0] * MB
    return orc.assign(n, cap_bytes=cap, first_cap_bytes=cap, order=REVERSE)


def pin_timeline_exercise4(orc):
    g = read_golden("lecture15_exercise4.txt")
    r = _exercise3_plan(orc)
    ready = [t / 10 for t in g["ready_tenths_p0_p1_p2_p3_p4"]]
    t = orc.overlap_timeline(ready, r["bucket_of"], r["bucket_order"], r["bucket_bytes"], g["alpha_tenths"][0] / 10,
                             0.1 / 10 ** 6)
    assert [round(x * 10) for x in t["start_ms"]] == g["bucket_start_tenths"]
    assert [round(x * 10) for x in t["end_ms"]] == g["bucket_end_tenths"]
    assert round(t["step_ms"] * 10) == g["step_tenths"][0]
    assert round(t["serial_ms"] * 10) == g["serial_tenths"][0]
    one = _exercise3_plan(orc, single=True)
    t1 = orc.overlap_timeline(ready, one["bucket_of"], one["bucket_order"], one["bucket_bytes"],
                              g["alpha_tenths"][0] / 10, 0.1 / 10 ** 6)
    assert one["nbuckets"] == 1 and round(t1["step_ms"] * 10) == g["single_bucket_step_tenths"][0]


def pin_timeline_properties(orc):
    """The step lies between the backward alone and the serial step; with free
    communication it equals the backward; the last bucket issued cannot start before
    its last gradient ("the last bucket is always exposed", Lecture 15 section 3.1)."""
    rng = np.random.default_rng(31)
    for trial in range(100):
        P = int(rng.integers(1, 15))
        n = [int(v) for v in rng.integers(1, 50, P)]
        r = orc.assign(n, cap_bytes=int(rng.integers(4, 200)), first_cap_bytes=int(rng.integers(4, 200)))
        ready = np.sort(rng.random(P) * 10)[::-1].copy()   # backward: last parameter first
        a, b = float(rng.random()), float(rng.random()) * 0.05
        t = orc.overlap_timeline(ready, r["bucket_of"], r["bucket_order"], r["bucket_bytes"], a, b)
        assert ready.max() - 1e-12 <= t["step_ms"] <= t["serial_ms"] + 1e-9
        last = r["bucket_order"][-1]
        assert t["start_ms"][last] >= max(ready[p] for p in range(P) if r["bucket_of"][p] == last) - 1e-12
        z = orc.overlap_timeline(ready, r["bucket_of"], r["bucket_order"], r["bucket_bytes"], 0.0, 0.0)
        assert abs(z["step_ms"] - ready.max()) < 1e-12


def pin_rebuild_linear12(orc):
    """Gradients observed in exactly reversed parameter order: the rebuilt buckets are the
    printed ones (DDP chapter 17.13)."""
    g = read_golden("linear12_bucket_bytes.txt")
    n = WL.numels(WL.linear12())
    r = orc.assign_sequence(n, list(range(len(n) - 1, -1, -1)), cap_bytes=g["cap_bytes"][0],
                            first_cap_bytes=g["first_cap_bytes"][0])
    assert list(r["bucket_bytes"]) == g["rebuilt_bucket_bytes"]
    assert sorted(r["members"][0]) == g["rebuilt_bucket0_params"]
    assert list(r["bucket_order"]) == [0, 1, 2]


def pin_rebuild_characterised(orc):
    """Any observed order: buckets are consecutive runs of the sequence (per dtype) that
    close on reaching the cap, the first under the first cap."""
    rng = np.random.default_rng(32)
    for trial in range(200):
        P = int(rng.integers(1, 14))
        numels = [int(v) for v in rng.integers(0, 40, P)]
        dtypes = [int(v) for v in rng.integers(0, 2, P)] if trial % 2 else [0] * P
        seq = [int(v) for v in rng.permutation(P)]
        cap, first = int(rng.integers(1, 120)), int(rng.integers(1, 120))
        r = orc.assign_sequence(numels, seq, dtypes, cap, first, 1, 1)
        pos = {p: k for k, p in enumerate(seq)}
        for g in sorted(set(dtypes)):
            gb = sorted((m for m in r["members"] if dtypes[m[0]] == g), key=lambda m: pos[m[0]])
            assert [p for m in gb for p in m] == [p for p in seq if dtypes[p] == g]
            for k, m in enumerate(gb):
                c = first if k == 0 else cap
                by = sum(numels[p] * 4 for p in m)
                if k < len(gb) - 1:
                    assert by >= c and by - numels[m[-1]] * 4 < c
                else:
                    assert by - numels[m[-1]] * 4 < c


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


# ---------------------------------------------------------------------------
# the local-used bitmap (find_unused_parameters)
# ---------------------------------------------------------------------------
def pin_bitmap_lecture_two_ranks(orc):
    """Lecture 15 section 4.2, two processes: a parameter that only rank 0 used is still
    all-reduced, rank 1 contributing zero, so rank 0 ends with exactly half of its own
    gradient; a parameter no rank used keeps its .grad untouched; one both used is the
    plain mean.  Parameters a (both), b (rank 0 only), c (neither)."""
    local = np.array([[1, 1, 0], [1, 0, 0]], np.uint8)
    count, glob = orc.used_allreduce(local)
    assert list(count) == [2, 1, 0] and list(glob) == [1, 1, 0]
    a = [np.array([0.5, -1.25], np.float32), np.array([1.5, 0.25], np.float32)]
    b0 = np.array([3.0, -0.75, 1e-3], np.float32)
    c = np.array([9.0], np.float32)
    grads = [[a[0], b0, c], [a[1], np.full(3, 123.0, np.float32), c]]
    offs, sizes = [0, 2, 5], [2, 3, 1]
    buf = orc.pack(grads, offs, 6, used=local)
    buf, _ = orc.ring(buf, ALLREDUCE)
    outs = [[np.full(k, -7.0, np.float32) for k in sizes] for _ in range(2)]
    orc.unpack(buf, offs, sizes, ALLREDUCE, global_used=glob, outs=outs)
    for w in range(2):
        assert list(outs[w][0]) == [1.0, -0.5]
        assert np.array_equal(outs[w][1], b0 / np.float32(2))
        assert list(outs[w][2]) == [-7.0]


def pin_bitmap_library(orc):
    """Against numpy's count_nonzero / any over the replica axis, with nonzero bytes
    other than 1 (any nonzero byte marks use), W from 1 to 64, ragged P, P = 0."""
    rng = np.random.default_rng(41)
    for W, P in [(1, 7), (2, 1), (3, 33), (4, 391), (8, 161), (16, 5), (64, 70), (5, 0)]:
        vals = np.array([0, 0, 0, 1, 1, 2, 0x80, 0xFF], np.uint8)
        local = vals[rng.integers(0, len(vals), (W, P))]
        count, glob = orc.used_allreduce(local)
        assert np.array_equal(count, np.count_nonzero(local, axis=0).astype(np.int32))
        assert np.array_equal(glob, np.any(local != 0, axis=0).astype(np.uint8))


def pin_bitmap_replica_symmetry(orc):
    """The all-reduce treats the ranks alike: permuting them changes nothing; the count
    lies in [0, W] and equals W exactly where every rank used the parameter."""
    rng = np.random.default_rng(42)
    W, P = 6, 50
    local = (rng.random((W, P)) < 0.6).astype(np.uint8)
    count, glob = orc.used_allreduce(local)
    for perm in ([5, 4, 3, 2, 1, 0], [1, 2, 3, 4, 5, 0]):
        c2, g2 = orc.used_allreduce(local[perm])
        assert np.array_equal(c2, count) and np.array_equal(g2, glob)
    assert count.min() >= 0 and count.max() <= W
    assert np.array_equal(count == W, local.all(axis=0))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
