"""Seeded synthetic workloads for the gradient-bucket reduction.

This module is shared by the tests, the benchmark and the oracle's callers.
It holds only two things, and none of the reduction's arithmetic:

* parameter shape lists of the models the DDP pages use as workloads
  (a small MLP, ResNet-50, GPT-2 small, BERT-large), written from the
  published architecture hyper-parameters, in ``model.parameters()`` order;
* a counter-based random generator (splitmix64, Vigna 2015) that gives the
  gradient value of element ``i`` of parameter ``p`` on replica ``w`` at
  micro-step ``m`` without generating anything before it, so a full-size GPU
  input and a sampled CPU check see the same numbers.

The same generator is written twice, once over numpy ``uint64`` (exact
wrap-around) and once over torch ``int64`` (two's complement, logical shifts
emulated by masking) so that large inputs can be produced directly in device
memory; tests check the two against each other bit for bit.

Value distributions (all exactly reproducible, no transcendental functions):

* ``dyadic12``  uniform integer k in [-4096, 4096], value k * 2**-12
  (sums of a few of these are exact in fp32);
* ``uniform``   24-bit uniform in [-1, 1): m * 2**-23 - 1, m in [0, 2**24);
* ``normal``    N(0, sigma) stood in for by the Irwin-Hall sum of four 16-bit
  uniform integers, centred and scaled to unit variance, times sigma
  (float64, one rounding), then rounded to fp32 (and from fp32 to bf16,
  round-to-nearest-even, for bf16 workloads).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# ---------------------------------------------------------------------------
# counter-based generator: splitmix64
# ---------------------------------------------------------------------------
_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1


def _finalize_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    """Key of one stream: output number ``stream`` of splitmix64 seeded with ``seed``."""
    return _finalize_int(seed + (stream + 1) * _GAMMA)


def stream_id(param: int, replica: int = 0, micro: int = 0) -> int:
    """Stream number of one parameter's gradient on one replica at one micro-step."""
    return (micro * 256 + replica) * 65536 + param


def bits_np(key: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the splitmix64 sequence seeded with ``key``."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(key) + idx * np.uint64(_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
        z = z ^ (z >> np.uint64(31))
    return z


def bits_at_np(key: int, indices: np.ndarray) -> np.ndarray:
    """Sequence outputs at arbitrary indices (for sampled checks)."""
    with np.errstate(over="ignore"):
        idx = np.asarray(indices, dtype=np.uint64) + np.uint64(1)
        z = np.uint64(key) + idx * np.uint64(_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
        z = z ^ (z >> np.uint64(31))
    return z


def _s64(x: int) -> int:
    x &= _MASK64
    return x - (1 << 64) if x >> 63 else x


def _lsr_t(z, k: int):
    # logical right shift of an int64 tensor holding uint64 bits
    return (z >> k) & ((1 << (64 - k)) - 1)


def bits_torch(key: int, start: int, count: int, device):
    import torch

    idx = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    z = idx * _s64(_GAMMA) + _s64(key)
    z = (z ^ _lsr_t(z, 30)) * _s64(_M1)
    z = (z ^ _lsr_t(z, 27)) * _s64(_M2)
    z = z ^ _lsr_t(z, 31)
    return z


# ---------------------------------------------------------------------------
# bits -> values
# ---------------------------------------------------------------------------
# unit-variance scale of the centred sum of four uniform 16-bit integers
_IH4_MEAN = 4 * 65535 / 2  # 131070
_IH4_INV_STD = 1.0 / math.sqrt(4 * (65536.0 * 65536.0 - 1.0) / 12.0)


def f32_to_bf16_bits_np(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern (uint16), round to nearest even; NaN kept quiet."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    r = np.where(nan, (u >> np.uint32(16)) | np.uint32(0x40), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32_np(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def values_np(bits: np.ndarray, dist: str, sigma: float = 1.0) -> np.ndarray:
    """Map generator outputs to fp32 values (numpy)."""
    if dist == "dyadic12":
        k = ((bits >> np.uint64(32)) * np.uint64(8193)) >> np.uint64(32)
        return ((k.astype(np.float64) - 4096.0) * (2.0 ** -12)).astype(np.float32)
    if dist == "uniform":
        m = (bits >> np.uint64(40)).astype(np.float64)
        return (m * (2.0 ** -23) - 1.0).astype(np.float32)
    if dist == "normal":
        m16 = np.uint64(0xFFFF)
        s = (bits & m16) + ((bits >> np.uint64(16)) & m16) + ((bits >> np.uint64(32)) & m16) + (bits >> np.uint64(48))
        z = (s.astype(np.float64) - _IH4_MEAN) * (_IH4_INV_STD * sigma)
        return z.astype(np.float32)
    if dist == "zero":
        return np.zeros(bits.shape, dtype=np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def values_torch(bits, dist: str, sigma: float = 1.0):
    """Map generator outputs to fp32 values (torch, any device); same bits as ``values_np``."""
    import torch

    if dist == "dyadic12":
        k = (_lsr_t(bits, 32) * 8193) >> 32
        return ((k.to(torch.float64) - 4096.0) * (2.0 ** -12)).to(torch.float32)
    if dist == "uniform":
        m = _lsr_t(bits, 40).to(torch.float64)
        return (m * (2.0 ** -23) - 1.0).to(torch.float32)
    if dist == "normal":
        s = (bits & 0xFFFF) + ((bits >> 16) & 0xFFFF) + ((bits >> 32) & 0xFFFF) + _lsr_t(bits, 48)
        z = (s.to(torch.float64) - _IH4_MEAN) * (_IH4_INV_STD * sigma)
        return z.to(torch.float32)
    if dist == "zero":
        return torch.zeros(bits.shape, dtype=torch.float32, device=bits.device)
    raise ValueError(f"unknown distribution {dist!r}")


# ---------------------------------------------------------------------------
# parameter shape lists, model.parameters() order
# ---------------------------------------------------------------------------
def mlp3() -> list[tuple[int, ...]]:
    """3-layer MLP 512 -> 256 -> 256 -> 10 (weights stored [in, out] as listed)."""
    return [(512, 256), (256,), (256, 256), (256,), (256, 10), (10,)]


def linear12() -> list[tuple[int, ...]]:
    """Twelve Linear(1024, 1024) layers: weight then bias per layer."""
    out: list[tuple[int, ...]] = []
    for _ in range(12):
        out += [(1024, 1024), (1024,)]
    return out


def resnet50() -> list[tuple[int, ...]]:
    """ResNet-50 (bottleneck blocks [3, 4, 6, 3], 1000 classes): conv, BN and fc parameters."""
    out: list[tuple[int, ...]] = [(64, 3, 7, 7), (64,), (64,)]
    inplanes = 64
    for planes, blocks in ((64, 3), (128, 4), (256, 6), (512, 3)):
        for b in range(blocks):
            out += [(planes, inplanes, 1, 1), (planes,), (planes,)]
            out += [(planes, planes, 3, 3), (planes,), (planes,)]
            out += [(planes * 4, planes, 1, 1), (planes * 4,), (planes * 4,)]
            if b == 0:
                out += [(planes * 4, inplanes, 1, 1), (planes * 4,), (planes * 4,)]
            inplanes = planes * 4
    out += [(1000, 2048), (1000,)]
    return out


def bert_large(vocab: int = 30522, d: int = 1024, ffn: int = 4096, layers: int = 24,
               positions: int = 512, token_types: int = 2) -> list[tuple[int, ...]]:
    """BERT-large encoder with embeddings and pooler (no pre-training heads)."""
    out: list[tuple[int, ...]] = [(vocab, d), (positions, d), (token_types, d), (d,), (d,)]
    for _ in range(layers):
        out += [(d, d), (d,), (d, d), (d,), (d, d), (d,)]   # query, key, value
        out += [(d, d), (d,), (d,), (d,)]                   # attention output dense + LayerNorm
        out += [(ffn, d), (ffn,), (d, ffn), (d,), (d,), (d,)]  # intermediate, output dense + LayerNorm
    out += [(d, d), (d,)]                                   # pooler
    return out


BERT_LAYER_PARAMS = 16
BERT_FIRST_LAYER_PARAM = 5


def gpt2_small(vocab: int = 50257, d: int = 768, ctx: int = 1024, layers: int = 12) -> list[tuple[int, ...]]:
    """GPT-2 small (LM head tied to the token embedding, so not listed)."""
    out: list[tuple[int, ...]] = [(vocab, d), (ctx, d)]
    for _ in range(layers):
        out += [(d,), (d,), (d, 3 * d), (3 * d,), (d, d), (d,)]   # ln_1, c_attn, attn c_proj
        out += [(d,), (d,), (d, 4 * d), (4 * d,), (4 * d, d), (d,)]  # ln_2, c_fc, mlp c_proj
    out += [(d,), (d,)]
    return out


def numels(shapes) -> list[int]:
    return [int(np.prod(s)) if len(s) else 1 for s in shapes]


# ---------------------------------------------------------------------------
# workload configurations
# ---------------------------------------------------------------------------
F32, BF16 = 0, 1            # dtype codes (match the library's and the oracle's)
REVERSE, FWD_THEN_REVERSE, MEGATRON = 0, 1, 2
ALLREDUCE, REDUCE_SCATTER = 0, 1
MiB = 1 << 20


@dataclass
class Workload:
    name: str
    shapes: list
    W: int
    mode: int
    order: int
    cap_bytes: int
    first_cap_bytes: int
    pad_multiple: int
    dtype: int                 # grad dtype code
    dist: str
    sigma: float
    seed: int
    micro_steps: int = 1       # > 1: no_sync accumulation of this many micro-steps
    unused: list = field(default_factory=list)   # params unused on every replica
    grad_reduce_in_fp32: int = 1
    partial_unused: float = 0.0  # seeded fraction of the other (replica, param) pairs left unused

    @property
    def numels(self) -> list[int]:
        return numels(self.shapes)

    @property
    def nparams(self) -> int:
        return len(self.shapes)

    def dist_of(self, p: int) -> str:
        return "zero" if p in self.unused else self.dist


def c1_mlp() -> Workload:
    return Workload("mlp3_w4_allreduce", mlp3(), 4, ALLREDUCE, REVERSE, 25 * MiB, 1 * MiB, 1,
                    F32, "dyadic12", 1.0, 1001)


def c2_resnet50() -> Workload:
    return Workload("resnet50_w8_allreduce", resnet50(), 8, ALLREDUCE, REVERSE, 25 * MiB, 1 * MiB, 1,
                    F32, "normal", 1e-3, 1002)


def c3_gpt2() -> Workload:
    W = 8
    cap = max(40_000_000, 1_000_000 * W)
    return Workload("gpt2_small_w8_reduce_scatter", gpt2_small(), W, REDUCE_SCATTER, MEGATRON, cap, cap, W,
                    BF16, "normal", 1e-2, 1003)


def c4_bert_large(unused_layer: int = 11) -> Workload:
    first = BERT_FIRST_LAYER_PARAM + unused_layer * BERT_LAYER_PARAMS
    return Workload("bert_large_w4_nosync4_allreduce", bert_large(), 4, ALLREDUCE, REVERSE, 25 * MiB, 1 * MiB, 1,
                    F32, "normal", 1e-3, 1004, micro_steps=4,
                    unused=list(range(first, first + BERT_LAYER_PARAMS)))


def c6_bert_find_unused() -> Workload:
    """BERT-large, W = 4: encoder layer 11 unused by every replica and, as with experts
    that receive no tokens on some ranks, 5% of the other (replica, parameter) pairs
    unused locally -- the find_unused_parameters case."""
    wl = c4_bert_large()
    wl.name = "bert_large_w4_find_unused_allreduce"
    wl.micro_steps = 1
    wl.seed = 1006
    wl.partial_unused = 0.05
    return wl


def c5_sweep_points() -> list[tuple[int, int]]:
    """(bucket bytes, W) of the bandwidth sweep: 1 KiB .. 1 GiB in powers of 4, W in {2, 4, 8, 16}."""
    return [(1024 * 4 ** k, W) for k in range(11) for W in (2, 4, 8, 16)]


def c5_bucket(nbytes: int, W: int) -> Workload:
    n = nbytes // 4
    return Workload(f"sweep_{nbytes}B_w{W}", [(n,)], W, ALLREDUCE, REVERSE, 1 << 62, 1 << 62, 1,
                    F32, "uniform", 1.0, 1005)


ALL = {"c1": c1_mlp, "c2": c2_resnet50, "c3": c3_gpt2, "c4": c4_bert_large, "c6": c6_bert_find_unused}

USED_MAP_STREAM = 1 << 40   # generator stream of the local-used bitmaps (beyond every gradient stream)


POWERSGD_Q_STREAM = 1 << 41   # generator streams of PowerSGD's initial Q matrices (one per tensor)


def powersgd_q0_np(seed: int, tensor: int, n: int, r: int) -> np.ndarray:
    """The initial Q of one tensor (N x R, fp32): the hook's random normal draw,
    stood in for by the generator's ``normal`` values (unit variance)."""
    bits = bits_np(stream_key(seed, POWERSGD_Q_STREAM + tensor), 0, n * r)
    return values_np(bits, "normal", 1.0).reshape(n, r)


def c7_resnet50_powersgd(rank: int = 4) -> Workload:
    """ResNet-50, W = 8, DDP buckets, every bucket reduced through the PowerSGD hook
    at the given rank (the page's example rank is 4)."""
    wl = c2_resnet50()
    wl.name = f"resnet50_w8_powersgd_r{rank}"
    wl.seed = 1007
    return wl


def local_used_np(wl: Workload) -> np.ndarray:
    """[W, P] uint8 local-used bitmap of one iteration: 0 on every replica for the
    parameters in ``wl.unused``; 0 for the seeded fraction ``wl.partial_unused`` of
    the remaining (replica, parameter) pairs; 1 elsewhere."""
    W, P = wl.W, wl.nparams
    used = np.ones((W, P), np.uint8)
    if wl.partial_unused > 0 and P > 0:
        r = bits_np(stream_key(wl.seed, USED_MAP_STREAM), 0, W * P) >> np.uint64(11)
        u = r.astype(np.float64) * 2.0 ** -53
        used[(u < wl.partial_unused).reshape(W, P)] = 0
    if wl.unused:
        used[:, list(wl.unused)] = 0
    return used


# ---------------------------------------------------------------------------
# gradient generation
# ---------------------------------------------------------------------------
def grad_np(wl: Workload, p: int, w: int, m: int = 0, start: int = 0, count: int | None = None) -> np.ndarray:
    """Gradient of parameter p on replica w at micro-step m as fp32 (bf16 workloads: the
    bf16-rounded values widened back to fp32)."""
    n = wl.numels[p]
    count = n - start if count is None else count
    b = bits_np(stream_key(wl.seed, stream_id(p, w, m)), start, count)
    v = values_np(b, wl.dist_of(p), wl.sigma)
    if wl.dtype == BF16:
        v = bf16_bits_to_f32_np(f32_to_bf16_bits_np(v))
    return v


def grad_raw_np(wl: Workload, p: int, w: int, m: int = 0) -> np.ndarray:
    """Gradient in its storage type: float32, or uint16 bf16 bit patterns."""
    b = bits_np(stream_key(wl.seed, stream_id(p, w, m)), 0, wl.numels[p])
    v = values_np(b, wl.dist_of(p), wl.sigma)
    return f32_to_bf16_bits_np(v) if wl.dtype == BF16 else v


def grad_at_np(wl: Workload, p: int, w: int, m: int, indices: np.ndarray) -> np.ndarray:
    """Sampled gradient values (fp32, bf16-rounded for bf16 workloads) at element indices."""
    b = bits_at_np(stream_key(wl.seed, stream_id(p, w, m)), indices)
    v = values_np(b, wl.dist_of(p), wl.sigma)
    if wl.dtype == BF16:
        v = bf16_bits_to_f32_np(f32_to_bf16_bits_np(v))
    return v


def grad_torch(wl: Workload, p: int, w: int, m: int = 0, device="cpu"):
    """The same gradient generated with torch on ``device``, in its storage dtype."""
    import torch

    b = bits_torch(stream_key(wl.seed, stream_id(p, w, m)), 0, wl.numels[p], device)
    v = values_torch(b, wl.dist_of(p), wl.sigma)
    if wl.dtype == BF16:
        v = v.to(torch.bfloat16)
    return v


def bucket_np(nbytes: int, W: int, seed: int = 1005, dist: str = "uniform") -> np.ndarray:
    """W replicas of one fp32 bucket (the sweep's input), shape [W, nbytes/4]."""
    n = nbytes // 4
    out = np.empty((W, n), dtype=np.float32)
    for w in range(W):
        out[w] = values_np(bits_np(stream_key(seed, stream_id(0, w)), 0, n), dist)
    return out


def bucket_torch(nbytes: int, W: int, device, seed: int = 1005, dist: str = "uniform", stride: int | None = None):
    import torch

    n = nbytes // 4
    stride = n if stride is None else stride
    out = torch.zeros((W, stride), dtype=torch.float32, device=device)
    for w in range(W):
        out[w, :n] = values_torch(bits_torch(stream_key(seed, stream_id(0, w)), 0, n, device), dist)
    return out
