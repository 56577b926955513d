"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws numbers and rounds
them to the storage type, so that the CUDA library and the CPU oracle see the
same bytes.

Recipe
------
* Uniform 64-bit words come from SplitMix64 (Steele, Lea & Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014): the state advances
  by 0x9E3779B97F4A7C15 and each word is the state passed through the
  published 30/27/31 xor-shift-multiply finaliser.
* Word w becomes a uniform u = ((w >> 11) + 1) * 2^-53 in (0, 1].
* Normals come from the Box-Muller transform on consecutive pairs (u1, u2):
  r = sqrt(-2 ln u1); element 2t = r cos(2 pi u2), element 2t+1 = r sin(2 pi u2).
  All of this is fp64.
* bf16 tensors are the fp64 normals rounded once, to nearest-even, to bf16
  (no intermediate fp32 rounding).  fp32 tensors are rounded once to fp32.
* Tensor seeds: 0x5EED0000 + 16 * config_id + tensor_id with Q=0, K=1, V=2,
  dO=3.  The long-logit workload multiplies the rounded Q by 8 (exact in bf16).
* Block-varying magnitudes (FP8 block quantization tests): every 128 rows
  of a head multiplied by 2^e, e drawn uniformly from a small set by
  SplitMix64 from the seed xor 0xB10C (exact: powers of two).
* Block masks (block-sparse workloads): entry kept when a SplitMix64 uniform
  is below the density.

The named workloads are the five shapes the library is measured and checked
on (see ``WORKLOADS``).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TENSOR_IDS = {"Q": 0, "K": 1, "V": 2, "dO": 3}


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Words start .. start+count-1 of the SplitMix64 stream for `seed`."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + idx * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def normals(seed: int, start: int, count: int) -> np.ndarray:
    """fp64 standard normals start .. start+count-1 of the stream (start even)."""
    if start % 2:
        raise ValueError("start must be even (normals come in Box-Muller pairs)")
    npairs = (count + 1) // 2
    w = splitmix64(seed, start, 2 * npairs)
    u = ((w >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * math.pi * u2)
    out[1::2] = r * np.sin(2.0 * math.pi * u2)
    return out[:count]


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns (uint16), one round-to-nearest-even step.

    bf16 keeps 8 significant bits, fp64 has 53, so the low 45 bits of the
    fp64 pattern are rounded away.  Values are assumed finite and within the
    normal bf16 range (true for the normal draws used here).
    """
    b = np.ascontiguousarray(x, dtype=np.float64).view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    with np.errstate(over="ignore"):
        r = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    f32 = r.view(np.float64).astype(np.float32)  # exact: r has 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


@dataclass(frozen=True)
class Workload:
    name: str
    config_id: int
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    dtype: str          # "bf16" or "f32"
    q_mul: float = 1.0  # multiplier applied to Q after rounding
    backward: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def shape(self, tensor: str):
        H = self.Hkv if tensor in ("K", "V") else self.Hq
        return (self.B, H, self.N, self.d)

    def fwd_flops(self) -> float:
        f = 4.0 * self.N * self.N * self.d * self.Hq * self.B
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()


WORKLOADS = {
    "c1": Workload("c1: single head B1 H1 N256 d64 fp32, non-causal, forward only",
                   1, 1, 1, 1, 256, 64, False, "f32", backward=False),
    "c2": Workload("c2: B4 H16 N1024 d64 bf16, non-causal", 2, 4, 16, 16, 1024, 64, False, "bf16"),
    "c3": Workload("c3: B2 H32 N4096 d128 bf16, causal, Q x8", 3, 2, 32, 32, 4096, 128, True,
                   "bf16", q_mul=8.0),
    "c4": Workload("c4: GQA B1 Hq32 Hkv8 N16384 d128 bf16, causal", 4, 1, 32, 8, 16384, 128,
                   True, "bf16"),
    "c5": Workload("c5: long context B1 H8 N131072 d128 bf16, causal", 5, 1, 8, 8, 131072, 128,
                   True, "bf16"),
}


def tensor_seed(config_id: int, tensor: str) -> int:
    return 0x5EED0000 + 16 * config_id + TENSOR_IDS[tensor]


def make_tensor(seed: int, shape, dtype: str, mul: float = 1.0,
                chunk: int = 1 << 24) -> np.ndarray:
    """Seeded tensor of iid N(0,1) draws rounded once to `dtype`.

    Returns uint16 bf16 bit patterns for "bf16" and float32 for "f32".
    `mul` must be a power of two (it is applied after rounding and must be exact).
    """
    n = int(np.prod(shape))
    if dtype == "bf16":
        out = np.empty(n, dtype=np.uint16)
    elif dtype == "f32":
        out = np.empty(n, dtype=np.float32)
    else:
        raise ValueError(dtype)
    if mul != 1.0 and math.frexp(mul)[0] != 0.5:
        raise ValueError("mul must be a power of two")
    for s in range(0, n, chunk):
        cnt = min(chunk, n - s)
        x = normals(seed, s, cnt)
        if dtype == "bf16":
            bits = round_to_bf16_bits(x)
            if mul != 1.0:
                bits = round_to_bf16_bits(bf16_bits_to_f64(bits) * mul)
            out[s:s + cnt] = bits
        else:
            out[s:s + cnt] = (x.astype(np.float32) * np.float32(mul))
    return out.reshape(shape)


def make_blocky_tensor(seed: int, shape, block: int = 128, exps=(-1, 0, 1)) -> np.ndarray:
    """bf16 bits of make_tensor(seed, shape) with every `block` rows of each head
    multiplied by 2^e, e drawn uniformly from `exps` (exact: powers of two).

    Block quantization gives each 128-row block its own scale; varying the
    magnitude per block makes a wrong block index visible in the output."""
    base = make_tensor(seed, shape, "bf16")
    *lead, N, d = shape
    heads = int(np.prod(lead)) if lead else 1
    T = -(-N // block)
    words = splitmix64(seed ^ 0xB10C, 0, heads * T)
    e = np.asarray(exps, dtype=np.float64)[(words % np.uint64(len(exps))).astype(np.int64)].reshape(heads, T)
    mul = np.repeat(np.exp2(e), block, axis=1)[:, :N]
    x = bf16_bits_to_f64(base).reshape(heads, N, d) * mul[:, :, None]
    return round_to_bf16_bits(x).reshape(shape)


def random_block_mask(seed: int, heads: int, T: int, density: float) -> np.ndarray:
    """uint8 [heads, T, T] block mask, each entry kept with probability `density`
    (uniforms from the SplitMix64 stream of `seed`)."""
    u = (splitmix64(seed, 0, heads * T * T) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return (u < density).astype(np.uint8).reshape(heads, T, T)


def workload_tensors(w: Workload, names=("Q", "K", "V", "dO"), shape_override=None):
    """The seeded tensors of a workload as numpy arrays (bf16 bits or fp32)."""
    out = {}
    for t in names:
        shape = w.shape(t) if shape_override is None else shape_override[t]
        mul = w.q_mul if t == "Q" else 1.0
        out[t] = make_tensor(tensor_seed(w.config_id, t), shape, w.dtype, mul)
    return out


def to_f64(a: np.ndarray) -> np.ndarray:
    """Exact fp64 view of a generated tensor (bf16 bits or fp32)."""
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def sample_rows(seed: int, total: int, count: int, must=()) -> np.ndarray:
    """Seeded, sorted, distinct row indices in [0, total), always containing `must`."""
    words = splitmix64(seed, 0, 4 * count + 16)
    picks = list(dict.fromkeys(int(m) for m in must if 0 <= m < total))
    for w in words:
        if len(picks) >= min(count, total):
            break
        r = int(w % np.uint64(total))
        if r not in picks:
            picks.append(r)
    return np.array(sorted(picks), dtype=np.int64)
