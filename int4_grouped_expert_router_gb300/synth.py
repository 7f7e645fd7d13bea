"""Seeded synthetic inputs for the MoE decode block.

This module only draws random numbers and lays them out in the input formats the
library accepts (packed int4 bytes, f32 scales, f32/bf16 activations, router
weights and biases). It contains none of the routed-expert arithmetic, so both
the CPU oracle and the CUDA path can take their inputs from it.

Generator: a counter-based SplitMix64 stream (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014): the i-th 64-bit word
of stream ``seed`` is ``mix64(seed + (i + 1) * 0x9E3779B97F4A7C15)``. Because
word i depends only on (seed, i), any expert's bytes can be regenerated alone,
on the host with numpy or on a device with torch, and the two agree bit for bit
(integer arithmetic only; uniform floats use one exact int->double scaling).
Normals use the Box-Muller transform in float64 and are drawn on the host only.
"""
from __future__ import annotations

import zlib

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)
BASE_SEED = 20261202

_TWO_M53 = float(2.0 ** -53)


def stream_seed(base: int, *names) -> int:
    """Derive an independent 64-bit stream id from a base seed and a name path."""
    s = np.uint64(base & 0xFFFFFFFFFFFFFFFF)
    for n in names:
        h = np.uint64(zlib.crc32(str(n).encode()) & 0xFFFFFFFF)
        with np.errstate(over="ignore"):
            s = _mix64(s ^ (h * GOLDEN))
    return int(s)


def _mix64(z):
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * M1
        z = (z ^ (z >> np.uint64(27))) * M2
        return z ^ (z >> np.uint64(31))


def u64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Words start..start+n-1 of the counter-based SplitMix64 stream ``seed``."""
    ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + ctr * GOLDEN
    return _mix64(z)


def u64_torch(seed: int, n: int, device="cpu"):
    """Same words as :func:`u64` (start=0), computed with torch int64 ops on ``device``."""
    import torch

    def c(v):  # reinterpret an unsigned 64-bit constant as signed int64
        v &= 0xFFFFFFFFFFFFFFFF
        return v - (1 << 64) if v >= (1 << 63) else v

    def lsr(z, k):  # logical right shift on int64
        return (z >> k) & ((1 << (64 - k)) - 1)

    ctr = torch.arange(1, n + 1, dtype=torch.int64, device=device)
    z = ctr * c(0x9E3779B97F4A7C15) + c(seed)
    z = (z ^ lsr(z, 30)) * c(0xBF58476D1CE4E5B9)
    z = (z ^ lsr(z, 27)) * c(0x94D049BB133111EB)
    return z ^ lsr(z, 31)


def random_bytes(seed: int, nbytes: int) -> np.ndarray:
    """``nbytes`` uniform bytes (little-endian bytes of the u64 stream)."""
    w = u64(seed, (nbytes + 7) // 8)
    return w.astype("<u8").view(np.uint8)[:nbytes].copy()


def random_bytes_torch(seed: int, nbytes: int, device="cpu"):
    import torch

    w = u64_torch(seed, (nbytes + 7) // 8, device)
    b = w.view(torch.uint8)  # little-endian on every supported host and GPU
    return b[:nbytes].clone()


def uniform(seed: int, n: int, lo: float, hi: float, dtype=np.float32) -> np.ndarray:
    """U(lo, hi): the top 53 bits of each word scaled exactly to [0, 1), then f64 affine."""
    u = (u64(seed, n) >> np.uint64(11)).astype(np.float64) * _TWO_M53
    return (lo + (hi - lo) * u).astype(dtype)


def uniform_torch(seed: int, n: int, lo: float, hi: float, device="cpu"):
    import torch

    w = u64_torch(seed, n, device)
    top = ((w >> 11) & ((1 << 53) - 1)).to(torch.float64) * _TWO_M53
    return (lo + (hi - lo) * top).to(torch.float32)


def normal(seed: int, n: int, std: float = 1.0, dtype=np.float32) -> np.ndarray:
    """N(0, std^2) by Box-Muller on pairs of uniform words (host only)."""
    m = (n + 1) // 2
    w = u64(seed, 2 * m)
    u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * _TWO_M53  # (0, 1]
    u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * _TWO_M53
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return (std * z[:n]).astype(dtype)


def permutation(seed: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n) (sort of n random words; ties impossible in practice)."""
    return np.argsort(u64(seed, n), kind="stable")


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round f32 values to bfloat16 (round to nearest even); returns the uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = a.view(np.uint32).astype(np.uint64)
    rounding = ((b >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    out = ((b + rounding) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(a)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------------------------
# Workload recipes: shapes and value distributions of the decode layer and its variants.
# --------------------------------------------------------------------------------------------

def packed_row_bytes(cols: int) -> int:
    return (cols + 1) // 2


def scale_count(rows: int, cols: int, gs: int) -> int:
    return rows if gs == 0 else rows * ((cols + gs - 1) // gs)


def expert_tensor(seed: int, rows: int, cols: int, gs: int, scale_lo=0.005, scale_hi=0.02):
    """One int4 weight tensor: uniform packed bytes [rows x ceil(cols/2)] and U(lo, hi) f32 scales."""
    rb = packed_row_bytes(cols)
    packed = random_bytes(stream_seed(seed, "packed"), rows * rb).reshape(rows, rb)
    scales = uniform(stream_seed(seed, "scales"), scale_count(rows, cols, gs), scale_lo, scale_hi)
    return packed, scales


def expert_tensor_torch(seed: int, rows: int, cols: int, gs: int, device, scale_lo=0.005, scale_hi=0.02):
    """Same bytes and scales as :func:`expert_tensor`, generated on ``device`` with torch."""
    rb = packed_row_bytes(cols)
    packed = random_bytes_torch(stream_seed(seed, "packed"), rows * rb, device).reshape(rows, rb)
    scales = uniform_torch(stream_seed(seed, "scales"), scale_count(rows, cols, gs), scale_lo, scale_hi, device)
    return packed, scales


def gaussian_nibble_bytes(seed: int, nbytes: int, sigma: float = 2.5) -> np.ndarray:
    """Packed bytes whose nibbles follow a rounded normal centred between 7 and 8 (std ``sigma``, clipped
    to 0..15): the shape of int4-quantised weights, whose values crowd the middle of the code range."""
    z = normal(seed, 2 * nbytes, std=sigma).astype(np.float64)
    q = np.clip(np.floor(z + 8.0), 0, 15).astype(np.uint8)
    return (q[0::2] | (q[1::2] << 4)).astype(np.uint8)


def expert_seed(base: int, e: int, which: str) -> int:
    return stream_seed(base, "expert", e, which)


def zipf_bias(seed: int, E: int, s: float = 1.1, lam: float = 0.25) -> np.ndarray:
    """Router bias with a Zipf(s) expert-popularity skew: U(-0.1, 0.1) + lam * ln p_rank.

    p_rank is proportional to rank^-s, ranks assigned by a seeded permutation.
    """
    base = uniform(stream_seed(seed, "bias"), E, -0.1, 0.1).astype(np.float64)
    rank = np.empty(E, dtype=np.int64)
    rank[permutation(stream_seed(seed, "rank"), E)] = np.arange(1, E + 1)
    p = rank.astype(np.float64) ** (-s)
    p /= p.sum()
    return (base + lam * np.log(p)).astype(np.float32)


def router_inputs(seed: int, S: int, D: int, E: int, zipf: bool = False, zipf_lambda: float = 0.25):
    """x ~ N(0,1) [S x D] f32, Wr ~ N(0, 0.02^2) [E x D] f32, bias [E] f32 (Zipf-skewed if zipf)."""
    x = normal(stream_seed(seed, "x"), S * D).reshape(S, D)
    Wr = normal(stream_seed(seed, "Wr"), E * D, std=0.02).reshape(E, D)
    bias = zipf_bias(seed, E, lam=zipf_lambda) if zipf else uniform(stream_seed(seed, "bias"), E, -0.1, 0.1)
    return x, Wr, bias
