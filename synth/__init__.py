"""Seeded synthetic inputs for the GEMM / implicit-GEMM convolution workloads.

This module is the one piece of code that both the CPU oracle's tests and the
GPU path's tests and benchmark use.  It draws random numbers and nothing else:
it holds none of the arithmetic of the method (no products, sums, zero-point
corrections, rounding of results or index mapping of the convolution).

Generator
---------
Every value is a pure function of ``(seed, tensor_id, index)``: the 64-bit
SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) applied to ``seed ^ (tensor_id << 48) ^
index``.  It is counter based, so any element can be regenerated on its own
and the order of generation does not matter.

* uniform real in [0, 1):   ``(h >> 11) * 2**-53``
* uniform integer in [lo, hi] (inclusive): ``lo + (((h >> 11) * n) >> 53)``,
  ``n = hi - lo + 1``
* standard normal: Box-Muller on the hashes of counters ``2*i`` and
  ``2*i + 1``, in float64
* fp16 / fp32 values are drawn in float64 and rounded once to the target type
  (round to nearest, ties to even, by numpy's conversion)

Workloads (one per benchmark configuration; the seed is ``20261202 + cfg``):

1. fp16 GEMM 256^3, A and B uniform[-1, 1], fp32 C
2. int8 GEMM 1024^3 with zero points: A_q, B_q uint8 uniform[0, 255],
   zA = 128, zB = 121, scale = 1/4096
3. fp16 GEMM 4096^3, A and B N(0, 1), fp16 C
4. 3x3 convolution, x NHWC 256x14x14x256 N(0, 1), w KRSC 512x3x3x256 with
   std 1/sqrt(2304) = 1/48, pad 1, stride 1
5. int8 GEMM 8192^3: A_q uint8 uniform[0, 255] with per-row zA_i uniform
   integers in [100, 156]; B_q int8 uniform[-127, 127], zB = 0; per-column
   fp32 scale uniform[1e-4, 1e-3]
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "SEED_BASE", "seed_for", "splitmix64", "hashes", "uniform01",
    "uniform_f16", "normal_f16", "normal_bf16_bits", "uniform_int", "uniform_f32",
    "gemm_f16_inputs", "gemm_s8_inputs", "conv_inputs", "workload",
    "WORKLOADS",
]

SEED_BASE = 20261202

# tensor ids: which stream of the counter-based generator a tensor draws from
TID_A, TID_B, TID_ZA, TID_ZB, TID_SCALE, TID_X, TID_W = 1, 2, 3, 4, 5, 6, 7

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_CHUNK = 1 << 22


def seed_for(cfg: int) -> int:
    return SEED_BASE + int(cfg)


def splitmix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z += np.uint64(0x9E3779B97F4A7C15)
        z ^= z >> np.uint64(30)
        z *= np.uint64(0xBF58476D1CE4E5B9)
        z ^= z >> np.uint64(27)
        z *= np.uint64(0x94D049BB133111EB)
        z ^= z >> np.uint64(31)
    return z


def hashes(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    """Hashes of counters ``start .. start+count-1`` of stream ``(seed, tid)``."""
    key = np.uint64((int(seed) ^ (int(tid) << 48)) & 0xFFFFFFFFFFFFFFFF)
    idx = np.arange(start, start + count, dtype=np.uint64)
    return splitmix64(idx ^ key)


def _fill(n: int, fn, dtype) -> np.ndarray:
    out = np.empty(n, dtype=dtype)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = fn(s, c)
    return out


def uniform01(seed: int, tid: int, n: int) -> np.ndarray:
    return _fill(n, lambda s, c: (hashes(seed, tid, s, c) >> np.uint64(11)).astype(np.float64)
                 * (2.0 ** -53), np.float64)


def uniform_f16(seed: int, tid: int, shape, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))

    def fn(s, c):
        u = (hashes(seed, tid, s, c) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        return (lo + (hi - lo) * u).astype(np.float16)
    return _fill(n, fn, np.float16).reshape(shape)


def normal_f16(seed: int, tid: int, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))

    def fn(s, c):
        h = hashes(seed, tid, 2 * s, 2 * c)
        u1 = ((h[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
        u2 = (h[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return (std * z).astype(np.float16)
    return _fill(n, fn, np.float16).reshape(shape)


def normal_bf16_bits(seed: int, tid: int, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std) drawn in float64, rounded once to bfloat16 (RNE, by torch's
    conversion); returned as the uint16 bit patterns."""
    import torch
    n = int(np.prod(shape))

    def fn(s, c):
        h = hashes(seed, tid, 2 * s, 2 * c)
        u1 = ((h[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u2 = (h[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        z = std * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return _fill(n, fn, np.uint16).reshape(shape)


def uniform_int(seed: int, tid: int, shape, lo: int, hi: int, dtype) -> np.ndarray:
    """Uniform integers in [lo, hi] inclusive."""
    n = int(np.prod(shape))
    span = np.uint64(hi - lo + 1)

    def fn(s, c):
        h = hashes(seed, tid, s, c) >> np.uint64(11)
        with np.errstate(over="ignore"):
            r = (h * span) >> np.uint64(53)
        return (r.astype(np.int64) + lo).astype(dtype)
    return _fill(n, fn, dtype).reshape(shape)


def uniform_f32(seed: int, tid: int, shape, lo: float, hi: float) -> np.ndarray:
    n = int(np.prod(shape))

    def fn(s, c):
        u = (hashes(seed, tid, s, c) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        return (lo + (hi - lo) * u).astype(np.float32)
    return _fill(n, fn, np.float32).reshape(shape)


# --------------------------------------------------------------------------
# workload builders
# --------------------------------------------------------------------------

def gemm_f16_inputs(M: int, N: int, K: int, seed: int, dist: str = "uniform"):
    """A (M x K row-major) and Bt (N x K row-major, i.e. B column-major), fp16."""
    if dist == "uniform":
        A = uniform_f16(seed, TID_A, (M, K))
        Bt = uniform_f16(seed, TID_B, (N, K))
    elif dist == "normal":
        A = normal_f16(seed, TID_A, (M, K))
        Bt = normal_f16(seed, TID_B, (N, K))
    else:
        raise ValueError(dist)
    return {"A": A, "Bt": Bt}


def gemm_s8_inputs(M: int, N: int, K: int, seed: int, kind: str):
    """Quantised operands.

    kind "per_tensor": A_q, B_q uint8 in [0, 255], zA = 128, zB = 121,
    scale = 1/4096.
    kind "per_row": A_q uint8 in [0, 255], zA_i integers in [100, 156];
    B_q int8 in [-127, 127], zB = 0, scale_j fp32 in [1e-4, 1e-3].
    """
    if kind == "per_tensor":
        return {
            "A": uniform_int(seed, TID_A, (M, K), 0, 255, np.uint8), "a_signed": 0,
            "Bt": uniform_int(seed, TID_B, (N, K), 0, 255, np.uint8), "b_signed": 0,
            "zA": 128, "zA_row": None, "zB": 121, "zB_col": None,
            "scale": float(np.float32(1.0 / 4096.0)), "scale_col": None,
        }
    if kind == "per_row":
        return {
            "A": uniform_int(seed, TID_A, (M, K), 0, 255, np.uint8), "a_signed": 0,
            "Bt": uniform_int(seed, TID_B, (N, K), -127, 127, np.int8), "b_signed": 1,
            "zA": 0, "zA_row": uniform_int(seed, TID_ZA, (M,), 100, 156, np.int32),
            "zB": 0, "zB_col": None,
            "scale": 0.0, "scale_col": uniform_f32(seed, TID_SCALE, (N,), 1e-4, 1e-3),
        }
    raise ValueError(kind)


def conv_inputs(N: int, H: int, W: int, C: int, K: int, R: int, S: int, seed: int,
                w_std: float | None = None):
    """x NHWC fp16 N(0, 1); w KRSC fp16 N(0, w_std), w_std = 1/sqrt(R*S*C) by default."""
    if w_std is None:
        w_std = 1.0 / np.sqrt(R * S * C)
    return {"x": normal_f16(seed, TID_X, (N, H, W, C)),
            "w": normal_f16(seed, TID_W, (K, R, S, C), std=w_std)}


WORKLOADS = {
    1: dict(op="gemm_f16", M=256, N=256, K=256, dist="uniform", out="f32"),
    2: dict(op="gemm_s8_zp", M=1024, N=1024, K=1024, kind="per_tensor"),
    3: dict(op="gemm_f16", M=4096, N=4096, K=4096, dist="normal", out="f16"),
    4: dict(op="conv", N=256, H=14, W=14, C=256, K=512, R=3, S=3, pad=1, stride=1),
    5: dict(op="gemm_s8_zp", M=8192, N=8192, K=8192, kind="per_row"),
}


def workload(cfg: int):
    """Inputs and parameters of benchmark configuration ``cfg`` (1..5)."""
    p = dict(WORKLOADS[cfg])
    seed = seed_for(cfg)
    if p["op"] == "gemm_f16":
        p.update(gemm_f16_inputs(p["M"], p["N"], p["K"], seed, p["dist"]))
    elif p["op"] == "gemm_s8_zp":
        p.update(gemm_s8_inputs(p["M"], p["N"], p["K"], seed, p["kind"]))
    elif p["op"] == "conv":
        p.update(conv_inputs(p["N"], p["H"], p["W"], p["C"], p["K"], p["R"], p["S"], seed))
    p["seed"] = seed
    return p
