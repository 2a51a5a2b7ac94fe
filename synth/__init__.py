"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds none of the FP8 method's arithmetic: it only draws random
numbers and rounds them to the input dtypes (BF16 bit patterns, FP32).  Both
the CUDA library and the CPU oracle receive the very same arrays.

Generator (counter based, so any element can be drawn independently):

* ``splitmix64``: state_i = key + (i + 1) * 0x9E3779B97F4A7C15 (mod 2^64),
  output = mix(state_i) with Steele/Lea/Flood's SplitMix64 finaliser.
* ``key`` = mix(seed * 0xD1B54A32D192ED03 + stream), so that different
  ``(seed, stream)`` pairs give unrelated sequences.
* uniform u = (output >> 11) * 2^-53 in [0, 1).
* normals by Box-Muller in float64: element 2j and 2j+1 come from the pair
  (u_{2j}, u_{2j+1}): r = sqrt(-2 ln(1 - u_{2j})), n = r cos / r sin(2 pi u_{2j+1}).
* BF16 = round-to-nearest-even of the float32 value (float64 -> float32 by
  numpy, then the upper 16 bits with RNE).

Workload laws (the pages give shapes only as model classes; the laws are the
benchmark's):

* "N(0, sigma) + 0.1% outliers x f": every element is independently an
  outlier with probability 1e-3 (its own uniform stream) and is multiplied by
  f before rounding to BF16.
* "signed lognormal": |x| = exp(N(mu, sigma^2)) * scale, sign from a third
  uniform stream.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_SEEDMUL = 0xD1B54A32D192ED03
_MASK64 = (1 << 64) - 1

STREAM_NORMAL = 1
STREAM_OUTLIER = 2
STREAM_SIGN = 3

_CHUNK = 1 << 22


def _mix_scalar(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def _key(seed: int, stream: int) -> np.uint64:
    return np.uint64(_mix_scalar(seed * _SEEDMUL + stream))


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of stream ``(seed, stream)`` (uint64)."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(_key(seed, stream) + idx * _GOLDEN)


def uniform(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniform float64 in [0, 1) with 53 random bits."""
    return (splitmix64(seed, stream, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _normal_chunk(seed: int, start: int, count: int) -> np.ndarray:
    # Box-Muller over aligned pairs; ``start`` is even.
    u = uniform(seed, STREAM_NORMAL, start, count + (count & 1))
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    t = 2.0 * np.pi * u2
    out = np.empty(u.shape[0], dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:count]


def _chunked(n: int, fill) -> None:
    """Run ``fill(start, count)`` over fixed chunks on a thread pool (numpy releases the GIL)."""
    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        for s in starts:
            fill(s, min(_CHUNK, n - s))
        return
    workers = min(len(starts), os.cpu_count() or 1, 16)
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda s: fill(s, min(_CHUNK, n - s)), starts))


def standard_normal(seed: int, n: int) -> np.ndarray:
    """``n`` standard normals (float64), chunked to bound memory."""
    out = np.empty(n, dtype=np.float64)

    def fill(s, c):
        out[s:s + c] = _normal_chunk(seed, s, c)
    _chunked(n, fill)
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns (uint16), round to nearest even; NaN kept quiet."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    rounded = (u + (0x7FFF + ((u >> 16) & 1))) >> 16
    out = np.where(nan, (u >> 16) | 0x0040, rounded)
    return out.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_normal(shape, seed: int, std: float = 1.0, outlier_p: float = 0.0,
                outlier_scale: float = 1.0) -> np.ndarray:
    """BF16 bits of N(0, std) with independent outliers (prob ``outlier_p``) x ``outlier_scale``."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)

    def fill(s, c):
        v = _normal_chunk(seed, s, c) * std
        if outlier_p > 0.0:
            o = uniform(seed, STREAM_OUTLIER, s, c) < outlier_p
            v = np.where(o, v * outlier_scale, v)
        out[s:s + c] = f32_to_bf16_bits(v.astype(np.float32))
    _chunked(n, fill)
    return out.reshape(shape)


def bf16_signed_lognormal(shape, seed: int, mu: float, sigma: float,
                          scale: float = 1.0) -> np.ndarray:
    """BF16 bits of +-exp(N(mu, sigma^2)) * scale, sign uniform."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)

    def fill(s, c):
        mag = np.exp(mu + sigma * _normal_chunk(seed, s, c)) * scale
        neg = uniform(seed, STREAM_SIGN, s, c) < 0.5
        out[s:s + c] = f32_to_bf16_bits(np.where(neg, -mag, mag).astype(np.float32))
    _chunked(n, fill)
    return out.reshape(shape)


def f32_normal(shape, seed: int, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return (standard_normal(seed, n) * std).astype(np.float32).reshape(shape)


# ---------------------------------------------------------------------------
# The five benchmark workloads (shapes and laws; see the module docstring).
# ---------------------------------------------------------------------------

def tiny_fprop(seed: int = 0):
    """Tiny FP8 Linear fprop: X [256,512], W [256,512], N(0,1) + 0.1% outliers x100."""
    x = bf16_normal((256, 512), seed, 1.0, 1e-3, 100.0)
    w = bf16_normal((256, 512), seed + 1000, 1.0, 1e-3, 100.0)
    return x, w


def qkv_fprop(seed: int = 0, m: int = 8192, hidden: int = 4096, n_qkv: int = 6144):
    """Dense attention QKV projection (8B class): X [8192,4096] N(0,1)+0.1% x50, W [6144,4096] N(0,0.02)."""
    x = bf16_normal((m, hidden), seed, 1.0, 1e-3, 50.0)
    w = bf16_normal((n_qkv, hidden), seed + 1000, 0.02)
    return x, w


def mlp_step(seed: int = 0, m: int = 8192, hidden: int = 4096, ffn: int = 14336):
    """Dense SwiGLU MLP step: X [m,h] (N(0,1)+0.1% x50), W_gu [2f,h], W_down [h,f] N(0,0.02), dY [m,h] N(0,1e-3)."""
    x = bf16_normal((m, hidden), seed, 1.0, 1e-3, 50.0)
    w_gu = bf16_normal((2 * ffn, hidden), seed + 1000, 0.02)
    w_down = bf16_normal((hidden, ffn), seed + 2000, 0.02)
    dy = bf16_normal((m, hidden), seed + 3000, 1e-3)
    return x, w_gu, w_down, dy


def delayed_step_inputs(t: int, m: int = 16384, hidden: int = 4096, n_out: int = 4096):
    """Per-tensor delayed-scaling Linear, step t (seed t): drifting lognormal X and dY, fixed W."""
    drift = 1.5 ** (t // 8)
    x = bf16_signed_lognormal((m, hidden), t, 0.0, 1.5, drift)
    dy = bf16_signed_lognormal((m, n_out), 100000 + t, float(np.log(1e-3)), 2.5, drift)
    return x, dy


def delayed_weight(hidden: int = 4096, n_out: int = 4096):
    return bf16_normal((n_out, hidden), 7, 0.02)


def moe_inputs(tokens: int = 8192, hidden: int = 2048, experts: int = 128, ffn: int = 768,
               seed: int = 0):
    """MoE grouped expert GEMM (30B-A3B class): X [T,h], router logits [T,E], W_gu [E,2f,h], W_down [E,h,f]."""
    x = bf16_normal((tokens, hidden), seed, 1.0, 1e-3, 50.0)
    logits = f32_normal((tokens, experts), seed + 1)
    w_gu = bf16_normal((experts, 2 * ffn, hidden), seed + 2, 0.02)
    w_down = bf16_normal((experts, hidden, ffn), seed + 3, 0.02)
    return x, logits, w_gu, w_down
