"""Seeded synthetic inputs for the BF16 GEMM workloads.

This module is the one thing the CUDA path and the CPU oracle share: it makes
the bf16 bit patterns both of them consume.  It holds the input recipe only --
a counter-based generator, the three value distributions, the scaling and the
rounding of inputs to bf16 -- and none of the GEMM arithmetic.  It imports
neither the library nor the oracle.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used counter-style: output i of stream s is
mix(key(seed, s) + (i + 1) * 0x9E3779B97F4A7C15), where mix is the SplitMix64
finaliser.  The top 53 bits give a uniform u in [0, 1).

Distributions (per workload):
  - "uniform":  2u - 1, i.e. uniform on [-1, 1);
  - "normal":   Box-Muller on consecutive pairs (u1, u2):
                sqrt(-2 ln(1 - u1)) * (cos 2 pi u2, sin 2 pi u2);
  - "int4":     floor(9u) - 4, integers uniform on {-4, ..., 4} (exact in bf16).
Each value is multiplied by ``scale`` (1/sqrt(K) for the scaled workloads) in
binary64 and then rounded to bf16: binary64 -> binary32 by numpy, then
binary32 -> bf16 to nearest even on the bit pattern.  That two-step rounding
is part of the input recipe only; both sides receive the same resulting bits.

Storage: ``matrix(rows, cols, ...)`` returns a C-contiguous uint16 array of
shape (rows, cols).  A (M x K, row-major) is ``matrix(M, K, ...)``; B (K x N,
column-major) is stored as its transpose, ``matrix(N, K, ...)``, so each
column of B is contiguous along K.
"""
from __future__ import annotations

import math

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

STREAM_A = 0
STREAM_B = 1


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(seed * 0x100000001B3 + stream * 0x632BE59BD9B4E019) & 0xFFFFFFFFFFFFFFFF],
                        dtype=np.uint64)
        return _mix(base)[0]


def uniform01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of stream ``stream``, as binary64 in [0, 1)."""
    key = _key(seed, stream)
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = _mix(key + ctr * _GAMMA)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def _values(dist: str, seed: int, stream: int, start: int, count: int) -> np.ndarray:
    if dist == "uniform":
        return 2.0 * uniform01(seed, stream, start, count) - 1.0
    if dist == "int4":
        return np.floor(9.0 * uniform01(seed, stream, start, count)) - 4.0
    if dist == "normal":
        # values start..start+count-1 come from pairs start//2 .. ; take whole pairs
        p0 = start // 2
        p1 = (start + count + 1) // 2
        u = uniform01(seed, stream, 2 * p0, 2 * (p1 - p0))
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))
        t = (2.0 * math.pi) * u2
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        off = start - 2 * p0
        return z[off:off + count]
    raise ValueError(f"unknown distribution {dist!r}")


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """binary64 values -> bf16 bit patterns (via binary32, nearest even twice)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    w = f.view(np.uint32).astype(np.uint64)
    w = (w + np.uint64(0x7FFF) + ((w >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return w.astype(np.uint16)


def matrix(rows: int, cols: int, *, dist: str, seed: int, stream: int,
           scale: float = 1.0) -> np.ndarray:
    """A (rows x cols) C-contiguous uint16 array of bf16 bit patterns.

    Element (r, c) is value number r*cols + c of the stream, times ``scale``.
    """
    n = rows * cols
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        v = _values(dist, seed, stream, s, c)
        if scale != 1.0:
            v = v * scale
        out[s:s + c] = to_bf16_bits(v)
    return out.reshape(rows, cols)


# The workloads (distribution, scale) by name; the shapes live with the callers.
def workload_operands(M: int, N: int, K: int, *, dist: str, scaled: bool, seed: int):
    """(A, B_t): A is M x K row-major, B_t is B's column-major storage (N x K)."""
    scale = 1.0 / math.sqrt(K) if (scaled and K > 0) else 1.0
    A = matrix(M, K, dist=dist, seed=seed, stream=STREAM_A, scale=scale)
    Bt = matrix(N, K, dist=dist, seed=seed, stream=STREAM_B, scale=scale)
    return A, Bt


DEFAULT_SEED = 20261202
