"""Seeded synthetic inputs, shared by the CUDA path's tests and the oracle's.

This module only draws numbers; it holds none of the method's arithmetic
(no quantisation, no scaling, no GEMM).  Generator: a counter-based SplitMix64
stream (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014; the constants of Vigna's public-domain ``splitmix64.c``) feeding
the Box-Muller transform in fp64, rounded once to fp32.

A stream is identified by ``(seed, tensor_id, slice)``; element ``i`` of a
stream depends only on those and ``i``, so any sub-block can be regenerated
independently (used to draw a bounded sample of a large workload).
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids used by the tests, the smoke check and the benchmark
TID_A, TID_B, TID_X, TID_W = 1, 2, 3, 4

_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, tensor_id: int, slice_id: int) -> np.uint64:
    k = np.array([(seed & 0xFFFFFFFF) | ((tensor_id & 0xFFFF) << 32) | ((slice_id & 0xFFFF) << 48)],
                 dtype=np.uint64)
    return _mix(k + _GAMMA)[0]


def uniform_u64(seed: int, tensor_id: int, slice_id: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit outputs ``start .. start+count-1`` of a stream."""
    key = _key(seed, tensor_id, slice_id)
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(key + ctr * _GAMMA)


def normal(seed: int, tensor_id: int, slice_id: int, shape, sigma: float = 1.0,
           start: int = 0) -> np.ndarray:
    """fp32 N(0, sigma^2) values; element j of the flattened result is element
    ``start + j`` of the stream (pairs share one Box-Muller draw)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    pos = 0
    while pos < n:
        cnt = min(_CHUNK, n - pos)
        g0 = start + pos                   # first global index of this chunk
        p0 = g0 // 2                       # first Box-Muller pair touched
        p1 = (g0 + cnt + 1) // 2           # one past the last pair touched
        u = uniform_u64(seed, tensor_id, slice_id, 2 * p0, 2 * (p1 - p0))
        u1 = ((u[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)   # (0, 1]
        u2 = (u[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)           # [0, 1)
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        off = g0 - 2 * p0
        out[pos:pos + cnt] = (z[off:off + cnt] * sigma).astype(np.float32)
        pos += cnt
    return out.reshape(shape)


def normal_rows(seed: int, tensor_id: int, slice_id: int, n_cols: int, rows, sigma: float = 1.0):
    """Selected rows of a row-major [*, n_cols] normal matrix drawn by ``normal``."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, n_cols), dtype=np.float32)
    for i, r in enumerate(rows):
        out[i] = normal(seed, tensor_id, slice_id, (n_cols,), sigma, start=int(r) * n_cols)
    return out
