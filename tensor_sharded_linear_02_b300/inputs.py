"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds none of the sharded-linear arithmetic: it only draws
numbers.  Both the CUDA path and the host oracle are fed the exact bytes it
returns, generated once on the host.

Generator (counter-based, so any slice can be drawn independently):

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): the i-th output of stream ``s`` is the SplitMix64
  finaliser applied to ``s + (i+1) * 0x9E3779B97F4A7C15`` (mod 2^64).
* Uniform double in [0, 1): the top 53 bits of that output times 2^-53.
* Normal: Box-Muller on consecutive pairs (u1, u2):
  r = sqrt(-2 ln(1 - u1)), z0 = r cos(2 pi u2), z1 = r sin(2 pi u2); scaled by
  the standard deviation.
* bf16 values: the scaled normal rounded to float32, then to bf16 (both round
  to nearest even).  Any deterministic mapping would do for inputs; this one
  is stated so that the bytes can be reproduced.
* Integer values uniform in [lo, hi] (both ends included):
  lo + floor(u * (hi - lo + 1)), stored as float32.

Each tensor draws from its own stream, seed = base_seed * 1000 + index.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def stream_seed(base_seed: int, index: int) -> int:
    return (int(base_seed) * 1000 + int(index)) & 0xFFFFFFFFFFFFFFFF


def _splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def _uniform(seed: int, start: int, count: int) -> np.ndarray:
    z = _splitmix64(seed, start, count)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def _normal_chunk(seed: int, start_pair: int, npairs: int) -> np.ndarray:
    u = _uniform(seed, 2 * start_pair, 2 * npairs)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    t = 2.0 * np.pi * u2
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out


def _f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    u = x32.view(np.uint32).astype(np.uint64)
    nan = np.isnan(x32)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    out[nan] = np.uint16(0x7FC0)
    return out


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """float64 normals N(0, std^2) of the given shape from stream ``seed``."""
    n = int(np.prod(shape))
    npairs = (n + 1) // 2
    chunk_pairs = _CHUNK // 2
    starts = list(range(0, npairs, chunk_pairs))
    out = np.empty(2 * npairs, dtype=np.float64)

    def work(sp):
        cnt = min(chunk_pairs, npairs - sp)
        out[2 * sp: 2 * (sp + cnt)] = _normal_chunk(seed, sp, cnt) * std

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, starts))
    return out[:n].reshape(shape)


def bf16_normal(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, std^2) draws."""
    n = int(np.prod(shape))
    npairs = (n + 1) // 2
    chunk_pairs = _CHUNK // 2
    out = np.empty(2 * npairs, dtype=np.uint16)

    def work(sp):
        cnt = min(chunk_pairs, npairs - sp)
        z = (_normal_chunk(seed, sp, cnt) * std).astype(np.float32)
        out[2 * sp: 2 * (sp + cnt)] = _f32_to_bf16_bits(z)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(0, npairs, chunk_pairs)))
    return out[:n].reshape(shape)


def int_uniform(shape, seed: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """float32 integers uniform in [lo, hi] inclusive."""
    n = int(np.prod(shape))
    u = _uniform(seed, 0, n)
    v = lo + np.floor(u * (hi - lo + 1))
    return v.astype(np.float32).reshape(shape)


def f32_normal(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """float32 normals (rounded to nearest from the double draw)."""
    return normal(shape, seed, std).astype(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact: the low 16 bits are zero)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
