"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws numbers; it holds none of the attention arithmetic.

Recipe (the pages name no dataset; these stand in for real activations):

* Q, K, V and dO are iid N(0, 1): ``numpy.random.default_rng(seed)
  .standard_normal(shape, dtype=float32)``, rounded to bf16 by
  round-to-nearest-even on the bit pattern, and returned as uint16 bf16 bit
  patterns, so both the CUDA path and the oracle see the same bytes.  For
  fp16 runs the same float32 draws are rounded to IEEE binary16 (numpy's
  float32 -> float16 cast, round-to-nearest-even) and returned as float16.
* Seeds: Q = s, K = s + 1, V = s + 2, dO = s + 3.
* Packed variable-length batches draw their lengths with
  ``default_rng(seed).integers(lo, hi + 1, size=n)`` (both ends inclusive).
"""
from __future__ import annotations

import numpy as np


def bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Inputs are finite (normal draws), so no NaN special case is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def normal_bf16(shape, seed: int) -> np.ndarray:
    """iid N(0,1) drawn in float32 from ``default_rng(seed)``, as bf16 bit patterns."""
    x = np.random.default_rng(seed).standard_normal(size=shape, dtype=np.float32)
    return bf16_bits_rne(x)


def normal_f16(shape, seed: int) -> np.ndarray:
    """iid N(0,1) drawn in float32 from ``default_rng(seed)``, rounded to float16."""
    x = np.random.default_rng(seed).standard_normal(size=shape, dtype=np.float32)
    return x.astype(np.float16)


def varlen_lengths(seed: int, n: int = 16, lo: int = 256, hi: int = 8192) -> np.ndarray:
    """Sequence lengths drawn uniformly from [lo, hi] (inclusive)."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=n).astype(np.int64)


def cu_seqlens_of(lengths) -> np.ndarray:
    """Exclusive prefix sum [0, l0, l0+l1, ...] as int32."""
    lengths = np.asarray(lengths, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def attention_inputs(q_shape, kv_shape, seed: int, with_dout: bool = True, dtype: str = "bf16"):
    """Q, K, V (and dO) with the seed offsets of the recipe: bf16 bit patterns
    (dtype "bf16") or float16 arrays (dtype "f16")."""
    draws = {"bf16": normal_bf16, "f16": normal_f16}
    if dtype not in draws:
        raise ValueError(f"dtype must be 'bf16' or 'f16', got {dtype!r}")
    draw = draws[dtype]
    out = {
        "q": draw(q_shape, seed),
        "k": draw(kv_shape, seed + 1),
        "v": draw(kv_shape, seed + 2),
    }
    if with_dout:
        out["dout"] = draw(q_shape, seed + 3)
    return out
