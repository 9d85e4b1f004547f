"""Seeded synthetic inputs, shared by the tests, the bench and the smoke check.

This module holds no attention arithmetic: it draws i.i.d. normal numbers
from a fixed seed and rounds them to the storage type. The same host arrays
feed both the CUDA path (copied to the device) and the fp64 oracle, so both
sides see bit-identical inputs.

Recipe: numpy PCG64 seeded with (seed, stream), standard normal float32,
multiplied by ``scale`` (1/sqrt(d) for q, k, v), then rounded to the storage
type: round-to-nearest-even to bfloat16, or kept as float32. Arrays are
returned as float32 holding exactly representable values of the storage type.
"""

from __future__ import annotations

import numpy as np

# stream ids, so q, k, v and the upstream gradient of one seed are independent
STREAM_Q, STREAM_K, STREAM_V, STREAM_G = 0, 1, 2, 3


def round_to_bf16(x):
    """Round float32 values to the nearest bfloat16 (ties to even); float32 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1))
    rounded = ((bits + bias) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return rounded.view(np.float32).reshape(x.shape)


def normal(shape, seed, stream=0, scale=1.0, dtype="bf16"):
    """i.i.d. N(0, scale^2) values of ``shape``, rounded to ``dtype``.

    ``dtype`` is "bf16" or "f32"; the result is always a float32 array.
    """
    rng = np.random.Generator(np.random.PCG64([int(seed), int(stream)]))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "f32":
        return x
    raise ValueError(f"unknown dtype {dtype!r}")


def qkv(B, H, N, dk, dv, seed, dtype="bf16"):
    """q, k, v of shape [B,H,N,d], each N(0,1)/sqrt(d) rounded to ``dtype``."""
    q = normal((B, H, N, dk), seed, STREAM_Q, 1.0 / np.sqrt(dk), dtype)
    k = normal((B, H, N, dk), seed, STREAM_K, 1.0 / np.sqrt(dk), dtype)
    v = normal((B, H, N, dv), seed, STREAM_V, 1.0 / np.sqrt(dv), dtype)
    return q, k, v


def upstream_grad(B, H, N, dv, seed, dtype="bf16"):
    """dL/dout of shape [B,H,N,dv], N(0,1) rounded to ``dtype``."""
    return normal((B, H, N, dv), seed, STREAM_G, 1.0, dtype)


def decode_token(B, H, dk, dv, seed, step, dtype="bf16"):
    """q, k, v for decode step ``step``: [B,H,d] each, N(0,1)/sqrt(d)."""
    s = int(seed) * 1_000_003 + int(step)
    q = normal((B, H, dk), s, STREAM_Q, 1.0 / np.sqrt(dk), dtype)
    k = normal((B, H, dk), s, STREAM_K, 1.0 / np.sqrt(dk), dtype)
    v = normal((B, H, dv), s, STREAM_V, 1.0 / np.sqrt(dv), dtype)
    return q, k, v
