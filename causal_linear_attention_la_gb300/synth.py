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

from concurrent.futures import ThreadPoolExecutor

import numpy as np

# stream ids, so q, k, v and the upstream gradient of one seed are independent
STREAM_Q, STREAM_K, STREAM_V, STREAM_G = 0, 1, 2, 3


def round_to_bf16(x, inplace=False):
    """Round finite float32 values to the nearest bfloat16 (ties to even).

    Returns float32. Works on the bit pattern: add 0x7FFF plus the lowest kept
    bit, then clear the low 16 bits (no overflow for finite inputs).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not inplace:
        x = x.copy()
    bits = x.view(np.uint32)
    bias = bits >> np.uint32(16)
    bias &= np.uint32(1)
    bias += np.uint32(0x7FFF)
    bits += bias
    bits &= np.uint32(0xFFFF0000)
    return x


def normal(shape, seed, stream=0, scale=1.0, dtype="bf16"):
    """i.i.d. N(0, scale^2) values of ``shape``, rounded to ``dtype``.

    ``dtype`` is "bf16" or "f32"; the result is always a float32 array.
    """
    rng = np.random.Generator(np.random.PCG64([int(seed), int(stream)]))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    if dtype == "bf16":
        return round_to_bf16(x, inplace=True)
    if dtype == "f32":
        return x
    raise ValueError(f"unknown dtype {dtype!r}")


def qkv(B, H, N, dk, dv, seed, dtype="bf16"):
    """q, k, v of shape [B,H,N,d], each N(0,1)/sqrt(d) rounded to ``dtype``."""
    jobs = [((B, H, N, dk), STREAM_Q, dk), ((B, H, N, dk), STREAM_K, dk),
            ((B, H, N, dv), STREAM_V, dv)]
    if B * H * N * max(dk, dv) < (1 << 22):
        return tuple(normal(s, seed, st, 1.0 / np.sqrt(d), dtype) for s, st, d in jobs)
    # large tensors: the three independent streams in parallel threads
    with ThreadPoolExecutor(max_workers=3) as ex:
        futs = [ex.submit(normal, s, seed, st, 1.0 / np.sqrt(d), dtype) for s, st, d in jobs]
        return tuple(f.result() for f in futs)


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
