"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and
the benchmark.

This module holds none of the collectives' arithmetic: it only draws rank
buffers.  It imports neither the oracle nor the product library.  Every
generator is a pure function of its arguments (numpy PCG64 via
``default_rng(seed)``).

Workloads (values as synthetic gradients, the pages name no dataset):
  * uniform_int32: integers uniform in [-1000, 1000]  (int32 AllReduce case)
  * gradients_f32: N(0,1) * scale as float32         (scale 1e-3 or 1)
  * gradients_bf16: round-to-nearest-even bf16 of N(0,1) * scale, returned as
    uint16 bit patterns (the conversion is torch's float32 -> bfloat16 cast,
    used here as plumbing).
"""
import numpy as np


def uniform_int32(P, n, seed=0, lo=-1000, hi=1000):
    return np.random.default_rng(seed).integers(lo, hi + 1, size=(P, n), dtype=np.int32)


def gradients_f32(P, n, seed=0, scale=1e-3):
    x = np.random.default_rng(seed).standard_normal((P, n), dtype=np.float32)
    if scale != 1:
        x *= np.float32(scale)
    return x


def gradients_bf16(P, n, seed=0, scale=1e-2):
    """bf16 bit patterns (uint16) of N(0,1)*scale rounded to nearest even."""
    import torch
    x = gradients_f32(P, n, seed=seed, scale=scale)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def rank_buffers(dtype, P, n, seed=0, scale=None):
    """Dispatch on dtype name: int32 / float32 / bfloat16 (uint16 bits)."""
    if dtype == "int32":
        return uniform_int32(P, n, seed=seed)
    if dtype == "float32":
        return gradients_f32(P, n, seed=seed, scale=1e-3 if scale is None else scale)
    if dtype == "bfloat16":
        return gradients_bf16(P, n, seed=seed, scale=1e-2 if scale is None else scale)
    raise ValueError(dtype)


def sample_indices(n, count, seed=1, segment_edges=()):
    """Sorted distinct element indices: `count` uniform picks plus both sides
    of every given segment edge (first/last element of each segment and the
    last element of the vector), for sampled checks at full size."""
    rng = np.random.default_rng(seed)
    picks = set(int(i) for i in rng.integers(0, n, size=min(count, n))) if n > 0 else set()
    for e in segment_edges:
        for d in (-1, 0):
            j = int(e) + d
            if 0 <= j < n:
                picks.add(j)
    if n > 0:
        picks.update((0, n - 1))
    return np.array(sorted(picks), dtype=np.int64)
