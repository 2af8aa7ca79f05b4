"""Seeded synthetic inputs shared by the tests, ``bench.py`` and ``smoke()``.

This module draws random numbers and rounds them to the requested storage type;
it holds none of the method's arithmetic. Both the CUDA path and the oracle get
their inputs from here, each through its own copy of the data.

Seeds follow ``1000 * config + 10 * tensor_id + rank``. Large tensors are
drawn in fixed 8 Mi-element chunks, chunk c from PCG64(SeedSequence([seed, c])),
so the values do not depend on the number of threads used to draw them.
"""

from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np
import torch

CHUNK = 1 << 23


def seed_of(config, tensor_id, rank=0):
    return 1000 * config + 10 * tensor_id + rank


def _draw(seed, n, kind):
    def one(c):
        lo = c * CHUNK
        m = min(CHUNK, n - lo)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, c])))
        if kind == "normal":
            return g.standard_normal(m, dtype=np.float32)
        if kind == "uniform":
            return g.random(m, dtype=np.float32) * 2.0 - 1.0
        if kind == "smallint":
            return g.integers(-4, 5, m).astype(np.float32)
        raise ValueError(kind)

    chunks = (n + CHUNK - 1) // CHUNK
    if chunks <= 1:
        return one(0) if n else np.zeros(0, np.float32)
    workers = min(chunks, max(1, len(os.sched_getaffinity(0))))
    with ThreadPoolExecutor(workers) as ex:
        return np.concatenate(list(ex.map(one, range(chunks))))


def tensor(seed, shape, dtype, kind="normal", std=1.0):
    """A CPU ``torch.Tensor`` of ``shape`` and ``dtype``.

    ``kind``: "normal" (N(0, std^2)), "uniform" (U(-1, 1)), or "smallint"
    (integers in [-4, 4], exact in every supported type).
    """
    n = int(np.prod(shape)) if len(shape) else 1
    x = _draw(seed, n, kind)
    if kind == "normal" and std != 1.0:
        x *= np.float32(std)
    return torch.from_numpy(x.reshape(shape)).to(dtype)


def per_rank(config, tensor_id, nranks, shape, dtype, kind="normal", std=1.0):
    """One tensor per rank, rank r seeded with ``seed_of(config, tensor_id, r)``."""
    return [tensor(seed_of(config, tensor_id, r), shape, dtype, kind, std) for r in range(nranks)]


def as_f64(t):
    """The exact values of a tensor, as a float64 NumPy array (for the oracle)."""
    return t.detach().to("cpu", torch.float64).numpy()
