"""Shared helpers of the GPU parity tests (comparison against the oracle)."""

import numpy as np
import torch

# |gpu - ref| <= tol * (|ref| + 1), against the float64 oracle.
TOL = {torch.float32: 1e-5, torch.float16: 2e-2, torch.bfloat16: 2e-2}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(gpu, ref, dtype, what=""):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} != {ref.shape}"
    err = np.abs(g - ref) / (np.abs(ref) + 1.0)
    worst = float(err.max()) if err.size else 0.0
    if worst > TOL[dtype]:
        i = np.unravel_index(int(np.argmax(err)), err.shape)
        raise AssertionError(f"{what}: max scaled error {worst:.3e} > {TOL[dtype]} at {i}: gpu {g[i]} ref {ref[i]}")


def dev(tensors):
    return [t.cuda() for t in tensors]


def empty_like_list(n, shape, dtype):
    return [torch.full(shape, float("nan"), dtype=dtype, device="cuda") for _ in range(n)]
