"""Shared helpers for the GPU parity tests (comparison metric, sampling)."""
import numpy as np
import torch

import oracle

# Tolerances of the accuracy target: max relative error 1e-4 for fp32 inputs,
# 2e-2 for bf16 inputs with fp32 accumulation, for y and for the final states.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def to64(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu").to(torch.float64).numpy()


def normwise_rel(a, r, slice_dims=2):
    """Max over the leading (b, h) slices of max|a - r| / max|r|: the relative
    error measure used throughout (elementwise ratios are ill-posed because y
    is a weighted mean of zero-mean values and can be arbitrarily close to 0)."""
    a = to64(a)
    r = to64(r)
    assert a.shape == r.shape, (a.shape, r.shape)
    lead = int(np.prod(a.shape[:slice_dims]))
    a = a.reshape(lead, -1)
    r = r.reshape(lead, -1)
    if a.shape[1] == 0:
        return 0.0
    err = np.max(np.abs(a - r), axis=1)
    scale = np.maximum(np.max(np.abs(r), axis=1), 1e-30)
    if not np.all(np.isfinite(a)):
        return float("inf")
    return float(np.max(err / scale))


def assert_close(name, a, r, tol, slice_dims=2):
    e = normwise_rel(a, r, slice_dims)
    assert e <= tol, f"{name}: normwise relative error {e:.3e} > {tol:.1e}"
    return e


def oracle_prefill(q, k, v, s0=None, z0=None, eps=0.0):
    return oracle.prefill(q, k, v, s0, z0, eps)


def sample_heads(B, H, n, seed=0):
    """n distinct (b, h) pairs, always including the first and the last."""
    rng = np.random.default_rng(seed)
    flat = set([0, B * H - 1])
    while len(flat) < min(n, B * H):
        flat.add(int(rng.integers(0, B * H)))
    return sorted((f // H, f % H) for f in flat)
