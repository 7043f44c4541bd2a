"""Plain, slow fp64 CPU oracle for causal Taylor linear attention.

TEST INFRASTRUCTURE: only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The library's GPU path never
imports, links or runs anything here, and nothing here imports the library.

Two independent implementations live here:

* ``la_oracle.c`` (loaded through ctypes): the recurrent form, the prefix
  (JRT-RNN) form, the decode step and the blockwise form, all in fp64 with
  plain loops (see the citations at the top of that file);
* ``quadratic.py``: the O(N^2) closed form sum_j K(q_i,k_j) v_j / sum_j K(q_i,k_j)
  with K = 1 + q.k/sqrt(d') + (q.k)^2/(2 d'), in numpy, for small N.

Every function takes numpy arrays (any float dtype; converted exactly to
float64) in the dense row-major layouts

    q, k [B, H, N, dk]   v [B, H, N, dv]   s [B, H, D, dv]   z [B, H, D]

with D = 1 + dk + dk^2 and feature order (constant, linear a, quadratic a*dk+b).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .quadratic import kernel_closed_form, prefill_closed_form, prefix_closed_form

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_la_oracle.so")
_lib = None
_lock = threading.Lock()

__all__ = [
    "build", "feature_dim", "phi", "prefill", "prefix_prefill", "decode_step",
    "prefill_chunked", "max_threads", "kernel_closed_form", "prefill_closed_form",
    "prefix_closed_form",
]


def build(force: bool = False) -> str:
    """Compile la_oracle.c into a shared object beside it (gcc, OpenMP).

    -ffp-contract=off keeps every multiply and add separately rounded so the
    oracle gives the same bits on x86 and Arm hosts."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER(ctypes.c_double)
        L, D, I = ctypes.c_long, ctypes.c_double, ctypes.c_int
        lib.oracle_feature_dim.argtypes = [L]
        lib.oracle_feature_dim.restype = L
        lib.oracle_phi.argtypes = [P, L, P]
        lib.oracle_phi.restype = None
        lib.oracle_prefill.argtypes = [P, P, P, P, P, P, P, P, L, L, L, L, L, D, I]
        lib.oracle_prefill.restype = I
        lib.oracle_prefix_prefill.argtypes = [P, P, P, P, P, L, P, P, P, P, P,
                                              L, L, L, L, L, D, I]
        lib.oracle_prefix_prefill.restype = I
        LP = ctypes.POINTER(ctypes.c_long)
        lib.oracle_prefix_prefill_padded.argtypes = [P, P, P, P, P, L, P, P, LP, P, P, P,
                                                     L, L, L, L, L, D, I]
        lib.oracle_prefix_prefill_padded.restype = I
        lib.oracle_decode_step.argtypes = [P, P, P, P, P, P, P, P, L, L, L, L, D, I]
        lib.oracle_decode_step.restype = I
        lib.oracle_prefill_decay.argtypes = [P, P, P, P, P, P, P, P, P, L, L, L, L, L, D, I]
        lib.oracle_prefill_decay.restype = I
        lib.oracle_decode_step_decay.argtypes = [P, P, P, P, P, P, P, P, P, L, L, L, L, D, I]
        lib.oracle_decode_step_decay.restype = I
        lib.oracle_prefill_chunked.argtypes = [P, P, P, P, P, P, P, P, L, L, L, L,
                                               L, L, D, I]
        lib.oracle_prefill_chunked.restype = I
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = I
        _lib = lib
        return lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # a torch tensor: exact upcast on the CPU
        a = a.detach().to("cpu")
        import torch
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def feature_dim(dk: int) -> int:
    return 1 + dk + dk * dk


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def phi(x) -> np.ndarray:
    """phi(x) for a single vector x of length dk."""
    x = _f64(x).reshape(-1)
    out = np.empty(feature_dim(x.size), dtype=np.float64)
    _load().oracle_phi(_ptr(x), x.size, _ptr(out))
    return out


def _shapes(q, v):
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    return B, H, N, dk, dv


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"oracle returned error {rc}")


def prefix_prefill(q, k, v, ke=None, ve=None, s0=None, z0=None, eps=0.0,
                   nthreads: int = 0, left_pad=None):
    """Prefix linear attention; ke/ve [B,H,M,*] (None: plain causal).
    left_pad: per-batch-row count of leading padding positions (None: none).
    Returns (y [B,H,N,dv], s [B,H,D,dv], z [B,H,D]) in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    ke, ve, s0, z0 = _f64(ke), _f64(ve), _f64(s0), _f64(z0)
    B, H, N, dk, dv = _shapes(q, v)
    D = feature_dim(dk)
    assert k.shape == q.shape and v.shape[:3] == (B, H, N)
    M = 0 if ke is None else ke.shape[2]
    if ke is not None:
        assert ke.shape == (B, H, M, dk) and ve.shape == (B, H, M, dv)
    if s0 is not None:
        assert s0.shape == (B, H, D, dv)
    if z0 is not None:
        assert z0.shape == (B, H, D)
    y = np.empty((B, H, N, dv), dtype=np.float64)
    s = np.empty((B, H, D, dv), dtype=np.float64)
    z = np.empty((B, H, D), dtype=np.float64)
    lp = None
    if left_pad is not None:
        lp = np.ascontiguousarray(np.asarray(left_pad, dtype=np.int64).reshape(B))
        assert ctypes.sizeof(ctypes.c_long) == 8
    _check(_load().oracle_prefix_prefill_padded(
        _ptr(q), _ptr(k), _ptr(v), _ptr(ke), _ptr(ve), M, _ptr(s0), _ptr(z0),
        None if lp is None else lp.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
        _ptr(y), _ptr(s), _ptr(z), B, H, N, dk, dv, float(eps), int(nthreads)))
    return y, s, z


def prefill(q, k, v, s0=None, z0=None, eps=0.0, nthreads: int = 0, left_pad=None):
    """Causal prefill from an optional initial state; returns (y, s, z)."""
    return prefix_prefill(q, k, v, None, None, s0, z0, eps, nthreads, left_pad=left_pad)


def prefill_chunked(q, k, v, C: int, s0=None, z0=None, eps=0.0, nthreads: int = 0):
    """The blockwise form with block length C; returns (y, s, z)."""
    q, k, v, s0, z0 = _f64(q), _f64(k), _f64(v), _f64(s0), _f64(z0)
    B, H, N, dk, dv = _shapes(q, v)
    D = feature_dim(dk)
    y = np.empty((B, H, N, dv), dtype=np.float64)
    s = np.empty((B, H, D, dv), dtype=np.float64)
    z = np.empty((B, H, D), dtype=np.float64)
    _check(_load().oracle_prefill_chunked(
        _ptr(q), _ptr(k), _ptr(v), _ptr(s0), _ptr(z0), _ptr(y), _ptr(s), _ptr(z),
        B, H, N, dk, dv, int(C), float(eps), int(nthreads)))
    return y, s, z


def prefill_decay(q, k, v, gamma, s0=None, z0=None, eps=0.0, nthreads: int = 0):
    """Causal prefill with a fixed per-head decay gamma [H] in [0, 1];
    returns (y, s, z) in float64."""
    q, k, v, s0, z0 = _f64(q), _f64(k), _f64(v), _f64(s0), _f64(z0)
    B, H, N, dk, dv = _shapes(q, v)
    D = feature_dim(dk)
    g = np.ascontiguousarray(np.asarray(gamma, dtype=np.float64).reshape(H))
    y = np.empty((B, H, N, dv), dtype=np.float64)
    s = np.empty((B, H, D, dv), dtype=np.float64)
    z = np.empty((B, H, D), dtype=np.float64)
    _check(_load().oracle_prefill_decay(
        _ptr(q), _ptr(k), _ptr(v), _ptr(s0), _ptr(z0), _ptr(g), _ptr(y), _ptr(s), _ptr(z),
        B, H, N, dk, dv, float(eps), int(nthreads)))
    return y, s, z


def decode_step(q, k, v, s_in, z_in, eps=0.0, nthreads: int = 0, gamma=None):
    """One recurrent step; q,k [B,H,dk], v [B,H,dv]; gamma [H] per-head decay
    or None; returns (y, s, z)."""
    q, k, v, s_in, z_in = _f64(q), _f64(k), _f64(v), _f64(s_in), _f64(z_in)
    B, H, dk = q.shape
    dv = v.shape[-1]
    D = feature_dim(dk)
    y = np.empty((B, H, dv), dtype=np.float64)
    s = np.empty((B, H, D, dv), dtype=np.float64)
    z = np.empty((B, H, D), dtype=np.float64)
    g = None if gamma is None else np.ascontiguousarray(np.asarray(gamma, dtype=np.float64).reshape(H))
    _check(_load().oracle_decode_step_decay(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(s_in), _ptr(z_in), _ptr(s), _ptr(z),
        _ptr(y), B, H, dk, dv, float(eps), int(nthreads)))
    return y, s, z
