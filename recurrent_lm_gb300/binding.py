"""Thin Python binding of liblinattn.so (ctypes).

Argument marshalling only: shapes and dtypes are checked, outputs are
allocated with torch when the caller does not pass them, and every step of the
computation runs in the library's CUDA kernels on the current torch stream.
There is no CPU path: calling any function without the built library, or with
CPU tensors, raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblinattn.so")
D_FEAT, D_V, D_PHI = 16, 64, 273
D_COMPACT = 153  # rows of the compact state layout (1 + 16 + 16*17/2)


def feature_dim(dk: int) -> int:
    """D = 1 + d' + d'^2: rows of the state for feature dimension d'."""
    return 1 + dk + dk * dk

(LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_MISALIGNED, LA_ERR_CUDA, LA_ERR_TIMEOUT,
 LA_ERR_SCRATCH_TOO_SMALL) = range(7)
LA_DTYPE_F32, LA_DTYPE_BF16 = 0, 1

_lib = None
_lock = threading.Lock()


class LAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"liblinattn status {status}: {msg}")
        self.status = status


# (name, restype, argtypes) of every symbol declared in include/linattn.h
_VP, _FP, _I64, _I, _F, _SZ = (ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                               ctypes.c_int, ctypes.c_float, ctypes.c_size_t)
SIGNATURES = {
    "la_prefill": (_I, [_VP, _VP, _VP, _FP, _FP, _VP, _FP, _FP, _I64, _I64, _I64, _I, _I,
                        _I, _F, _VP]),
    "la_prefill_padded": (_I, [_VP, _VP, _VP, _FP, _FP, _VP, _VP, _FP, _FP, _I64, _I64, _I64, _I,
                               _I, _I, _F, _VP]),
    "la_prefill_decay": (_I, [_VP, _VP, _VP, _FP, _FP, _FP, _VP, _FP, _FP, _I64, _I64, _I64, _I,
                              _I, _I, _F, _VP]),
    "la_decode_step_decay": (_I, [_VP, _VP, _VP, _FP, _FP, _FP, _FP, _FP, _VP, _I64, _I64, _I, _I,
                                  _I, _F, _VP]),
    "la_prefix_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "la_prefill_host_workspace_size": (_SZ, [_I64, _I64, _I64, _I, _I]),
    "la_prefill_workspace_size": (_SZ, [_I64, _I64, _I64, _I, _I]),
    "la_prefill_decay_ws": (_I, [_VP, _VP, _VP, _FP, _FP, _FP, _VP, _FP, _FP, _VP, _SZ, _I64, _I64, _I64,
                                 _I, _I, _I, _F, _VP]),
    "la_prefill_split_info": (_I, [_I64, _I64, _I64, ctypes.POINTER(ctypes.c_int),
                                   ctypes.POINTER(ctypes.c_int)]),
    "la_prefill_ws": (_I, [_VP, _VP, _VP, _FP, _FP, _VP, _FP, _FP, _VP, _SZ, _I64, _I64, _I64, _I, _I,
                           _I, _F, _VP]),
    "la_prefill_host": (_I, [_VP, _VP, _VP, _FP, _FP, _VP, _FP, _FP, _VP, _SZ, _I64, _I64, _I64,
                             _I, _I, _I, _F, _VP]),
    "la_prefix_prefill": (_I, [_VP, _VP, _VP, _VP, _VP, _I64, _FP, _FP, _VP, _FP, _FP, _VP,
                               _SZ, _I64, _I64, _I64, _I, _I, _I, _F, _VP]),
    "la_prefix_prefill_padded": (_I, [_VP, _VP, _VP, _VP, _VP, _I64, _FP, _FP, _VP, _VP, _FP, _FP,
                                      _VP, _SZ, _I64, _I64, _I64, _I, _I, _I, _F, _VP]),
    "la_decode_step": (_I, [_VP, _VP, _VP, _FP, _FP, _FP, _FP, _VP, _I64, _I64, _I, _I, _I,
                            _F, _VP]),
    "la_prefix_prefill_noalloc": (_I, [_VP, _VP, _VP, _VP, _VP, _I64, _FP, _FP, _VP, _FP, _FP,
                                       _I64, _I64, _I64, _I, _I, _I, _F, _VP]),
    "la_noalloc_scratch_bytes": (_SZ, []),
    "la_state_to_compact": (_I, [_FP, _FP, _FP, _FP, _I64, _I64, _I, _I, _VP]),
    "la_state_from_compact": (_I, [_FP, _FP, _FP, _FP, _I64, _I64, _I, _I, _VP]),
    "la_prefill_compact": (_I, [_VP, _VP, _VP, _FP, _FP, _VP, _FP, _FP, _I64, _I64, _I64, _I, _I,
                                _I, _F, _VP]),
    "la_decode_step_compact": (_I, [_VP, _VP, _VP, _FP, _FP, _FP, _FP, _VP, _I64, _I64, _I, _I, _I,
                                    _F, _VP]),
    "la_status_string": (ctypes.c_char_p, [_I]),
    "la_check_device_status": (_I, [_VP]),
    "la_debug_timeout_probe": (_I, [_VP]),
    "la_version": (_I, []),
}


def load_library(path: str = LIB_PATH):
    """Load liblinattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first (python -m recurrent_lm_gb300.build); "
                "there is no fallback implementation")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().la_status_string(int(status)).decode()


def _raise(status: int):
    if status != LA_OK:
        raise LAError(status, status_string(status))


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return LA_DTYPE_BF16
    if t.dtype == torch.float32:
        return LA_DTYPE_F32
    raise TypeError(f"activations must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, shape, dtype):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _keep_for(t: torch.Tensor, stream):
    """A tensor allocated here (on the current stream) but used by work
    enqueued on another stream: tell the caching allocator, so that the block
    is not handed out again before that stream's work has finished with it."""
    if stream is not None and stream != torch.cuda.current_stream(t.device):
        t.record_stream(stream)


def _need_pad(left_pad, B):
    if left_pad is not None:
        _need(left_pad, "left_pad", (B,), torch.int32)


def prefill(q, k, v, s0=None, z0=None, *, eps: float = 0.0, y=None, s_out=None,
            z_out=None, want_state: bool = True, stream=None, left_pad=None, gamma=None,
            workspace=None, split: bool = True):
    """Causal prefill.  q,k [B,H,N,16], v [B,H,N,64] (bf16 or fp32, CUDA,
    contiguous); s0 [B,H,273,64], z0 [B,H,273] fp32 or None.
    left_pad: CUDA int32 [B] counts of leading padding positions per batch row
    (la_prefill_padded), or None.  gamma: CUDA fp32 [H] per-head decay in
    [0, 1] (la_prefill_decay), or None; not combined with left_pad.
    Without either, the call is la_prefill_ws with ``workspace`` (a CUDA uint8
    tensor of la_prefill_workspace_size bytes; allocated here if None), or
    la_prefill when split is False.  With bf16 and d' = 24 or 32 that workspace
    holds the tensor-core form's buffers (about 3.3 or 5.1 KB per head-token,
    e.g. 0.9 / 1.4 GB at B=4, H=16, N=4096); split=False runs the CUDA-core
    path, which needs none.
    Returns (y, s_out, z_out); the states are None when want_state is False."""
    lib = load_library()
    B, H, N, dk = q.shape
    D = feature_dim(dk)
    dt = q.dtype
    _need(q, "q", (B, H, N, dk), dt)
    _need(k, "k", (B, H, N, dk), dt)
    _need(v, "v", (B, H, N, D_V), dt)
    if s0 is not None or z0 is not None:
        _need(s0, "s0", (B, H, D, D_V), torch.float32)
        _need(z0, "z0", (B, H, D), torch.float32)
    if y is None:
        y = torch.empty((B, H, N, D_V), dtype=dt, device=q.device)
    _need(y, "y", (B, H, N, D_V), dt)
    if want_state:
        if s_out is None:
            s_out = torch.empty((B, H, D, D_V), dtype=torch.float32, device=q.device)
        if z_out is None:
            z_out = torch.empty((B, H, D), dtype=torch.float32, device=q.device)
    if s_out is not None:
        _need(s_out, "s_out", (B, H, D, D_V), torch.float32)
    if z_out is not None:
        _need(z_out, "z_out", (B, H, D), torch.float32)
    _need_pad(left_pad, B)
    if gamma is not None:
        if left_pad is not None:
            raise ValueError("left_pad and gamma cannot be combined")
        _need(gamma, "gamma", (H,), torch.float32)
        need = int(lib.la_prefill_workspace_size(B, H, N, dk, _dt(q))) if split else 0
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            _keep_for(workspace, stream)
        if workspace is not None:
            _need(workspace, "workspace", (workspace.numel(),), torch.uint8)
        _raise(lib.la_prefill_decay_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(s0), _ptr(z0), _ptr(gamma),
                                       _ptr(y), _ptr(s_out), _ptr(z_out), _ptr(workspace),
                                       0 if workspace is None else workspace.numel(), B, H, N, dk, D_V,
                                       _dt(q), float(eps), _stream(stream)))
    elif left_pad is None:
        # la_prefill_ws with a workspace from torch's caching allocator (it
        # balances the last wave of heads on the bf16 path); la_prefill when
        # the call has no workspace form
        need = int(lib.la_prefill_workspace_size(B, H, N, dk, _dt(q))) if split else 0
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            _keep_for(workspace, stream)
        if workspace is not None:
            _need(workspace, "workspace", (workspace.numel(),), torch.uint8)
            _raise(lib.la_prefill_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(s0), _ptr(z0), _ptr(y), _ptr(s_out),
                                     _ptr(z_out), _ptr(workspace), workspace.numel(), B, H, N, dk, D_V,
                                     _dt(q), float(eps), _stream(stream)))
        else:
            _raise(lib.la_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(s0), _ptr(z0), _ptr(y), _ptr(s_out),
                                  _ptr(z_out), B, H, N, dk, D_V, _dt(q), float(eps), _stream(stream)))
    else:
        _raise(lib.la_prefill_padded(_ptr(q), _ptr(k), _ptr(v), _ptr(s0), _ptr(z0), _ptr(left_pad),
                                     _ptr(y), _ptr(s_out), _ptr(z_out), B, H, N, dk, D_V, _dt(q),
                                     float(eps), _stream(stream)))
    return y, s_out, z_out


def prefill_workspace_size(B: int, H: int, N: int, dk: int = D_FEAT,
                           dtype: torch.dtype = torch.bfloat16) -> int:
    """Bytes of the workspace la_prefill_ws uses (0: the call has no use for one)."""
    dt = LA_DTYPE_BF16 if dtype == torch.bfloat16 else LA_DTYPE_F32
    return int(load_library().la_prefill_workspace_size(B, H, N, dk, dt))


def prefill_split_info(B: int, H: int, N: int):
    """(split_heads, split_chunk) that la_prefill_ws chooses on the current device."""
    r, c = ctypes.c_int(0), ctypes.c_int(0)
    _raise(load_library().la_prefill_split_info(B, H, N, ctypes.byref(r), ctypes.byref(c)))
    return r.value, c.value


def _need_host(t: torch.Tensor, name: str, shape, dtype):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name} must be a CPU tensor (prefill_host reads and writes host memory)")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def prefill_host_workspace_size(B: int, H: int, N: int, dk: int = D_FEAT,
                                dtype: torch.dtype = torch.bfloat16) -> int:
    dt = LA_DTYPE_BF16 if dtype == torch.bfloat16 else LA_DTYPE_F32
    return int(load_library().la_prefill_host_workspace_size(B, H, N, dk, dt))


def prefill_host(q, k, v, s0=None, z0=None, *, eps: float = 0.0, y=None, s_out=None, z_out=None,
                 want_state: bool = True, workspace=None, stream=None, device=None):
    """Causal prefill from and to host memory (la_prefill_host): q, k, v and
    s0, z0 are CPU tensors (pinned, for the copies to overlap the kernels);
    outputs are CPU tensors, pinned when allocated here.  ``workspace`` is a
    CUDA uint8 tensor of at least prefill_host_workspace_size(...) bytes on
    ``device`` (the current CUDA device if None; allocated here if not given).
    The call is asynchronous: the host outputs are valid once ``stream`` (the
    current stream if None) has completed the call's work."""
    lib = load_library()
    B, H, N, dk = q.shape
    D = feature_dim(dk)
    dt = q.dtype
    _need_host(q, "q", (B, H, N, dk), dt)
    _need_host(k, "k", (B, H, N, dk), dt)
    _need_host(v, "v", (B, H, N, D_V), dt)
    if s0 is not None or z0 is not None:
        _need_host(s0, "s0", (B, H, D, D_V), torch.float32)
        _need_host(z0, "z0", (B, H, D), torch.float32)
    if y is None:
        y = torch.empty((B, H, N, D_V), dtype=dt).pin_memory()
    _need_host(y, "y", (B, H, N, D_V), dt)
    if want_state:
        if s_out is None:
            s_out = torch.empty((B, H, D, D_V), dtype=torch.float32).pin_memory()
        if z_out is None:
            z_out = torch.empty((B, H, D), dtype=torch.float32).pin_memory()
    if s_out is not None:
        _need_host(s_out, "s_out", (B, H, D, D_V), torch.float32)
    if z_out is not None:
        _need_host(z_out, "z_out", (B, H, D), torch.float32)
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        need = prefill_host_workspace_size(B, H, N, dk, dt)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _keep_for(workspace, stream)
    _need(workspace, "workspace", (workspace.numel(),), torch.uint8)
    # the library works on the current device: make it the workspace's
    with torch.cuda.device(workspace.device):
        _raise(lib.la_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(s0), _ptr(z0), _ptr(y), _ptr(s_out),
                                   _ptr(z_out), _ptr(workspace), workspace.numel(), B, H, N, dk, D_V,
                                   _dt(q), float(eps), _stream(stream)))
    return y, s_out, z_out


def prefix_workspace_size(B: int, H: int, M: int) -> int:
    return int(load_library().la_prefix_workspace_size(B, H, M))


def prefix_prefill(q, k, v, k_e, v_e, s0=None, z0=None, *, eps: float = 0.0, y=None,
                   s_out=None, z_out=None, want_state: bool = True, workspace=None,
                   stream=None, left_pad=None):
    """JRT-RNN prefix linear attention (la_prefix_prefill).  k_e [B,H,M,16],
    v_e [B,H,M,64] with M <= N.  ``workspace`` is a CUDA uint8 tensor of at
    least prefix_workspace_size(B, H, M) bytes (allocated here if None).
    left_pad: CUDA int32 [B] counts of leading padding positions per batch row
    (la_prefix_prefill_padded), or None."""
    lib = load_library()
    B, H, N, _ = q.shape
    dt = q.dtype
    M = k_e.shape[2]
    _need(q, "q", (B, H, N, D_FEAT), dt)
    _need(k, "k", (B, H, N, D_FEAT), dt)
    _need(v, "v", (B, H, N, D_V), dt)
    _need(k_e, "k_e", (B, H, M, D_FEAT), dt)
    _need(v_e, "v_e", (B, H, M, D_V), dt)
    if s0 is not None or z0 is not None:
        _need(s0, "s0", (B, H, D_PHI, D_V), torch.float32)
        _need(z0, "z0", (B, H, D_PHI), torch.float32)
    if y is None:
        y = torch.empty((B, H, N, D_V), dtype=dt, device=q.device)
    if want_state:
        if s_out is None:
            s_out = torch.empty((B, H, D_PHI, D_V), dtype=torch.float32, device=q.device)
        if z_out is None:
            z_out = torch.empty((B, H, D_PHI), dtype=torch.float32, device=q.device)
    need = prefix_workspace_size(B, H, M)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
        _keep_for(workspace, stream)
    _need_pad(left_pad, B)
    if left_pad is None:
        _raise(lib.la_prefix_prefill(
            _ptr(q), _ptr(k), _ptr(v), _ptr(k_e), _ptr(v_e), M, _ptr(s0), _ptr(z0), _ptr(y),
            _ptr(s_out), _ptr(z_out), _ptr(workspace), workspace.numel(), B, H, N, D_FEAT, D_V,
            _dt(q), float(eps), _stream(stream)))
    else:
        _raise(lib.la_prefix_prefill_padded(
            _ptr(q), _ptr(k), _ptr(v), _ptr(k_e), _ptr(v_e), M, _ptr(s0), _ptr(z0), _ptr(left_pad),
            _ptr(y), _ptr(s_out), _ptr(z_out), _ptr(workspace), workspace.numel(), B, H, N, D_FEAT,
            D_V, _dt(q), float(eps), _stream(stream)))
    return y, s_out, z_out


def prefix_prefill_noalloc(q, k, v, k_e, v_e, s0=None, z0=None, *, eps: float = 0.0, y=None,
                           s_out=None, z_out=None, want_state: bool = True, stream=None):
    """la_prefix_prefill_noalloc: JRT-RNN prefix prefill for callers that cannot
    allocate device memory when they call; the library's fixed scratch buffer
    replaces the workspace (outputs are still allocated here when not given)."""
    lib = load_library()
    B, H, N, _ = q.shape
    dt = q.dtype
    M = k_e.shape[2]
    _need(q, "q", (B, H, N, D_FEAT), dt)
    _need(k, "k", (B, H, N, D_FEAT), dt)
    _need(v, "v", (B, H, N, D_V), dt)
    _need(k_e, "k_e", (B, H, M, D_FEAT), dt)
    _need(v_e, "v_e", (B, H, M, D_V), dt)
    if s0 is not None or z0 is not None:
        _need(s0, "s0", (B, H, D_PHI, D_V), torch.float32)
        _need(z0, "z0", (B, H, D_PHI), torch.float32)
    if y is None:
        y = torch.empty((B, H, N, D_V), dtype=dt, device=q.device)
    if want_state:
        if s_out is None:
            s_out = torch.empty((B, H, D_PHI, D_V), dtype=torch.float32, device=q.device)
        if z_out is None:
            z_out = torch.empty((B, H, D_PHI), dtype=torch.float32, device=q.device)
    _raise(lib.la_prefix_prefill_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k_e), _ptr(v_e), M, _ptr(s0), _ptr(z0), _ptr(y),
        _ptr(s_out), _ptr(z_out), B, H, N, D_FEAT, D_V, _dt(q), float(eps), _stream(stream)))
    return y, s_out, z_out


def noalloc_scratch_bytes() -> int:
    return int(load_library().la_noalloc_scratch_bytes())


def decode_step(q, k, v, s, z, *, eps: float = 0.0, y=None, s_out=None, z_out=None,
                inplace: bool = False, stream=None, gamma=None):
    """One decode step (la_decode_step).  q,k [B,H,16], v [B,H,64]; s [B,H,273,64],
    z [B,H,273] fp32.  With inplace=True the state is updated in s, z.
    gamma: CUDA fp32 [H] per-head decay (la_decode_step_decay), or None."""
    lib = load_library()
    B, H, dk = q.shape
    D = feature_dim(dk)
    dt = q.dtype
    _need(q, "q", (B, H, dk), dt)
    _need(k, "k", (B, H, dk), dt)
    _need(v, "v", (B, H, D_V), dt)
    _need(s, "s", (B, H, D, D_V), torch.float32)
    _need(z, "z", (B, H, D), torch.float32)
    if inplace:
        s_out, z_out = s, z
    if s_out is None:
        s_out = torch.empty_like(s)
    if z_out is None:
        z_out = torch.empty_like(z)
    if y is None:
        y = torch.empty((B, H, D_V), dtype=dt, device=q.device)
    if gamma is None:
        _raise(lib.la_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(z), _ptr(s_out),
                                  _ptr(z_out), _ptr(y), B, H, dk, D_V, _dt(q), float(eps),
                                  _stream(stream)))
    else:
        _need(gamma, "gamma", (H,), torch.float32)
        _raise(lib.la_decode_step_decay(_ptr(q), _ptr(k), _ptr(v), _ptr(gamma), _ptr(s), _ptr(z),
                                        _ptr(s_out), _ptr(z_out), _ptr(y), B, H, dk, D_V, _dt(q),
                                        float(eps), _stream(stream)))
    return y, s_out, z_out


def state_to_compact(s, z, *, s_c=None, z_c=None, stream=None):
    """la_state_to_compact: s [B,H,273,64], z [B,H,273] fp32 -> the compact
    layout s_c [B,H,153,64], z_c [B,H,153] (the antisymmetric part of the
    quadratic block is dropped)."""
    lib = load_library()
    B, H = s.shape[:2]
    _need(s, "s", (B, H, D_PHI, D_V), torch.float32)
    _need(z, "z", (B, H, D_PHI), torch.float32)
    if s_c is None:
        s_c = torch.empty((B, H, D_COMPACT, D_V), dtype=torch.float32, device=s.device)
    if z_c is None:
        z_c = torch.empty((B, H, D_COMPACT), dtype=torch.float32, device=s.device)
    _need(s_c, "s_c", (B, H, D_COMPACT, D_V), torch.float32)
    _need(z_c, "z_c", (B, H, D_COMPACT), torch.float32)
    _raise(lib.la_state_to_compact(_ptr(s), _ptr(z), _ptr(s_c), _ptr(z_c), B, H, D_FEAT, D_V,
                                   _stream(stream)))
    return s_c, z_c


def state_from_compact(s_c, z_c, *, s=None, z=None, stream=None):
    """la_state_from_compact: the compact layout -> the 273-row layout (cross
    terms split evenly between (a, b) and (b, a))."""
    lib = load_library()
    B, H = s_c.shape[:2]
    _need(s_c, "s_c", (B, H, D_COMPACT, D_V), torch.float32)
    _need(z_c, "z_c", (B, H, D_COMPACT), torch.float32)
    if s is None:
        s = torch.empty((B, H, D_PHI, D_V), dtype=torch.float32, device=s_c.device)
    if z is None:
        z = torch.empty((B, H, D_PHI), dtype=torch.float32, device=s_c.device)
    _need(s, "s", (B, H, D_PHI, D_V), torch.float32)
    _need(z, "z", (B, H, D_PHI), torch.float32)
    _raise(lib.la_state_from_compact(_ptr(s_c), _ptr(z_c), _ptr(s), _ptr(z), B, H, D_FEAT, D_V,
                                     _stream(stream)))
    return s, z


def prefill_compact(q, k, v, s0=None, z0=None, *, eps: float = 0.0, y=None, s_out=None,
                    z_out=None, want_state: bool = True, stream=None):
    """la_prefill_compact: causal prefill (bf16) with s0 [B,H,153,64], z0
    [B,H,153] and the final state in the compact layout."""
    lib = load_library()
    B, H, N, _ = q.shape
    dt = q.dtype
    _need(q, "q", (B, H, N, D_FEAT), dt)
    _need(k, "k", (B, H, N, D_FEAT), dt)
    _need(v, "v", (B, H, N, D_V), dt)
    if s0 is not None or z0 is not None:
        _need(s0, "s0", (B, H, D_COMPACT, D_V), torch.float32)
        _need(z0, "z0", (B, H, D_COMPACT), torch.float32)
    if y is None:
        y = torch.empty((B, H, N, D_V), dtype=dt, device=q.device)
    _need(y, "y", (B, H, N, D_V), dt)
    if want_state:
        if s_out is None:
            s_out = torch.empty((B, H, D_COMPACT, D_V), dtype=torch.float32, device=q.device)
        if z_out is None:
            z_out = torch.empty((B, H, D_COMPACT), dtype=torch.float32, device=q.device)
    if s_out is not None:
        _need(s_out, "s_out", (B, H, D_COMPACT, D_V), torch.float32)
    if z_out is not None:
        _need(z_out, "z_out", (B, H, D_COMPACT), torch.float32)
    _raise(lib.la_prefill_compact(_ptr(q), _ptr(k), _ptr(v), _ptr(s0), _ptr(z0), _ptr(y),
                                  _ptr(s_out), _ptr(z_out), B, H, N, D_FEAT, D_V, _dt(q),
                                  float(eps), _stream(stream)))
    return y, s_out, z_out


def decode_step_compact(q, k, v, s, z, *, eps: float = 0.0, y=None, s_out=None, z_out=None,
                        inplace: bool = False, stream=None):
    """la_decode_step_compact: one decode step on a compact state s
    [B,H,153,64], z [B,H,153] fp32 (in place with inplace=True)."""
    lib = load_library()
    B, H, _ = q.shape
    dt = q.dtype
    _need(q, "q", (B, H, D_FEAT), dt)
    _need(k, "k", (B, H, D_FEAT), dt)
    _need(v, "v", (B, H, D_V), dt)
    _need(s, "s", (B, H, D_COMPACT, D_V), torch.float32)
    _need(z, "z", (B, H, D_COMPACT), torch.float32)
    if inplace:
        s_out, z_out = s, z
    if s_out is None:
        s_out = torch.empty_like(s)
    if z_out is None:
        z_out = torch.empty_like(z)
    if y is None:
        y = torch.empty((B, H, D_V), dtype=dt, device=q.device)
    _raise(lib.la_decode_step_compact(_ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(z), _ptr(s_out),
                                      _ptr(z_out), _ptr(y), B, H, D_FEAT, D_V, _dt(q), float(eps),
                                      _stream(stream)))
    return y, s_out, z_out


def debug_timeout_probe(stream=None) -> None:
    """Enqueue the bounded-wait failure probe (la_debug_timeout_probe): about one
    second later the device status word holds a timeout, which the next
    check_device_status raises as LAError(LA_ERR_TIMEOUT)."""
    _raise(load_library().la_debug_timeout_probe(_stream(stream)))


def check_device_status(stream=None) -> None:
    """Synchronize and raise LAError(LA_ERR_TIMEOUT) if a bounded wait gave up."""
    _raise(load_library().la_check_device_status(_stream(stream)))
