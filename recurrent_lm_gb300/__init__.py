"""GB300 (sm_103a) causal Taylor linear attention: prefill, JRT-RNN prefix
prefill and recurrent decode, computed by the CUDA kernels of liblinattn.so.

The functions below only marshal arguments; see binding.py and
include/linattn.h.  The seeded workload generators live in ``inputs``.
"""
from .binding import (  # noqa: F401
    D_COMPACT, D_FEAT, D_PHI, D_V, LA_ERR_CUDA, LA_ERR_INVALID_ARG, LA_ERR_MISALIGNED,
    LA_ERR_SCRATCH_TOO_SMALL, LA_ERR_TIMEOUT, LA_ERR_UNSUPPORTED, LA_OK, LAError, LIB_PATH,
    check_device_status, debug_timeout_probe, decode_step, decode_step_compact, load_library,
    noalloc_scratch_bytes, prefill, prefill_compact, prefill_host, prefill_host_workspace_size,
    prefill_split_info, prefill_workspace_size,
    prefix_prefill, prefix_prefill_noalloc, prefix_workspace_size, state_from_compact,
    state_to_compact, status_string,
)
