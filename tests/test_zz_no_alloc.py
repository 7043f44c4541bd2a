"""la_prefix_prefill_noalloc: the prefix prefill for callers that cannot
allocate device memory when they call (a serving loop that must not trigger
the synchronisation an allocation implies, or a plug-in whose host process
owns all device memory).  It runs on the library's own fixed scratch buffer
instead of a caller workspace, so its results must match the ordinary entry
point's.  This file is collected last on purpose, and must pass both alone in
a fresh process and after the other tests."""
import ctypes

import pytest
import torch

import recurrent_lm_gb300 as la
from recurrent_lm_gb300 import binding, build, inputs
from helpers import TOL, assert_close

DEV = "cuda:0"


@pytest.mark.gpu
def test_noalloc_prefix_matches_workspace_prefix_on_two_calls():
    """Two calls in a row through the C ABI, each on different inputs (so the
    second finds the first one's data in the shared buffer), each compared
    with la_prefix_prefill given its own workspace."""
    cases = [(2, 4, 3000, 2500, 61), (1, 3, 700, 129, 62)]
    for B, H, N, M, seed in cases:
        q, k, v, ke, ve = inputs.qkv(B, H, N, seed=seed, M=M)
        s0, z0 = inputs.random_state(B, H, seed=seed + 100)
        args = [t.to(DEV) for t in (q, k, v, ke, ve, s0, z0)]
        assert la.prefix_workspace_size(B, H, M) <= la.noalloc_scratch_bytes()
        ref = la.prefix_prefill(*args)
        got = la.prefix_prefill_noalloc(*args)
        torch.cuda.synchronize()
        la.check_device_status()
        for name, a, r in zip("ysz", got, ref):
            assert_close(f"{name} (B={B} H={H} N={N} M={M})", a, r, TOL[torch.bfloat16])


def test_noalloc_rejects_problems_larger_than_its_buffer():
    """Too large for the fixed buffer: an error before any work (fake,
    never-dereferenced pointers; no GPU needed)."""
    build.build()
    lib = binding.load_library()
    B, H, M = 64, 16, 16384
    assert lib.la_prefix_workspace_size(B, H, M) > lib.la_noalloc_scratch_bytes()
    p = [ctypes.c_void_p(0x7F0000000000 + i * (1 << 36)) for i in range(10)]
    rc = lib.la_prefix_prefill_noalloc(p[0], p[1], p[2], p[3], p[4], M, p[5], p[6], p[7], p[8],
                                       p[9], B, H, 32768, 16, 64, 1, 0.0, None)
    assert rc == binding.LA_ERR_SCRATCH_TOO_SMALL
    assert "scratch" in binding.status_string(rc)
