"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/*.h declares, and rejects bad arguments on the host before
any CUDA call (fake, never-dereferenced pointer values are used for that)."""
import ctypes
import glob
import os
import re

import pytest

from recurrent_lm_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"LA_API\s+[\w\s\*]*?\b(la_\w+)\s*\(", text))
    return names


def test_header_declares_the_three_calls():
    names = declared_functions()
    assert {"la_prefill", "la_prefix_prefill", "la_decode_step"} <= names
    assert len(names) >= 6


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in binding.SIGNATURES, f"binding has no signature for {name}"


def test_status_strings(lib):
    for s in range(6):
        assert binding.status_string(s)
    assert "unknown" in binding.status_string(99)
    assert lib.la_version() >= 100


# Fake device addresses: 16-byte aligned, far apart, never dereferenced
# because every call below fails validation before touching the device.
A = 0x7f0000000000
STEP = 1 << 36


def fake(i, misalign=0):
    return ctypes.c_void_p(A + i * STEP + misalign)


def call_prefill(lib, B=1, H=1, N=8, dk=16, dv=64, dtype=1, ptrs=None, s0=True):
    p = ptrs or [fake(i) for i in range(8)]
    if not s0:
        p[3] = None
        p[4] = None
    return lib.la_prefill(*p, B, H, N, dk, dv, dtype, 0.0, None)


def test_prefill_rejects_unsupported_dims(lib):
    assert call_prefill(lib, dk=12) == binding.LA_ERR_UNSUPPORTED  # d' in {8, 16, 24, 32} only
    assert call_prefill(lib, dk=64) == binding.LA_ERR_UNSUPPORTED
    assert call_prefill(lib, dv=32) == binding.LA_ERR_UNSUPPORTED
    assert call_prefill(lib, dtype=7) == binding.LA_ERR_UNSUPPORTED


def test_prefill_rejects_bad_shapes(lib):
    assert call_prefill(lib, B=0) == binding.LA_ERR_INVALID_ARG
    assert call_prefill(lib, H=-1) == binding.LA_ERR_INVALID_ARG
    assert call_prefill(lib, N=-5) == binding.LA_ERR_INVALID_ARG
    assert call_prefill(lib, B=1 << 20, H=1 << 20) == binding.LA_ERR_INVALID_ARG


def test_prefill_rejects_null_and_half_state(lib):
    p = [fake(i) for i in range(8)]
    p[0] = None  # q
    assert call_prefill(lib, ptrs=p) == binding.LA_ERR_INVALID_ARG
    p = [fake(i) for i in range(8)]
    p[4] = None  # z0 without s0
    assert call_prefill(lib, ptrs=p) == binding.LA_ERR_INVALID_ARG


def test_prefill_rejects_misaligned(lib):
    for i in range(8):
        p = [fake(j) for j in range(8)]
        p[i] = fake(i, misalign=4)
        assert call_prefill(lib, ptrs=p) == binding.LA_ERR_MISALIGNED, i


def test_prefill_rejects_overlap(lib):
    p = [fake(i) for i in range(8)]
    p[5] = ctypes.c_void_p(p[2].value + 64)  # y inside v
    assert call_prefill(lib, ptrs=p) == binding.LA_ERR_INVALID_ARG
    p = [fake(i) for i in range(8)]
    p[6] = ctypes.c_void_p(p[3].value)       # s_out == s0 (prefill is not in place)
    assert call_prefill(lib, ptrs=p) == binding.LA_ERR_INVALID_ARG


def test_prefix_rejects_m_greater_than_n(lib):
    p = [fake(i) for i in range(12)]
    rc = lib.la_prefix_prefill(p[0], p[1], p[2], p[3], p[4], 9, p[5], p[6], p[7], p[8], p[9],
                               p[10], 1 << 40, 1, 1, 8, 16, 64, 1, 0.0, None)
    assert rc == binding.LA_ERR_INVALID_ARG
    rc = lib.la_prefix_prefill(p[0], p[1], p[2], p[3], p[4], -1, p[5], p[6], p[7], p[8], p[9],
                               p[10], 1 << 40, 1, 1, 8, 16, 64, 1, 0.0, None)
    assert rc == binding.LA_ERR_INVALID_ARG


def test_prefix_rejects_small_or_misaligned_workspace(lib):
    need = lib.la_prefix_workspace_size(2, 3, 5000)
    assert need > 0 and need % 256 == 0
    assert lib.la_prefix_workspace_size(2, 3, 0) == 0
    p = [fake(i) for i in range(12)]
    # smaller than the prefix partial states (at least 3 segments x 6 heads x 70,980 B):
    # rejected; between that and `need` the call runs without split heads
    rc = lib.la_prefix_prefill(p[0], p[1], p[2], p[3], p[4], 5000, p[5], p[6], p[7], p[8], p[9],
                               p[10], 6 * 3 * 70980 - 1, 2, 3, 8000, 16, 64, 1, 0.0, None)
    assert rc == binding.LA_ERR_INVALID_ARG
    assert need > 6 * 3 * 70980
    ws = ctypes.c_void_p(p[10].value + 16)   # 16- but not 256-byte aligned
    rc = lib.la_prefix_prefill(p[0], p[1], p[2], p[3], p[4], 5000, p[5], p[6], p[7], p[8], p[9],
                               ws, need, 2, 3, 8000, 16, 64, 1, 0.0, None)
    assert rc == binding.LA_ERR_MISALIGNED


def test_decode_rejects_bad_args(lib):
    p = [fake(i) for i in range(8)]
    assert lib.la_decode_step(*p, 4, 2, 16, 32, 1, 0.0, None) == binding.LA_ERR_UNSUPPORTED
    assert lib.la_decode_step(*p, 0, 2, 16, 64, 1, 0.0, None) == binding.LA_ERR_INVALID_ARG
    q = list(p); q[3] = None
    assert lib.la_decode_step(*q, 4, 2, 16, 64, 1, 0.0, None) == binding.LA_ERR_INVALID_ARG
    q = list(p); q[7] = fake(7, misalign=8)
    assert lib.la_decode_step(*q, 4, 2, 16, 64, 1, 0.0, None) == binding.LA_ERR_MISALIGNED
    q = list(p); q[5] = ctypes.c_void_p(p[3].value + 256)   # s_out partially overlaps s_in
    assert lib.la_decode_step(*q, 4, 2, 16, 64, 1, 0.0, None) == binding.LA_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 4, 16, dtype=torch.bfloat16)
    v = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        binding.prefill(q, q, v)


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    mod = importlib.import_module("recurrent_lm_gb300.binding")
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(RuntimeError, match="missing"):
            mod.load_library(str(tmp_path / "nope.so"))
    finally:
        mod._lib = saved


def test_padded_calls_reject_null_misaligned_or_overlapping_pads(lib):
    """la_prefill_padded / la_prefix_prefill_padded: the pad counts are a
    required 4-byte aligned device array that no output may overlap."""
    p = [fake(i) for i in range(8)]
    q, k, v, s0, z0, y, so, zo = p
    args = (1, 1, 8, 16, 64, 1, 0.0, None)
    assert lib.la_prefill_padded(q, k, v, s0, z0, None, y, so, zo, *args) == binding.LA_ERR_INVALID_ARG
    assert lib.la_prefill_padded(q, k, v, s0, z0, fake(9, misalign=2), y, so, zo,
                                 *args) == binding.LA_ERR_MISALIGNED
    inside_y = ctypes.c_void_p(y.value + 32)
    assert lib.la_prefill_padded(q, k, v, s0, z0, inside_y, y, so, zo, *args) == binding.LA_ERR_INVALID_ARG
    ke, ve, ws = fake(10), fake(11), fake(12)
    pargs = (1, 1, 8, 16, 64, 1, 0.0, None)
    assert lib.la_prefix_prefill_padded(q, k, v, ke, ve, 4, s0, z0, None, y, so, zo, ws, 1 << 30,
                                        *pargs) == binding.LA_ERR_INVALID_ARG
    assert lib.la_prefix_prefill_padded(q, k, v, ke, ve, 4, s0, z0, fake(9, misalign=1), y, so, zo, ws,
                                        1 << 30, *pargs) == binding.LA_ERR_MISALIGNED
    assert lib.la_prefix_prefill_padded(q, k, v, ke, ve, 9, s0, z0, fake(9), y, so, zo, ws, 1 << 30,
                                        *pargs) == binding.LA_ERR_INVALID_ARG  # M > N


def test_padding_decay_and_prefix_need_d16(lib):
    """The general-d' path covers la_prefill and la_decode_step; the padded,
    decayed and prefix calls exist for d' = 16 only."""
    p = [fake(i) for i in range(8)]
    q, k, v, s0, z0, y, so, zo = p
    assert lib.la_prefill_padded(q, k, v, s0, z0, fake(9), y, so, zo, 1, 1, 8, 8, 64, 1, 0.0,
                                 None) == binding.LA_ERR_UNSUPPORTED
    assert lib.la_prefill_decay(q, k, v, s0, z0, fake(9), y, so, zo, 1, 1, 8, 24, 64, 1, 0.0,
                                None) == binding.LA_ERR_UNSUPPORTED
    assert lib.la_prefix_prefill(q, k, v, fake(10), fake(11), 4, s0, z0, y, so, zo, fake(12), 1 << 30,
                                 1, 1, 8, 32, 64, 1, 0.0, None) == binding.LA_ERR_UNSUPPORTED
    assert lib.la_decode_step_decay(q, k, v, fake(9), s0, z0, so, zo, y, 1, 1, 8, 64, 1, 0.0,
                                    None) == binding.LA_ERR_UNSUPPORTED


def test_host_prefill_workspace_size(lib):
    need = lib.la_prefill_host_workspace_size(2, 3, 300, 16, 1)
    assert need > 0 and need % 256 == 0
    # three slices of one row in flight: q, k, v, y and both states per slice
    per_row = 2 * 300 * (16 + 16 + 64 + 64) + 4 * (273 * 64 + 273) * 2
    assert 3 * per_row <= need <= 3 * per_row + 3 * 8 * 256
    assert lib.la_prefill_host_workspace_size(0, 3, 300, 16, 1) == 0
    assert lib.la_prefill_host_workspace_size(2, 3, 300, 12, 1) == 0
    assert lib.la_prefill_host_workspace_size(2, 3, 300, 16, 1) < lib.la_prefill_host_workspace_size(2, 3, 300, 16, 0)


def test_prefill_workspace_size_general_dk(lib):
    """d' = 24, 32 with bf16 (dtype 1): the workspace of the tensor-core form,
    at least its buffers per token of whole 128-token chunks (features of q and
    k, [v | 1 | 0], chunk states in fp32 and bf16, the numerator, P) plus the
    cuBLASLt workspace; none for fp32 or an empty sequence."""
    for dk, dp in ((24, 328), (32, 568)):
        B, H, N = 2, 3, 300
        tokens = B * H * 384  # three chunks
        per_token = 2 * 2 * dp + 2 * 80 + (4 + 2) * dp * 80 / 128 + 4 * 80 + 2 * 128
        need = lib.la_prefill_workspace_size(B, H, N, dk, 1)
        assert tokens * per_token + (32 << 20) <= need <= tokens * per_token + (32 << 20) + 8 * 256
        assert lib.la_prefill_workspace_size(B, H, N, dk, 0) == 0
        assert lib.la_prefill_workspace_size(B, H, 0, dk, 1) == 0
    assert lib.la_prefill_workspace_size(2, 3, 300, 12, 1) == 0
    # past 2^31 head-tokens (whole chunks) the form is not offered: la_prefill_ws
    # then runs la_prefill
    assert lib.la_prefill_workspace_size(1 << 12, 16, (1 << 15) + 1, 24, 1) == 0
    assert lib.la_prefill_workspace_size(1 << 12, 16, 1 << 15, 24, 1) > 0


def call_host(lib, p, ws, ws_bytes, B=2, H=3, N=300, dk=16, dtype=1):
    return lib.la_prefill_host(p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], ws, ws_bytes, B, H, N,
                               dk, 64, dtype, 0.0, None)


def test_host_prefill_rejects_bad_args(lib):
    need = lib.la_prefill_host_workspace_size(2, 3, 300, 16, 1)
    p = [fake(i) for i in range(8)]
    ws = fake(9)
    assert call_host(lib, p, ws, need - 1) == binding.LA_ERR_INVALID_ARG     # workspace too small
    assert call_host(lib, p, None, need) == binding.LA_ERR_INVALID_ARG       # no workspace
    assert call_host(lib, p, fake(9, misalign=16), need) == binding.LA_ERR_MISALIGNED
    assert call_host(lib, p, ws, need, dk=12) == binding.LA_ERR_UNSUPPORTED
    q = list(p); q[4] = None                                                 # s0 without z0
    assert call_host(lib, q, ws, need) == binding.LA_ERR_INVALID_ARG
    q = list(p); q[5] = ctypes.c_void_p(p[0].value + 64)                     # y overlaps q
    assert call_host(lib, q, ws, need) == binding.LA_ERR_INVALID_ARG
    # host buffers need no alignment: a misaligned q still reaches the workspace check
    q = list(p); q[0] = fake(0, misalign=2)
    assert call_host(lib, q, ws, need - 1) == binding.LA_ERR_INVALID_ARG
    # the workspace must not overlap an input or an output (device-resident
    # buffers are accepted, so they could)
    assert call_host(lib, p, ctypes.c_void_p(p[0].value + 256), need) == binding.LA_ERR_INVALID_ARG
    assert call_host(lib, p, ctypes.c_void_p(p[6].value), need) == binding.LA_ERR_INVALID_ARG


def test_compact_calls_reject_bad_args(lib):
    """The compact-state calls: d' = 16 and d_v = 64 only, bf16 only for the
    prefill, required pointers, 16-byte alignment, no overlap (the overlap
    ranges use the 153-row sizes)."""
    p = [fake(i) for i in range(8)]
    # decode: dims, shapes, NULL, alignment, partial overlap of the compact state
    assert lib.la_decode_step_compact(*p, 4, 2, 8, 64, 1, 0.0, None) == binding.LA_ERR_UNSUPPORTED
    assert lib.la_decode_step_compact(*p, 4, 2, 16, 32, 1, 0.0, None) == binding.LA_ERR_UNSUPPORTED
    assert lib.la_decode_step_compact(*p, 0, 2, 16, 64, 1, 0.0, None) == binding.LA_ERR_INVALID_ARG
    q = list(p); q[4] = None
    assert lib.la_decode_step_compact(*q, 4, 2, 16, 64, 1, 0.0, None) == binding.LA_ERR_INVALID_ARG
    q = list(p); q[6] = fake(6, misalign=4)
    assert lib.la_decode_step_compact(*q, 4, 2, 16, 64, 1, 0.0, None) == binding.LA_ERR_MISALIGNED
    # s_out starts inside s_in's last head: 153 rows * 64 * 4 B per head, 8 heads
    q = list(p); q[5] = ctypes.c_void_p(p[3].value + 8 * 153 * 256 - 256)
    assert lib.la_decode_step_compact(*q, 4, 2, 16, 64, 1, 0.0, None) == binding.LA_ERR_INVALID_ARG
    q = list(p); q[5] = ctypes.c_void_p(p[3].value + 8 * 153 * 256)   # just past it: fine up to the device
    assert lib.la_decode_step_compact(*q, 4, 2, 16, 64, 1, 0.0, None) not in (
        binding.LA_ERR_INVALID_ARG, binding.LA_ERR_MISALIGNED, binding.LA_ERR_UNSUPPORTED)
    # prefill: fp32 activations and d' != 16 are unsupported; half state is invalid
    assert lib.la_prefill_compact(*p, 1, 1, 8, 16, 64, 0, 0.0, None) == binding.LA_ERR_UNSUPPORTED
    assert lib.la_prefill_compact(*p, 1, 1, 8, 8, 64, 1, 0.0, None) == binding.LA_ERR_UNSUPPORTED
    q = list(p); q[4] = None
    assert lib.la_prefill_compact(*q, 1, 1, 8, 16, 64, 1, 0.0, None) == binding.LA_ERR_INVALID_ARG
    q = list(p); q[6] = ctypes.c_void_p(p[3].value)
    assert lib.la_prefill_compact(*q, 1, 1, 8, 16, 64, 1, 0.0, None) == binding.LA_ERR_INVALID_ARG
    # conversions
    c = [fake(i) for i in range(4)]
    for fn in (lib.la_state_to_compact, lib.la_state_from_compact):
        assert fn(*c, 2, 3, 16, 48, None) == binding.LA_ERR_UNSUPPORTED
        assert fn(*c, 2, 3, 24, 64, None) == binding.LA_ERR_UNSUPPORTED
        assert fn(*c, 0, 3, 16, 64, None) == binding.LA_ERR_INVALID_ARG
        for i in range(4):
            d = list(c); d[i] = None
            assert fn(*d, 2, 3, 16, 64, None) == binding.LA_ERR_INVALID_ARG
            d = list(c); d[i] = fake(i, misalign=8)
            assert fn(*d, 2, 3, 16, 64, None) == binding.LA_ERR_MISALIGNED
        d = list(c); d[2] = ctypes.c_void_p(c[0].value + 1024)
        assert fn(*d, 2, 3, 16, 64, None) == binding.LA_ERR_INVALID_ARG
