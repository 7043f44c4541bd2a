"""GPU tests of la_prefill_host: the prefill with activations and states in
host memory, pipelined over slices of (b, h) rows on internal streams.

Each (b, h) row is computed by the same kernel whether it runs in a slice or
in one launch over all rows, so the host path must match the device path bit
for bit; the fp32 case is also compared with the oracle."""
import pytest
import torch

import oracle
import recurrent_lm_gb300 as la
from recurrent_lm_gb300 import inputs
from helpers import TOL, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def pinned(*ts):
    return [None if t is None else t.contiguous().pin_memory() for t in ts]


def device_run(q, k, v, s0=None, z0=None, want_state=True):
    args = [None if t is None else t.to(DEV) for t in (q, k, v, s0, z0)]
    y, s, z = la.prefill(*args, want_state=want_state)
    torch.cuda.synchronize()
    return [None if t is None else t.cpu() for t in (y, s, z)]


def host_run(q, k, v, s0=None, z0=None, want_state=True):
    y, s, z = la.prefill_host(*pinned(q, k, v, s0, z0), want_state=want_state)
    torch.cuda.current_stream().synchronize()
    return y, s, z


@pytest.mark.parametrize("B,H,N", [(2, 3, 300), (1, 1, 129), (3, 5, 64), (16, 16, 1024)])
def test_host_equals_device_bf16_with_state(B, H, N):
    """Slices of one row (B*H < 8), several rows, a ragged last slice and the
    three in-flight buffers reused several times."""
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=900 + N, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(B, H, seed=901)
    ref = device_run(q, k, v, s0, z0)
    got = host_run(q, k, v, s0, z0)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_host_without_state_matches_device():
    q, k, v, _, _ = inputs.qkv(4, 4, 200, seed=902, dtype=torch.bfloat16)
    yr, _, _ = device_run(q, k, v, want_state=False)
    y, s, z = host_run(q, k, v, want_state=False)
    assert s is None and z is None
    assert torch.equal(y, yr)


def test_host_fp32_matches_oracle():
    q, k, v, _, _ = inputs.qkv(1, 2, 256, seed=903, dtype=torch.float32)
    s0, z0 = inputs.random_state(1, 2, seed=904)
    y, s, z = host_run(q, k, v, s0, z0)
    yr, sr, zr = oracle.prefill(q, k, v, s0, z0)
    tol = TOL[torch.float32]
    assert_close("y", y, yr, tol)
    assert_close("s", s, sr, tol)
    assert_close("z", z, zr, tol)


def test_host_general_feature_dim():
    q, k, v, _, _ = inputs.qkv(2, 2, 100, seed=905, dtype=torch.bfloat16, dk=8)
    ref = device_run(q, k, v)
    got = host_run(q, k, v)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_host_zero_length_copies_state():
    q = torch.empty(2, 3, 0, 16, dtype=torch.bfloat16)
    v = torch.empty(2, 3, 0, 64, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(2, 3, seed=906)
    y, s, z = host_run(q, q, v, s0, z0)
    assert y.numel() == 0 and torch.equal(s, s0) and torch.equal(z, z0)


def test_host_pageable_memory_is_correct():
    """Without page-locked buffers the copies do not overlap, but the result is the same."""
    q, k, v, _, _ = inputs.qkv(2, 2, 150, seed=907, dtype=torch.bfloat16)
    ref = device_run(q, k, v)
    y, s, z = la.prefill_host(q, k, v, y=torch.empty(2, 2, 150, 64, dtype=torch.bfloat16),
                              s_out=torch.empty(2, 2, 273, 64), z_out=torch.empty(2, 2, 273))
    torch.cuda.current_stream().synchronize()
    for a, b in zip((y, s, z), ref):
        assert torch.equal(a, b)


def test_host_rejects_small_workspace():
    q, k, v, _, _ = inputs.qkv(1, 2, 64, seed=908, dtype=torch.bfloat16)
    ws = torch.empty(1024, dtype=torch.uint8, device=DEV)
    with pytest.raises(la.LAError) as e:
        la.prefill_host(*pinned(q, k, v), workspace=ws)
    assert e.value.status == la.LA_ERR_INVALID_ARG


def test_host_prefill_on_a_side_stream():
    """The workspace allocated by the binding is used on the caller's stream,
    not the current one: with other allocations and work on the current
    stream meanwhile, the side-stream call still matches the device path."""
    q, k, v, _, _ = inputs.qkv(4, 4, 700, seed=905, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(4, 4, seed=906)
    ref = device_run(q, k, v, s0, z0)
    side = torch.cuda.Stream()
    hq, hk, hv, hs0, hz0 = pinned(q, k, v, s0, z0)
    outs = []
    for _ in range(3):
        outs.append(la.prefill_host(hq, hk, hv, hs0, hz0, stream=side))
        # current-stream work that would reuse a freed workspace block
        junk = torch.full((1 << 22,), 7, dtype=torch.uint8, device=DEV)
        junk.add_(1)
    side.synchronize()
    torch.cuda.synchronize()
    for y, s, z in outs:
        assert torch.equal(y, ref[0]) and torch.equal(s, ref[1]) and torch.equal(z, ref[2])
