"""GPU parity of the per-head decayed prefill and decode step
(la_prefill_decay, la_decode_step_decay) against the fp64 oracle.

Reading (length-generalization notes, sec. 2.1 Eq. (1) with A_t = gamma_h I):
s_i = gamma s_(i-1) + phi(k_i) v_i^T, z likewise; the initial state reaches
position i as gamma^(i+1) s0."""
import math

import numpy as np
import pytest
import torch

import oracle
import recurrent_lm_gb300 as la
from recurrent_lm_gb300 import inputs
from helpers import TOL, assert_close, normwise_rel, sample_heads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GAMMAS4 = [1.0, 0.999, 0.95, 0.5]


def gdev(g):
    return torch.tensor(g, dtype=torch.float32, device=DEV)


def check(got, ref, tol, what=""):
    for name, a, r in zip("ysz", got, ref):
        assert_close(name + what, a, r, tol)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N", [1, 127, 300, 1000])
def test_decayed_prefill(dtype, N):
    """Per-head rates from 1 (no decay) to 0.5, ragged lengths across chunk
    boundaries, non-zero initial state."""
    q, k, v, _, _ = inputs.qkv(2, 4, N, seed=1100 + N, dtype=dtype)
    s0, z0 = inputs.random_state(2, 4, seed=1101)
    g32 = torch.tensor(GAMMAS4, dtype=torch.float32)
    got = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV), gamma=g32.to(DEV))
    la.check_device_status()
    ref = oracle.prefill_decay(q, k, v, g32.double().numpy(), s0, z0)
    check(got, ref, TOL[dtype], f" N={N}")


@pytest.mark.parametrize("N", [2999, 4100])
def test_decayed_prefill_across_epochs(N):
    """bf16 decayed prefill over 24 to 33 chunks with rates from 1 down to 0.3
    (for 0.3 the state before a chunk is below 2^-200 of its value after 128
    tokens), ragged N: y and the final state against the oracle."""
    g = [1.0, 0.999, 0.9375, 0.8, 0.6, 0.55, 0.3, 0.99]
    q, k, v, _, _ = inputs.qkv(1, len(g), N, seed=1150 + N, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(1, len(g), seed=1151)
    g32 = torch.tensor(g, dtype=torch.float32)
    got = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV), gamma=g32.to(DEV))
    la.check_device_status()
    ref = oracle.prefill_decay(q, k, v, g32.double().numpy(), s0, z0)
    check(got, ref, TOL[torch.bfloat16], f" N={N}")


@pytest.mark.parametrize("N", [333, 1000])
def test_decayed_prefill_small_rates(N):
    """bf16 decayed prefill with rates on both sides of 1/4, where the
    intra-chunk factors change from a per-row times per-key product to a
    power-table read, down to 0 (each token sees only itself): against the
    oracle, ragged N."""
    g = [0.26, 0.25, 0.2499, 0.1, 0.01, 0.0, 1.0, 0.4]
    q, k, v, _, _ = inputs.qkv(1, len(g), N, seed=1160 + N, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(1, len(g), seed=1161)
    g32 = torch.tensor(g, dtype=torch.float32)
    got = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV), gamma=g32.to(DEV))
    la.check_device_status()
    ref = oracle.prefill_decay(q, k, v, g32.double().numpy(), s0, z0)
    check(got, ref, TOL[torch.bfloat16], f" N={N}")


def test_decay_of_one_is_the_plain_prefill():
    q, k, v, _, _ = inputs.qkv(2, 3, 700, seed=1110)
    s0, z0 = inputs.random_state(2, 3, seed=1111)
    dev = [t.to(DEV) for t in (q, k, v, s0, z0)]
    a = la.prefill(*dev, gamma=gdev([1.0, 1.0, 1.0]))
    b = la.prefill(*dev)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert normwise_rel(x, y) <= 1e-6


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decayed_decode_steps(dtype):
    """State from a decayed oracle prefill, then 24 decayed decode steps in
    place; every y and the final state against the oracle."""
    B, H = 2, 4
    g = np.array(GAMMAS4)
    qs, ks, vs, _, _ = inputs.qkv(B, H, 500, seed=1120, dtype=dtype)
    _, s_r, z_r = oracle.prefill_decay(qs, ks, vs, g)
    s = torch.from_numpy(s_r).float().to(DEV)
    z = torch.from_numpy(z_r).float().to(DEV)
    s_r, z_r = s.double().cpu().numpy(), z.double().cpu().numpy()
    gd = gdev(GAMMAS4)
    for step in range(24):
        q, k, v = (t[:, :H].to(dtype) for t in inputs.decode_step_inputs(5, step, B=B))
        y, _, _ = la.decode_step(q.contiguous().to(DEV), k.contiguous().to(DEV), v.contiguous().to(DEV), s, z,
                                 inplace=True, gamma=gd)
        y_r, s_r, z_r = oracle.decode_step(q, k, v, s_r, z_r, gamma=g)
        assert_close(f"y step {step}", y, y_r, TOL[dtype])
    la.check_device_status()
    assert_close("s", s, s_r, TOL[dtype])
    assert_close("z", z, z_r, TOL[dtype])


def test_out_of_range_decay_is_clamped_and_reported():
    q, k, v, _, _ = inputs.qkv(1, 4, 200, seed=1130)
    dev = [t.to(DEV) for t in (q, k, v)]
    got = la.prefill(*dev, gamma=gdev([1.5, -0.25, float("nan"), 0.5]))
    with pytest.raises(la.LAError) as e:
        la.check_device_status()
    assert e.value.status == la.binding.LA_ERR_INVALID_ARG
    want = la.prefill(*dev, gamma=gdev([1.0, 0.0, 0.0, 0.5]))
    la.check_device_status()
    for x, y in zip(got, want):
        assert torch.equal(x, y)


def test_decayed_long_prefill_full_size_sampled_heads():
    """Long-prefill workload at full size (B=16, H=16, N=32768, s0 from a
    seeded state) with per-head rates 1 - 2^-(4 + h); sampled heads."""
    w = inputs.WORKLOADS[3]
    q, k, v, _, _ = inputs.workload_inputs(3)
    s0, z0 = inputs.random_state(w.B, w.H, seed=1140, tokens=4096.0)
    g = np.array([1.0 - 2.0 ** -(4 + h) for h in range(w.H)])
    y, s, z = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV),
                         gamma=torch.tensor(g, dtype=torch.float32, device=DEV))
    la.check_device_status()
    g32 = torch.tensor(g, dtype=torch.float32).double().numpy()  # the rates the kernel saw
    for b, h in sample_heads(w.B, w.H, 3, seed=43):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.prefill_decay(q[sl], k[sl], v[sl], g32[h:h + 1], s0[sl], z0[sl])
        for name, a, r in zip("ysz", (y[sl], s[sl], z[sl]), ref):
            assert_close(f"{name} (b={b} h={h})", a, r, TOL[torch.bfloat16])
