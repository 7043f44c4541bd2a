"""GPU parity of la_decode_step and la_prefix_prefill against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import recurrent_lm_gb300 as la
from recurrent_lm_gb300 import inputs
from helpers import TOL, assert_close, sample_heads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_steps_from_oracle_state(dtype):
    """Decode workload at reduced batch (B=2, H=16): state from a seeded
    2048-token oracle prefill, then 64 steps with fresh N(0,1) q,k,v, each
    step in place; every step's y and the final state against the oracle."""
    B, H = 2, 16
    qs, ks, vs, _, _ = inputs.qkv(B, H, 2048, seed=2005, dtype=dtype)
    _, s_r, z_r = oracle.prefill(qs, ks, vs)
    s = torch.from_numpy(s_r).float().to(DEV)
    z = torch.from_numpy(z_r).float().to(DEV)
    s_r = s.double().cpu().numpy()
    z_r = z.double().cpu().numpy()
    tol = TOL[dtype]
    for step in range(64):
        q, k, v = inputs.decode_step_inputs(5, step, B=B)
        q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
        y, _, _ = la.decode_step(q.to(DEV), k.to(DEV), v.to(DEV), s, z, inplace=True)
        y_r, s_r, z_r = oracle.decode_step(q, k, v, s_r, z_r)
        assert_close(f"y step {step}", y, y_r, tol)
    torch.cuda.synchronize()
    assert_close("s", s, s_r, tol)
    assert_close("z", z, z_r, tol)


def test_decode_out_of_place_leaves_input():
    B, H = 3, 5
    s0, z0 = inputs.random_state(B, H, seed=11)
    q, k, v = inputs.decode_step_inputs(5, 0, B=B)
    q, k, v = (t[:, :H].contiguous() for t in (q, k, v))
    s_in, z_in = s0.to(DEV), z0.to(DEV)
    y, s_out, z_out = la.decode_step(q.to(DEV), k.to(DEV), v.to(DEV), s_in, z_in)
    torch.cuda.synchronize()
    assert torch.equal(s_in.cpu(), s0) and torch.equal(z_in.cpu(), z0)
    y_r, s_r, z_r = oracle.decode_step(q, k, v, s0, z0)
    assert_close("y", y, y_r, TOL[torch.bfloat16])
    assert_close("s", s_out, s_r, TOL[torch.bfloat16])
    assert_close("z", z_out, z_r, TOL[torch.bfloat16])


def test_decode_equals_prefill_of_same_tokens():
    """n decode steps from s0 == oracle prefill of those n tokens from s0."""
    B, H, n = 2, 4, 12
    q, k, v, _, _ = inputs.qkv(B, H, n, seed=21, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(B, H, seed=22)
    s, z = s0.to(DEV), z0.to(DEV)
    ys = []
    for i in range(n):
        y, _, _ = la.decode_step(q[:, :, i].contiguous().to(DEV), k[:, :, i].contiguous().to(DEV),
                                 v[:, :, i].contiguous().to(DEV), s, z, inplace=True)
        ys.append(y)
    torch.cuda.synchronize()
    yr, sr, zr = oracle.prefill(q, k, v, s0, z0)
    assert_close("y", torch.stack(ys, dim=2), yr, TOL[torch.bfloat16])
    assert_close("s", s, sr, TOL[torch.bfloat16])
    assert_close("z", z, zr, TOL[torch.bfloat16])


def test_decode_full_batch_sampled_heads():
    """Full decode batch (B=128, H=16), in place, 3 steps; the state of the
    sampled heads comes from the oracle, the rest from a seeded random state."""
    w = inputs.WORKLOADS[5]
    B, H = w.B, w.H
    s0, z0 = inputs.random_state(B, H, seed=55, tokens=2048.0)
    heads = sample_heads(B, H, 6, seed=5)
    qs, ks, vs, _, _ = inputs.qkv(1, len(heads), 2048, seed=2005, dtype=torch.bfloat16)
    _, so, zo = oracle.prefill(qs, ks, vs)
    so32 = torch.from_numpy(so[0]).float()
    zo32 = torch.from_numpy(zo[0]).float()
    for j, (b, h) in enumerate(heads):
        s0[b, h] = so32[j]
        z0[b, h] = zo32[j]
    s, z = s0.to(DEV), z0.to(DEV)
    s_r = so32[None].double().numpy()
    z_r = zo32[None].double().numpy()
    for step in range(3):
        q, k, v = inputs.decode_step_inputs(5, step)
        y, _, _ = la.decode_step(q.to(DEV), k.to(DEV), v.to(DEV), s, z, inplace=True)
        qq = torch.stack([q[b, h] for b, h in heads])[None]
        kk = torch.stack([k[b, h] for b, h in heads])[None]
        vv = torch.stack([v[b, h] for b, h in heads])[None]
        y_r, s_r, z_r = oracle.decode_step(qq, kk, vv, s_r, z_r)
        ys = torch.stack([y[b, h] for b, h in heads])[None]
        assert_close(f"y step {step}", ys, y_r, TOL[torch.bfloat16])
    torch.cuda.synchronize()
    ss = torch.stack([s[b, h] for b, h in heads])[None]
    zs = torch.stack([z[b, h] for b, h in heads])[None]
    assert_close("s", ss, s_r, TOL[torch.bfloat16])
    assert_close("z", zs, z_r, TOL[torch.bfloat16])


def test_decode_graph_pipeline_full_batch():
    """The benchmark's decode pipeline: B=128, H=16, the state from a 2048-token
    GPU prefill, then T=128 consecutive in-place decode steps captured in one
    CUDA graph and replayed.  The oracle runs its own prefill of the 8 sampled
    heads' 2048 tokens (checked against the GPU's), then every step's y and
    the final state of those heads are checked against the oracle's steps."""
    w = inputs.WORKLOADS[5]
    B, H, T = w.B, w.H, 128
    qs, ks, vs = inputs.s0_sequence(5)
    _, s, z = la.prefill(qs.to(DEV), ks.to(DEV), vs.to(DEV))
    torch.cuda.synchronize()
    heads = sample_heads(B, H, 8, seed=6)
    pick = lambda t: torch.stack([t[b, h] for b, h in heads])[None]
    _, s_r, z_r = oracle.prefill(pick(qs), pick(ks), pick(vs))
    tol = TOL[torch.bfloat16]
    assert_close("prefill s", pick(s), s_r, tol)
    assert_close("prefill z", pick(z), z_r, tol)
    steps = [inputs.decode_step_inputs(5, i) for i in range(T)]
    qd = torch.stack([t[0] for t in steps]).to(DEV)
    kd = torch.stack([t[1] for t in steps]).to(DEV)
    vd = torch.stack([t[2] for t in steps]).to(DEV)
    yd = torch.empty((T, B, H, 64), dtype=torch.bfloat16, device=DEV)
    # one call before capture (per-device set-up), on a copy of the state
    la.decode_step(qd[0], kd[0], vd[0], s.clone(), z.clone(), y=yd[0], inplace=True)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(T):
                la.decode_step(qd[i], kd[i], vd[i], s, z, y=yd[i], inplace=True)
    graph.replay()
    torch.cuda.synchronize()
    la.check_device_status()
    for i, (q, k, v) in enumerate(steps):
        qq, kk, vv = (torch.stack([t[b, h] for b, h in heads])[None] for t in (q, k, v))
        y_r, s_r, z_r = oracle.decode_step(qq, kk, vv, s_r, z_r)
        assert_close(f"y step {i}", torch.stack([yd[i, b, h] for b, h in heads])[None], y_r, tol)
    assert_close("s", torch.stack([s[b, h] for b, h in heads])[None], s_r, tol)
    assert_close("z", torch.stack([z[b, h] for b, h in heads])[None], z_r, tol)


# ------------------------------------------------------------------ prefix
def run_prefix(q, k, v, ke, ve, s0=None, z0=None):
    dev = [t.to(DEV) if t is not None else None for t in (q, k, v, ke, ve, s0, z0)]
    got = la.prefix_prefill(*dev)
    torch.cuda.synchronize()
    ref = oracle.prefix_prefill(q, k, v, ke, ve, s0, z0)
    return got, ref


def check(got, ref, tol, what=""):
    for name, a, r in zip("ysz", got, ref):
        assert_close(name + what, a, r, tol)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N,M", [(64, 1), (300, 300), (700, 129), (5000, 4100), (2100, 2048),
                                 (257, 0)])
def test_prefix_edge_lengths(dtype, N, M):
    """M in {0, 1, N}, M across the 2048-token reduction segments, ragged N."""
    q, k, v, ke, ve = inputs.qkv(1, 3, N, seed=400 + M, dtype=dtype, M=max(M, 1))
    ke, ve = ke[:, :, :M].contiguous(), ve[:, :, :M].contiguous()
    got, ref = run_prefix(q, k, v, ke, ve)
    check(got, ref, TOL[dtype], f" N={N} M={M}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_prefix_with_initial_state(dtype):
    q, k, v, ke, ve = inputs.qkv(2, 2, 333, seed=501, dtype=dtype, M=150)
    s0, z0 = inputs.random_state(2, 2, seed=502)
    got, ref = run_prefix(q, k, v, ke, ve, s0, z0)
    check(got, ref, TOL[dtype])


def test_prefix_full_size_sampled_heads():
    """JRT-RNN prefix workload at full size (B=16, H=16, N=32768, M=16384)."""
    w = inputs.WORKLOADS[4]
    q, k, v, ke, ve = inputs.workload_inputs(4)
    y, s, z = la.prefix_prefill(q.to(DEV), k.to(DEV), v.to(DEV), ke.to(DEV), ve.to(DEV))
    torch.cuda.synchronize()
    heads = sample_heads(w.B, w.H, 3, seed=4)

    def pick(t):
        return torch.stack([t[b, h] for b, h in heads])[None]

    ref = oracle.prefix_prefill(pick(q), pick(k), pick(v), pick(ke), pick(ve))
    tol = TOL[torch.bfloat16]
    for name, a, r in zip("ysz", (y, s, z), ref):
        assert_close(name, pick(a), r, tol)
    assert torch.isfinite(y.float()).all()


def test_timeout_status_is_clear_after_normal_calls():
    la.prefill(*(t.to(DEV) for t in inputs.qkv(1, 1, 10, seed=1)[:3]))
    la.check_device_status()


def test_prefix_bitwise_deterministic():
    """The split-M prefix reduction sums segments in a fixed order: repeated
    calls give identical bits (256 heads, 3 segments, non-zero s0)."""
    q, k, v, ke, ve = inputs.qkv(16, 16, 2100, seed=77, M=5000 - 2900)
    s0, z0 = inputs.random_state(16, 16, seed=78, tokens=512.0)
    args = [t.to(DEV) for t in (q, k, v, ke, ve, s0, z0)]
    first = la.prefix_prefill(*args)
    again = la.prefix_prefill(*args)
    torch.cuda.synchronize()
    for x, y in zip(first, again):
        assert torch.equal(x, y)
