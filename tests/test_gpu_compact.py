"""GPU parity of the compact-state calls (la_state_to_compact,
la_state_from_compact, la_prefill_compact, la_decode_step_compact) against
the fp64 oracle.

The oracle computes in the 273-row layout (oracle.prefill, oracle.decode_step)
and the tests fold its states symmetrically with oracle.compact.fold_state
(BASED reading notes, sec. 2.3: the 153-feature symmetric form) before
comparing them with the library's compact states.
"""
import numpy as np
import pytest
import torch

import oracle
import recurrent_lm_gb300 as la
from oracle import compact
from recurrent_lm_gb300 import inputs
from helpers import TOL, assert_close, sample_heads, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def fold(s, z):
    return compact.fold_state(to64(s), to64(z))


def dev32(a):
    return torch.from_numpy(np.ascontiguousarray(a)).float().to(DEV)


def oracle_state(B, H, N, seed):
    """A state the recurrence builds: the oracle's prefill of a seeded sequence."""
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=seed, dtype=torch.bfloat16)
    _, s, z = oracle.prefill(q, k, v)
    return s, z


# ------------------------------------------------------------------ conversions
@pytest.mark.parametrize("B,H", [(2, 3), (3, 5), (1, 300)])
def test_state_conversions(B, H):
    """to_compact against the oracle's fold (of a state with an antisymmetric
    part, which is dropped), from_compact against its unfold, and the round
    trip compact -> 273 -> compact."""
    s0, z0 = inputs.random_state(B, H, seed=71)
    s_c, z_c = la.state_to_compact(s0.to(DEV), z0.to(DEV))
    torch.cuda.synchronize()
    rs, rz = fold(s0, z0)
    assert_close("s_c", s_c, rs, 1e-6)
    assert_close("z_c", z_c, rz, 1e-6)
    s, z = la.state_from_compact(s_c, z_c)
    torch.cuda.synchronize()
    us, uz = compact.unfold_state(to64(s_c), to64(z_c))
    assert_close("s", s, us, 1e-6)
    assert_close("z", z, uz, 1e-6)
    s_c2, z_c2 = la.state_to_compact(s, z)
    torch.cuda.synchronize()
    assert_close("round trip s_c", s_c2, to64(s_c), 1e-6)
    assert_close("round trip z_c", z_c2, to64(z_c), 1e-6)


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_compact_steps(dtype):
    """B=2, H=16: the folded state of a 2048-token oracle prefill, then 64
    in-place compact steps; every y and the final state against the oracle's
    273-row steps (state folded for the comparison)."""
    B, H = 2, 16
    s_r, z_r = oracle_state(B, H, 2048, seed=2005)
    s_c0, z_c0 = compact.fold_state(s_r, z_r)
    s, z = dev32(s_c0), dev32(z_c0)
    # the oracle starts from the fp32 values the library was given
    s_r, z_r = compact.unfold_state(to64(s), to64(z))
    tol = TOL[dtype]
    for step in range(64):
        q, k, v = inputs.decode_step_inputs(5, step, B=B)
        q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
        y, _, _ = la.decode_step_compact(q.to(DEV), k.to(DEV), v.to(DEV), s, z, inplace=True)
        y_r, s_r, z_r = oracle.decode_step(q, k, v, s_r, z_r)
        assert_close(f"y step {step}", y, y_r, tol)
    torch.cuda.synchronize()
    fs, fz = compact.fold_state(s_r, z_r)
    assert_close("s_c", s, fs, tol)
    assert_close("z_c", z, fz, tol)


@pytest.mark.parametrize("B,H", [(11, 16), (3, 5), (1, 1)])
def test_decode_compact_out_of_place_every_head(B, H):
    """Out of place (the input state is left as it was), more heads than SMs
    and odd head counts; every head against the oracle, fp32 activations."""
    s0, z0 = inputs.random_state(B, H, seed=12 + B)
    # a state the recurrence could build: symmetric quadratic block
    s0c, z0c = compact.fold_state(to64(s0), to64(z0))
    s_in, z_in = dev32(s0c), dev32(z0c)
    s_keep, z_keep = s_in.clone(), z_in.clone()
    q, k, v = inputs.decode_step_inputs(5, 3, B=B)
    q, k, v = (t[:, :H].contiguous().float() for t in (q, k, v))
    y, s_out, z_out = la.decode_step_compact(q.to(DEV), k.to(DEV), v.to(DEV), s_in, z_in)
    torch.cuda.synchronize()
    assert torch.equal(s_in, s_keep) and torch.equal(z_in, z_keep)
    s_r, z_r = compact.unfold_state(to64(s_keep), to64(z_keep))
    y_r, s1, z1 = oracle.decode_step(q, k, v, s_r, z_r)
    fs, fz = compact.fold_state(s1, z1)
    tol = TOL[torch.float32]
    assert_close("y", y, y_r, tol)
    assert_close("s_c", s_out, fs, tol)
    assert_close("z_c", z_out, fz, tol)


def test_decode_compact_graph_pipeline_full_batch():
    """The benchmark's compact decode pipeline: B=128, H=16, the compact state
    from a 2048-token la_prefill_compact, then T=128 in-place compact steps in
    one CUDA graph.  The oracle runs its own prefill of 8 sampled heads
    (checked against the GPU's compact state), then every step's y and the
    final state of those heads against the oracle's steps."""
    w = inputs.WORKLOADS[5]
    B, H, T = w.B, w.H, 128
    qs, ks, vs = inputs.s0_sequence(5)
    _, s, z = la.prefill_compact(qs.to(DEV), ks.to(DEV), vs.to(DEV))
    torch.cuda.synchronize()
    heads = sample_heads(B, H, 8, seed=7)
    pick = lambda t: torch.stack([t[b, h] for b, h in heads])[None]
    _, s_r, z_r = oracle.prefill(pick(qs), pick(ks), pick(vs))
    tol = TOL[torch.bfloat16]
    fs, fz = compact.fold_state(s_r, z_r)
    assert_close("prefill s_c", pick(s), fs, tol)
    assert_close("prefill z_c", pick(z), fz, tol)
    steps = [inputs.decode_step_inputs(5, i) for i in range(T)]
    qd = torch.stack([t[0] for t in steps]).to(DEV)
    kd = torch.stack([t[1] for t in steps]).to(DEV)
    vd = torch.stack([t[2] for t in steps]).to(DEV)
    yd = torch.empty((T, B, H, 64), dtype=torch.bfloat16, device=DEV)
    la.decode_step_compact(qd[0], kd[0], vd[0], s.clone(), z.clone(), y=yd[0], inplace=True)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(T):
                la.decode_step_compact(qd[i], kd[i], vd[i], s, z, y=yd[i], inplace=True)
    graph.replay()
    torch.cuda.synchronize()
    la.check_device_status()
    for i, (q, k, v) in enumerate(steps):
        y_r, s_r, z_r = oracle.decode_step(pick(q), pick(k), pick(v), s_r, z_r)
        assert_close(f"y step {i}", pick(yd[i]), y_r, tol)
    fs, fz = compact.fold_state(s_r, z_r)
    assert_close("s_c", pick(s), fs, tol)
    assert_close("z_c", pick(z), fz, tol)


# ------------------------------------------------------------------ prefill
@pytest.mark.parametrize("N", [1, 127, 128, 300, 2100])
def test_prefill_compact_from_folded_state(N):
    """bf16 prefill with a compact s0 (the folded state of a 500-token oracle
    prefill): y and the compact final state against the oracle's 273-row
    prefill from the unfolded s0 (final state folded)."""
    B, H = 2, 3
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=3100 + N, dtype=torch.bfloat16)
    s0, z0 = oracle_state(B, H, 500, seed=3000)
    s0c, z0c = compact.fold_state(s0, z0)
    s_c0, z_c0 = dev32(s0c), dev32(z0c)
    y, s_c, z_c = la.prefill_compact(q.to(DEV), k.to(DEV), v.to(DEV), s_c0, z_c0)
    torch.cuda.synchronize()
    s_u, z_u = compact.unfold_state(to64(s_c0), to64(z_c0))
    y_r, s_r, z_r = oracle.prefill(q, k, v, s_u, z_u)
    tol = TOL[torch.bfloat16]
    fs, fz = compact.fold_state(s_r, z_r)
    assert_close("y", y, y_r, tol)
    assert_close("s_c", s_c, fs, tol)
    assert_close("z_c", z_c, fz, tol)


def test_prefill_compact_zero_state_and_empty():
    """Zero initial state (NULL), and N = 0 (the compact s0 is copied)."""
    B, H, N = 1, 4, 700
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=3200, dtype=torch.bfloat16)
    y, s_c, z_c = la.prefill_compact(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    y_r, s_r, z_r = oracle.prefill(q, k, v)
    tol = TOL[torch.bfloat16]
    fs, fz = compact.fold_state(s_r, z_r)
    assert_close("y", y, y_r, tol)
    assert_close("s_c", s_c, fs, tol)
    assert_close("z_c", z_c, fz, tol)
    e = torch.empty((B, H, 0, 16), dtype=torch.bfloat16, device=DEV)
    ev = torch.empty((B, H, 0, 64), dtype=torch.bfloat16, device=DEV)
    _, s_c2, z_c2 = la.prefill_compact(e, e.clone(), ev, s_c, z_c)
    torch.cuda.synchronize()
    assert torch.equal(s_c2, s_c) and torch.equal(z_c2, z_c)


def test_prefill_compact_antisymmetric_part_is_invisible():
    """A 273-row s0 with an antisymmetric part: la_prefill from it and
    la_prefill_compact from its GPU-folded form give y within the bf16
    tolerance of the oracle's y from the original s0, and the compact final
    state is the fold of the oracle's."""
    B, H, N = 2, 2, 400
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=3300, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(B, H, seed=3301, tokens=300.0)
    s_c0, z_c0 = la.state_to_compact(s0.to(DEV), z0.to(DEV))
    y, s_c, z_c = la.prefill_compact(q.to(DEV), k.to(DEV), v.to(DEV), s_c0, z_c0)
    y_full, _, _ = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV))
    torch.cuda.synchronize()
    y_r, s_r, z_r = oracle.prefill(q, k, v, s0, z0)
    tol = TOL[torch.bfloat16]
    fs, fz = compact.fold_state(s_r, z_r)
    assert_close("y", y, y_r, tol)
    assert_close("y (273-row call)", y_full, y_r, tol)
    assert_close("s_c", s_c, fs, tol)
    assert_close("z_c", z_c, fz, tol)


def test_prefill_compact_unsupported_for_fp32():
    q = torch.zeros((1, 1, 8, 16), device=DEV)
    v = torch.zeros((1, 1, 8, 64), device=DEV)
    with pytest.raises(la.LAError) as e:
        la.prefill_compact(q, q.clone(), v)
    assert e.value.status == la.LA_ERR_UNSUPPORTED
