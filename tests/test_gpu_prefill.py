"""GPU parity of la_prefill against the fp64 oracle (through the C-ABI).

Inputs are seeded and synthetic (recurrent_lm_gb300.inputs); the oracle gets
the same values upcast exactly to fp64 (bf16 inputs: the bf16-rounded values),
so the comparison measures kernel error, not input quantisation."""
import numpy as np
import pytest
import torch

import oracle
import recurrent_lm_gb300 as la
from recurrent_lm_gb300 import inputs
from helpers import TOL, assert_close, normwise_rel, sample_heads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_both(q, k, v, s0=None, z0=None, eps=0.0):
    dev = [t.to(DEV) if t is not None else None for t in (q, k, v, s0, z0)]
    y, s, z = la.prefill(*dev, eps=eps)
    torch.cuda.synchronize()
    yr, sr, zr = oracle.prefill(q, k, v, s0, z0, eps)
    return (y, s, z), (yr, sr, zr)


def check(got, ref, tol, what=""):
    y, s, z = got
    yr, sr, zr = ref
    assert_close(f"y{what}", y, yr, tol)
    assert_close(f"s{what}", s, sr, tol)
    assert_close(f"z{what}", z, zr, tol)


def test_small_fp32_workload():
    """fp32, B=1, H=2, N=256, q,k,v ~ N(0,1), zero initial state: <= 1e-4."""
    q, k, v, _, _ = inputs.workload_inputs(1)
    got, ref = run_both(q, k, v)
    check(got, ref, TOL[torch.float32])


def test_based_layer_bf16_workload():
    """bf16, B=8, H=16, N=2048, inputs scaled by 1/sqrt2, zero s0: <= 2e-2."""
    q, k, v, _, _ = inputs.workload_inputs(2)
    got, ref = run_both(q, k, v)
    check(got, ref, TOL[torch.bfloat16])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N", [1, 2, 3, 17, 64, 65, 127, 128, 129, 255, 383])
def test_ragged_lengths(dtype, N):
    """Lengths below, at and across chunk boundaries, with a non-zero s0."""
    q, k, v, _, _ = inputs.qkv(2, 3, N, seed=300 + N, dtype=dtype)
    s0, z0 = inputs.random_state(2, 3, seed=77)
    got, ref = run_both(q, k, v, s0, z0)
    check(got, ref, TOL[dtype], f" N={N}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_zero_length_copies_state(dtype):
    q = torch.empty(2, 3, 0, 16, dtype=dtype)
    v = torch.empty(2, 3, 0, 64, dtype=dtype)
    s0, z0 = inputs.random_state(2, 3, seed=5)
    y, s, z = la.prefill(q.to(DEV), q.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV))
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert torch.equal(s.cpu(), s0) and torch.equal(z.cpu(), z0)
    y, s, z = la.prefill(q.to(DEV), q.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    assert torch.count_nonzero(s) == 0 and torch.count_nonzero(z) == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_state_passing_split_equals_oracle_whole(dtype):
    """Run 300 tokens, feed (s, z) back as s0, run 211 more: matches one oracle
    run over all 511 tokens (state passing)."""
    q, k, v, _, _ = inputs.qkv(1, 4, 511, seed=41, dtype=dtype)
    q_, k_, v_ = (t.to(DEV) for t in (q, k, v))
    y1, s1, z1 = la.prefill(q_[:, :, :300].contiguous(), k_[:, :, :300].contiguous(),
                            v_[:, :, :300].contiguous())
    y2, s2, z2 = la.prefill(q_[:, :, 300:].contiguous(), k_[:, :, 300:].contiguous(),
                            v_[:, :, 300:].contiguous(), s1, z1)
    torch.cuda.synchronize()
    yr, sr, zr = oracle.prefill(q, k, v)
    tol = TOL[dtype]
    assert_close("y", torch.cat([y1, y2], dim=2), yr, tol)
    assert_close("s", s2, sr, tol)
    assert_close("z", z2, zr, tol)


def test_eps_is_used():
    q, k, v, _, _ = inputs.qkv(1, 2, 50, seed=9, dtype=torch.float32)
    got, ref = run_both(q, k, v, eps=0.75)
    check(got, ref, TOL[torch.float32])


def test_q_or_k_zero_gives_running_mean():
    """K = 1 when q = 0: y_i is the running mean of v (closed form, no oracle)."""
    N = 300
    _, k, v, _, _ = inputs.qkv(1, 2, N, seed=12, dtype=torch.bfloat16)
    q = torch.zeros_like(k)
    y, _, _ = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    mean = torch.cumsum(v.double(), dim=2) / torch.arange(1, N + 1).double()[None, None, :, None]
    assert normwise_rel(y, mean) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_bitwise_deterministic(dtype):
    """Repeated calls give identical bits.  The bf16 case uses 256 heads
    (more CTAs than SMs), a ragged length and a non-zero s0, the setting in
    which a synchronisation mistake between the kernel's roles would show."""
    B, H, N, reps = (2, 2, 700, 2) if dtype == torch.float32 else (16, 16, 4000, 4)
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=3, dtype=dtype)
    s0, z0 = inputs.random_state(B, H, seed=4, tokens=4096.0)
    args = [t.to(DEV) for t in (q, k, v, s0, z0)]
    first = la.prefill(*args)
    for _ in range(reps - 1):
        again = la.prefill(*args)
        torch.cuda.synchronize()
        for x, y in zip(first, again):
            assert torch.equal(x, y)


def test_outputs_stay_inside_their_buffers():
    """Guard bands: every output is a view into a larger NaN-filled buffer;
    the margins must be untouched after the call."""
    B, H, N = 2, 2, 200
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=8, dtype=torch.bfloat16)
    pad = 4096

    def guarded(n, dtype):
        buf = torch.full((n + 2 * pad,), float("nan"), dtype=dtype, device=DEV)
        return buf, buf[pad:pad + n]

    yb, yv = guarded(B * H * N * 64, torch.bfloat16)
    sb, sv = guarded(B * H * 273 * 64, torch.float32)
    zb, zv = guarded(B * H * 273, torch.float32)
    la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), y=yv.view(B, H, N, 64),
               s_out=sv.view(B, H, 273, 64), z_out=zv.view(B, H, 273))
    torch.cuda.synchronize()
    for buf, view in ((yb, yv), (sb, sv), (zb, zv)):
        assert torch.isnan(buf[:pad].float()).all() and torch.isnan(buf[-pad:].float()).all()
        assert torch.isfinite(view.float()).all()


def _heads(t, heads):
    return torch.stack([t[b, h] for b, h in heads])[None]


def test_long_prefill_full_size_sampled_heads():
    """Long prefill with state passing at full size (B=16, H=16, N=32768), the
    call the benchmark times.  s0/z0 are the GPU's final state of a separately
    seeded 4096-token sequence, as in the benchmark; that run is compared with
    the oracle first, then the long prefill from the GPU's s0 is compared with
    the oracle run from the same fp32 s0, on 16 sampled heads."""
    w = inputs.WORKLOADS[3]
    q, k, v, _, _ = inputs.workload_inputs(3)
    qs, ks, vs = inputs.s0_sequence(3)
    heads = sample_heads(w.B, w.H, 16, seed=3)
    tol = TOL[torch.bfloat16]
    _, s0, z0 = la.prefill(qs.to(DEV), ks.to(DEV), vs.to(DEV))
    torch.cuda.synchronize()
    _, s0r, z0r = oracle.prefill(_heads(qs, heads), _heads(ks, heads), _heads(vs, heads))
    assert_close("s0 (4096-token run)", _heads(s0, heads), s0r, tol)
    assert_close("z0 (4096-token run)", _heads(z0, heads), z0r, tol)
    y, s, z = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0, z0)
    torch.cuda.synchronize()
    yr, sr, zr = oracle.prefill(_heads(q, heads), _heads(k, heads), _heads(v, heads),
                                _heads(s0, heads).cpu(), _heads(z0, heads).cpu())
    assert_close("y", _heads(y, heads), yr, tol)
    assert_close("s", _heads(s, heads), sr, tol)
    assert_close("z", _heads(z, heads), zr, tol)
    assert torch.isfinite(y.float()).all()


@pytest.mark.parametrize("B,H,N", [(11, 16, 4096 + 77), (1, 153, 3 * 128 + 5), (2, 100, 1000)])
def test_more_heads_than_sms_every_head(B, H, N):
    """More heads than SMs (176, 153 and 200 heads: two waves of CTAs, the
    second partly filled), ragged lengths, a non-zero s0: every head matches
    the oracle, y, s and z."""
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=900 + H, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(B, H, seed=901, tokens=1024.0)
    got, ref = run_both(q, k, v, s0, z0)
    check(got, ref, TOL[torch.bfloat16], f" B={B} H={H} N={N}")


def test_output_without_final_state_is_identical():
    """Asking for no final state (s_out, z_out NULL) gives the same y bits as
    asking for it."""
    B, H, N = 11, 16, 2000
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=31, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(B, H, seed=32, tokens=512.0)
    args = [t.to(DEV) for t in (q, k, v, s0, z0)]
    y1, s1, _ = la.prefill(*args)
    y2, s2, _ = la.prefill(*args, want_state=False)
    torch.cuda.synchronize()
    assert s1 is not None and s2 is None
    assert torch.equal(y1, y2)
