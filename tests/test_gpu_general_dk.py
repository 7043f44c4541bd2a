"""GPU parity of the general feature-dimension path (d' in {8, 24, 32}, D =
1 + d' + d'^2) of la_prefill and la_decode_step against the fp64 oracle, which
implements the same map for any d' (BASED notes, sec. 2.3)."""
import pytest
import torch

import oracle
import recurrent_lm_gb300 as la
from recurrent_lm_gb300 import inputs
from helpers import TOL, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def check(got, ref, tol, what=""):
    for name, a, r in zip("ysz", got, ref):
        assert_close(name + what, a, r, tol)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk", [8, 24, 32])
@pytest.mark.parametrize("N", [1, 37, 300])
def test_general_dk_prefill(dtype, dk, N):
    D = oracle.feature_dim(dk)
    q, k, v, _, _ = inputs.qkv(2, 3, N, seed=1200 + dk + N, dtype=dtype, dk=dk)
    s0, z0 = inputs.random_state(2, 3, seed=1201 + dk, D=D)
    got = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.prefill(q, k, v, s0, z0)
    check(got, ref, TOL[dtype], f" dk={dk} N={N}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk", [8, 24, 32])
def test_general_dk_decode_in_place_equals_prefill(dtype, dk):
    """n decode steps in place (the state buffers are also the outputs) equal
    the oracle's prefill of those n tokens from the same initial state."""
    D, n = oracle.feature_dim(dk), 9
    q, k, v, _, _ = inputs.qkv(2, 2, n, seed=1300 + dk, dtype=dtype, dk=dk)
    s0, z0 = inputs.random_state(2, 2, seed=1301 + dk, D=D)
    s, z = s0.to(DEV), z0.to(DEV)
    ys = []
    for i in range(n):
        y, _, _ = la.decode_step(q[:, :, i].contiguous().to(DEV), k[:, :, i].contiguous().to(DEV),
                                 v[:, :, i].contiguous().to(DEV), s, z, inplace=True)
        ys.append(y)
    torch.cuda.synchronize()
    yr, sr, zr = oracle.prefill(q, k, v, s0, z0)
    check((torch.stack(ys, dim=2), s, z), (yr, sr, zr), TOL[dtype], f" dk={dk}")


def test_general_dk_zero_length_copies_state():
    D = oracle.feature_dim(24)
    s0, z0 = inputs.random_state(1, 2, seed=1400, D=D)
    e = torch.empty((1, 2, 0, 24), device=DEV)
    ev = torch.empty((1, 2, 0, 64), device=DEV)
    _, s, z = la.prefill(e, e, ev, s0.to(DEV), z0.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(s.cpu(), s0) and torch.equal(z.cpu(), z0)


@pytest.mark.parametrize("N", [128, 1000, 4100])
def test_dk8_tensor_core_prefill(N):
    """bf16 at d' = 8 runs the tensor-core kernel on the padded map (q, k read
    16 wide, the upper 8 columns zero): every chunk size class, a non-symmetric
    initial state, against the oracle's d' = 8 map."""
    D = oracle.feature_dim(8)
    q, k, v, _, _ = inputs.qkv(2, 3, N, seed=1500 + N, dtype=torch.bfloat16, dk=8)
    s0, z0 = inputs.random_state(2, 3, seed=1501, D=D)
    got = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV))
    torch.cuda.synchronize()
    la.check_device_status()
    ref = oracle.prefill(q, k, v, s0, z0)
    check(got, ref, TOL[torch.bfloat16], f" N={N}")


def test_dk8_split_heads():
    """d' = 8 with split heads (la_prefill_ws): every split head against the
    oracle."""
    B, H, N = 10, 16, 4096
    r, _ = la.prefill_split_info(B, H, N)
    assert r > 0
    D = oracle.feature_dim(8)
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=1510, dtype=torch.bfloat16, dk=8)
    s0, z0 = inputs.random_state(B, H, seed=1511, D=D)
    y, s, z = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV))
    torch.cuda.synchronize()
    la.check_device_status()
    idx = list(range(B * H - r, B * H)) + [0]
    sel = lambda t: torch.stack([t[i // H, i % H] for i in idx])[None]
    ref = oracle.prefill(sel(q), sel(k), sel(v), sel(s0), sel(z0))
    check((sel(y), sel(s), sel(z)), ref, TOL[torch.bfloat16])


@pytest.mark.parametrize("dk", [24, 32])
@pytest.mark.parametrize("N", [128, 1000, 2100])
def test_dk24_32_tensor_core_prefill(dk, N):
    """bf16 at d' = 24, 32 through la_prefill_ws (the compact symmetric map,
    chunk states and read-out on the tensor cores): one chunk, ragged chunk
    counts, a non-symmetric initial state (its antisymmetric part passes
    through to s_out), against the oracle's full map."""
    D = oracle.feature_dim(dk)
    q, k, v, _, _ = inputs.qkv(2, 3, N, seed=1600 + dk + N, dtype=torch.bfloat16, dk=dk)
    s0, z0 = inputs.random_state(2, 3, seed=1601 + dk, D=D)
    ws = la.prefill_workspace_size(2, 3, N, dk)
    assert ws > 0
    got = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV))
    torch.cuda.synchronize()
    la.check_device_status()
    ref = oracle.prefill(q, k, v, s0, z0)
    check(got, ref, TOL[torch.bfloat16], f" dk={dk} N={N}")


@pytest.mark.parametrize("dk", [24, 32])
def test_dk24_32_tensor_core_agrees_with_cuda_cores(dk):
    """The tensor-core path (la_prefill_ws) and the CUDA-core path (la_prefill)
    on the same bf16 inputs, without an initial state: the same y and state up
    to bf16 rounding."""
    q, k, v, _, _ = inputs.qkv(2, 2, 777, seed=1700 + dk, dtype=torch.bfloat16, dk=dk)
    args = [t.to(DEV) for t in (q, k, v)]
    a = la.prefill(*args)
    b = la.prefill(*args, split=False)
    torch.cuda.synchronize()
    for name, x, r in zip("ysz", a, b):
        assert_close(name, x, r.double().cpu().numpy(), 1e-2)


def test_dk24_small_workspace_runs_the_cuda_core_path():
    """la_prefill_ws with a workspace one byte short of la_prefill_workspace_size
    runs exactly la_prefill (the CUDA-core path): bitwise the same outputs."""
    dk = 24
    q, k, v, _, _ = inputs.qkv(1, 2, 300, seed=1800, dtype=torch.bfloat16, dk=dk)
    s0, z0 = inputs.random_state(1, 2, seed=1801, D=oracle.feature_dim(dk))
    args = [t.to(DEV) for t in (q, k, v, s0, z0)]
    need = la.prefill_workspace_size(1, 2, 300, dk)
    short = torch.empty(need - 1, dtype=torch.uint8, device=DEV)
    a = la.prefill(*args, workspace=short)
    b = la.prefill(*args, split=False)
    torch.cuda.synchronize()
    for x, r in zip(a, b):
        assert torch.equal(x, r)


@pytest.mark.parametrize("dk", [24, 32])
def test_dk24_32_tensor_core_bench_size_sampled_heads(dk):
    """The bench leg's workload (B=4, H=16, N=4096 with s0) through the
    tensor-core form in one call; three sampled heads (first, middle, last) of
    y and the final state against the oracle."""
    B, H, N = 4, 16, 4096
    D = oracle.feature_dim(dk)
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=1900 + dk, dtype=torch.bfloat16, dk=dk)
    s0, z0 = inputs.random_state(B, H, seed=1901 + dk, D=D)
    y, s, z = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV))
    torch.cuda.synchronize()
    la.check_device_status()
    idx = [0, (B * H) // 2 + 3, B * H - 1]
    sel = lambda t: torch.stack([t[i // H, i % H] for i in idx])[None]
    ref = oracle.prefill(sel(q), sel(k), sel(v), sel(s0), sel(z0))
    check((sel(y), sel(s), sel(z)), ref, TOL[torch.bfloat16], f" dk={dk}")


@pytest.mark.parametrize("dk", [24, 32])
def test_dk24_32_tensor_core_without_states(dk):
    """No initial state and no state outputs (NULL s0/z0 and s_out/z_out):
    y against the oracle from a zero state."""
    q, k, v, _, _ = inputs.qkv(2, 2, 640, seed=2000 + dk, dtype=torch.bfloat16, dk=dk)
    y, s, z = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), want_state=False)
    torch.cuda.synchronize()
    la.check_device_status()
    assert s is None and z is None
    yr, _, _ = oracle.prefill(q, k, v)
    assert_close("y", y, yr, TOL[torch.bfloat16])
