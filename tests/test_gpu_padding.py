"""GPU parity of the left-padded calls (la_prefill_padded,
la_prefix_prefill_padded) against the fp64 oracle with the same padding.

Reading ("Just read twice" notes, sec. 2.7 and 4.7): row b's first p_b
positions are padding, kept out of the prefix sum (j < min(p_b, M)) and of
the causal sums (i < p_b); y is zero there."""
import pytest
import torch

import oracle
import recurrent_lm_gb300 as la
from recurrent_lm_gb300 import inputs
from helpers import TOL, assert_close, sample_heads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def pads_dev(pads):
    return torch.tensor(pads, dtype=torch.int32, device=DEV)


def check(got, ref, tol, what=""):
    for name, a, r in zip("ysz", got, ref):
        assert_close(name + what, a, r, tol)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_padded_prefill(dtype):
    """Pads of 0, 1, inside the first chunk, across a chunk boundary and the
    whole row, ragged N, non-zero initial state."""
    N, pads = 700, [0, 1, 100, 129, 300, 700]
    B = len(pads)
    q, k, v, _, _ = inputs.qkv(B, 3, N, seed=900, dtype=dtype)
    s0, z0 = inputs.random_state(B, 3, seed=901)
    got = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV), left_pad=pads_dev(pads))
    la.check_device_status()
    ref = oracle.prefill(q, k, v, s0, z0, left_pad=pads)
    check(got, ref, TOL[dtype])
    y = got[0].cpu()
    for b, p in enumerate(pads):
        assert torch.count_nonzero(y[b, :, :p]) == 0, b


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_padded_prefix_prefill(dtype):
    """JRT-RNN prefix with pads below M, equal to M, above M, and zero, across
    the 2048-token prefix segments."""
    N, M, pads = 2600, 2300, [0, 300, 2100, 2300, 2500]
    B = len(pads)
    q, k, v, ke, ve = inputs.qkv(B, 2, N, seed=910, dtype=dtype, M=M)
    s0, z0 = inputs.random_state(B, 2, seed=911)
    args = [t.to(DEV) for t in (q, k, v, ke, ve, s0, z0)]
    got = la.prefix_prefill(*args, left_pad=pads_dev(pads))
    la.check_device_status()
    ref = oracle.prefix_prefill(q, k, v, ke, ve, s0, z0, left_pad=pads)
    check(got, ref, TOL[dtype])


def test_zero_pads_are_bitwise_the_unpadded_call():
    q, k, v, ke, ve = inputs.qkv(2, 4, 1000, seed=920, M=700)
    s0, z0 = inputs.random_state(2, 4, seed=921)
    args = [t.to(DEV) for t in (q, k, v, ke, ve, s0, z0)]
    a = la.prefix_prefill(*args, left_pad=pads_dev([0, 0]))
    b = la.prefix_prefill(*args)
    c = la.prefill(args[0], args[1], args[2], args[5], args[6], left_pad=pads_dev([0, 0]))
    d = la.prefill(args[0], args[1], args[2], args[5], args[6])
    torch.cuda.synchronize()
    for x, y in list(zip(a, b)) + list(zip(c, d)):
        assert torch.equal(x, y)


def test_out_of_range_pads_are_clamped_and_reported():
    """Counts outside [0, N] are an argument error found on the device: the
    kernels clamp them (no access outside the buffers) and the next status
    check reports LA_ERR_INVALID_ARG."""
    N = 300
    q, k, v, _, _ = inputs.qkv(2, 2, N, seed=930)
    dev = [t.to(DEV) for t in (q, k, v)]
    got = la.prefill(*dev, left_pad=pads_dev([-5, N + 40]))
    with pytest.raises(la.LAError) as e:
        la.check_device_status()
    assert e.value.status == la.binding.LA_ERR_INVALID_ARG
    la.check_device_status()  # cleared
    want = la.prefill(*dev, left_pad=pads_dev([0, N]))
    torch.cuda.synchronize()
    for x, y in zip(got, want):
        assert torch.equal(x, y)


def test_padded_prefix_full_size_sampled_heads():
    """JRT-RNN prefix workload at full size (B=16, H=16, N=32768, M=16384)
    with seeded pads in [0, M]; sampled heads against the oracle."""
    w = inputs.WORKLOADS[4]
    q, k, v, ke, ve = inputs.workload_inputs(4)
    g = torch.Generator().manual_seed(940)
    pads = torch.randint(0, w.M + 1, (w.B,), generator=g, dtype=torch.int32)
    pads[0] = w.M  # a row whose whole prefix is padding
    y, s, z = la.prefix_prefill(q.to(DEV), k.to(DEV), v.to(DEV), ke.to(DEV), ve.to(DEV),
                                left_pad=pads.to(DEV))
    la.check_device_status()
    heads = sample_heads(w.B, w.H, 3, seed=41)

    def pick(t):
        return torch.stack([t[b, h] for b, h in heads])[None]

    for b, h in heads:
        ref = oracle.prefix_prefill(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1],
                                    ke[b:b + 1, h:h + 1], ve[b:b + 1, h:h + 1],
                                    left_pad=[int(pads[b])])
        for name, a, r in zip("ysz", (y[b:b + 1, h:h + 1], s[b:b + 1, h:h + 1], z[b:b + 1, h:h + 1]), ref):
            assert_close(f"{name} (b={b} h={h} pad={int(pads[b])})", a, r, TOL[torch.bfloat16])
