"""GPU parity of the split heads of the bf16 prefill.

With a workspace (la_prefill_ws, and the prefix call, whose workspace holds
the hand-over), the heads of the last wave run as two pieces along the
sequence, the second starting from the state the first hands over (the
blockwise state carry of the BASED reading notes, sec. 2.5, across two CTAs).
Every split head, and whole heads on both sides of them, are checked against
the fp64 oracle, which has no notion of pieces.
"""
import numpy as np
import pytest
import torch

import oracle
import recurrent_lm_gb300 as la
from recurrent_lm_gb300 import inputs
from helpers import TOL, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def heads_of(t, idx, H):
    return torch.stack([t[i // H, i % H] for i in idx])[None]


def check_heads(got, ref_fn, idx, H, tol, what=""):
    for name, a, r in zip("ysz", got, ref_fn()):
        assert_close(name + what, heads_of(a, idx, H), r, tol)


def test_split_plan_on_this_device():
    """The long-prefill workload splits its last wave: B*H - SMs heads, at a
    chunk that balances one piece per SM against the others (> 0, < n)."""
    P = sms()
    r, n1 = la.prefill_split_info(16, 16, 32768)
    if 256 % P == 0 or 256 < P:
        assert r == 0
        return
    assert r == 256 - (256 // P) * P
    assert 0 < n1 < 256
    assert la.prefill_split_info(16, 16, 2048) == (0, 0)      # too short to pay
    assert la.prefill_split_info(1, 16, 32768) == (0, 0)      # one wave


@pytest.mark.parametrize("B,H,N", [(16, 16, 8192), (10, 16, 4096), (11, 16, 5000)])
def test_split_prefill_every_split_head(B, H, N):
    """bf16 prefill with s0 through la_prefill_ws: every split head (both
    pieces and the hand-over at the split chunk) and the whole heads next to
    them, against the oracle; ragged N included."""
    r, n1 = la.prefill_split_info(B, H, N)
    assert r > 0, "this case is meant to split"
    BH = B * H
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=4100 + N, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(B, H, seed=4101, tokens=256.0)
    got = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV))
    torch.cuda.synchronize()
    la.check_device_status()
    idx = sorted(set(range(BH - r, BH)) | {0, BH - r - 1})
    ref = lambda: oracle.prefill(heads_of(q, idx, H), heads_of(k, idx, H), heads_of(v, idx, H),
                                 heads_of(s0, idx, H), heads_of(z0, idx, H))
    check_heads(got, ref, idx, H, TOL[torch.bfloat16])


def test_split_and_unsplit_agree():
    """la_prefill_ws and la_prefill on the same inputs: the same y up to the
    rounding of the handed-over state (well inside the bf16 tolerance), and
    bitwise the same on the heads that are not split."""
    B, H, N = 10, 16, 4096
    r, _ = la.prefill_split_info(B, H, N)
    assert r > 0
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=4200, dtype=torch.bfloat16)
    args = [t.to(DEV) for t in (q, k, v)]
    y1, s1, z1 = la.prefill(*args)
    y2, s2, z2 = la.prefill(*args, split=False)
    torch.cuda.synchronize()
    BH = B * H
    whole = [i for i in range(BH - r)]
    assert torch.equal(heads_of(y1, whole, H), heads_of(y2, whole, H))
    assert torch.equal(heads_of(s1, whole, H), heads_of(s2, whole, H))
    split = list(range(BH - r, BH))
    assert_close("y", heads_of(y1, split, H), heads_of(y2, split, H).double().cpu().numpy(), 1e-2)
    assert_close("s", heads_of(s1, split, H), heads_of(s2, split, H).double().cpu().numpy(), 1e-3)


@pytest.mark.parametrize("padded", [False, True])
def test_split_prefix_prefill(padded):
    """The JRT-RNN prefix call splits the same way (its second pieces start
    from a state that already holds s0 and the prefix sum); with left padding
    too (uniform pads in [0, N], so some first pieces are all padding)."""
    B, H, N, M = 16, 16, 8192, 4096
    r, _ = la.prefill_split_info(B, H, N)
    assert r > 0
    q, k, v, ke, ve = inputs.qkv(B, H, N, seed=4300, dtype=torch.bfloat16, M=M)
    s0, z0 = inputs.random_state(B, H, seed=4301, tokens=128.0)
    pad = None
    if padded:
        pad = torch.from_numpy(np.random.default_rng(4302).integers(0, N + 1, size=B).astype(np.int32))
        pad[-1] = 7000  # the last row's first pieces (8 chunks at this size) are all padding
    dev = [t.to(DEV) for t in (q, k, v, ke, ve, s0, z0)]
    got = la.prefix_prefill(*dev, left_pad=None if pad is None else pad.to(DEV))
    torch.cuda.synchronize()
    la.check_device_status()
    BH = B * H
    idx = sorted(set(range(BH - r, BH, 3)) | {BH - 1, BH - r, 0})
    sel = lambda t: heads_of(t, idx, H)
    lp = None if pad is None else np.array([int(pad[i // H]) for i in idx])
    if lp is None:
        ref = lambda: oracle.prefix_prefill(sel(q), sel(k), sel(v), sel(ke), sel(ve), sel(s0), sel(z0))
        check_heads(got, ref, idx, H, TOL[torch.bfloat16])
    else:
        # the oracle takes one pad per batch row: check head by head
        for j, i in enumerate(idx):
            one = lambda t: t[i // H, i % H][None, None]
            ref = oracle.prefix_prefill(one(q), one(k), one(v), one(ke), one(ve), one(s0), one(z0),
                                        left_pad=[lp[j]])
            for name, a, rr in zip("ysz", got, ref):
                assert_close(f"{name} head {i}", a[i // H, i % H][None, None], rr, TOL[torch.bfloat16])


def test_split_decayed_prefill():
    """The decayed prefill splits the same way (la_prefill_decay_ws): every
    split head against the oracle, with per-head rates from 1 down to 0.5 and
    a non-symmetric s0, whose antisymmetric part the pieces hand over decayed
    by their own lengths."""
    B, H, N = 16, 16, 8192
    r, _ = la.prefill_split_info(B, H, N)
    assert r > 0
    q, k, v, _, _ = inputs.qkv(B, H, N, seed=4400, dtype=torch.bfloat16)
    s0, z0 = inputs.random_state(B, H, seed=4401, tokens=128.0)
    g = [1.0 - 2.0 ** -(4 + h) for h in range(H - 2)] + [1.0, 0.5]
    g32 = torch.tensor(g, dtype=torch.float32)
    got = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV), s0.to(DEV), z0.to(DEV), gamma=g32.to(DEV))
    torch.cuda.synchronize()
    la.check_device_status()
    BH = B * H
    idx = sorted(set(range(BH - r, BH, 2)) | {BH - 1, BH - r, 0})
    for i in idx:
        b, h = i // H, i % H
        one = lambda t: t[b, h][None, None]
        ref = oracle.prefill_decay(one(q), one(k), one(v), g32[h:h + 1].double().numpy(), one(s0), one(z0))
        for name, a, rr in zip("ysz", got, ref):
            assert_close(f"{name} head {i}", a[b, h][None, None], rr, TOL[torch.bfloat16])
