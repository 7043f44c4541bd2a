"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle itself.

Each test names the property it pins and the passage it comes from (page
title and section).  Pages:
  BASED  = "BASED: Simple linear attention language models balance the
           recall-throughput tradeoff" (reading notes)
  JRT    = "Just read twice: closing the recall gap for recurrent language
           models" (reading notes)
  LENGEN = "Understanding and Improving Length Generalization in Recurrent
           Models" (reading notes)
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import quadratic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


def rnd(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def rel(a, r):
    return float(np.max(np.abs(a - r)) / max(np.max(np.abs(r)), 1e-300))


# ---------------------------------------------------------------- feature map
def test_feature_dims():
    """BASED sec. 2.3 table: full expansion 1 + d' + d'^2 = 273 at d' = 16."""
    assert oracle.feature_dim(16) == 273
    assert oracle.phi(np.zeros(16)).shape == (273,)
    assert oracle.phi(np.zeros(8)).shape == (73,)


def test_phi_explicit_entries():
    """BASED sec. 2.3: phi = [1, xbar, vec(xbar xbar^T)/sqrt2], xbar = x/d'^(1/4)."""
    x = rnd(16)
    p = oracle.phi(x)
    xb = x / 2.0
    assert p[0] == 1.0
    assert np.array_equal(p[1:17], xb)
    for a in (0, 3, 15):
        for b in (0, 7, 15):
            assert p[17 + 16 * a + b] == pytest.approx(xb[a] * xb[b] / math.sqrt(2), rel=1e-15)


@pytest.mark.parametrize("dk", [8, 24, 32])
def test_phi_explicit_entries_general_dk(dk):
    """The same map at other d' (the pages' feature-dimension ablations):
    1 + d' + d'^2 entries, xbar = x / d'^(1/4), quadratic entry (a, b) at row
    1 + d' + a d' + b."""
    x = rnd(dk)
    p = oracle.phi(x)
    xb = x / dk ** 0.25
    assert p.shape == (1 + dk + dk * dk,)
    assert p[0] == 1.0
    assert np.allclose(p[1:1 + dk], xb, rtol=1e-15, atol=0)
    for a in (0, dk // 2, dk - 1):
        for b in (0, dk // 3, dk - 1):
            assert p[1 + dk + dk * a + b] == pytest.approx(xb[a] * xb[b] / math.sqrt(2), rel=1e-14)


def test_phi_kernel_identity():
    """BASED sec. 2.3: phi(qbar).phi(kbar) = 1 + q.k/sqrt(d') + (q.k)^2/(2d')
    on 10^4 random pairs (d' = 16) and for d' in {1, 2, 8, 24, 32}."""
    for dk, n in ((16, 10000), (1, 500), (2, 500), (8, 500), (24, 300), (32, 300)):
        q = rnd(n, dk)
        k = rnd(n, dk)
        lhs = np.array([oracle.phi(q[i]) @ oracle.phi(k[i]) for i in range(n)])
        rhs = quadratic.kernel_closed_form(q, k)
        assert np.max(np.abs(lhs - rhs) / np.abs(rhs)) < 1e-13


def test_kernel_positive_minimum():
    """BASED sec. 2.3: 1 + t + t^2/2 = ((t+1)^2 + 1)/2 >= 1/2 with equality at
    t = -1, i.e. q.k = -sqrt(d') = -4 at d' = 16."""
    q = np.zeros(16); k = np.zeros(16)
    q[0] = 2.0; k[0] = -2.0                      # q.k = -4
    assert oracle.phi(q) @ oracle.phi(k) == pytest.approx(0.5, abs=1e-15)
    q = rnd(20000, 16, scale=3.0); k = rnd(20000, 16, scale=3.0)
    vals = np.array([oracle.phi(q[i]) @ oracle.phi(k[i]) for i in range(0, 20000, 7)])
    assert vals.min() >= 0.5 - 1e-12


# ---------------------------------------------------------- hand-worked cases
def test_golden_dk1_by_hand():
    """tests/golden/hand_worked_dk1.json: two tokens at d' = 1 worked by hand."""
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_dk1.json")))
    q = np.array(g["q"])[None, None]; k = np.array(g["k"])[None, None]
    v = np.array(g["v"])[None, None]
    y, s, z = oracle.prefill(q, k, v)
    np.testing.assert_allclose(y[0, 0], np.array(g["y"]), rtol=1e-15)
    np.testing.assert_allclose(s[0, 0], np.array(g["s"]), rtol=1e-15)
    np.testing.assert_allclose(z[0, 0], np.array(g["z"]), rtol=1e-15)


def test_golden_dk16_by_hand():
    """tests/golden/hand_worked_dk16.json: three tokens at d' = 16 by hand."""
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_dk16.json")))
    N, dk, dv = 3, g["dk"], g["dv"]
    q = np.zeros((1, 1, N, dk)); k = np.zeros((1, 1, N, dk))
    for i in range(N):
        for a, val in g["q_nonzero"][i]:
            q[0, 0, i, a] = val
        for a, val in g["k_nonzero"][i]:
            k[0, 0, i, a] = val
    v = np.array(g["v"])[None, None]
    y, s, z = oracle.prefill(q, k, v)
    np.testing.assert_allclose(y[0, 0], np.array(g["y"]), rtol=1e-15, atol=1e-15)
    s_ref = np.zeros((273, dv)); z_ref = np.zeros(273)
    for f, row in g["s_nonzero"].items():
        s_ref[int(f)] = row
    for f, val in g["z_nonzero"].items():
        z_ref[int(f)] = val
    np.testing.assert_allclose(s[0, 0], s_ref, rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(z[0, 0], z_ref, rtol=1e-15, atol=1e-15)


def test_tiny_brute_force():
    """BASED sec. 2.2, Eq. (1): for N in {1,2,3} the outputs are the K-weighted
    means written out token by token with scalar loops."""
    dk, dv = 16, 5
    for N in (1, 2, 3):
        q = rnd(1, 1, N, dk); k = rnd(1, 1, N, dk); v = rnd(1, 1, N, dv)
        y, _, _ = oracle.prefill(q, k, v)
        for i in range(N):
            w = []
            for j in range(i + 1):
                t = sum(q[0, 0, i, a] * k[0, 0, j, a] for a in range(dk))
                w.append(1.0 + t / 4.0 + t * t / 32.0)
            for c in range(dv):
                ref = sum(w[j] * v[0, 0, j, c] for j in range(i + 1)) / sum(w)
                assert y[0, 0, i, c] == pytest.approx(ref, rel=1e-12, abs=1e-14)
        # one token: y_1 = v_1 up to a few ulps of fp64 rounding
        assert rel(y[0, 0, 0], v[0, 0, 0]) < 1e-14


# ------------------------------------------------------- recurrence vs forms
def test_recurrent_equals_quadratic_closed_form():
    """BASED sec. 2.2, Eq. (1) = Eqs. (2)-(3): recurrent form equals the O(N^2)
    closed form, at the small fp32 workload's shape (B=1, H=2, N=256)."""
    q = rnd(1, 2, 256, 16); k = rnd(1, 2, 256, 16); v = rnd(1, 2, 256, 64)
    y, _, _ = oracle.prefill(q, k, v)
    y_ref = quadratic.prefill_closed_form(q, k, v)
    assert rel(y, y_ref) < 1e-12


def test_running_mean_when_kernel_is_one():
    """q = 0 or k = 0 makes K = 1 (BASED sec. 2.3), so y_i = mean(v_1..v_i)."""
    N = 40
    v = rnd(1, 1, N, 8)
    mean = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    for q, k in ((np.zeros((1, 1, N, 16)), rnd(1, 1, N, 16)),
                 (rnd(1, 1, N, 16), np.zeros((1, 1, N, 16)))):
        y, _, _ = oracle.prefill(q, k, v)
        assert rel(y, mean) < 1e-13


@pytest.mark.parametrize("C", [1, 16, 64, 100])
def test_chunked_equals_recurrent(C):
    """BASED sec. 2.5: the blockwise form is an exact re-association of the
    recurrence, for block lengths that do and do not divide N, with s0."""
    N = 203
    q = rnd(1, 2, N, 16); k = rnd(1, 2, N, 16); v = rnd(1, 2, N, 64)
    s0 = rnd(1, 2, 273, 64, scale=5.0); z0 = np.abs(rnd(1, 2, 273)) + 1.0
    y, s, z = oracle.prefill(q, k, v, s0, z0)
    yc, sc, zc = oracle.prefill_chunked(q, k, v, C, s0, z0)
    assert rel(yc, y) < 1e-12 and rel(sc, s) < 1e-12 and rel(zc, z) < 1e-12


# ------------------------------------------------------------ state invariants
def test_state_invariants():
    """BASED sec. 2.5 (order-0 term = prefix sum of v) and the definition of z:
    z_N[0] = z0[0] + N, s_N[0,:] = s0[0,:] + sum v, z_N[1+a] = z0[1+a] + sum k_a/2,
    and the quadratic block of s - s0 is symmetric in (a, b)."""
    N = 97
    q = rnd(2, 3, N, 16); k = rnd(2, 3, N, 16); v = rnd(2, 3, N, 64)
    s0 = rnd(2, 3, 273, 64); z0 = np.abs(rnd(2, 3, 273)) + 1.0
    _, s, z = oracle.prefill(q, k, v, s0, z0)
    np.testing.assert_allclose(z[..., 0], z0[..., 0] + N, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s[..., 0, :], s0[..., 0, :] + v.sum(axis=2), atol=1e-11)
    np.testing.assert_allclose(z[..., 1:17], z0[..., 1:17] + k.sum(axis=2) / 2.0, atol=1e-11)
    dq = (s - s0)[..., 17:, :].reshape(2, 3, 16, 16, 64)
    np.testing.assert_allclose(dq, np.swapaxes(dq, 2, 3), atol=1e-11)
    # quadratic block of z: sum_j kbar_a kbar_b / sqrt2
    zq = (z - z0)[..., 17:].reshape(2, 3, 16, 16)
    gram = np.einsum("bhna,bhnc->bhac", k / 2.0, k / 2.0) / math.sqrt(2.0)
    np.testing.assert_allclose(zq, gram, atol=1e-11)


def test_state_passing_split_equals_whole():
    """LENGEN sec. 2.5, Eq. (4) with A_t = I: running N1 tokens, then N2 tokens
    from the resulting state, equals one run over N1 + N2 tokens."""
    N1, N2 = 70, 53
    q = rnd(1, 2, N1 + N2, 16); k = rnd(1, 2, N1 + N2, 16); v = rnd(1, 2, N1 + N2, 64)
    y, s, z = oracle.prefill(q, k, v)
    y1, s1, z1 = oracle.prefill(q[:, :, :N1], k[:, :, :N1], v[:, :, :N1])
    y2, s2, z2 = oracle.prefill(q[:, :, N1:], k[:, :, N1:], v[:, :, N1:], s1, z1)
    assert rel(np.concatenate([y1, y2], axis=2), y) < 1e-12
    assert rel(s2, s) < 1e-12 and rel(z2, z) < 1e-12


def test_initial_state_against_closed_form():
    """LENGEN sec. 2.5, Eq. (4): an initial state adds phi(q_i).s0 to every
    numerator and phi(q_i).z0 to every denominator.  s0/z0 come from a prefix
    sequence, so the reference is the closed form over the concatenation."""
    Np, N = 37, 51
    q = rnd(1, 1, Np + N, 16); k = rnd(1, 1, Np + N, 16); v = rnd(1, 1, Np + N, 8)
    _, s0, z0 = oracle.prefill(q[:, :, :Np], k[:, :, :Np], v[:, :, :Np])
    y, _, _ = oracle.prefill(q[:, :, Np:], k[:, :, Np:], v[:, :, Np:], s0, z0)
    y_ref = quadratic.prefill_closed_form(q, k, v)[:, :, Np:]
    assert rel(y, y_ref) < 1e-12


def test_decode_steps_equal_prefill():
    """BASED sec. 2.2: decode is one step of the same recurrence, so n decode
    steps from (s0, z0) reproduce the prefill of those n tokens."""
    n = 9
    q = rnd(2, 2, n, 16); k = rnd(2, 2, n, 16); v = rnd(2, 2, n, 64)
    s0 = rnd(2, 2, 273, 64); z0 = np.abs(rnd(2, 2, 273)) + 3.0
    y, s, z = oracle.prefill(q, k, v, s0, z0)
    ss, zz = s0, z0
    for i in range(n):
        yi, ss, zz = oracle.decode_step(q[:, :, i], k[:, :, i], v[:, :, i], ss, zz)
        assert rel(yi, y[:, :, i]) < 1e-13
    assert rel(ss, s) < 1e-13 and rel(zz, z) < 1e-13


def test_eps_enters_denominator_only():
    """The eps the implementation adds (BASED sec. 2.3) shifts the denominator."""
    q = rnd(1, 1, 5, 16); k = rnd(1, 1, 5, 16); v = rnd(1, 1, 5, 4)
    y0, _, _ = oracle.prefill(q, k, v)
    y1, _, _ = oracle.prefill(q, k, v, eps=0.5)
    y_ref = quadratic.prefill_closed_form(q, k, v, eps=0.5)
    assert rel(y1, y_ref) < 1e-13 and not np.allclose(y0, y1)


# ------------------------------------------------------------------- prefix
def test_prefix_zero_length_is_causal():
    """JRT sec. 2.6: with an empty prefix (M = 0) PLA is plain causal LA."""
    q = rnd(1, 2, 33, 16); k = rnd(1, 2, 33, 16); v = rnd(1, 2, 33, 64)
    ke = np.zeros((1, 2, 0, 16)); ve = np.zeros((1, 2, 0, 64))
    a = oracle.prefix_prefill(q, k, v, ke, ve)
    b = oracle.prefill(q, k, v)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_prefix_against_closed_form():
    """JRT sec. 2.6, Eq. (3) (denominator typo corrected): y_i =
    phi(q_i)(s_E + s_D,i) / phi(q_i)(z_E + z_D,i), checked against the kernel
    closed form with the non-causal sum over all M prefix keys."""
    M, N = 29, 41
    q = rnd(2, 2, N, 16); k = rnd(2, 2, N, 16); v = rnd(2, 2, N, 16)
    ke = rnd(2, 2, M, 16); ve = rnd(2, 2, M, 16)
    y, _, _ = oracle.prefix_prefill(q, k, v, ke, ve)
    y_ref = quadratic.prefix_closed_form(q, k, v, ke, ve)
    assert rel(y, y_ref) < 1e-12


def test_prefix_self_prefix_full_length():
    """JRT sec. 2.6: with k_e = k, v_e = v and M = N the prefix sum equals the
    causal sum at the last position, so y_N(prefix) = y_N(causal)."""
    N = 45
    q = rnd(1, 2, N, 16); k = rnd(1, 2, N, 16); v = rnd(1, 2, N, 64)
    yp, _, _ = oracle.prefix_prefill(q, k, v, k, v)
    yc, _, _ = oracle.prefill(q, k, v)
    assert rel(yp[:, :, -1], yc[:, :, -1]) < 1e-13


def test_prefix_merge_eq4():
    """JRT sec. 2.6, Eq. (4): the state after the prefix prefill is
    s0 + s_E + s_D,N, where s_E is the final state of running the encoder set
    alone and s_D,N that of the causal set alone."""
    M, N = 23, 31
    q = rnd(1, 2, N, 16); k = rnd(1, 2, N, 16); v = rnd(1, 2, N, 64)
    ke = rnd(1, 2, M, 16); ve = rnd(1, 2, M, 64)
    s0 = rnd(1, 2, 273, 64); z0 = np.abs(rnd(1, 2, 273)) + 1.0
    _, s, z = oracle.prefix_prefill(q, k, v, ke, ve, s0, z0)
    _, sE, zE = oracle.prefill(ke, ke, ve)
    _, sD, zD = oracle.prefill(q, k, v)
    assert rel(s, s0 + sE + sD) < 1e-13 and rel(z, z0 + zE + zD) < 1e-13


def test_cost_ratio_prefix_vs_causal():
    """JRT sec. 2.8 / Table 5: JRT-RNN prefill costs about 1.24x Based.  With
    M = N/2 the prefix only runs the state update (half of the 2*D*(d_v+1)
    readout + update flops per token), so the algorithmic ratio is 1.25."""
    D, dv = 273, 64
    per_token = 2 * D * (dv + 1) * 2       # readout + update
    per_prefix_token = 2 * D * (dv + 1)   # update only
    N, M = 32768, 16384
    ratio = (N * per_token + M * per_prefix_token) / (N * per_token)
    assert ratio == pytest.approx(1.25)
    assert per_token == 70980


# ---------------------------------------------------------------- left padding
def _padded_case(M, N, pads, seed_scale=1.0):
    B = len(pads)
    q = rnd(B, 2, N, 16); k = rnd(B, 2, N, 16); v = rnd(B, 2, N, 8)
    ke = rnd(B, 2, M, 16) if M else None
    ve = rnd(B, 2, M, 8) if M else None
    return q, k, v, ke, ve


def test_left_padding_against_closed_form_on_the_valid_suffix():
    """JRT sec. 2.7 and 4.7: a prompt shorter than M is left-padded and the
    padding is kept out of the prefix linear-attention state (and out of the
    causal state).  So row b with p_b padding positions gives, at every valid
    position, the kernel closed form over its valid tokens alone: prefix keys
    j in [p_b, M) and causal keys j in [p_b, i]; padded outputs are zero."""
    M, N, pads = 13, 21, [0, 5, 13, 17]
    q, k, v, ke, ve = _padded_case(M, N, pads)
    y, _, _ = oracle.prefix_prefill(q, k, v, ke, ve, left_pad=pads)
    for b, p in enumerate(pads):
        pe = min(p, M)
        ref = quadratic.prefix_closed_form(q[b:b + 1, :, p:], k[b:b + 1, :, p:], v[b:b + 1, :, p:],
                                           ke[b:b + 1, :, pe:] if pe < M else None,
                                           ve[b:b + 1, :, pe:] if pe < M else None)
        assert rel(y[b:b + 1, :, p:], ref) < 1e-12, b
        assert np.all(y[b, :, :p] == 0.0)


def test_left_padding_state_is_the_valid_tokens_state():
    """JRT sec. 2.6 Eq. (4) with the padding masked: the final state is
    s0 + (sum over valid prefix tokens) + (sum over valid causal tokens),
    i.e. what plain prefills of the valid tokens alone accumulate."""
    M, N, pads = 9, 15, [3, 0, 15]
    q, k, v, ke, ve = _padded_case(M, N, pads)
    s0 = rnd(3, 2, 273, 8); z0 = np.abs(rnd(3, 2, 273)) + 1.0
    _, s, z = oracle.prefix_prefill(q, k, v, ke, ve, s0, z0, left_pad=pads)
    for b, p in enumerate(pads):
        pe = min(p, M)
        sE = np.zeros((1, 2, 273, 8)); zE = np.zeros((1, 2, 273))
        if pe < M:
            _, sE, zE = oracle.prefill(ke[b:b + 1, :, pe:], ke[b:b + 1, :, pe:], ve[b:b + 1, :, pe:])
        sD = np.zeros_like(sE); zD = np.zeros_like(zE)
        if p < N:
            _, sD, zD = oracle.prefill(q[b:b + 1, :, p:], k[b:b + 1, :, p:], v[b:b + 1, :, p:])
        assert rel(s[b:b + 1], s0[b:b + 1] + sE + sD) < 1e-13
        assert rel(z[b:b + 1], z0[b:b + 1] + zE + zD) < 1e-13
    # a fully padded row keeps its initial state exactly
    assert np.array_equal(s[2], s0[2]) and np.array_equal(z[2], z0[2])


def test_zero_padding_is_no_padding_and_bad_pads_are_rejected():
    """p_b = 0 everywhere is the unpadded call bit for bit; p_b outside
    [0, N] is an error."""
    M, N = 7, 11
    q, k, v, ke, ve = _padded_case(M, N, [0, 0])
    a = oracle.prefix_prefill(q, k, v, ke, ve, left_pad=[0, 0])
    b = oracle.prefix_prefill(q, k, v, ke, ve)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    with pytest.raises(RuntimeError):
        oracle.prefix_prefill(q, k, v, ke, ve, left_pad=[0, N + 1])
    with pytest.raises(RuntimeError):
        oracle.prefill(q, k, v, left_pad=[-1, 0])


# ---------------------------------------------------------------- per-head decay
def test_decay_one_is_no_decay_and_zero_keeps_only_the_current_token():
    """LENGEN sec. 2.1 Eq. (1) with A_t = gamma I.  gamma = 1 is the plain
    recurrence (bit for bit); gamma = 0 keeps only the current token, so
    y_i = K(q_i,k_i) v_i / K(q_i,k_i) = v_i and the final state is
    phi(k_N) v_N^T."""
    N = 23
    q = rnd(1, 2, N, 16); k = rnd(1, 2, N, 16); v = rnd(1, 2, N, 8)
    s0 = rnd(1, 2, 273, 8); z0 = np.abs(rnd(1, 2, 273)) + 1.0
    a = oracle.prefill_decay(q, k, v, [1.0, 1.0], s0, z0)
    b = oracle.prefill(q, k, v, s0, z0)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    y, s, z = oracle.prefill_decay(q, k, v, [0.0, 0.0], s0, z0)
    assert rel(y, v) < 1e-13
    ph = np.stack([oracle.phi(k[0, h, -1]) for h in range(2)])
    assert rel(s[0], ph[:, :, None] * v[0, :, -1][:, None, :]) < 1e-15
    assert rel(z[0], ph) < 1e-15


def test_decay_against_closed_form():
    """LENGEN sec. 2.5 Eq. (4) with A_t = gamma I: token j reaches position i
    with weight gamma^(i-j) and the initial state with gamma^(i+1); checked
    against the decayed kernel closed form, per-head gammas."""
    N = 37
    q = rnd(2, 3, N, 16); k = rnd(2, 3, N, 16); v = rnd(2, 3, N, 8)
    s0 = rnd(2, 3, 273, 8) * 0.1; z0 = np.abs(rnd(2, 3, 273)) + 2.0
    gam = [0.5, 0.9, 0.999]
    y, _, _ = oracle.prefill_decay(q, k, v, gam, s0, z0)
    y_ref = quadratic.prefill_decay_closed_form(q, k, v, gam, s0, z0)
    assert rel(y, y_ref) < 1e-12


def test_decay_running_mean_when_kernel_is_one():
    """q = 0 makes every kernel value 1, so y_i is the exponentially weighted
    mean sum_j gamma^(i-j) v_j / sum_j gamma^(i-j) (a closed form)."""
    N, gam = 40, 0.8
    q = np.zeros((1, 1, N, 16)); k = rnd(1, 1, N, 16); v = rnd(1, 1, N, 4)
    y, _, _ = oracle.prefill_decay(q, k, v, [gam])
    for i in range(N):
        w = gam ** (i - np.arange(i + 1))
        assert rel(y[0, 0, i], (w[:, None] * v[0, 0, :i + 1]).sum(0) / w.sum()) < 1e-13


def test_decay_state_passing_and_decode():
    """The decayed recurrence splits at any point (LENGEN sec. 2.5): run(N1)
    then run(N2) from its state equals run(N1+N2), and n decode steps equal
    the prefill of those n tokens."""
    N1, N2, gam = 11, 9, [0.93, 0.6]
    q = rnd(1, 2, N1 + N2, 16); k = rnd(1, 2, N1 + N2, 16); v = rnd(1, 2, N1 + N2, 8)
    y, s, z = oracle.prefill_decay(q, k, v, gam)
    _, s1, z1 = oracle.prefill_decay(q[:, :, :N1], k[:, :, :N1], v[:, :, :N1], gam)
    y2, s2, z2 = oracle.prefill_decay(q[:, :, N1:], k[:, :, N1:], v[:, :, N1:], gam, s1, z1)
    assert rel(y2, y[:, :, N1:]) < 1e-13 and rel(s2, s) < 1e-13 and rel(z2, z) < 1e-13
    sd, zd = s1, z1
    for i in range(N1, N1 + N2):
        yd, sd, zd = oracle.decode_step(q[:, :, i], k[:, :, i], v[:, :, i], sd, zd, gamma=gam)
        assert rel(yd, y[:, :, i]) < 1e-13
    assert rel(sd, s) < 1e-13 and rel(zd, z) < 1e-13


def test_decay_outside_unit_interval_is_rejected():
    q = rnd(1, 1, 4, 16)
    with pytest.raises(RuntimeError):
        oracle.prefill_decay(q, q, rnd(1, 1, 4, 8), [1.5])
    with pytest.raises(RuntimeError):
        oracle.prefill_decay(q, q, rnd(1, 1, 4, 8), [-0.1])
