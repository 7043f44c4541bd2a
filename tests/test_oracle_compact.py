"""Pins for the oracle's symmetric-compact feature map and state folding
(oracle.compact), checked against the kernel's closed form, the 273-feature
map of the C oracle, hand-worked values and brute force -- never against
themselves.

Page: "BASED: Simple linear attention language models balance the
recall-throughput tradeoff" (reading notes), sec. 2.3 (the feature-dimension
table with the 153-feature symmetric form) and sec. 2.5 (decode reads and
writes the whole state).
"""
import math

import numpy as np
import pytest

import oracle
from oracle import compact, quadratic

RNG = np.random.default_rng(777)


def rnd(*shape):
    return RNG.standard_normal(shape)


def rel(a, r):
    return float(np.max(np.abs(a - r)) / max(np.max(np.abs(r)), 1e-300))


def test_compact_dims():
    """BASED sec. 2.3 table: 1 + d' + d'(d'+1)/2 = 153 at d' = 16, 1.78x fewer
    rows than the 273 of the full expansion."""
    assert compact.compact_dim(16) == 153
    assert compact.compact_dim(8) == 45
    assert compact.phi_compact(np.zeros(16)).shape == (153,)
    assert round(273 / 153, 2) == 1.78


def test_compact_kernel_identity():
    """phi_c(q).phi_c(k) = 1 + q.k/sqrt(d') + (q.k)^2/(2 d') (the closed form of
    BASED sec. 2.3) on random pairs, d' in {16, 8, 2, 1}."""
    for dk, n in ((16, 4000), (8, 500), (2, 500), (1, 200)):
        q, k = rnd(n, dk), rnd(n, dk)
        got = np.sum(compact.phi_compact(q) * compact.phi_compact(k), axis=-1)
        want = quadratic.kernel_closed_form(q, k)
        assert rel(got, want) < 1e-13, dk


def test_compact_by_hand_dk2():
    """d' = 2, xbar = (1, 2) (x = 2^(1/4) xbar): phi_c = [1, 1, 2, 1/sqrt2, 2, 4/sqrt2]."""
    x = 2 ** 0.25 * np.array([1.0, 2.0])
    want = [1.0, 1.0, 2.0, 1 / math.sqrt(2), 2.0, 4 / math.sqrt(2)]
    assert np.allclose(compact.phi_compact(x), want, rtol=1e-14, atol=0)


def test_compact_row_order():
    """Row layout (constant, linear, upper triangle row-major): (0,0) is row 17,
    (0,1) 18, (0,15) 32, (1,1) 33, (15,15) 152; a one-hot xbar = e_a has its
    square at row compact_row(a, a) with value 1/sqrt2 and nothing else
    quadratic; xbar = e_a + e_b puts exactly 1 at compact_row(a, b)."""
    assert [compact.compact_row(16, a, b) for a, b in ((0, 0), (0, 1), (0, 15), (1, 1), (15, 15))] == \
        [17, 18, 32, 33, 152]
    assert compact.compact_row(16, 7, 3) == compact.compact_row(16, 3, 7)
    for a in (0, 5, 15):
        x = np.zeros(16)
        x[a] = 2.0  # xbar = e_a
        p = compact.phi_compact(x)
        nz = set(np.flatnonzero(p).tolist())
        assert nz == {0, 1 + a, compact.compact_row(16, a, a)}
        assert p[compact.compact_row(16, a, a)] == pytest.approx(1 / math.sqrt(2), rel=1e-15)
    for a, b in ((0, 1), (3, 12), (14, 15)):
        x = np.zeros(16)
        x[a] = x[b] = 2.0
        p = compact.phi_compact(x)
        assert p[compact.compact_row(16, a, b)] == pytest.approx(1.0, rel=1e-15)


def test_fold_of_a_recurrent_state_is_the_compact_recurrence():
    """fold(s) of the C oracle's prefill state equals sum_j phi_c(k_j) v_j^T
    (and z likewise) summed directly, brute force over 40 tokens."""
    q, k, v = rnd(1, 2, 40, 16), rnd(1, 2, 40, 16), rnd(1, 2, 40, 64)
    _, s, z = oracle.prefill(q, k, v)
    s_c, z_c = compact.fold_state(s, z)
    pk = compact.phi_compact(k)                     # [1,2,40,153]
    assert rel(s_c, np.einsum("bhnf,bhnc->bhfc", pk, v)) < 1e-13
    assert rel(z_c, pk.sum(axis=2)) < 1e-13


def test_fold_keeps_every_readout():
    """phi(q).s = phi_c(q).fold(s) for ANY state, symmetric or not (so the
    dropped antisymmetric part never reaches an output)."""
    s, z = rnd(273, 64), rnd(273)
    s_c, z_c = compact.fold_state(s, z)
    for _ in range(20):
        q = rnd(16)
        pf, pc = oracle.phi(q), compact.phi_compact(q)
        assert rel(pc @ s_c, pf @ s) < 1e-12
        assert abs(pc @ z_c - pf @ z) <= 1e-12 * np.abs(pf * z).sum()


def test_fold_unfold_round_trips():
    """fold(unfold(c)) = c; unfold(fold(s)) is s with its quadratic block
    symmetrised; a purely antisymmetric block folds to zero."""
    s_c, z_c = rnd(2, 153, 64), rnd(2, 153)
    s2, z2 = compact.fold_state(*compact.unfold_state(s_c, z_c))
    assert rel(s2, s_c) < 1e-15 and rel(z2, z_c) < 1e-15
    s, z = rnd(273, 64), rnd(273)
    su, zu = compact.unfold_state(*compact.fold_state(s, z))
    Q = s[17:].reshape(16, 16, 64)
    assert rel(su[17:].reshape(16, 16, 64), (Q + Q.transpose(1, 0, 2)) / 2) < 1e-15
    assert np.array_equal(su[:17], s[:17])
    A = Q - Q.transpose(1, 0, 2)
    s_anti = np.concatenate([np.zeros((17, 64)), A.reshape(256, 64)])
    fa, _ = compact.fold_state(s_anti, np.zeros(273))
    assert np.max(np.abs(fa)) < 1e-15 * np.max(np.abs(A))


def test_compact_decode_equals_full_decode():
    """decode_step_compact on fold(s) gives the y and the folded state of the C
    oracle's 273-feature decode step on s."""
    q, k, v = rnd(2, 3, 64, 16), rnd(2, 3, 64, 16), rnd(2, 3, 64, 64)
    _, s, z = oracle.prefill(q, k, v)
    qd, kd, vd = rnd(2, 3, 16), rnd(2, 3, 16), rnd(2, 3, 64)
    y, s1, z1 = oracle.decode_step(qd, kd, vd, s, z)
    yc, sc1, zc1 = compact.decode_step_compact(qd, kd, vd, *compact.fold_state(s, z))
    f_s, f_z = compact.fold_state(s1, z1)
    assert rel(yc, y) < 1e-12
    assert rel(sc1, f_s) < 1e-12 and rel(zc1, f_z) < 1e-12
