"""The O(N^2) closed form of causal Taylor linear attention, in numpy fp64.

TEST INFRASTRUCTURE (see the package docstring).  This module never builds a
feature vector: it evaluates the kernel K(q, k) = 1 + q.k/sqrt(d') +
(q.k)^2/(2 d') directly, which is the right-hand side of the identity
phi(qbar)^T phi(kbar) = K(q, k) on the BASED reading-notes page (sec. 2.3),
and the attention-sum form y_i = sum_{j<=i} K(q_i,k_j) v_j / sum_{j<=i} K(q_i,k_j)
of sec. 2.2, Eq. (1).  An initial state enters only through the two numbers it
contributes to each position, phi(qbar_i)^T s0 and phi(qbar_i)^T z0, which the
caller passes in (``init_num`` [B,H,N,dv], ``init_den`` [B,H,N]); the prefix
form of the "Just read twice" page (sec. 2.6, Eq. (3)) adds the non-causal sum
over the M prefix keys to every position.
"""
from __future__ import annotations

import numpy as np


def kernel_closed_form(q, k):
    """K(q, k) = 1 + q.k / sqrt(d') + (q.k)^2 / (2 d') for [..., d'] arrays."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    dk = q.shape[-1]
    t = np.sum(q * k, axis=-1)
    return 1.0 + t / np.sqrt(dk) + t * t / (2.0 * dk)


def _gram_kernel(q, k):
    """K(q_i, k_j) for all pairs: [B,H,Nq,d'] x [B,H,Nk,d'] -> [B,H,Nq,Nk]."""
    dk = q.shape[-1]
    t = np.einsum("bhid,bhjd->bhij", q, k)
    return 1.0 + t / np.sqrt(dk) + t * t / (2.0 * dk)


def prefix_closed_form(q, k, v, ke=None, ve=None, init_num=None, init_den=None,
                       eps=0.0):
    """y_i = [init_num_i + sum_{j<=M} K(q_i,ke_j) ve_j + sum_{j<=i} K(q_i,k_j) v_j]
           / [init_den_i + sum_{j<=M} K(q_i,ke_j)    + sum_{j<=i} K(q_i,k_j) + eps]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    N = q.shape[2]
    A = _gram_kernel(q, k)
    A = A * np.tril(np.ones((N, N)))[None, None]
    num = np.einsum("bhij,bhjc->bhic", A, v)
    den = A.sum(axis=-1)
    if ke is not None and ke.shape[2] > 0:
        ke = np.asarray(ke, dtype=np.float64)
        ve = np.asarray(ve, dtype=np.float64)
        AE = _gram_kernel(q, ke)
        num = num + np.einsum("bhij,bhjc->bhic", AE, ve)
        den = den + AE.sum(axis=-1)
    if init_num is not None:
        num = num + np.asarray(init_num, dtype=np.float64)
    if init_den is not None:
        den = den + np.asarray(init_den, dtype=np.float64)
    return num / (den + eps)[..., None]


def prefill_closed_form(q, k, v, init_num=None, init_den=None, eps=0.0):
    """Causal closed form (BASED page, sec. 2.2, Eq. (1))."""
    return prefix_closed_form(q, k, v, None, None, init_num, init_den, eps)


def prefill_decay_closed_form(q, k, v, gamma, s0=None, z0=None, eps=0.0):
    """Causal form with a fixed per-head decay, written as sums over tokens
    (length-generalization page, sec. 2.5, Eq. (4) with A_t = gamma I): for
    0-based positions i, j
      y_i = [gamma^(i+1) phi(q_i)^T s0 + sum_{j<=i} gamma^(i-j) K(q_i,k_j) v_j]
          / [gamma^(i+1) phi(q_i)^T z0 + sum_{j<=i} gamma^(i-j) K(q_i,k_j) + eps].
    gamma has shape [H]; phi(q)^T s0 uses the explicit feature map _phi_np."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, dk = q.shape
    g = np.asarray(gamma, dtype=np.float64).reshape(1, H, 1, 1)
    idx = np.arange(N)
    diff = (idx[:, None] - idx[None, :]).astype(np.float64)
    mask = (diff >= 0).astype(np.float64)
    decay = np.where(diff[None, None] >= 0, g ** np.maximum(diff, 0)[None, None], 0.0)
    A = _gram_kernel(q, k) * decay * mask[None, None]
    num = np.einsum("bhij,bhjc->bhic", A, v)
    den = A.sum(axis=-1)
    if s0 is not None:
        lam = g[..., 0] ** (idx + 1.0)[None, None]          # [1,H,N]
        phq = _phi_np(q)                                   # [B,H,N,D]
        num = num + lam[..., None] * np.einsum("bhid,bhdc->bhic", phq, np.asarray(s0, np.float64))
        den = den + lam * np.einsum("bhid,bhd->bhi", phq, np.asarray(z0, np.float64))
    return num / (den + eps)[..., None]


def _phi_np(x):
    """phi(x) = [1, xbar, vec(xbar xbar^T)/sqrt(2)], xbar = x / d'^(1/4), over
    the last axis (BASED page, sec. 2.3), written out with numpy."""
    x = np.asarray(x, dtype=np.float64)
    dk = x.shape[-1]
    xb = x / dk ** 0.25
    quad = (xb[..., :, None] * xb[..., None, :]).reshape(*x.shape[:-1], dk * dk) / np.sqrt(2.0)
    return np.concatenate([np.ones(x.shape[:-1] + (1,)), xb, quad], axis=-1)
