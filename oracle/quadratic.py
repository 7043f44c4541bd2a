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
