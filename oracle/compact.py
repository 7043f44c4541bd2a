"""Symmetric-compact form of the Taylor feature map, in plain fp64 numpy.

TEST INFRASTRUCTURE: like the rest of ``oracle``, only the tests, the smoke
check and the benchmark's CPU-baseline leg may use this module.

BASED reading notes ("Simple linear attention language models balance the
recall-throughput tradeoff"), sec. 2.3: the quadratic block vec(xbar xbar^T)
/ sqrt(2) of phi holds every cross product xbar_a xbar_b (a != b) twice, so
the kernel phi(q).phi(k) = 1 + q.k/sqrt(d') + (q.k)^2/(2 d') is also reached
with 1 + d' + d'(d'+1)/2 features (153 at d' = 16):

    phi_c(x) = [1, xbar_a, xbar_a^2 / sqrt(2) for a = b, xbar_a xbar_b for a < b]

The page's table gives the count and the scalings (squares / sqrt 2, cross
terms once, unscaled); the row order is this library's: constant, linear
a = 0..d'-1, then the upper triangle a <= b row-major.  The passage is cut off
mid-sentence on the page; this reading is the one whose inner product is the
kernel above, which the pins check.

States: s [.., D, dv] (D = 1 + d' + d'^2, the phi layout) folds into the
compact layout s_c [.., Dc, dv] by
    s_c[aa] = s[aa],   s_c[ab] = (s[ab] + s[ba]) / sqrt(2)   (a < b),
so phi_c(q).fold(s) = phi(q).s for every s (the antisymmetric part of s is
invisible to a symmetric phi(q) and is dropped); unfold splits a cross term
evenly.
"""
from __future__ import annotations

import numpy as np


def compact_dim(dk: int) -> int:
    """1 + d' + d'(d'+1)/2 features."""
    return 1 + dk + dk * (dk + 1) // 2


def compact_pairs(dk: int):
    """(a, b), a <= b, of the quadratic compact rows, in row order."""
    return [(a, b) for a in range(dk) for b in range(a, dk)]


def compact_row(dk: int, a: int, b: int) -> int:
    """Row of the quadratic feature (min(a,b), max(a,b)) in the compact layout."""
    a, b = min(a, b), max(a, b)
    return 1 + dk + compact_pairs(dk).index((a, b))


def phi_compact(x) -> np.ndarray:
    """phi_c over the last axis of x (fp64); xbar = x / d'^(1/4)."""
    x = np.asarray(x, dtype=np.float64)
    dk = x.shape[-1]
    xb = x / dk ** 0.25
    quad = []
    for a, b in compact_pairs(dk):
        p = xb[..., a] * xb[..., b]
        quad.append(p / np.sqrt(2.0) if a == b else p)
    return np.concatenate([np.ones(x.shape[:-1] + (1,)), xb, np.stack(quad, axis=-1)], axis=-1)


def _rows(dk: int):
    """(compact row, phi row, mirrored phi row or None) for every compact row."""
    out = [(0, 0, None)] + [(1 + a, 1 + a, None) for a in range(dk)]
    for a, b in compact_pairs(dk):
        r1 = 1 + dk + a * dk + b
        r2 = None if a == b else 1 + dk + b * dk + a
        out.append((compact_row(dk, a, b), r1, r2))
    return out


def fold_state(s, z, dk: int = 16):
    """phi-layout state (s [.., D, dv], z [.., D]) -> compact layout (fp64)."""
    s = np.asarray(s, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    Dc = compact_dim(dk)
    s_c = np.empty(s.shape[:-2] + (Dc, s.shape[-1]))
    z_c = np.empty(z.shape[:-1] + (Dc,))
    for rc, r1, r2 in _rows(dk):
        if r2 is None:
            s_c[..., rc, :] = s[..., r1, :]
            z_c[..., rc] = z[..., r1]
        else:
            s_c[..., rc, :] = (s[..., r1, :] + s[..., r2, :]) / np.sqrt(2.0)
            z_c[..., rc] = (z[..., r1] + z[..., r2]) / np.sqrt(2.0)
    return s_c, z_c


def unfold_state(s_c, z_c, dk: int = 16):
    """Compact layout -> phi layout, cross terms split evenly (fp64)."""
    s_c = np.asarray(s_c, dtype=np.float64)
    z_c = np.asarray(z_c, dtype=np.float64)
    D = 1 + dk + dk * dk
    s = np.empty(s_c.shape[:-2] + (D, s_c.shape[-1]))
    z = np.empty(z_c.shape[:-1] + (D,))
    for rc, r1, r2 in _rows(dk):
        if r2 is None:
            s[..., r1, :] = s_c[..., rc, :]
            z[..., r1] = z_c[..., rc]
        else:
            s[..., r1, :] = s[..., r2, :] = s_c[..., rc, :] / np.sqrt(2.0)
            z[..., r1] = z[..., r2] = z_c[..., rc] / np.sqrt(2.0)
    return s, z


def decode_step_compact(q, k, v, s_c, z_c, eps: float = 0.0):
    """One recurrent step on a compact state (BASED notes, sec. 2.2 Eq. (2) for
    one token, with phi_c): s_c += phi_c(k) v^T, z_c += phi_c(k), then
    y = phi_c(q).s_c / (phi_c(q).z_c + eps).  q, k [B,H,dk], v [B,H,dv];
    returns (y, s_c, z_c) in fp64."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    pk, pq = phi_compact(k), phi_compact(q)
    s = np.asarray(s_c, dtype=np.float64) + pk[..., :, None] * v[..., None, :]
    z = np.asarray(z_c, dtype=np.float64) + pk
    num = np.einsum("bhd,bhdc->bhc", pq, s)
    den = np.einsum("bhd,bhd->bh", pq, z) + eps
    return num / den[..., None], s, z
