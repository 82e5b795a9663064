"""Independent NumPy twin of the C oracle -- TEST INFRASTRUCTURE.

Written separately from ``attn_ref.c`` (vectorised NumPy, the normaliser taken
from ``scipy.special.logsumexp``) so that the two pin each other on small
inputs: a dropped term, a wrong sign, index or a transposed operand in either
one shows up as a disagreement.  fp64 throughout.  Only for small S (it builds
the full score matrix).
"""
from __future__ import annotations

import numpy as np
from scipy.special import logsumexp


def attention(q, k, v, j0: int = 0, j1: int | None = None):
    """Softmax attention over keys [j0, j1): q, k, v are [..., S, D]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S, D = q.shape[-2], q.shape[-1]
    j1 = S if j1 is None else j1
    ks = k[..., j0:j1, :]
    vs = v[..., j0:j1, :]
    scores = np.einsum("...id,...jd->...ij", q, ks) / np.sqrt(D)
    lse = logsumexp(scores, axis=-1)
    probs = np.exp(scores - lse[..., None])
    out = np.einsum("...ij,...jd->...id", probs, vs)
    return out, lse


def lse_merge(partials, lses):
    """Log-sum-exp merge over axis 0; -inf partials carry zero weight."""
    partials = np.asarray(partials, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    lse = logsumexp(lses, axis=0)
    finite = np.isfinite(lse)
    w = np.zeros_like(lses)
    w[:, finite] = np.exp(lses[:, finite] - lse[finite])
    contrib = np.where((w > 0)[..., None], w[..., None] * np.nan_to_num(partials), 0.0)
    return contrib.sum(axis=0), lse


def cfg_combine(eps_c, eps_u, w):
    eps_c = np.asarray(eps_c, dtype=np.float64)
    eps_u = np.asarray(eps_u, dtype=np.float64)
    return (1.0 - w) * eps_u + w * eps_c


def relmae_sums(eps_c, eps_u):
    """(sum |eps_c - eps_u|, sum |eps_u|) with NumPy's pairwise summation."""
    eps_c = np.asarray(eps_c, dtype=np.float64)
    eps_u = np.asarray(eps_u, dtype=np.float64)
    return float(np.abs(eps_c - eps_u).sum()), float(np.abs(eps_u).sum())
