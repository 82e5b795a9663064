"""Helpers for the GPU parity tests: oracle references and tolerance checks.

Tolerances:
  attention O (bf16 out)  max-abs <= 2e-2, mean-abs <= 2e-3 against fp64
  attention LSE           max-abs <= 1e-3
  fp32 merge / CFG        max-abs <= 1e-5 * max|ref| (norm-wise relative)

The attention bounds are absolute and are applied as such to every workload
(no ``abs_ref``).  Edge-case inputs drawn with a larger spread give outputs up
to ~20, where bf16 itself cannot hold 2e-2 (half an ulp at 16 is 0.0625).  For
those the caller passes ``abs_ref`` = the oracle's attention over |v| (the
same weights applied to |v_j|), and each element gets the bound that the
kernel's two roundings to bf16 imply: P_ij rounded to bf16 moves O_i by at
most 2^-8 sum_j w_ij |v_j|, and the bf16 output by at most 2^-8 |O_i|, so

    |O_gpu - O_ref| <= 2e-2 + 2^-8 (|O_ref| + abs_ref)      elementwise,

with the mean-abs bound scaled by max(1, mean|O_ref|).  An element whose
output and weighted |v| are small keeps (about) the plain 2e-2 bound however
large the rest of the tensor is.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3
F32_REL = 1e-5


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


BF16_ROUND = 2.0 ** -8   # largest relative error of a round-to-nearest bf16 value


def check_attention(o_gpu, lse_gpu, o_ref, lse_ref, what="", abs_ref=None):
    o = f64(o_gpu).reshape(o_ref.shape)
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    if abs_ref is None:
        assert err.max() <= O_MAX_ABS, f"{what}: O max-abs {err.max():.3e}"
        assert err.mean() <= O_MEAN_ABS, f"{what}: O mean-abs {err.mean():.3e}"
    else:
        a = np.asarray(abs_ref, dtype=np.float64).reshape(o_ref.shape)
        bound = O_MAX_ABS + BF16_ROUND * (np.abs(o_ref) + a)
        worst = int(np.argmax(err - bound))
        assert (err <= bound).all(), \
            f"{what}: O error {err.flat[worst]:.3e} > bound {bound.flat[worst]:.3e} at flat index {worst}"
        mean_scale = max(1.0, float(np.abs(o_ref).mean()))
        assert err.mean() <= O_MEAN_ABS * mean_scale, f"{what}: O mean-abs {err.mean():.3e}"
    if lse_gpu is not None:
        l = f64(lse_gpu).reshape(lse_ref.shape)
        lerr = np.abs(l - lse_ref)
        assert lerr.max() <= LSE_MAX_ABS, f"{what}: LSE max-abs {lerr.max():.3e}"
    return float(err.max()), float(err.mean())


def check_f32(got, ref, what="", rel=F32_REL):
    g = f64(got).reshape(ref.shape) if isinstance(got, torch.Tensor) else got
    scale = max(float(np.abs(ref).max()), 1e-30)
    err = float(np.abs(g - ref).max())
    assert err <= rel * scale, f"{what}: max-abs {err:.3e} > {rel} * {scale:.3e}"
    return err


def sample_rows(BH: int, S: int, count: int, seed: int) -> np.ndarray:
    """Flat rows (bh * S + i) spread over heads and tiles, always including
    the first and last rows of the sequence and rows on both sides of every
    128-row tile edge in head 0."""
    rng = np.random.default_rng(seed)
    fixed = [0, S - 1] + [e + d for e in range(128, S, 128) for d in (-1, 0) if 0 <= e + d < S][:16]
    rows = set(int(r) for r in fixed)
    rows.update(int((BH - 1) * S + r) for r in (0, S - 1))
    while len(rows) < count:
        rows.add(int(rng.integers(0, BH * S)))
    return np.array(sorted(rows), dtype=np.int64)


def oracle_rows(q, k, v, rows):
    """Oracle (O, LSE) for sampled flat rows, converting one head at a time."""
    B, H, S, D = q.shape
    qf, kf, vf = q.reshape(B * H, S, D), k.reshape(B * H, S, D), v.reshape(B * H, S, D)
    out = np.empty((rows.size, D))
    lse = np.empty((rows.size,))
    heads = rows // S
    for bh in np.unique(heads):
        sel = np.nonzero(heads == bh)[0]
        qh, kh, vh = (f64(x[bh])[None] for x in (qf, kf, vf))
        o, l = oracle.attention_rows(qh, kh, vh, rows[sel] - bh * S)
        out[sel] = o
        lse[sel] = l
    return out, lse


def abs_weighted(q, k, v, j0=0, j1=None):
    """The oracle's attention of q over keys [j0, j1) applied to |v|: per output
    element, sum_j w_ij |v_jd|, the scale of the bf16 rounding of P (see the
    module docstring).  q, k, v: float64 arrays [..., S, D]."""
    return oracle.attention(q, k, np.abs(v), j0, j1)[0]
