"""Pins for the fp64 oracle: checks against what the mathematics fixes.

Each pin takes an ``OracleLib`` and raises ``AssertionError`` if it disagrees
with a closed form, an invariant, a special case that reduces to a library
routine (``scipy.special``), or the independent NumPy twin (``oracle.brute``).
The same pins are run on copies of the oracle with planted mistakes
(``test_oracle_mutants.py``) to show that a plausible slip -- a dropped term, a
wrong sign, index or stride, a swapped operand -- fails at least one of them.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import expit, logsumexp

from oracle import brute, chunk_bounds

TOL = 1e-12


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    both_nan = np.isnan(a) & np.isnan(b)
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    ok = both_nan | same_inf
    err = np.nan_to_num(np.where(ok, 0.0, np.abs(a - b)), nan=np.inf)
    ref = np.abs(np.where(ok | np.isnan(b), 0.0, b))
    scale = max(1.0, float(ref.max())) if b.size else 1.0
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol * scale, \
        f"{what}: max err {worst:.3e} > {tol:.1e} * {scale:.3g}"


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def pin_brute_twin(impl):
    """C oracle == NumPy twin on small inputs (S <= 64, D in {1, 8, 64, 72}),
    with distinct heads so a wrong head stride shows."""
    rng = np.random.default_rng(11)
    for S in (1, 5, 33, 64):
        for D in (1, 8, 64, 72):
            q, k, v = (_rand(rng, 2, 3, S, D, std=1.5) for _ in range(3))
            o, l = impl.attention(q, k, v)
            ob, lb = brute.attention(q, k, v)
            _close(o, ob, what=f"O S={S} D={D}")
            _close(l, lb, what=f"LSE S={S} D={D}")
            if S > 3:
                o, l = impl.attention(q, k, v, 1, S - 2)
                ob, lb = brute.attention(q, k, v, 1, S - 2)
                _close(o, ob, what=f"O range S={S} D={D}")
                _close(l, lb, what=f"LSE range S={S} D={D}")


def pin_single_key(impl):
    """S = 1: the softmax has one term, so O = v_0 and LSE = q.k / sqrt(D)."""
    rng = np.random.default_rng(12)
    for D in (1, 8, 72):
        q, k, v = (_rand(rng, 4, 1, D) for _ in range(3))
        o, l = impl.attention(q, k, v)
        _close(o, v, what="O")
        _close(l, np.einsum("bid,bid->bi", q, k) / math.sqrt(D), what="LSE")


def pin_zero_query(impl):
    """Q = 0: every score is 0, so LSE = ln S and O is the mean of the values."""
    rng = np.random.default_rng(13)
    S, D = 37, 16
    k, v = _rand(rng, 2, S, D), _rand(rng, 2, S, D)
    q = np.zeros_like(k)
    o, l = impl.attention(q, k, v)
    _close(l, np.full((2, S), math.log(S)), what="LSE")
    _close(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape), what="O")


def pin_constant_v(impl):
    """All value rows equal u: the weights sum to one, so O = u for any Q, K."""
    rng = np.random.default_rng(14)
    S, D = 50, 24
    q, k = _rand(rng, 3, S, D, std=3.0), _rand(rng, 3, S, D, std=3.0)
    u = _rand(rng, 3, 1, D)
    v = np.repeat(u, S, axis=1)
    o, _ = impl.attention(q, k, v)
    _close(o, np.broadcast_to(u, o.shape), what="O")


def pin_shift_invariance(impl):
    """k_j -> k_j + u for every j adds q_i.u / sqrt(D) to every score of row i:
    O is unchanged and LSE_i grows by exactly that amount."""
    rng = np.random.default_rng(15)
    S, D = 29, 12
    q, k, v = (_rand(rng, 2, S, D) for _ in range(3))
    u = _rand(rng, 2, 1, D)
    o1, l1 = impl.attention(q, k, v)
    o2, l2 = impl.attention(q, k + u, v)
    _close(o2, o1, tol=1e-11, what="O")
    _close(l2, l1 + np.einsum("bid,bjd->bi", q, u) / math.sqrt(D), tol=1e-11, what="LSE")


def pin_permutation(impl):
    """Permuting the key/value rows jointly leaves O and LSE unchanged."""
    rng = np.random.default_rng(16)
    S, D = 41, 8
    q, k, v = (_rand(rng, 2, S, D) for _ in range(3))
    perm = rng.permutation(S)
    o1, l1 = impl.attention(q, k, v)
    o2, l2 = impl.attention(q, k[:, perm], v[:, perm])
    _close(o2, o1, what="O")
    _close(l2, l1, what="LSE")


def pin_two_key_logistic(impl):
    """Two keys: softmax reduces to the logistic function.  With s_a, s_b the
    scaled scores, O = expit(s_a - s_b) v_a + expit(s_b - s_a) v_b and
    LSE = logaddexp(s_a, s_b).  D = 4 so the 1/sqrt(D) scale is distinct from
    1/D and 1; the two query rows differ so a swapped Q/K shows."""
    D = 4
    q = np.array([[[1.0, 1.0, 1.0, 1.0], [0.5, -2.0, 0.0, 1.0]]])
    k = np.array([[[1.0, 1.0, 1.0, 1.0], [0.0, 0.0, 0.0, 0.0]]])
    v = np.array([[[1.0, -1.0, 2.0, 0.0], [3.0, 5.0, -7.0, 1.0]]])
    s = np.einsum("bid,bjd->bij", q, k) / 2.0  # sqrt(4) = 2
    o, l = impl.attention(q, k, v)
    for i in range(2):
        sa, sb = s[0, i, 0], s[0, i, 1]
        want = expit(sa - sb) * v[0, 0] + expit(sb - sa) * v[0, 1]
        _close(o[0, i], want, what=f"O row {i}")
        _close(l[0, i], np.logaddexp(sa, sb), what=f"LSE row {i}")


def pin_chunked_equals_unchunked(impl):
    """Chunking the keys and merging by LSE reproduces unchunked attention, for
    every chunk count 1..16, for random contiguous partitions, and for any order
    of the chunks in the merge."""
    rng = np.random.default_rng(17)
    S, D = 48, 16
    q, k, v = (_rand(rng, 2, S, D, std=2.0) for _ in range(3))
    o_ref, l_ref = impl.attention(q, k, v)
    for n in range(1, 17):
        o, l = impl.attention_chunked(q, k, v, chunk_bounds(S, n))
        _close(o, o_ref, what=f"O n={n}")
        _close(l, l_ref, what=f"LSE n={n}")
    for _ in range(20):
        n = int(rng.integers(2, 17))
        cuts = np.sort(rng.choice(np.arange(1, S), size=n - 1, replace=False))
        edges = [0, *cuts.tolist(), S]
        bounds = list(zip(edges[:-1], edges[1:]))
        order = rng.permutation(len(bounds))
        o, l = impl.attention_chunked(q, k, v, [bounds[i] for i in order])
        _close(o, o_ref, what="O random partition")
        _close(l, l_ref, what="LSE random partition")


def pin_merge_identities(impl):
    """n = 1 is the identity; merging (O, L) with itself gives (O, L + ln 2)."""
    rng = np.random.default_rng(18)
    rows, D = 33, 10
    o = _rand(rng, rows, D)
    l = _rand(rng, rows, std=5.0)
    m1, l1 = impl.lse_merge(o[None], l[None])
    _close(m1, o, what="O n=1")
    _close(l1, l, what="LSE n=1")
    m2, l2 = impl.lse_merge(np.stack([o, o]), np.stack([l, l]))
    _close(m2, o, what="O self-merge")
    _close(l2, l + math.log(2.0), what="LSE self-merge")


def pin_merge_brute(impl):
    """Merge == NumPy twin (scipy logsumexp normaliser) on random partials, and
    a weighted average: the weights exp(LSE_c - LSE) sum to one."""
    rng = np.random.default_rng(19)
    for n in (1, 2, 5, 16):
        p = _rand(rng, n, 40, 7)
        ls = _rand(rng, n, 40, std=4.0)
        o, l = impl.lse_merge(p, ls)
        ob, lb = brute.lse_merge(p, ls)
        _close(o, ob, what=f"O n={n}")
        _close(l, lb, what=f"LSE n={n}")
        _close(l, logsumexp(ls, axis=0), what=f"LSE logsumexp n={n}")


def pin_merge_neg_inf(impl):
    """A partial with LSE = -inf has weight zero and its O_c is never read (a NaN
    there must not leak); a row whose partials are all -inf gives O = 0 and
    LSE = -inf."""
    rng = np.random.default_rng(20)
    rows, D = 6, 4
    p = _rand(rng, 3, rows, D)
    ls = _rand(rng, 3, rows)
    ls[1, :] = -np.inf
    p[1, :, :] = np.nan
    o, l = impl.lse_merge(p, ls)
    o2, l2 = impl.lse_merge(p[[0, 2]], ls[[0, 2]])
    _close(o, o2, what="O with -inf chunk")
    _close(l, l2, what="LSE with -inf chunk")
    ls_all = np.full((2, rows), -np.inf)
    o3, l3 = impl.lse_merge(np.full((2, rows, D), np.nan), ls_all)
    assert np.all(o3 == 0.0), "all -inf rows must give O = 0"
    assert np.all(np.isneginf(l3)), "all -inf rows must give LSE = -inf"


def pin_cfg(impl):
    """w = 1 gives eps_c, w = 0 gives eps_u, the result is affine in w, and it
    matches the twin's (1 - w) eps_u + w eps_c."""
    rng = np.random.default_rng(21)
    ec, eu = _rand(rng, 4, 8, 8), _rand(rng, 4, 8, 8)
    _close(impl.cfg_combine(ec, eu, 1.0), ec, what="w=1")
    _close(impl.cfg_combine(ec, eu, 0.0), eu, what="w=0")
    a, b = impl.cfg_combine(ec, eu, 2.0), impl.cfg_combine(ec, eu, 5.0)
    _close(impl.cfg_combine(ec, eu, 4.5), a + (b - a) * (4.5 - 2.0) / 3.0, what="affine in w")
    _close(impl.cfg_combine(ec, eu, 4.5), brute.cfg_combine(ec, eu, 4.5), what="twin")


def pin_cfg_relmae(impl):
    """rel-MAE sums: exact values on integer inputs (every partial sum is an
    exact integer in fp64); eps_c = eps_u gives 0, eps_c = 2 eps_u gives a
    ratio of exactly 1, eps_c = -eps_u exactly 2; the ratio is scale
    invariant; the fused combine equals the plain one; the sums match the
    NumPy twin.  The ratio: 8 / 10 on the integer case; 0 / 0 gives 0 and
    x / 0 gives +inf (all-zero unconditional noise)."""
    u = np.array([1.0, -2.0, 3.0, -4.0])
    c = np.array([2.0, 0.0, 3.0, 1.0])          # |c - u| = 1, 2, 0, 5
    _, (d, b) = impl.cfg_relmae(c, u, 4.5)
    assert (d, b) == (8.0, 10.0), (d, b)
    assert impl.cfg_relmae_ratio(c, u) == 0.8
    z = np.zeros(5)
    assert impl.cfg_relmae_ratio(z, z) == 0.0
    assert impl.cfg_relmae_ratio(np.array([0.0, 0.0, -0.5, 0.0, 0.0]), z) == math.inf
    rng = np.random.default_rng(24)
    u = _rand(rng, 3, 16, 16)
    _, (d, b) = impl.cfg_relmae(u, u, 2.0)
    assert d == 0.0 and b > 0.0
    _, (d, b) = impl.cfg_relmae(2.0 * u, u, 2.0)
    assert d == b, (d, b)
    _, (d, b) = impl.cfg_relmae(-u, u, 2.0)
    assert d == 2.0 * b, (d, b)
    assert impl.cfg_relmae_ratio(u, u) == 0.0
    assert impl.cfg_relmae_ratio(2.0 * u, u) == 1.0
    assert impl.cfg_relmae_ratio(-u, u) == 2.0
    c = _rand(rng, 3, 16, 16)
    out, (d, b) = impl.cfg_relmae(c, u, 4.5)
    _, (d3, b3) = impl.cfg_relmae(3.0 * c, 3.0 * u, 4.5)
    _close(d3 / b3, d / b, what="scale invariance")
    _close(out, impl.cfg_combine(c, u, 4.5), what="fused combine")
    db, bb = brute.relmae_sums(c, u)
    _close([d, b], [db, bb], what="twin")


def pin_one_hot(impl):
    """One key whose score exceeds every other by more than 55 takes all the
    weight: O equals its value row to within exp(-55) relative."""
    rng = np.random.default_rng(22)
    S, D, star = 20, 16, 7
    q0 = _rand(rng, D)
    q = np.repeat(q0[None, None, :], S, axis=1)      # every query row is q0
    k = _rand(rng, 1, S, D) * 0.01                     # |score| < 1 for these
    k[0, star] = q0 * (60.0 * math.sqrt(D) / float(q0 @ q0))  # score exactly 60
    v = _rand(rng, 1, S, D)
    o, l = impl.attention(q, k, v)
    _close(o[0], np.repeat(v[0, star][None], S, axis=0), what="O")
    _close(l[0], np.full(S, 60.0), tol=1e-20 + math.exp(-55.0), what="LSE")


def pin_rows_match_full(impl):
    """The sampled-row entry point agrees with the full computation."""
    rng = np.random.default_rng(23)
    q, k, v = (_rand(rng, 2, 3, 30, 8) for _ in range(3))
    o, l = impl.attention(q, k, v, 4, 27)
    rows = np.array([0, 5, 29, 30, 77, 179])
    orow, lrow = impl.attention_rows(q, k, v, rows, 4, 27)
    _close(orow, o.reshape(-1, 8)[rows], what="O rows")
    _close(lrow, l.reshape(-1)[rows], what="LSE rows")


PINS = [
    pin_brute_twin, pin_single_key, pin_zero_query, pin_constant_v,
    pin_shift_invariance, pin_permutation, pin_two_key_logistic,
    pin_chunked_equals_unchunked, pin_merge_identities, pin_merge_brute,
    pin_merge_neg_inf, pin_cfg, pin_cfg_relmae, pin_one_hot, pin_rows_match_full,
]
