"""Property-based GPU parity: random small shapes and chunk counts against the
fp64 oracle (hypothesis, derandomised so every run draws the same cases).

Shapes: B*H in 1..4, S in 1..700 (single keys, ragged tails, chunks shorter
than a 128-key tile, chunk boundaries off tile boundaries), D in {64, 72, 128},
1 <= n_kv_chunks <= min(S, 16), inputs N(0, std^2) with std in {0.5, 1, 2}.
Also random LSE merges of 1..16 partials with some empty (-inf) chunks, random
key ranges [j0, j1) of the range entry point, and the Torus-style chunked path
with K/V streamed from pinned host memory."""
import numpy as np
import pytest
import torch
from hypothesis import HealthCheck, given, settings, strategies as st

import oracle
from parity_util import abs_weighted, check_attention, check_f32, f64
from sequence_attention_attn_b300 import dit_attn, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SETTINGS = settings(max_examples=40, deadline=None, derandomize=True, database=None,
                    suppress_health_check=[HealthCheck.too_slow, HealthCheck.data_too_large])


@st.composite
def attn_case(draw):
    B = draw(st.integers(1, 2))
    H = draw(st.integers(1, 2))
    S = draw(st.one_of(st.integers(1, 140), st.integers(120, 700)))
    D = draw(st.sampled_from([64, 72, 128]))
    n = draw(st.integers(1, min(S, 16)))
    std = draw(st.sampled_from([0.5, 1.0, 2.0]))
    seed = draw(st.integers(0, 2**31 - 1))
    return B, H, S, D, n, std, seed


@SETTINGS
@given(attn_case())
def test_attention_random_shapes(case):
    B, H, S, D, n, std, seed = case
    q, k, v = workloads.make_random_qkv(B, H, S, D, seed=seed, std=std)
    qf, kf, vf = f64(q), f64(k), f64(v)
    o_ref, l_ref = oracle.attention(qf, kf, vf)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    out, lse = dit_attn.attention(qd, kd, vd, n_kv_chunks=n)
    torch.cuda.synchronize()
    assert dit_attn.dit_last_device_status() == 0
    check_attention(out, lse, o_ref, l_ref, f"B={B} H={H} S={S} D={D} n={n} std={std}",
                    abs_ref=abs_weighted(qf, kf, vf))


@SETTINGS
@given(attn_case())
def test_partials_random_shapes(case):
    B, H, S, D, n, std, seed = case
    q, k, v = workloads.make_random_qkv(B, H, S, D, seed=seed, std=std)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    parts, lses = dit_attn.attention_partials(qd, kd, vd, n)
    torch.cuda.synchronize()
    assert dit_attn.dit_last_device_status() == 0
    qf, kf, vf = f64(q), f64(k), f64(v)
    for c, (j0, j1) in enumerate(oracle.chunk_bounds(S, n)):
        o_c, l_c = oracle.attention(qf, kf, vf, j0, j1)
        check_attention(parts[c], lses[c], o_c.reshape(-1, D), l_c.reshape(-1), f"S={S} D={D} chunk {c}/{n}",
                        abs_ref=abs_weighted(qf, kf, vf, j0, j1).reshape(-1, D))


@SETTINGS
@given(st.integers(1, 16), st.integers(1, 300), st.sampled_from([1, 3, 4, 64, 72, 128]),
       st.sampled_from([0.0, 0.2]), st.integers(0, 2**31 - 1))
def test_merge_random(n, rows, D, empty, seed):
    p, l = workloads.make_merge(n, rows, D, seed=seed, neg_inf_frac=empty)
    ref_o, ref_l = oracle.lse_merge(p.numpy(), l.numpy())
    pd, ld = p.to(DEV), l.to(DEV)
    out, lse = dit_attn.merge(pd, ld)
    o = f64(out)
    assert np.isfinite(o).all()
    check_f32(o, ref_o, f"merge n={n} rows={rows} D={D}")
    fin = np.isfinite(ref_l)
    assert (np.isneginf(f64(lse)) == ~fin).all()
    if fin.any():
        assert np.abs(f64(lse)[fin] - ref_l[fin]).max() <= 1e-5 * max(1.0, np.abs(ref_l[fin]).max())


@st.composite
def range_case(draw):
    B = draw(st.integers(1, 2))
    H = draw(st.integers(1, 2))
    S = draw(st.one_of(st.integers(1, 140), st.integers(120, 700)))
    D = draw(st.sampled_from([64, 72, 128]))
    j0 = draw(st.integers(0, S - 1))
    j1 = draw(st.integers(j0 + 1, S))
    std = draw(st.sampled_from([0.5, 1.0, 2.0]))
    seed = draw(st.integers(0, 2**31 - 1))
    return B, H, S, D, j0, j1, std, seed


@SETTINGS
@given(range_case())
def test_key_range_random(case):
    B, H, S, D, j0, j1, std, seed = case
    q, k, v = workloads.make_random_qkv(B, H, S, D, seed=seed, std=std)
    qf, kf, vf = f64(q), f64(k), f64(v)
    o_ref, l_ref = oracle.attention(qf, kf, vf, j0, j1)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    out, lse = dit_attn.attention_range(qd, kd, vd, j0, j1)
    torch.cuda.synchronize()
    assert dit_attn.dit_last_device_status() == 0
    check_attention(out, lse, o_ref.reshape(-1, D), l_ref.reshape(-1),
                    f"B={B} H={H} S={S} D={D} [{j0},{j1}) std={std}",
                    abs_ref=abs_weighted(qf, kf, vf, j0, j1).reshape(-1, D))


@settings(max_examples=15, deadline=None, derandomize=True, database=None,
          suppress_health_check=[HealthCheck.too_slow, HealthCheck.data_too_large])
@given(attn_case())
def test_torus_random(case):
    B, H, S, D, n, std, seed = case
    q, k, v = workloads.make_random_qkv(B, H, S, D, seed=seed, std=std)
    qf, kf, vf = f64(q), f64(k), f64(v)
    o_ref, l_ref = oracle.attention(qf, kf, vf)
    out, lse = dit_attn.attention_torus(q.to(DEV), k.pin_memory(), v.pin_memory(), n,
                                        copy_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert dit_attn.dit_last_device_status() == 0
    check_attention(out, lse, o_ref.reshape(-1, D), l_ref.reshape(-1),
                    f"torus B={B} H={H} S={S} D={D} n={n} std={std}",
                    abs_ref=abs_weighted(qf, kf, vf).reshape(-1, D))
