"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs (every workload, every chunk count it lists), plus edge
cases (ragged tails, chunks shorter than a tile, S = 1, every head size)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import (abs_weighted, check_attention, check_f32, f64, oracle_rows, sample_rows)
from sequence_attention_attn_b300 import dit_attn, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def to_dev(*ts):
    return [t.to(DEV) for t in ts]


def assert_no_device_error():
    assert dit_attn.dit_last_device_status() == 0, "a device-side wait ran out"


# ------------------------------------------------------------ CFG combine
@pytest.mark.parametrize("name", ["tiny", "pixart_1024"])
def test_cfg_combine_workloads(name):
    cfg = workloads.BY_NAME[name]
    if name == "pixart_1024":
        # one [2, 4, 128, 128] buffer: index 0 = cond, 1 = uncond
        g = torch.Generator().manual_seed(workloads.seed_for(cfg, 100))
        buf = torch.randn((2,) + cfg.cfg_shape, generator=g)
        eps_c, eps_u = buf[0].contiguous(), buf[1].contiguous()
    else:
        eps_c, eps_u = workloads.make_cfg(cfg.cfg_shape, workloads.seed_for(cfg, 100))
    ref = oracle.cfg_combine(eps_c.numpy(), eps_u.numpy(), cfg.cfg_w)
    c, u = to_dev(eps_c, eps_u)
    out = dit_attn.combine(c, u, cfg.cfg_w)
    check_f32(out, ref, f"cfg {name}")
    assert_no_device_error()


@pytest.mark.parametrize("numel", [1, 3, 4, 5, 1023, 4096 + 3, 1 << 20])
def test_cfg_combine_sizes_and_alias(numel):
    eps_c, eps_u = workloads.make_cfg((numel,), 7 + numel)
    ref = oracle.cfg_combine(eps_c.numpy(), eps_u.numpy(), 4.5)
    c, u = to_dev(eps_c, eps_u)
    check_f32(dit_attn.combine(c, u, 4.5), ref, f"cfg numel={numel}")
    dit_attn.cfg_combine(c, u, 4.5, c)  # in place over eps_c
    check_f32(c, ref, "cfg in place")
    c1, u1 = to_dev(eps_c, eps_u)
    check_f32(dit_attn.combine(c1, u1, 1.0), eps_c.double().numpy(), "w=1")
    check_f32(dit_attn.combine(c1, u1, 0.0), eps_u.double().numpy(), "w=0")


# ----------------------------------------------- CFG combine + rel-MAE
def check_relmae(eps_c, eps_u, w, what):
    ref_out, (ref_d, ref_b) = oracle.cfg_relmae(eps_c.numpy(), eps_u.numpy(), w)
    ref_ratio = oracle.cfg_relmae_ratio(eps_c.numpy(), eps_u.numpy())
    c, u = to_dev(eps_c, eps_u)
    out = torch.empty_like(c)
    sums = torch.full((3,), float("nan"), dtype=torch.float64, device=DEV)
    dit_attn.cfg_combine_relmae(c, u, w, out, sums)
    check_f32(out, ref_out, f"{what} combine")
    # the fused combine is the plain combine, bit for bit
    assert torch.equal(out, dit_attn.combine(c, u, w)), what
    d, b, ratio = sums.tolist()
    assert abs(d - ref_d) <= 1e-5 * ref_d + 1e-30, (what, d, ref_d)
    assert abs(b - ref_b) <= 1e-5 * ref_b, (what, b, ref_b)
    # the ratio is computed on the device
    assert abs(ratio - ref_ratio) <= 1e-5 * ref_ratio + 1e-30, (what, ratio, ref_ratio)
    assert_no_device_error()


@pytest.mark.parametrize("name", ["tiny", "pixart_1024"])
def test_cfg_relmae_workloads(name):
    cfg = workloads.BY_NAME[name]
    eps_c, eps_u = workloads.make_cfg(cfg.cfg_shape, workloads.seed_for(cfg, 100))
    check_relmae(eps_c, eps_u, cfg.cfg_w, f"relmae {name}")


@pytest.mark.parametrize("numel", [1, 3, 4, 5, 1023, 4096 + 3, 1 << 20, (1 << 24) + 7])
def test_cfg_relmae_sizes(numel):
    eps_c, eps_u = workloads.make_cfg((numel,), 11 + numel)
    check_relmae(eps_c, eps_u, 4.5, f"relmae numel={numel}")


def test_cfg_relmae_closed_forms_and_alias():
    _, eps_u = workloads.make_cfg((4096 + 1,), 5)
    for c, want in ((eps_u.clone(), 0.0), (2.0 * eps_u, 1.0), (-eps_u, 2.0)):
        cd, ud = to_dev(c, eps_u)
        out, rel = dit_attn.combine_relmae(cd, ud, 4.5)
        assert abs(rel - want) <= 1e-6, (want, rel)
    # all-zero unconditional noise: identical paths give 0, any difference +inf
    zero = torch.zeros(777, device=DEV)
    assert dit_attn.combine_relmae(zero, zero, 4.5)[1] == 0.0
    bump = zero.clone()
    bump[500] = -0.25
    assert dit_attn.combine_relmae(bump, zero, 4.5)[1] == float("inf")
    # two calls in a row on one buffer: each starts from zero
    c, u = to_dev(*workloads.make_cfg((1 << 16,), 9))
    sums = torch.empty(3, dtype=torch.float64, device=DEV)
    o = torch.empty_like(c)
    dit_attn.cfg_combine_relmae(c, u, 4.5, o, sums)
    first = sums.clone()
    dit_attn.cfg_combine_relmae(c, u, 4.5, o, sums)
    assert torch.allclose(first, sums, rtol=1e-12, atol=0.0)
    c, u = to_dev(*workloads.make_cfg((1000,), 6))
    ref = dit_attn.combine(c, u, 4.5)
    sums = torch.empty(3, dtype=torch.float64, device=DEV)
    dit_attn.cfg_combine_relmae(c, u, 4.5, c, sums)       # in place over eps_c
    assert torch.equal(c, ref)


# ------------------------------------------------------------- LSE merge
@pytest.mark.parametrize("n,rows,D", [(1, 100, 64), (2, 777, 72), (5, 300, 128), (16, 4096, 64),
                                      (3, 50, 7), (16, 333, 1)])
def test_merge_random(n, rows, D):
    p, l = workloads.make_merge(n, rows, D, seed=n * 1000 + rows + D)
    ref_o, ref_l = oracle.lse_merge(p.numpy(), l.numpy())
    pd, ld = to_dev(p, l)
    out, lse = dit_attn.merge(pd, ld)
    check_f32(out, ref_o, f"merge O n={n} D={D}")
    assert np.abs(f64(lse) - ref_l).max() <= 1e-5 * max(1.0, np.abs(ref_l).max())
    assert_no_device_error()


def test_merge_neg_inf_partials():
    n, rows, D = 4, 513, 64
    p, l = workloads.make_merge(n, rows, D, seed=5, neg_inf_frac=0.3)
    l[:, :7] = float("-inf")                 # rows with no weight at all
    p[1][torch.isinf(l[1])] = float("nan")   # never read when its LSE is -inf
    ref_o, ref_l = oracle.lse_merge(p.numpy(), l.numpy())
    pd, ld = to_dev(p, l)
    out, lse = dit_attn.merge(pd, ld)
    o = f64(out)
    assert np.isfinite(o).all()
    assert (o[:7] == 0).all() and np.isneginf(f64(lse)[:7]).all()
    check_f32(o[7:], ref_o[7:], "merge with -inf")
    fin = np.isfinite(ref_l)
    assert np.abs(f64(lse)[fin] - ref_l[fin]).max() <= 1e-5 * max(1.0, np.abs(ref_l[fin]).max())


def test_merge_video_workload_sampled():
    cfg = workloads.BY_NAME["video"]
    rows = cfg.rows
    p, l = workloads.make_merge(cfg.merge_n, rows, cfg.D, seed=workloads.seed_for(cfg, 200),
                                device=DEV)
    out, lse = dit_attn.merge(p, l)
    pick = sample_rows(1, rows, 2048, seed=3)
    ref_o, ref_l = oracle.lse_merge(f64(p[:, pick]), f64(l[:, pick]))
    check_f32(out[pick], ref_o, "video merge O")
    assert np.abs(f64(lse[pick]) - ref_l).max() <= 1e-5 * max(1.0, np.abs(ref_l).max())
    assert_no_device_error()


# -------------------------------------------------------------- attention
def run_attention(q, k, v, n):
    qd, kd, vd = to_dev(q, k, v)
    out, lse = dit_attn.attention(qd, kd, vd, n_kv_chunks=n)
    torch.cuda.synchronize()
    assert_no_device_error()
    return out, lse


@pytest.mark.parametrize("n", [1, 2, 4])
def test_attention_tiny_full(n):
    cfg = workloads.BY_NAME["tiny"]
    q, k, v = workloads.make_qkv(cfg)
    o_ref, l_ref = oracle.attention_chunked(f64(q), f64(k), f64(v), oracle.chunk_bounds(cfg.S, n))
    out, lse = run_attention(q, k, v, n)
    check_attention(out, lse, o_ref, l_ref, f"tiny n={n}")


@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_attention_dit_xl2_full(n):
    cfg = workloads.BY_NAME["dit_xl2_512"]
    q, k, v = workloads.make_qkv(cfg)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v))
    out, lse = run_attention(q, k, v, n)
    check_attention(out, lse, o_ref, l_ref, f"dit_xl2 n={n}")


@pytest.mark.parametrize("name,n", [("pixart_1024", 1), ("pixart_1024", 4), ("pixart_1024", 8),
                                    ("flux_mmdit", 1), ("flux_mmdit", 2), ("flux_mmdit", 4),
                                    ("flux_mmdit", 8), ("video", 1), ("video", 8), ("video", 16)])
def test_attention_full_size_sampled(name, n):
    cfg = workloads.BY_NAME[name]
    q, k, v = workloads.make_qkv(cfg)
    out, lse = run_attention(q, k, v, n)
    rows = sample_rows(cfg.B * cfg.H, cfg.S, 384, seed=cfg.index * 10 + n)
    o_ref, l_ref = oracle_rows(q, k, v, rows)
    D = cfg.D
    check_attention(out.reshape(-1, D)[torch.as_tensor(rows, device=DEV)],
                    lse.reshape(-1)[torch.as_tensor(rows, device=DEV)], o_ref, l_ref, f"{name} n={n}")


def test_attention_offsets_past_32_bits_sampled():
    # B*H*S*D = 2.18e9 elements (4.4 GB per tensor): element offsets of the
    # last heads pass 2^31 and byte offsets pass 2^32.
    B, H, S, D = 1, 520, 65536, 64
    q, k, v = workloads.make_random_qkv(B, H, S, D, seed=77, device=DEV)
    out, lse = dit_attn.attention(q, k, v, n_kv_chunks=4)
    torch.cuda.synchronize()
    assert_no_device_error()
    rng = np.random.default_rng(3)
    rows = []
    for bh in (0, 260, H - 2, H - 1):
        rows += [bh * S + r for r in (0, 1, 127, 128, S // 4, S // 4 + 1, S - 129, S - 1)]
        rows += [bh * S + int(r) for r in rng.integers(0, S, 4)]
    rows = np.array(sorted(set(rows)), dtype=np.int64)
    o_ref, l_ref = oracle_rows(q, k, v, rows)
    idx = torch.as_tensor(rows, device=DEV)
    check_attention(out.reshape(-1, D)[idx], lse.reshape(-1)[idx], o_ref, l_ref, "offsets past 32 bits")
    del q, k, v, out, lse
    torch.cuda.empty_cache()


EDGE_S = [1, 2, 100, 127, 128, 129, 255, 257, 383, 640]


def edge_chunk_counts(S):
    return sorted({1, min(S, 3), min(S, 7), S if S <= 16 else 16})


@pytest.mark.parametrize("S", EDGE_S)
@pytest.mark.parametrize("D", [64, 72, 128])
def test_attention_edge_lengths(S, D):
    q, k, v = workloads.make_random_qkv(1, 3, S, D, seed=S * 7 + D, std=1.5)
    qf, kf, vf = f64(q), f64(k), f64(v)
    o_ref, l_ref = oracle.attention(qf, kf, vf)
    a_ref = abs_weighted(qf, kf, vf)
    for n in edge_chunk_counts(S):
        out, lse = run_attention(q, k, v, n)
        check_attention(out, lse, o_ref, l_ref, f"S={S} D={D} n={n}", abs_ref=a_ref)


@pytest.mark.parametrize("S", EDGE_S)
@pytest.mark.parametrize("D", [64, 72, 128])
def test_attention_edge_lengths_unit_std(S, D):
    # the same shapes with N(0, 1) inputs, held to the plain absolute bounds
    q, k, v = workloads.make_random_qkv(1, 3, S, D, seed=S * 11 + D + 1, std=1.0)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v))
    for n in edge_chunk_counts(S):
        out, lse = run_attention(q, k, v, n)
        check_attention(out, lse, o_ref, l_ref, f"std 1 S={S} D={D} n={n}")


@pytest.mark.parametrize("D", [64, 72, 128])
def test_attention_chunks_shorter_than_a_tile(D):
    # 40 chunks of 6-7 keys: every tile is cut at a chunk end; then one key
    # per chunk, merged on chip and as S one-key partials merged afterwards
    S = 260
    q, k, v = workloads.make_random_qkv(2, 2, S, D, seed=99 + D, std=2.0)
    qf, kf, vf = f64(q), f64(k), f64(v)
    o_ref, l_ref = oracle.attention(qf, kf, vf)
    a_ref = abs_weighted(qf, kf, vf)
    out, lse = run_attention(q, k, v, 40)
    check_attention(out, lse, o_ref, l_ref, f"D={D} n=40", abs_ref=a_ref)
    out, lse = run_attention(q, k, v, S)
    check_attention(out, lse, o_ref, l_ref, f"D={D} n=S", abs_ref=a_ref)
    parts, lses = dit_attn.attention_partials(*to_dev(q, k, v), S)
    merged, mlse = dit_attn.merge(parts, lses)
    torch.cuda.synchronize()
    assert_no_device_error()
    check_attention(merged.to(torch.bfloat16), mlse, o_ref, l_ref, f"D={D} n=S partials+merge", abs_ref=a_ref)


# D = 128 with every chunk at least one tile long and chunk ends inside tiles:
# the merged launch takes the grid walk (a straddling tile computed once, its
# row sum split at the chunk end).  Ends inside tiles only (1000/3, 1152/2),
# inside and on tile boundaries (1344/3: 448, 896), almost every tile
# straddling (2000/15: 133-134 keys), a ragged last tile throughout but 1152.
@pytest.mark.parametrize("S,n", [(1000, 3), (1152, 2), (1344, 3), (2000, 15)])
def test_attention_grid_walk_d128(S, n):
    q, k, v = workloads.make_random_qkv(2, 2, S, 128, seed=S + n)
    qf, kf, vf = f64(q), f64(k), f64(v)
    o_ref, l_ref = oracle.attention(qf, kf, vf)
    out, lse = run_attention(q, k, v, n)
    check_attention(out, lse, o_ref, l_ref, f"grid walk S={S} n={n}")
    # the same chunks as partials, merged afterwards
    parts, lses = dit_attn.attention_partials(*to_dev(q, k, v), n)
    merged, mlse = dit_attn.merge(parts, lses)
    torch.cuda.synchronize()
    assert_no_device_error()
    assert (out.float().cpu() - merged.reshape(out.shape).cpu()).abs().max().item() <= 2e-2
    assert (lse.cpu() - mlse.reshape(lse.shape).cpu()).abs().max().item() <= 1e-3


@pytest.mark.parametrize("D", [64, 72, 128])
def test_attention_sharp_softmax(D):
    # large logits: the reference max moves often and by a lot, so O is
    # rescaled in TMEM (at D = 72 including its 16-column tail block)
    q, k, v = workloads.make_random_qkv(1, 4, 512, D, seed=5 + D, std=4.0)
    qf, kf, vf = f64(q), f64(k), f64(v)
    o_ref, l_ref = oracle.attention(qf, kf, vf)
    a_ref = abs_weighted(qf, kf, vf)
    for n in (1, 3):
        out, lse = run_attention(q, k, v, n)
        check_attention(out, lse, o_ref, l_ref, f"sharp D={D} n={n}", abs_ref=a_ref)


@pytest.mark.parametrize("D", [64, 72, 128])
def test_attention_without_lse_output(D):
    q, k, v = workloads.make_random_qkv(1, 2, 300, D, seed=8)
    o_ref, _ = oracle.attention(f64(q), f64(k), f64(v))
    qd, kd, vd = to_dev(q, k, v)
    out, lse = dit_attn.attention(qd, kd, vd, 2, with_lse=False)
    assert lse is None
    check_attention(out, None, o_ref, None, f"no lse D={D}")
    # the LSE output changes nothing else
    out2, _ = dit_attn.attention(qd, kd, vd, 2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


# ------------------------------------------------- partials + standalone merge
@pytest.mark.parametrize("name,n", [("tiny", 2), ("tiny", 4), ("dit_xl2_512", 8)])
def test_partials_then_merge(name, n):
    cfg = workloads.BY_NAME[name]
    q, k, v = workloads.make_qkv(cfg)
    qd, kd, vd = to_dev(q, k, v)
    parts, lses = dit_attn.attention_partials(qd, kd, vd, n)
    torch.cuda.synchronize()
    assert_no_device_error()
    qf, kf, vf = f64(q), f64(k), f64(v)
    for c, (j0, j1) in enumerate(oracle.chunk_bounds(cfg.S, n)):
        o_c, l_c = oracle.attention(qf, kf, vf, j0, j1)
        check_attention(parts[c], lses[c], o_c.reshape(-1, cfg.D), l_c.reshape(-1), f"{name} chunk {c}")
    out, lse = dit_attn.merge(parts, lses)
    o_ref, l_ref = oracle.attention(qf, kf, vf)
    check_attention(out, lse, o_ref.reshape(-1, cfg.D), l_ref.reshape(-1), f"{name} merged")
    # the merge of the GPU partials is exactly the oracle merge of those partials
    m_ref, ml_ref = oracle.lse_merge(f64(parts), f64(lses))
    check_f32(out, m_ref, f"{name} merge of gpu partials")


@pytest.mark.parametrize("D", [64, 72, 128])
def test_repeatable_bitwise(D):
    q, k, v = to_dev(*workloads.make_random_qkv(1, 3, 700, D, seed=21))
    a, la = dit_attn.attention(q, k, v, 3)
    b, lb = dit_attn.attention(q, k, v, 3)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_bounded_wait_times_out_without_fault():
    """A wait that nothing satisfies gives up after ~1 s: the kernel returns,
    the status word reports the timeout once, and the context stays usable."""
    import time
    assert dit_attn.dit_last_device_status() == 0
    t0 = time.perf_counter()
    dit_attn.dit_selftest_bounded_wait()
    assert dit_attn.dit_last_device_status() == -6      # DIT_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 30.0
    assert dit_attn.dit_last_device_status() == 0       # read-and-clear
    cfg = workloads.BY_NAME["tiny"]
    q, k, v = workloads.make_qkv(cfg)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v))
    out, lse = run_attention(q, k, v, 2)                # still works afterwards
    check_attention(out, lse, o_ref, l_ref, "after timeout")


def test_attention_chain_on_its_own_output_d72():
    """At D = 72 the merged output leaves the kernel through TMA stores.  Two
    launches back to back, the second reading the first one's output as its
    queries (programmatic dependent launch: it may start before the first has
    finished and waits for its writes), then a third on the second's."""
    B, H, S, D = 2, 3, 300, 72
    q, k, v = workloads.make_random_qkv(B, H, S, D, seed=4242)
    qd, kd, vd = to_dev(q, k, v)
    o1, o2, o3 = (torch.empty_like(qd) for _ in range(3))
    l1, l2, l3 = (torch.empty((B, H, S), dtype=torch.float32, device=DEV) for _ in range(3))
    torch.cuda.synchronize()
    dit_attn.dit_attn_fwd(qd, kd, vd, o1, l1, 1)
    dit_attn.dit_attn_fwd(o1, kd, vd, o2, l2, 3)
    dit_attn.dit_attn_fwd(o2, kd, vd, o3, l3, 1)
    torch.cuda.synchronize()
    assert_no_device_error()
    kf, vf = f64(k), f64(v)
    for qin, o, l, what in ((q, o1, l1, "first"), (o1, o2, l2, "second"), (o2, o3, l3, "third")):
        o_ref, l_ref = oracle.attention(f64(qin), kf, vf)
        check_attention(o, l, o_ref, l_ref, f"D=72 chain: {what} launch")


def test_dependent_launch_chain_without_sync():
    """Short kernels may start while the previous kernel in the stream is
    finishing (programmatic dependent launch); each still waits for that
    kernel's writes before reading.  A chain where every launch consumes the
    previous one's output, with no host synchronisation in between, must
    match the oracle applied step by step."""
    B, H, S, D = 1, 2, 200, 64
    q, k, v = workloads.make_random_qkv(B, H, S, D, seed=321)
    qd, kd, vd = to_dev(q, k, v)
    n = 3
    parts = torch.empty((n, B * H * S, D), dtype=torch.float32, device=DEV)
    lses = torch.empty((n, B * H * S), dtype=torch.float32, device=DEV)
    merged = torch.empty((B * H * S, D), dtype=torch.float32, device=DEV)
    mlse = torch.empty((B * H * S,), dtype=torch.float32, device=DEV)
    c1 = torch.empty_like(merged)
    c2 = torch.empty_like(merged)
    other = torch.randn(merged.shape, generator=torch.Generator().manual_seed(5)).to(DEV)
    q2 = torch.empty_like(qd)
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    # partials -> merge -> two CFG combines on the merge output, all back to
    # back; then (bf16 cast by torch) an attention whose queries are that result
    dit_attn.dit_attn_fwd_partials(qd, kd, vd, parts, lses, n)
    dit_attn.dit_attn_merge(parts, lses, merged, mlse)
    dit_attn.cfg_combine(merged, other, 2.0, c1)
    dit_attn.cfg_combine(c1, merged, 0.25, c2)
    q2.copy_(c2.view(B, H, S, D))
    dit_attn.dit_attn_fwd(q2, kd, vd, out, lse, 2)
    torch.cuda.synchronize()
    assert_no_device_error()
    qf, kf, vf = f64(q), f64(k), f64(v)
    m_ref, _ = oracle.lse_merge(f64(parts), f64(lses))
    check_f32(merged, m_ref, "chain: merge of the partials")
    c1_ref = oracle.cfg_combine(f64(merged), f64(other), 2.0)
    check_f32(c1, c1_ref, "chain: first combine")
    c2_ref = oracle.cfg_combine(f64(c1), f64(merged), 0.25)
    check_f32(c2, c2_ref, "chain: second combine")
    o_ref, l_ref = oracle.attention(f64(q2), kf, vf)
    check_attention(out, lse, o_ref, l_ref, "chain: attention on the combined queries")
    o1_ref, _ = oracle.attention(qf, kf, vf)
    check_attention(merged.view(B, H, S, D), None, o1_ref, None, "chain: merged attention")
