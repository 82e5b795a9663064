"""GPU parity of the key-range attention and of the Torus-style chunked
attention (each K/V chunk computed as soon as its copy has landed, then the
LSE merge) against the fp64 oracle, through the C ABI."""
import pytest
import torch

import oracle
from parity_util import abs_weighted, check_attention, f64, oracle_rows, sample_rows
from sequence_attention_attn_b300 import dit_attn, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def assert_no_device_error():
    assert dit_attn.dit_last_device_status() == 0, "a device-side wait ran out"


# ------------------------------------------------------- one key range
def range_cases(S):
    cases = {(0, S), (0, 1), (S - 1, S), (0, min(S, 5)), (S // 3, S - S // 4)}
    if S > 140:
        cases |= {(5, 133), (128, min(S, 256)), (127, 129), (1, S - 1)}
    return sorted(c for c in cases if 0 <= c[0] < c[1] <= S)


@pytest.mark.parametrize("S", [1, 100, 257, 640])
@pytest.mark.parametrize("D", [64, 72, 128])
def test_range_matches_oracle(S, D):
    q, k, v = workloads.make_random_qkv(2, 2, S, D, seed=31 * S + D, std=1.5)
    qf, kf, vf = f64(q), f64(k), f64(v)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    for j0, j1 in range_cases(S):
        out, lse = dit_attn.attention_range(qd, kd, vd, j0, j1)
        torch.cuda.synchronize()
        assert_no_device_error()
        o_ref, l_ref = oracle.attention(qf, kf, vf, j0, j1)
        check_attention(out, lse, o_ref.reshape(-1, D), l_ref.reshape(-1), f"S={S} D={D} [{j0},{j1})",
                        abs_ref=abs_weighted(qf, kf, vf, j0, j1).reshape(-1, D))


def test_range_ignores_keys_outside_the_range():
    # Rows outside [j0, j1) -- before j0 and in the masked tail of the last
    # tile alike -- are rewritten with other finite values: the result must
    # not change by a single bit.
    S, D, j0, j1 = 700, 64, 130, 300
    q, k, v = (t.to(DEV) for t in workloads.make_random_qkv(1, 3, S, D, seed=4))
    out_a, lse_a = dit_attn.attention_range(q, k, v, j0, j1)
    k2, v2 = k.clone(), v.clone()
    for t in (k2, v2):
        t[:, :, :j0] = 7.0
        t[:, :, j1:] = -3.0
    out_b, lse_b = dit_attn.attention_range(q, k2, v2, j0, j1)
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)


@pytest.mark.parametrize("D", [64, 72, 128])
def test_range_reads_no_key_row_outside_the_range(D):
    # Every key and value row outside [j0, j1) is NaN: the range kernel must
    # read none of them (the last tile's tail past j1 is zero-filled, not read).
    S = 700
    q, k, v = workloads.make_random_qkv(1, 3, S, D, seed=40 + D)
    qf, kf, vf = f64(q), f64(k), f64(v)
    qd = q.to(DEV)
    for j0, j1 in ((130, 300), (0, 5), (127, 129), (600, 700), (0, 700)):
        kd, vd = k.to(DEV), v.to(DEV)
        for t in (kd, vd):
            t[:, :, :j0] = float("nan")
            t[:, :, j1:] = float("nan")
        out, lse = dit_attn.attention_range(qd, kd, vd, j0, j1)
        torch.cuda.synchronize()
        assert_no_device_error()
        o_ref, l_ref = oracle.attention(qf, kf, vf, j0, j1)
        check_attention(out, lse, o_ref.reshape(-1, D), l_ref.reshape(-1), f"NaN outside [{j0},{j1}) D={D}")


def test_ranges_merge_to_full_attention():
    # uneven ranges, none aligned to a tile: the merge of the range results is
    # the attention over all keys
    cfg = workloads.BY_NAME["dit_xl2_512"]
    q, k, v = workloads.make_qkv(cfg)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    cuts = [0, 3, 200, 201, 515, 1024]
    parts, lses = zip(*(dit_attn.attention_range(qd, kd, vd, a, b) for a, b in zip(cuts, cuts[1:])))
    out, lse = dit_attn.merge(torch.stack(parts), torch.stack(lses))
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v))
    check_attention(out, lse, o_ref.reshape(-1, cfg.D), l_ref.reshape(-1), "ranges merged")


# ---------------------------------------------- Torus-style overlap
def sources(q, k, v, where):
    if where == "pinned":
        return k.pin_memory(), v.pin_memory()
    return k.to(DEV), v.to(DEV)


@pytest.mark.parametrize("where", ["pinned", "device"])
@pytest.mark.parametrize("copy", ["side", "same"])
@pytest.mark.parametrize("name,n", [("tiny", 1), ("tiny", 3), ("dit_xl2_512", 4), ("dit_xl2_512", 16)])
def test_torus_matches_oracle(name, n, where, copy):
    cfg = workloads.BY_NAME[name]
    q, k, v = workloads.make_qkv(cfg)
    ks, vs = sources(q, k, v, where)
    side = torch.cuda.Stream() if copy == "side" else None
    out, lse = dit_attn.attention_torus(q.to(DEV), ks, vs, n, copy_stream=side)
    torch.cuda.synchronize()
    assert_no_device_error()
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v))
    check_attention(out, lse, o_ref.reshape(-1, cfg.D), l_ref.reshape(-1), f"torus {name} n={n} {where} {copy}")


def test_torus_equals_partials_then_merge_bitwise():
    # each chunk is the same kernel over the same key range as the partials
    # entry point, and the merge is the same kernel
    cfg = workloads.BY_NAME["dit_xl2_512"]
    q, k, v = (t.to(DEV) for t in workloads.make_qkv(cfg))
    for n in (2, 5, 8):
        parts, lses = dit_attn.attention_partials(q, k, v, n)
        ref_out, ref_lse = dit_attn.merge(parts, lses)
        out, lse = dit_attn.attention_torus(q, k, v, n, copy_stream=torch.cuda.Stream())
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), n


def test_torus_reads_only_landed_rows():
    # The landing buffers start as NaN.  Chunks of 40 keys end inside a
    # 128-key tile and chunk c is computed as soon as its own rows have
    # landed, while later chunks' rows may still be NaN: the result must not
    # depend on them.
    S, D, n = 1000, 64, 25
    q, k, v = workloads.make_random_qkv(1, 4, S, D, seed=12)
    qd = q.to(DEV)
    ks, vs = k.pin_memory(), v.pin_memory()
    kd = torch.full_like(qd, float("nan"))
    vd = torch.full_like(qd, float("nan"))
    rows = 4 * S
    parts = torch.empty((n, rows, D), dtype=torch.float32, device=DEV)
    lses = torch.empty((n, rows), dtype=torch.float32, device=DEV)
    out = torch.empty((rows, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((rows,), dtype=torch.float32, device=DEV)
    side = torch.cuda.Stream()
    for _ in range(3):
        kd.fill_(float("nan"))
        vd.fill_(float("nan"))
        dit_attn.dit_attn_fwd_torus(qd, ks, vs, kd, vd, parts, lses, out, lse, n, copy_stream=side)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    assert torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v))
    check_attention(out, lse, o_ref.reshape(-1, D), l_ref.reshape(-1), "torus NaN landing buffers")


def test_torus_video_workload_sampled():
    cfg = workloads.BY_NAME["video"]
    q, k, v = workloads.make_qkv(cfg)
    ks, vs = k.pin_memory(), v.pin_memory()
    out, lse = dit_attn.attention_torus(q.to(DEV), ks, vs, 8, copy_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert_no_device_error()
    rows = sample_rows(cfg.B * cfg.H, cfg.S, 256, seed=77)
    o_ref, l_ref = oracle_rows(q, k, v, rows)
    idx = torch.as_tensor(rows, device=DEV)
    check_attention(out[idx], lse[idx], o_ref, l_ref, "torus video n=8")


def test_torus_argument_checks_in_binding():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device=DEV)
    pageable = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="pinned"):
        dit_attn.attention_torus(q, pageable, pageable, 2)
    with pytest.raises(dit_attn.DitError):
        dit_attn.attention_torus(q, q.clone(), q.clone(), 65)
    # a source that is the other landing buffer is rejected before any copy
    k, v = torch.empty_like(q), torch.empty_like(q)
    rows = 128
    parts = torch.empty((2, rows, 64), dtype=torch.float32, device=DEV)
    lses = torch.empty((2, rows), dtype=torch.float32, device=DEV)
    out = torch.empty((rows, 64), dtype=torch.float32, device=DEV)
    with pytest.raises(dit_attn.DitError):
        dit_attn.dit_attn_fwd_torus(q, v, q.clone(), k, v, parts, lses, out, None, 2)
    with pytest.raises(dit_attn.DitError):
        dit_attn.dit_attn_fwd_torus(q, q.clone(), k, k, v, parts, lses, out, None, 2)
