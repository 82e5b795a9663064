"""GPU parity of the chunk-parallel attention launch (dit_attn_fwd_split:
one CTA per query-tile pair and chunk, then the log-sum-exp merge of the
chunks to bf16) against the fp64 oracle, through the C ABI: the workloads at
full size, one device's share of their heads under a head-parallel split,
ragged lengths, and the workspace's reuse."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import abs_weighted, check_attention, f64, oracle_rows, sample_rows
from sequence_attention_attn_b300 import dit_attn, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def run_split(q, k, v, n_split):
    out, lse = dit_attn.attention_split(q, k, v, n_split)
    torch.cuda.synchronize()
    assert dit_attn.dit_last_device_status() == 0, "a device-side wait ran out"
    return out, lse


@pytest.mark.parametrize("n_split", [1, 2, 4, 8])
def test_split_dit_xl2_full(n_split):
    cfg = workloads.BY_NAME["dit_xl2_512"]
    q, k, v = workloads.make_qkv(cfg)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v))
    out, lse = run_split(*(t.to(DEV) for t in (q, k, v)), n_split)
    check_attention(out, lse, o_ref, l_ref, f"dit_xl2 split={n_split}")


@pytest.mark.parametrize("name,n_split", [("pixart_1024", 2), ("flux_mmdit", 3), ("video", 4)])
def test_split_full_size_sampled(name, n_split):
    cfg = workloads.BY_NAME[name]
    q, k, v = workloads.make_qkv(cfg)
    out, lse = run_split(*(t.to(DEV) for t in (q, k, v)), n_split)
    rows = sample_rows(cfg.B * cfg.H, cfg.S, 256, seed=cfg.index * 10 + n_split)
    o_ref, l_ref = oracle_rows(q, k, v, rows)
    idx = torch.as_tensor(rows, device=DEV)
    check_attention(out.reshape(-1, cfg.D)[idx], lse.reshape(-1)[idx], o_ref, l_ref, f"{name} split={n_split}")


@pytest.mark.parametrize("name,heads", [("dit_xl2_512", 2), ("pixart_1024", 2), ("flux_mmdit", 3)])
def test_split_head_share(name, heads):
    # one device's share of the heads under an 8-way head split: the launch
    # the chunk-parallel form is for
    cfg = workloads.BY_NAME[name]
    q, k, v = (t[:, :heads].contiguous() for t in workloads.make_qkv(cfg))
    rows = sample_rows(cfg.B * heads, cfg.S, 256, seed=cfg.index + heads)
    o_ref, l_ref = oracle_rows(q, k, v, rows)
    idx = torch.as_tensor(rows, device=DEV)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    for n_split in (2, 4):
        out, lse = run_split(qd, kd, vd, n_split)
        check_attention(out.reshape(-1, cfg.D)[idx], lse.reshape(-1)[idx], o_ref, l_ref,
                        f"{name} heads={heads} split={n_split}")


@pytest.mark.parametrize("S", [1, 100, 129, 257, 1000])
@pytest.mark.parametrize("D", [64, 72, 128])
def test_split_edge_lengths(S, D):
    q, k, v = workloads.make_random_qkv(1, 3, S, D, seed=S * 17 + D, std=1.5)
    qf, kf, vf = f64(q), f64(k), f64(v)
    o_ref, l_ref = oracle.attention(qf, kf, vf)
    a_ref = abs_weighted(qf, kf, vf)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    for n_split in sorted({1, min(S, 2), min(S, 3), min(S, 40), S}):
        out, lse = run_split(qd, kd, vd, n_split)
        check_attention(out, lse, o_ref, l_ref, f"S={S} D={D} split={n_split}", abs_ref=a_ref)


def test_split_matches_the_merged_launch_on_the_same_chunks():
    # the same partition as dit_attn_fwd with n_kv_chunks = n_split, merged on
    # chip there and by the merge kernel here: equal up to rounding
    cfg = workloads.BY_NAME["pixart_1024"]
    q, k, v = (t.to(DEV) for t in workloads.make_qkv(cfg))
    for n in (1, 4):
        a, la = dit_attn.attention(q, k, v, n_kv_chunks=n)
        b, lb = run_split(q, k, v, n)
        d = (a.float() - b.float()).abs()
        assert d.max().item() <= 2e-2 and d.mean().item() <= 2e-4, (n, d.max().item(), d.mean().item())
        assert (la - lb).abs().max().item() <= 1e-4, n


def test_split_reuses_a_garbage_workspace():
    # nothing in the workspace is read before it is written: a workspace full
    # of NaN bytes gives the right result, and calls in a row give the same bits
    B, H, S, D, n_split = 2, 2, 1000, 72, 3
    q, k, v = workloads.make_random_qkv(B, H, S, D, seed=9)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v))
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    nbytes = dit_attn.dit_attn_split_workspace_bytes(B, H, S, D, n_split)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(3):
        out = torch.empty_like(qd)
        lse = torch.empty((B, H, S), dtype=torch.float32, device=DEV)
        dit_attn.dit_attn_fwd_split(qd, kd, vd, out, lse, n_split, ws)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert dit_attn.dit_last_device_status() == 0
    check_attention(outs[0][0], outs[0][1], o_ref, l_ref, "garbage workspace")
    for out, lse in outs[1:]:
        assert torch.equal(out, outs[0][0]) and torch.equal(lse, outs[0][1])


def test_split_rejects_bad_workspace():
    B, H, S, D = 1, 2, 256, 64
    q, k, v = workloads.make_random_qkv(B, H, S, D, seed=1, device=DEV)
    out = torch.empty_like(q)
    nbytes = dit_attn.dit_attn_split_workspace_bytes(B, H, S, D, 2)
    small = torch.empty(nbytes - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(dit_attn.DitError):
        dit_attn.dit_attn_fwd_split(q, k, v, out, None, 2, small)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    with pytest.raises(dit_attn.DitError):
        dit_attn.dit_attn_fwd_split(q, k, v, out, None, S + 1, ws)
    torch.cuda.synchronize()
    assert dit_attn.dit_last_device_status() == 0
