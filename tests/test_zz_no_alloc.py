"""cfg_combine_relmae_static, the entry point that takes no workspace and
allocates nothing (its per-block sums live in a fixed device array of the
library), against the existing cfg_combine_relmae through the C ABI, with two
calls in a row on the same inputs.  The file name puts it last in collection,
so it also runs after every other test in one process."""
import pytest
import torch

import oracle
from sequence_attention_attn_b300 import dit_attn, workloads

DEV = "cuda:0"
INVALID, MISALIGNED = -1, -3
NAN = float("nan")


def test_static_relmae_rejects_bad_arguments_on_host():
    # rejected before any CUDA call: the (never dereferenced) pointers are fake
    f = dit_attn.lib().cfg_combine_relmae_static
    A, B, O, S = 0x7F0000000000, 0x7F1000000000, 0x7F2000000000, 0x7F3000000000
    assert f(A, B, 1.5, O, dit_attn.RELMAE_STATIC_MAX_NUMEL + 1, S, None) == INVALID
    assert f(A, B, 1.5, O, 0, S, None) == INVALID
    assert f(None, B, 1.5, O, 16, S, None) == INVALID
    assert f(A, B, float("inf"), O, 16, S, None) == INVALID
    assert f(A + 8, B, 1.5, O, 16, S, None) == MISALIGNED      # eps_c not 16-byte aligned
    assert f(A, B, 1.5, O, 16, S + 4, None) == MISALIGNED      # sums not 8-byte aligned
    assert f(A, B, 1.5, A + 16, 16, S, None) == INVALID        # out overlaps eps_c, not equal to it
    assert f(A, B, 1.5, O, 16, B + 8, None) == INVALID         # sums inside eps_u


def run_both(c, u, w):
    out_a = torch.full_like(c, NAN)
    sums_a = torch.full((3,), NAN, dtype=torch.float64, device=DEV)
    dit_attn.cfg_combine_relmae(c, u, w, out_a, sums_a)
    outs, sums = [], []
    for _ in range(2):
        o = torch.full_like(c, NAN)
        s = torch.full((3,), NAN, dtype=torch.float64, device=DEV)
        dit_attn.cfg_combine_relmae_static(c, u, w, o, s)
        outs.append(o)
        sums.append(s)
    torch.cuda.synchronize()
    assert dit_attn.dit_last_device_status() == 0
    return out_a, sums_a, outs, sums


def check_against_existing(out_a, sums_a, outs, sums, what):
    for o in outs:
        assert torch.equal(o, out_a), f"{what}: combine differs from cfg_combine_relmae"
    # a fixed summation order: the two calls agree bit for bit
    assert torch.equal(sums[0], sums[1]), (what, sums[0].tolist(), sums[1].tolist())
    d, b, r = sums[0].tolist()
    da, ba, ra = sums_a.tolist()
    # both add fp32 per-thread sums in fp64, over different partitions
    assert abs(d - da) <= 1e-5 * da, (what, d, da)
    assert abs(b - ba) <= 1e-5 * ba, (what, b, ba)
    assert abs(r - ra) <= 1e-5 * ra, (what, r, ra)
    assert r == d / b, what


@pytest.mark.gpu
@pytest.mark.parametrize("numel", [1, 5, 4099, 65536 * 3 + 1, (1 << 20) + 7, 3 * (1 << 24) + 2])
def test_static_relmae_matches_existing_twice(numel):
    eps_c, eps_u = workloads.make_cfg((numel,), seed=numel % 9973 + 17)
    c, u = eps_c.to(DEV), eps_u.to(DEV)
    out_a, sums_a, outs, sums = run_both(c, u, 4.5)
    check_against_existing(out_a, sums_a, outs, sums, f"numel={numel}")
    # and the oracle (fp64 sums of the same definition)
    ref_ratio = oracle.cfg_relmae_ratio(eps_c.numpy(), eps_u.numpy())
    assert abs(sums[0][2].item() - ref_ratio) <= 1e-5 * ref_ratio


@pytest.mark.gpu
def test_static_relmae_at_its_maximum_size_and_in_place():
    numel = dit_attn.RELMAE_STATIC_MAX_NUMEL  # 4096 slabs, every slot of the array
    c, u = workloads.make_cfg((numel,), seed=5, device=DEV)
    out_a, sums_a, outs, sums = run_both(c, u, 7.5)
    check_against_existing(out_a, sums_a, outs, sums, "maximum numel")
    del outs
    # out aliasing eps_c, on the latent shape of the video workload
    c2, u2 = workloads.make_cfg((16, 13, 60, 90), seed=6, device=DEV)
    want = c2.clone()
    s_ref = torch.empty(3, dtype=torch.float64, device=DEV)
    dit_attn.cfg_combine_relmae(want, u2, 4.5, want, s_ref)
    s = torch.empty(3, dtype=torch.float64, device=DEV)
    dit_attn.cfg_combine_relmae_static(c2, u2, 4.5, c2, s)
    torch.cuda.synchronize()
    assert torch.equal(c2, want)
    assert abs(s[2].item() - s_ref[2].item()) <= 1e-5 * s_ref[2].item()
    assert dit_attn.dit_last_device_status() == 0


@pytest.mark.gpu
def test_static_relmae_rejects_numel_above_maximum():
    # the binding's error names the limit; nothing is launched
    c = torch.empty(dit_attn.RELMAE_STATIC_MAX_NUMEL + 4, dtype=torch.float32, device=DEV)
    s = torch.empty(3, dtype=torch.float64, device=DEV)
    with pytest.raises(dit_attn.DitError, match="maximum"):
        dit_attn.cfg_combine_relmae_static(c, c, 1.0, c, s)
