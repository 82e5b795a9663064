"""GPU parity on seeded random shapes: batch, heads, sequence length, head
dimension, chunk count, split count and input scale drawn per case; the
merged launch, the partials + merge path and the chunk-parallel launch
against the fp64 oracle.  The draws are fixed by the case number, so a failure
names a reproducible shape.  DIT_FUZZ_CASES sets the number of cases (24 by
default)."""
import os

import numpy as np
import pytest
import torch

import oracle
from parity_util import abs_weighted, check_attention, f64
from sequence_attention_attn_b300 import dit_attn, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def draw(case: int):
    rng = np.random.default_rng(1000 + case)
    B = int(rng.integers(1, 3))
    H = int(rng.integers(1, 5))
    S = int(rng.integers(1, 2600))
    D = int(rng.choice([64, 72, 128]))
    n = int(rng.integers(1, min(S, 64) + 1))
    std = float(rng.choice([0.5, 1.0, 2.0, 3.0]))
    n_split = int(rng.integers(1, min(S, 8) + 1))
    return B, H, S, D, n, std, n_split


@pytest.mark.parametrize("case", range(int(os.environ.get("DIT_FUZZ_CASES", "24"))))
def test_random_shape(case):
    B, H, S, D, n, std, n_split = draw(case)
    what = f"case {case}: B={B} H={H} S={S} D={D} n={n} split={n_split} std={std}"
    q, k, v = workloads.make_random_qkv(B, H, S, D, seed=7000 + case, std=std)
    qf, kf, vf = f64(q), f64(k), f64(v)
    o_ref, l_ref = oracle.attention_chunked(qf, kf, vf, oracle.chunk_bounds(S, n))
    a_ref = abs_weighted(qf, kf, vf)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    out, lse = dit_attn.attention(qd, kd, vd, n_kv_chunks=n)
    parts, lses = dit_attn.attention_partials(qd, kd, vd, n)
    merged, mlse = dit_attn.merge(parts, lses)
    sout, slse = dit_attn.attention_split(qd, kd, vd, n_split)
    torch.cuda.synchronize()
    assert dit_attn.dit_last_device_status() == 0, what
    check_attention(out, lse, o_ref, l_ref, what + " merged", abs_ref=a_ref)
    check_attention(merged.to(torch.bfloat16), mlse, o_ref, l_ref, what + " partials+merge", abs_ref=a_ref)
    check_attention(sout, slse, o_ref, l_ref, what + " chunk-parallel", abs_ref=a_ref)
