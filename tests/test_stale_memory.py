"""GPU parity of the attention launches (merged, partials + merge,
chunk-parallel) when the memory under their buffers held NaN just before:
blocks filled with NaN are freed, the inputs are copied from pageable host
memory into them (the copy is the last operation before the launch), and the
output, LSE, partial and workspace buffers are left uninitialised.  A
launch that read past its inputs, read an output buffer or left part of it
unwritten would show non-finite values here.  Repeated three times in one
process, so the later calls run on memory the earlier ones released."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import abs_weighted, check_attention, f64
from sequence_attention_attn_b300 import dit_attn, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def upload_over_nan(*ts):
    junk = [torch.full(t.shape, float("nan"), dtype=t.dtype, device=DEV) for t in ts]
    torch.cuda.synchronize()
    del junk
    return [t.to(DEV) for t in ts]


@pytest.mark.parametrize("D", [64, 72, 128])
def test_merged_and_partials_over_stale_nan_memory(D):
    cases = []
    for S in (100, 129, 257, 1000):
        q, k, v = workloads.make_random_qkv(1, 3, S, D, seed=S * 31 + D, std=1.5)
        qf, kf, vf = f64(q), f64(k), f64(v)
        o_ref, l_ref = oracle.attention(qf, kf, vf)
        cases.append((S, q, k, v, qf, kf, vf, o_ref, l_ref, abs_weighted(qf, kf, vf)))
    for rep in range(3):
        for S, q, k, v, qf, kf, vf, o_ref, l_ref, a_ref in cases:
            for n in sorted({1, 3, min(S, 40)}):
                qd, kd, vd = upload_over_nan(q, k, v)
                out, lse = dit_attn.attention(qd, kd, vd, n_kv_chunks=n)
                torch.cuda.synchronize()
                assert dit_attn.dit_last_device_status() == 0
                check_attention(out, lse, o_ref, l_ref, f"rep={rep} S={S} D={D} n={n} merged", abs_ref=a_ref)
                qd, kd, vd = upload_over_nan(q, k, v)
                parts, lses = dit_attn.attention_partials(qd, kd, vd, n)
                merged, mlse = dit_attn.merge(parts, lses)
                torch.cuda.synchronize()
                assert dit_attn.dit_last_device_status() == 0
                m = merged.cpu().numpy().reshape(o_ref.shape)
                assert np.isfinite(m).all(), f"rep={rep} S={S} D={D} n={n}: non-finite merge"
                check_attention(merged.to(torch.bfloat16), mlse, o_ref, l_ref,
                                f"rep={rep} S={S} D={D} n={n} partials+merge", abs_ref=a_ref)
                qd, kd, vd = upload_over_nan(q, k, v)
                sout, slse = dit_attn.attention_split(qd, kd, vd, n)
                torch.cuda.synchronize()
                assert dit_attn.dit_last_device_status() == 0
                check_attention(sout, slse, o_ref, l_ref, f"rep={rep} S={S} D={D} n={n} split", abs_ref=a_ref)
