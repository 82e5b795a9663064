"""Write ``tiny_oracle.json``: oracle outputs on the seeded tiny workload.

A regression record of the fp64 oracle (calls only ``oracle/`` and the seeded
input generator), so that any later change to the oracle's arithmetic shows up
as a diff of this file.  Regenerate with ``python tests/golden/make_golden.py``.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from sequence_attention_attn_b300 import workloads  # noqa: E402

PROBE_ROWS = [0, 1, 127, 128, 255, 256, 300, 511]


def compute():
    cfg = workloads.BY_NAME["tiny"]
    q, k, v = (t.float().numpy().astype(np.float64) for t in workloads.make_qkv(cfg))
    out = {"workload": "tiny B=1 H=2 S=256 D=64", "seed": workloads.seed_for(cfg),
           "probe_rows": PROBE_ROWS, "chunks": {}}
    for n in cfg.chunk_counts:
        o, l = oracle.attention_chunked(q, k, v, oracle.chunk_bounds(cfg.S, n))
        o2 = o.reshape(-1, cfg.D)
        l2 = l.reshape(-1)
        out["chunks"][str(n)] = {
            "lse": [float(l2[r]) for r in PROBE_ROWS],
            "o_first4": [[float(x) for x in o2[r, :4]] for r in PROBE_ROWS],
            "o_sum": float(o2.sum()),
            "o_abs_sum": float(np.abs(o2).sum()),
            "lse_sum": float(l2.sum()),
        }
    ec, eu = workloads.make_cfg(cfg.cfg_shape, workloads.seed_for(cfg, 100))
    c = oracle.cfg_combine(ec.numpy(), eu.numpy(), cfg.cfg_w)
    out["cfg"] = {"w": cfg.cfg_w, "sum": float(c.sum()), "abs_sum": float(np.abs(c).sum()),
                  "first4": [float(x) for x in c.reshape(-1)[:4]]}
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(compute(), f, indent=1)
        f.write("\n")
