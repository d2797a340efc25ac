"""Write tests/golden/tiny_oracle.json from the oracle alone.

Run from the repository root:  python tests/golden/make_golden.py
The fixture records the oracle's outputs on the seeded ``tiny`` workload
(CPU generator, seed 0) so that an unintended change to the oracle's
arithmetic shows up as a test failure.  It calls only ``oracle`` and the
input generators.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads  # noqa: E402


def summary():
    cfg = workloads.CONFIGS["tiny"]
    inp = workloads.make_inputs(cfg, seed=0)
    out = oracle.fused_topk_kl(inp["hidden"], inp["W"], inp["topk_idx"],
                               inp["topk_logit"], cfg.T)
    return {
        "config": "tiny", "seed": 0, "generator": "torch CPU",
        "loss": out["loss"],
        "lse_first4": out["lse"][:4].tolist(),
        "grad_hidden_fro": float(np.linalg.norm(out["grad_hidden"])),
        "grad_W_fro": float(np.linalg.norm(out["grad_W"])),
        "grad_hidden_00": float(out["grad_hidden"][0, 0]),
        "grad_W_00": float(out["grad_W"][0, 0]),
    }


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(path, "w") as f:
        json.dump(summary(), f, indent=1)
    print("wrote", path)
