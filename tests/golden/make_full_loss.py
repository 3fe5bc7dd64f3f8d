"""Writes tests/golden/full_loss.json: the fp64 oracle's total loss over every position of the
four full-size bf16 workloads (seed 0), with fingerprints of the inputs it saw.

Run from the repository root:  python tests/golden/make_full_loss.py [workload ...]
It calls only ``oracle`` and ``synthetic``; no value comes from the CUDA path. The oracle
walks each workload in blocks of 1024 positions (its result does not depend on the block
size: the loss is a sum of per-position terms), which takes minutes per workload.
"""
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import fckl_oracle as orc  # noqa: E402
import synthetic  # noqa: E402

OUT = os.path.join(HERE, "full_loss.json")
WORKLOADS = ["n8192_d3072_v128256", "n32768_d3072_v128256", "n65536_d2880_v201088",
             "n262144_d3072_v128256"]


def fingerprint(x):
    """Sums that change if the seeded generators give other inputs on another machine."""
    return {"H_sum": float(x["H"].astype(np.float64).sum()),
            "H_abs_sum": float(np.abs(x["H"].astype(np.float64)).sum()),
            "W_abs_sum": float(np.abs(x["W"].astype(np.float64)).sum()),
            "idx_sum": int(x["idx"].astype(np.int64).sum()),
            "logp_sum": float(x["logp"].astype(np.float64).sum())}


def one(name, seed=0, block=1024):
    w = synthetic.WORKLOADS[name]
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype=w.dtype, seed=seed)
    t0 = time.time()
    loss, lse, rl = orc.forward(x["H"], x["W"], x["idx"], x["logp"], chunk=block)
    return {"workload": name, "seed": seed, "N": w.N, "d": w.d, "V": w.V, "K": w.K,
            "inputs": fingerprint(x), "loss": loss, "lse_sum": float(lse.sum()),
            "lse_head": lse[:4].tolist(), "row_loss_head": rl[:4].tolist(),
            "oracle_seconds": round(time.time() - t0, 1)}


def main(names):
    out = {}
    if os.path.exists(OUT):
        with open(OUT) as f:
            out = json.load(f)
    out["about"] = ("fp64 oracle: total (sum) loss over every position of each full-size bf16 workload, "
                    "unweighted, seed 0; inputs from the seeded generators, fingerprinted")
    for name in names:
        out[name] = one(name)
        print(name, out[name]["loss"], out[name]["oracle_seconds"], "s", flush=True)
        with open(OUT, "w") as f:
            json.dump(out, f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    main(sys.argv[1:] or WORKLOADS)
