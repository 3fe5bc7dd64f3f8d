"""Writes tests/golden/tiny_oracle.json from the fp64 oracle and the seeded generators.

Run from the repository root:  python tests/golden/make_golden.py
It calls only ``oracle`` and ``synthetic``; no value comes from the CUDA path.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import fckl_oracle as orc  # noqa: E402
import synthetic  # noqa: E402


def main():
    w = synthetic.WORKLOADS["tiny_n64_d256_v4096"]
    seed, scale = 0, 1.0
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype=w.dtype, seed=seed)
    loss, lse, dH, dW = orc.forward_backward(x["H"], x["W"], x["idx"], x["logp"],
                                             grad_scale=scale, chunk=w.chunk)
    out = {
        "about": "fp64 oracle on the tiny workload (N=64, d=256, V=4096, K=16, fp32), seed 0",
        "workload": w.name, "seed": seed, "grad_scale": scale,
        "idx_row0": x["idx"][0, :8].tolist(),
        "logp_row0": [float(v) for v in x["logp"][0, :4]],
        "H_row0": [float(v) for v in x["H"][0, :4]],
        "loss": loss,
        "lse_head": lse[:8].tolist(),
        "dH_row0": dH[0, :8].tolist(),
        "dW_hit_row": dW[x["idx"][0, 0], :8].tolist(),
    }
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
