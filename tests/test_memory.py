"""Peak device memory of the fused loss grows linearly in the number of positions.

The pages' point of the fused, chunked loss is that peak memory follows the sequence length
instead of sequence x vocabulary ("扩展到长上下文" in "Hugging Face：让知识蒸馏廉价到可大规模运行").
At a fixed chunk the only buffers that grow with N are H, dH, the teacher cache, lse and the
per-position losses; the fit's slope must match those bytes and the points must lie on a line.
"""
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_peak_memory_linear_up_to_262144_positions():
    import argparse
    import bench
    args = argparse.Namespace(workload="n262144_d3072_v128256", seed=0)
    line = bench.memory_sweep(args)
    assert line["points"][-1]["N"] == 262144
    assert line["max_rel_residual"] <= 0.02
    slope, want = line["fit_bytes_per_position"], line["analytic_bytes_per_position"]
    assert abs(slope - want) <= 0.10 * want, (slope, want)
