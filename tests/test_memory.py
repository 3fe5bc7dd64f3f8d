"""Peak device memory of the fused loss grows linearly in the number of positions.

The pages' point of the fused, chunked loss is that peak memory follows the sequence length
instead of sequence x vocabulary ("扩展到长上下文" in "Hugging Face：让知识蒸馏廉价到可大规模运行").
At a fixed chunk the only buffers that grow with N are H, dH, the teacher cache, lse and the
per-position losses; the fit's slope must match those bytes and the points must lie on a line.
Both ways of running the backward are checked: separate calls (logits recomputed) and the
one call (what the backward needs of the logits kept in the gradient slab, at no extra cost),
also with the workspace that overlaps consecutive chunks (one more chunk's buffers, a constant).
"""
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_peak_memory_linear_up_to_262144_positions():
    import argparse
    import bench
    args = argparse.Namespace(workload="n262144_d3072_v128256", seed=0)
    line = bench.memory_sweep(args)
    want = line["analytic_bytes_per_position"]
    for key in ("separate_calls", "one_call", "one_call_overlap"):
        f = line[key]
        assert f["points"][-1]["N"] == 262144
        assert f["max_rel_residual"] <= 0.02
        slope = f["fit_bytes_per_position"]
        assert abs(slope - want) <= 0.10 * want, (key, slope, want)
    # the one call holds nothing beyond the separate calls' buffers; with the overlap
    # workspace it holds one more chunk's buffers, a constant
    extra = line["one_call"]["fit_intercept_gib"] - line["separate_calls"]["fit_intercept_gib"]
    assert abs(extra) <= 0.05, extra
    extra = line["one_call_overlap"]["fit_intercept_gib"] - line["one_call"]["fit_intercept_gib"]
    assert abs(extra - line["second_buffer_set_gib"]) <= 0.05, (extra, line["second_buffer_set_gib"])
