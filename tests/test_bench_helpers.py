"""bench.py's host logic on CPU: the roofline denominators, the DRAM traffic taken from the
committed ncu summary (only while it describes the current kernel sources), the workload
configuration and the oracle sample sizing. No GPU: nothing here launches a kernel.
"""
import os

import pytest

import bench
import synthetic


def test_traffic_is_read_only_for_the_profiled_sources(monkeypatch):
    path = os.path.join(bench.ROOT, "profiles", "bwd_dW_gemm_n32768_d3072_v128256.md")
    text = open(path).read()
    real = bench.profile_traffic("bwd_dW_gemm", "n32768_d3072_v128256")
    if "source_hash: " + bench.kernel_source_hash() in text:
        assert real is not None and 3.0e9 < real < 4.5e9  # a dW launch moves ~3.7 GB
    else:  # the engine changed since the capture
        assert real is None
    # once the engine sources differ from the ones the summary was taken on, no traffic
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0123456789abcdef")
    assert bench.profile_traffic("bwd_dW_gemm", "n32768_d3072_v128256") is None
    assert bench.profile_traffic("no_such_kernel", "n32768_d3072_v128256") is None


def test_peaks_prefer_the_measured_file(monkeypatch):
    monkeypatch.setattr(bench, "ROOT", os.path.join(bench.ROOT, "no_such_directory"))
    peaks, src = bench.measured_peaks()
    assert src == "fallback" and bench.peak_value(peaks, "bf16_tflops_sustained") == 1700.0
    measured = {"hbm_gbs": 6782.8, "bf16_tflops": 1915.7, "bf16_tflops_sustained": 1706.9}
    assert bench.peak_value(measured, "bf16_tflops_sustained") == 1706.9
    assert bench.peak_value(measured, "bf16_tflops") == 1915.7
    assert bench.peak_value({"other": 1.0}, "hbm_gbs") == bench.FALLBACK["hbm_gbs"]


def test_config_names_the_workload_and_path():
    w = synthetic.WORKLOADS["n32768_d3072_v128256"]
    c = bench.config_of(w)
    assert c["workload"] == w.name and (c["N"], c["d"], c["V"], c["K"], c["chunk"]) == (32768, 3072, 128256, 100, 2048)
    assert c["api"] == "fused" and "kept" in c["logits"] and "L2" in c["l2"]
    assert "recomputed" in bench.config_of(w, "separate")["logits"]
    assert w.flops() == 8.0 * w.N * w.d * w.V


def test_oracle_sample_is_sized_from_two_calibration_runs(monkeypatch):
    w = synthetic.WORKLOADS["n32768_d3072_v128256"]
    calls = []

    def fake_time(w_, x, W, n):  # a fixed 2 s per call plus 10 ms per position
        calls.append(n)
        return 2.0 + 0.01 * n

    monkeypatch.setattr(bench, "sample_rows_oracle", fake_time)
    n = bench.calibrated_sample_size(w, {}, None, 15.0)
    assert len(calls) == 2 and calls[1] == 2 * calls[0]
    # (15 s - 2 s) / 10 ms = 1300 positions, within the 4x clamp of the plain estimate
    assert abs(n - 1300) <= 2

    # noisy timings (the larger run no slower): never more than 4x the plain rate's answer
    monkeypatch.setattr(bench, "sample_rows_oracle", lambda w_, x, W, n: 3.0)
    n0 = bench.oracle_sample_size(w, target_s=1.0)
    n = bench.calibrated_sample_size(w, {}, None, 15.0)
    assert n <= 4 * int(2 * n0 * 15.0 / 3.0) + 1


def test_cpu_sample_is_the_first_positions_of_the_benched_inputs():
    """The oracle's CPU sample slices the workload's own inputs: its first n positions are
    the benched positions 0..n-1, bit for bit (the teacher cache's redraws of rows with a
    repeated id depend on the row count, so regenerating at n rows would give other rows)."""
    import numpy as np
    w = synthetic.WORKLOADS["n8192_d3072_v128256"]
    x, W = bench.cpu_inputs(w, 0)
    full = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype=w.dtype, seed=0)
    assert x["H"].shape == (w.N, w.d) and W.shape == (w.V, w.d)
    for k in ("H", "idx", "logp"):
        assert np.array_equal(x[k][:100], full[k][:100])
    assert np.array_equal(W, full["W"])


def test_path_summary_counts_and_kernel_roofline():
    """The step's 8NdV count and executed FLOPs come from the step time; the roofline from the
    dominant kernel's own launches: tensor-bound at chunk 2048, HBM-bound (dW's fp32
    read-modify-write) at chunk 1024."""
    for name, bound in (("n32768_d3072_v128256", "tensor"), ("n8192_d3072_v128256", "hbm")):
        w = synthetic.WORKLOADS[name]
        chunks = -(-w.N // w.chunk)
        steps, t_ms = 4, 4 * 50.0
        prof = {"bwd_dW_gemm": (steps * chunks * 1.0, steps * chunks), "fwd_logits_keep": (10.0, steps * chunks)}
        s = bench.path_summary(w, "fused", t_ms, steps, 1, prof, 1700.0, "measured", 6700.0)
        assert abs(s["tflops_8NdV"] - w.flops() / 0.05 / 1e12) < 1e-6 * s["tflops_8NdV"]
        assert abs(s["tflops_executed"] - 0.75 * s["tflops_8NdV"]) < 1e-6 * s["tflops_8NdV"]
        r = s["roofline"]
        assert r["kernel"] == "bwd_dW_gemm" and r["bound"] == bound
        f, b = bench.kernel_work(w, "bwd_dW_gemm")
        assert abs(r["flops_per_launch"] - f / chunks) < 1e-3 * r["flops_per_launch"]
        assert abs(r["tensor_frac"] - f / chunks / 1e-3 / 1e12 / 1700.0) < 1e-9
        assert abs(r["hbm_frac"] - b / chunks / 1e-3 / 1e9 / 6700.0) < 1e-9
        sep = bench.path_summary(w, "separate", t_ms, steps, 1, prof, 1700.0, "measured", 6700.0)
        assert sep["tflops_executed"] == sep["tflops_8NdV"]
        # with the clocks: the tensor-bound fraction is also given at the peak's clock
        c = bench.path_summary(w, "fused", t_ms, steps, 1, prof, 1700.0, "measured", 6700.0, 1450.0, 1507.0)
        if bound == "tensor":
            assert abs(c["roofline"]["frac_at_peak_clock"] - r["frac"] * 1507.0 / 1450.0) < 1e-12
        else:
            assert "frac_at_peak_clock" not in c["roofline"]
    assert bench.peak_clock_mhz({"clocks_under_load": {"sm_mhz_median": 1507.0}}) == 1507.0
    assert bench.peak_clock_mhz({}) is None
