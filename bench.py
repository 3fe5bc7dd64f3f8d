"""Benchmark of the fused, chunked top-K KL loss: forward + backward on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one forward + backward over the whole workload (all chunks), inputs resident in
HBM: one fckl_forward_backward call (--api fused, the default: each chunk's backward forms G
from what its forward kept in the gradient slab) or fckl_forward then fckl_backward (--api
separate: the backward recomputes each chunk's logits); the other structure is timed too over
the same steps and reported in a sub-object of the line. Prints one JSON line (rank 0). Under
torchrun each rank runs its own replica of the workload, or with --dp its own positions of a
data-parallel step (W replicated, dW and the loss all-reduced every step); the whole-job value
is the positions of all ranks over the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle, as it stands, on the host cores, on a
bounded sample of positions of the same workload (the pages ship no runnable code).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

DEFAULT_WORKLOAD = "n32768_d3072_v128256"
METRIC = "fused KL fwd+bwd positions/s & TFLOP/s (8NdV) vs BF16 roofline; peak GiB"
UNIT = "positions/s"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_KERNELS = ("fwd_logits_lse", "fwd_logits_keep", "bwd_logit_grad", "bwd_dH_gemm", "bwd_dW_gemm")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--positions", type=int, default=0,
                    help="run only the first P positions of the workload (profiling, memory sweeps)")
    ap.add_argument("--memory-sweep", action="store_true",
                    help="peak device memory of one forward+backward at N = W.N/8, W.N/4, W.N/2, W.N "
                         "(default workload n262144_d3072_v128256), with a linear fit")
    ap.add_argument("--topk", action="store_true",
                    help="time the teacher top-K cache builder (fckl_teacher_topk) on the workload's shapes")
    ap.add_argument("--api", default="fused", choices=["fused", "separate"],
                    help="one fckl_forward_backward call per step, or fckl_forward then fckl_backward")
    ap.add_argument("--recompute", action="store_true",
                    help="--topk: project each chunk twice instead of keeping its logits from pass 1")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cublas", action="store_true",
                    help="skip the same-shape cuBLAS GEMMs timed (after the timed region) for context")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dp", action="store_true",
                    help="under torchrun: data-parallel step (each rank its own positions, W replicated, dW and "
                         "the loss all-reduced inside the timed step) instead of independent replicas")
    ap.add_argument("--no-other-path", action="store_true",
                    help="time only --api's path (by default the other structure is timed too, over the same "
                         "steps, and reported as a sub-object of the line)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def sample_rows_oracle(w, x_rows, W_full, n_rows):
    """One oracle forward+backward over the first n_rows positions (full V and d)."""
    from oracle import fckl_oracle as orc
    sl = slice(0, n_rows)
    t0 = time.perf_counter()
    loss, lse, _ = orc.forward(x_rows["H"][sl], W_full, x_rows["idx"][sl], x_rows["logp"][sl], w.chunk)
    dH, dW = orc.backward(x_rows["H"][sl], W_full, x_rows["idx"][sl], x_rows["logp"][sl], 1.0, w.chunk)
    return time.perf_counter() - t0


def cpu_inputs(w, seed):
    """The workload's inputs exactly as the device sees them (bf16 values widened to fp32 for
    bf16 workloads): positions of a CPU sample are sliced from these, so a sample of n
    positions is the first n positions of the benched workload."""
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype=w.dtype, seed=seed)
    return {"H": x["H"], "idx": x["idx"], "logp": x["logp"]}, x["W"]


def oracle_sample_size(w, target_s=15.0):
    """Rows of a CPU sample taking roughly target_s seconds (cost is linear in rows)."""
    per_row_flops = 8.0 * w.d * w.V
    guess = int(target_s * 100e9 / per_row_flops)  # ~100 GFLOP/s fp64 BLAS as a first guess
    return max(8, min(w.N, guess))


def calibrated_sample_size(w, x, W, target_s):
    """Rows of an oracle sample taking about target_s seconds on this host. A call costs a
    fixed part (e.g. converting W) plus a part linear in rows; two short timed runs of the
    oracle itself, at n0 and 2 n0 rows, separate the two. Never more rows than ``x`` holds."""
    n_max = len(x["H"]) if x else w.N
    n0 = max(8, min(n_max // 2, oracle_sample_size(w, target_s=1.0)))
    t1 = sample_rows_oracle(w, x, W, n0)
    t2 = sample_rows_oracle(w, x, W, 2 * n0)
    naive = 2 * n0 * target_s / max(t2, 1e-3)  # as if the whole cost grew with rows
    per_row = (t2 - t1) / n0
    est = (target_s - max(t1 - per_row * n0, 0.0)) / per_row if per_row > 0 else 4 * naive
    # timing noise can make the slope look tiny: never more than 4x the plain rate's answer
    return max(8, min(n_max, int(min(max(est, naive), 4 * naive))))


def cpu_baseline(w, x, W):
    """The fp64 oracle, as it stands, timed on the host cores on the first n positions of the
    benched inputs ``x`` (n sized for about 15 s)."""
    n = calibrated_sample_size(w, x, W, target_s=15.0)
    t = sample_rows_oracle(w, x, W, n)
    return {"value": n / t, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
            "sample": f"fp64 oracle forward+backward on the first {n} of the {w.N} benched positions "
                      f"(full V={w.V}, d={w.d}, K={w.K}), {t:.1f} s (sized by two short calibration runs to about 15 s)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = synthetic.WORKLOADS[args.workload]
    n = max(8, oracle_sample_size(w, target_s=6.0))
    x, W = cpu_inputs(w, args.seed)
    for _ in range(args.warmup):
        sample_rows_oracle(w, x, W, min(n, 8))
    times = [sample_rows_oracle(w, x, W, n) for _ in range(args.steps)]
    t = sum(times)
    value = n * args.steps / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": config_of(w, args.api),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                             "sample": f"each step: fp64 oracle forward+backward on the first {n} of the "
                                       f"{w.N} positions of the workload (full V, d)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, api="fused", dp_world=0):
    par = (f"dp{dp_world}: {w.N} positions per rank, W replicated, dW and loss all-reduced every step"
           if dp_world > 1 else "replicas")
    return {"workload": w.name, "N": w.N, "d": w.d, "V": w.V, "K": w.K, "chunk": w.chunk,
            "input_dtype": w.dtype, "parallelism": par, "api": api,
            "logits": ("kept by the forward (fp16 exp(z - tile max) in the gradient slab)" if api == "fused"
                       else "recomputed in the backward"),
            "workspace": ("overlap (fckl_overlap_workspace_bytes): each chunk's G pass runs on a second stream "
                          "beside the next chunk's forward" if api == "fused"
                          else "the first fckl_workspace_bytes of the same workspace (chunks in sequence)"),
            "l2": "inputs larger than L2 (W alone is %.0f MB)" % (w.V * w.d * 2 / 1e6)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


def peak_value(peaks, key):
    for k, v in peaks.items():
        if k == key and isinstance(v, (int, float)):
            return float(v)
    for k, v in peaks.items():
        if key in k and isinstance(v, (int, float)):
            return float(v)
    return FALLBACK[key]


def kernel_source_hash():
    """Hash of the GEMM engine's sources (the kernels whose DRAM traffic the committed ncu
    summaries record); a summary whose hash differs no longer describes the current kernels."""
    h = hashlib.sha256()
    cdir = os.path.join(ROOT, "chunked_kl_loss_gb300", "csrc")
    for name in ("ptx.cuh", "tc_gemm.cuh"):
        with open(os.path.join(cdir, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profile_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m or not t or m.group(1) != kernel_source_hash():
        return None
    return float(t.group(1))


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            try:
                pw.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w": statistics.median(pw) if pw else None}


def max_over_ranks(value, device=None):
    """The largest of every rank's value (the slowest rank's time); the value itself on one
    process. Works with the nccl (CUDA tensors) and gloo (CPU tensors) backends."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cublas_context(w, dev, H, W_dev, idx, logp, reps=5):
    """cuBLAS bf16 GEMMs (torch.matmul) of the three per-chunk product shapes, for context
    beside the fused kernels: the same FLOPs without the epilogues. Timed with CUDA events,
    median of `reps` after one warm-up; TFLOP/s per shape. The library's own products are
    timed the same way (short isolated bursts: one chunk's fckl_forward_backward, per-kernel
    events, median of `reps`), so the two sets compare at the same clock conditions."""
    import torch
    import chunked_kl_loss_gb300 as fckl
    c = min(w.chunk, w.N)
    g = torch.Generator(device=dev).manual_seed(1)
    Hc = torch.randn(c, w.d, device=dev, generator=g).to(torch.bfloat16)
    W = torch.randn(w.V, w.d, device=dev, generator=g).to(torch.bfloat16)
    G = torch.randn(c, w.V, device=dev, generator=g).to(torch.bfloat16)
    shapes = {"logits [chunk,d]x[d,V]": lambda: torch.matmul(Hc, W.t()),
              "dH [chunk,V]x[V,d]": lambda: torch.matmul(G, W),
              "dW [V,chunk]x[chunk,d]": lambda: torch.matmul(G.t(), Hc)}
    out = {}
    for name, fn in shapes.items():
        fn()
        times = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        out[name] = {"ms": ms, "tflops": 2.0 * c * w.d * w.V / (ms / 1e3) / 1e12}
    del Hc, W, G
    torch.cuda.empty_cache()
    # the library's products on one chunk, same timing discipline
    dt = fckl.BF16 if w.dtype == "bf16" else fckl.F32
    ws = fckl.Workspace(c, w.d, w.V, w.K, c, dt, dev)
    Hs, idxs, logps = H[:c], idx[:c], logp[:c]
    fckl.forward_backward(Hs, W_dev, idxs, logps, c, ws=ws)
    per = {"fwd_logits_keep": [], "bwd_dH_gemm": [], "bwd_dW_gemm": []}
    for _ in range(reps):
        fckl.profile_enable(True)
        fckl.profile_read()
        fckl.forward_backward(Hs, W_dev, idxs, logps, c, ws=ws)
        prof = fckl.profile_read()
        fckl.profile_enable(False)
        for k in per:
            per[k].append(prof[k][0])
    fckl.check(ws)
    out["fused (this library), same bursts"] = {
        k: {"ms": statistics.median(v), "tflops": 2.0 * c * w.d * w.V / (statistics.median(v) / 1e3) / 1e12}
        for k, v in per.items()}
    return out


def kernel_work(w, kname):
    """Algorithmic work of one step's launches of a product kernel: (FLOPs, DRAM bytes) per
    step. Bytes count each operand once and each output once (dW's reduce-add launches read and
    write dW: every chunk after the first); re-reads served by L2 are not algorithmic."""
    n_chunks = -(-w.N // w.chunk)
    rows = [min(w.chunk, w.N - c * w.chunk) for c in range(n_chunks)]
    d, V = w.d, w.V
    flops = sum(2.0 * r * d * V for r in rows)
    Hc = sum(2.0 * r * d for r in rows)          # bf16 hidden states of each chunk
    Wb = n_chunks * 2.0 * V * d                   # W read once per chunk
    slab = sum(2.0 * r * V for r in rows)         # one pass over the bf16/fp16 slab
    if kname == "bwd_dW_gemm":
        byts = slab + Hc + 4.0 * V * d + (n_chunks - 1) * 8.0 * V * d
    elif kname == "bwd_dH_gemm":
        byts = slab + Wb + sum(4.0 * r * d for r in rows)
    elif kname in ("fwd_logits_keep", "bwd_logit_grad"):
        byts = Hc + Wb + slab
    else:  # fwd_logits_lse: statistics only
        byts = Hc + Wb + sum(12.0 * r * (-(-V // 256)) for r in rows)
    return flops, byts


def peak_clock_mhz(peaks):
    """Median SM clock under load while the sustained peak was measured, or None."""
    c = peaks.get("clocks_under_load") if isinstance(peaks, dict) else None
    v = c.get("sm_mhz_median") if isinstance(c, dict) else None
    return float(v) if isinstance(v, (int, float)) and v > 0 else None


def path_summary(w, api, t_ms, steps, world, prof, peak_sus, peak_src, hbm_peak=None, run_mhz=None,
                 peak_mhz=None):
    """Throughput of one timed path and the roofline of its dominant kernel.

    tflops_8NdV is the metric's count (8 N d V FLOPs per step: the four products of the
    recomputing structure) over the step time; it is a count, not a roofline fraction, since
    the one call runs only three of the four products. The roofline fraction is taken on the
    executed products only (tflops_executed) and, per kernel, on the dominant kernel's own
    FLOPs over its CUDA-event time."""
    ms_step = t_ms / steps
    products = 3 if api == "fused" else 4  # with kept logits the backward's logits product is not run
    tfl = w.flops() / (ms_step / 1e3) / 1e12
    tfl_exec = w.flops() * products / 4 / (ms_step / 1e3) / 1e12
    kname, (kms, kn) = max(prof.items(), key=lambda kv: kv[1][0])
    roof = None
    if kname in GEMM_KERNELS and kn > 0:
        # the kernel's own roofline: whichever of its FLOPs at the tensor peak and its
        # algorithmic bytes at the HBM peak takes longer
        f_step, b_step = kernel_work(w, kname)
        per_step = kn / steps
        flops_per_launch, bytes_per_launch = f_step / per_step, b_step / per_step
        t_launch = kms / kn / 1e3
        k_tfl = flops_per_launch / t_launch / 1e12
        k_gbs = bytes_per_launch / t_launch / 1e9
        hbm = hbm_peak or FALLBACK["hbm_gbs"]
        tensor_bound = flops_per_launch / (peak_sus * 1e12) >= bytes_per_launch / (hbm * 1e9)
        roof = {"kernel": kname, "bound": "tensor" if tensor_bound else "hbm",
                "achieved": k_tfl if tensor_bound else k_gbs, "peak": peak_sus if tensor_bound else hbm,
                "unit": "TFLOP/s" if tensor_bound else "GB/s",
                "frac": k_tfl / peak_sus if tensor_bound else k_gbs / hbm,
                "traffic": profile_traffic(kname, w.name),
                "peak_source": (f"{peak_src} bf16 sustained (kernel timed inside a long step)" if tensor_bound
                                else f"{peak_src} HBM copy bandwidth"),
                "flops_per_launch": flops_per_launch, "algorithmic_bytes_per_launch": bytes_per_launch,
                "tensor_frac": k_tfl / peak_sus, "hbm_frac": k_gbs / hbm, "avg_launch_ms": kms / kn}
        if tensor_bound and run_mhz and peak_mhz:
            # context for box-to-box differences under the power cap: the same fraction at the
            # clock the sustained peak was measured at (frac itself is the measured one)
            roof.update({"run_sm_mhz": run_mhz, "peak_sm_mhz": peak_mhz,
                         "frac_at_peak_clock": k_tfl / peak_sus * peak_mhz / run_mhz})
    total = max(1e-9, sum(u[0] for u in prof.values()))
    return {"value": world * w.N * steps / (t_ms / 1e3), "ms_per_step": ms_step,
            "tflops_8NdV": tfl,
            "tflops_8NdV_note": ("count: 8NdV FLOPs over the step time; this path executes "
                                 f"{products} of the 4 products (2NdV each)"),
            "tflops_executed": tfl_exec, "tflops_executed_frac_of_sustained": tfl_exec / peak_sus,
            "roofline": roof,
            "kernel_shares": {k: round(v[0] / total, 4) for k, v in prof.items() if v[1]},
            "kernel_ms_per_step": sum(v[0] for v in prof.values()) / steps,
            "kernel_shares_note": ("shares of the summed per-kernel event time" + (
                "; the G pass (bwd_grad_from_logits) runs on a second stream beside the next chunk's forward, "
                "so the summed time exceeds the step and both kernels' event times include the overlap"
                if api == "fused" else ""))}


def replica_seed(seed, rank):
    """Each rank runs its own replica of the workload on its own seeded inputs."""
    return seed + 1000 * rank


def run_ours(args):
    import torch
    import chunked_kl_loss_gb300 as fckl

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)  # before the process group: NCCL binds to the current device
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local_rank)
    fckl.load()
    w = synthetic.WORKLOADS[args.workload]
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype="f32", seed=replica_seed(args.seed, rank))
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    host = {
        "H": torch.from_numpy(x["H"]).to(tdt).pin_memory(),
        "W": torch.from_numpy(x["W"]).to(tdt).pin_memory(),
        "idx": torch.from_numpy(x["idx"]).pin_memory(),
        "logp": torch.from_numpy(x["logp"]).pin_memory(),
    }
    del x
    torch.cuda.reset_peak_memory_stats(dev)
    base_alloc = torch.cuda.memory_allocated(dev)
    H, W, idx, logp = (host[k].to(dev) for k in ("H", "W", "idx", "logp"))
    dt = fckl.BF16 if w.dtype == "bf16" else fckl.F32
    # the one call overlaps consecutive chunks with this workspace; the separate calls use
    # its first part (fckl_workspace_bytes)
    ws = fckl.Workspace(w.N, w.d, w.V, w.K, w.chunk, dt, dev, kind="loss_overlap")
    dH = torch.empty_like(H)
    dW = torch.empty(w.V, w.d, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(api):
        if api == "fused":
            loss, _, _, _ = fckl.forward_backward(H, W, idx, logp, w.chunk, ws=ws, stream=stream, dH=dH, dW=dW)
        else:
            loss, lse = fckl.forward(H, W, idx, logp, w.chunk, ws=ws, stream=stream)
            fckl.backward(H, W, idx, logp, lse, w.chunk, ws=ws, stream=stream, dH=dH, dW=dW)
        if args.dp:  # the data-parallel exchange: sum dW and the loss over the ranks
            fckl.allreduce_loss_and_dW(loss, dW)
        return loss

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(api):
        """W warm-up steps, then exactly K timed steps between barriers, with CUDA events on
        the launch stream, the library's per-kernel events and the clock sampler."""
        for _ in range(args.warmup):
            step(api)
        fckl.check(ws)
        barrier()
        clocks = ClockSampler(local_rank)
        clocks.start()
        fckl.profile_enable(True)
        fckl.profile_read()
        launches0 = fckl.launch_count()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step(api)
        e1.record(stream)
        barrier()
        elapsed = e0.elapsed_time(e1)
        n_launch = fckl.launch_count() - launches0
        prof_ = fckl.profile_read()
        fckl.profile_enable(False)
        clk_ = clocks.stop()
        fckl.check(ws)
        return elapsed, n_launch, prof_, clk_

    elapsed_ms, launches, prof, clk = timed(args.api)
    peak_bytes = torch.cuda.max_memory_allocated(dev) - base_alloc
    other = None
    if not args.no_other_path:  # the other structure over the same steps, same inputs
        other_api = "separate" if args.api == "fused" else "fused"
        o_ms, o_launch, o_prof, o_clk = timed(other_api)
        other = (other_api, max_over_ranks(o_ms, dev), o_launch, o_prof, o_clk)

    t_max = max_over_ranks(elapsed_ms, dev)
    cublas = cublas_context(w, dev, H, W, idx, logp) if (rank == 0 and not args.no_cublas) else None

    # end to end through the public API from pinned host buffers: every step copies its inputs
    # from pinned host memory and reads its loss back. The copies of step i+1 run on a second
    # stream into the other of two device input sets while step i computes, as a training
    # loop that prefetches its next batch would; all of them fall inside the timed region.
    e2e = None
    if not args.no_e2e:
        loss_host = torch.empty(args.steps + 1, dtype=torch.float32).pin_memory()
        bufs = [{k: torch.empty_like(host[k], device=dev) for k in host} for _ in range(2)]
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]

        def issue_copy(i):
            j = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(freed[j])  # step i-2, the last reader of set j, is done
                for k in host:
                    bufs[j][k].copy_(host[k], non_blocking=True)
                copied[j].record(copy_stream)

        def e2e_run(n):
            for j in range(2):
                freed[j].record(stream)
            issue_copy(0)
            for i in range(n):
                if i + 1 < n:
                    issue_copy(i + 1)
                j = i % 2
                stream.wait_event(copied[j])
                b = bufs[j]
                if args.api == "fused":
                    loss, _, _, _ = fckl.forward_backward(b["H"], b["W"], b["idx"], b["logp"], w.chunk, ws=ws,
                                                          stream=stream, dH=dH, dW=dW)
                else:
                    loss, lse = fckl.forward(b["H"], b["W"], b["idx"], b["logp"], w.chunk, ws=ws, stream=stream)
                    fckl.backward(b["H"], b["W"], b["idx"], b["logp"], lse, w.chunk, ws=ws, stream=stream, dH=dH,
                                  dW=dW)
                if args.dp:
                    fckl.allreduce_loss_and_dW(loss, dW)
                freed[j].record(stream)
                loss_host[i:i + 1].copy_(loss, non_blocking=True)

        e2e_run(2)
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        copy_stream.wait_event(f0)  # the first copy starts inside the timed region
        e2e_run(args.steps)
        f1.record(stream)
        barrier()
        e2e_ms = max_over_ranks(f0.elapsed_time(f1), dev)
        h2d = sum(host[k].numel() * host[k].element_size() for k in host)
        e2e = {"value": world * w.N * args.steps / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": 4, "ms_per_step": e2e_ms / args.steps,
               "copies": "step i+1's inputs copied on a second stream while step i computes (two device input "
                         "sets); every step's copies and loss read-back inside the timed region"}

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        return 0

    peaks, peak_src = measured_peaks()
    peak_sus = peak_value(peaks, "bf16_tflops_sustained")
    hbm_peak = peak_value(peaks, "hbm_gbs")
    pk_mhz = peak_clock_mhz(peaks)
    head = path_summary(w, args.api, t_max, args.steps, world, prof, peak_sus, peak_src, hbm_peak,
                        (clk or {}).get("sm_mhz"), pk_mhz)
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded generators; no dataset)",
        "config": config_of(w, args.api, world if args.dp else 0),
        "tflops_8NdV": head["tflops_8NdV"], "tflops_8NdV_note": head["tflops_8NdV_note"],
        "tflops_executed": head["tflops_executed"],
        "tflops_executed_frac_of_sustained": head["tflops_executed_frac_of_sustained"],
        "peak_gib": peak_bytes / 2**30,
        "gpu_launches": launches,
        "roofline": head["roofline"],
        "kernel_shares": head["kernel_shares"],
        "kernel_ms_per_step": head["kernel_ms_per_step"],
        "clocks": clk,
        "e2e": e2e,
        "cublas_context": cublas,
    }
    if other is not None:
        o_api, o_ms, o_launch, o_prof, o_clk = other
        o = path_summary(w, o_api, o_ms, args.steps, world, o_prof, peak_sus, peak_src, hbm_peak,
                         (o_clk or {}).get("sm_mhz"), pk_mhz)
        o.update({"api": o_api, "logits": config_of(w, o_api)["logits"], "gpu_launches": o_launch,
                  "clocks": o_clk, "steps": args.steps, "warmup": args.warmup})
        line[o_api] = o
    if not args.no_cpu_baseline and world == 1:
        n_host = min(w.N, 16384)  # the oracle's sample is far smaller; slice the benched inputs
        xs = {"H": host["H"][:n_host].float().numpy(), "idx": host["idx"][:n_host].numpy(),
              "logp": host["logp"][:n_host].numpy()}
        line["cpu_baseline"] = cpu_baseline(w, xs, host["W"].float().numpy())
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def bytes_per_position(w):
    """Device bytes that scale with N: H and dH (d bf16 each), the cache (K int32 + K fp32),
    lse (fp32) and the per-position loss kept in the workspace (fp32)."""
    return 2 * w.d + 2 * w.d + 8 * w.K + 4 + 4


def memory_sweep(args):
    """Peak device memory of one forward + backward for growing N at a fixed chunk."""
    import torch
    import chunked_kl_loss_gb300 as fckl
    fckl.load()
    w = synthetic.WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype="f32", seed=args.seed)
    Hh = torch.from_numpy(x["H"]).to(torch.bfloat16)
    W = torch.from_numpy(x["W"]).to(dev).to(torch.bfloat16)
    idx_h, logp_h = torch.from_numpy(x["idx"]), torch.from_numpy(x["logp"])
    del x
    def peak_of(n, fused, kind="loss"):
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)  # W already resident
        torch.cuda.reset_peak_memory_stats(dev)
        H = Hh[:n].to(dev)
        idx, logp = idx_h[:n].to(dev), logp_h[:n].to(dev)
        ws = fckl.Workspace(n, w.d, w.V, w.K, w.chunk, fckl.BF16, dev, kind=kind)
        if fused:
            fckl.forward_backward(H, W, idx, logp, w.chunk, ws=ws)
        else:
            loss, lse = fckl.forward(H, W, idx, logp, w.chunk, ws=ws)
            fckl.backward(H, W, idx, logp, lse, w.chunk, ws=ws)
        fckl.check(ws)
        return torch.cuda.max_memory_allocated(dev) - base + W.numel() * 2

    def fit(points):
        n_arr = np.array([p[0] for p in points], dtype=np.float64)
        y = np.array([p[1] for p in points], dtype=np.float64)
        b, a = np.polyfit(n_arr, y, 1)
        resid = np.abs(y - (a + b * n_arr)) / y
        return {"points": [{"N": int(n), "peak_gib": pk / 2**30} for n, pk in points],
                "fit_intercept_gib": a / 2**30, "fit_bytes_per_position": b, "max_rel_residual": float(resid.max())}

    sizes = (w.N // 8, w.N // 4, w.N // 2, w.N)
    sep = fit([(n, peak_of(n, False)) for n in sizes])
    fused = fit([(n, peak_of(n, True)) for n in sizes])
    overlap = fit([(n, peak_of(n, True, "loss_overlap")) for n in sizes])
    second_set = (fckl.overlap_workspace_bytes(w.N, w.d, w.V, w.K, w.chunk, fckl.BF16)
                  - fckl.workspace_bytes(w.N, w.d, w.V, w.K, w.chunk, fckl.BF16))
    line = {"metric": "peak device memory of one forward+backward vs N (GiB)", "workload": w.name,
            "chunk": w.chunk, "analytic_bytes_per_position": bytes_per_position(w),
            "separate_calls": sep, "one_call": fused, "one_call_overlap": overlap,
            "second_buffer_set_gib": second_set / 2**30}
    print(json.dumps(line), flush=True)
    return line


def topk_bench(args):
    """Teacher top-K cache build over the workload: teacher hidden states and output matrix
    with the shapes (and generators) of H and W, K cached tokens per position."""
    import torch
    import chunked_kl_loss_gb300 as fckl
    fckl.load()
    w = synthetic.WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    Ht = torch.from_numpy(synthetic.hidden_states(w.N, w.d, args.seed + 10)).to(dev).to(torch.bfloat16)
    Wt = torch.from_numpy(synthetic.output_projection(w.V, w.d, args.seed + 11)).to(dev).to(torch.bfloat16)
    keep = not args.recompute
    ws = fckl.Workspace(w.N, w.d, w.V, w.K, w.chunk, fckl.BF16, dev, kind="topk_overlap" if keep else "topk_min")
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        fckl.teacher_topk(Ht, Wt, w.K, w.chunk, ws=ws, stream=stream, keep_logits=keep)
    fckl.check(ws)
    torch.cuda.synchronize(dev)
    fckl.profile_enable(True)
    fckl.profile_read()
    n0 = fckl.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        fckl.teacher_topk(Ht, Wt, w.K, w.chunk, ws=ws, stream=stream, keep_logits=keep)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    prof = fckl.profile_read()
    fckl.profile_enable(False)
    fckl.check(ws)
    peaks, src = measured_peaks()
    peak = peak_value(peaks, "bf16_tflops_sustained")
    kname, (kms, kn) = max(prof.items(), key=lambda kv: kv[1][0])
    fl = 2.0 * w.N * w.d * w.V * args.steps / kn
    products = 1 if keep else 2
    cfg = config_of(w, "teacher_topk")
    cfg["logits"] = "kept from pass 1" if keep else "projected again in pass 2"
    cfg["workspace"] = ("fckl_topk_overlap_workspace_bytes: the chunk's fp32 logits kept for pass 2, which with the "
                        "selection runs on a second stream beside the next chunk's pass 1" if keep
                        else "fckl_topk_workspace_bytes: the minimum, logits projected twice")
    line = {"metric": "teacher top-K cache build positions/s", "value": w.N / (ms / 1e3),
            "unit": UNIT, "ms_per_step": ms, "steps": args.steps, "warmup": args.warmup,
            "tflops_executed": 2.0 * products * w.N * w.d * w.V / (ms / 1e3) / 1e12, "dtype": "bf16",
            "config": cfg, "gpu_launches": fckl.launch_count() - n0,
            "roofline": {"kernel": kname, "bound": "tensor", "achieved": fl / (kms / kn / 1e3) / 1e12,
                         "peak": peak, "unit": "TFLOP/s", "frac": fl / (kms / kn / 1e3) / 1e12 / peak,
                         "peak_source": f"{src} bf16 sustained"},
            "kernel_shares": {k: round(v[0] / max(1e-9, sum(u[0] for u in prof.values())), 4)
                              for k, v in prof.items() if v[1]}}
    if not args.no_cpu_baseline:
        from oracle import fckl_oracle as orc
        Ws = synthetic.round_bf16(synthetic.output_projection(w.V, w.d, args.seed + 11))

        def timed(n):
            Hs = synthetic.round_bf16(synthetic.hidden_states(n, w.d, args.seed + 10))
            t0 = time.perf_counter()
            orc.teacher_topk(Hs, Ws, w.K, chunk=w.chunk)
            return time.perf_counter() - t0

        n0 = max(8, int(1.0 * 100e9 / (2.0 * w.d * w.V)))  # a short run sets the host's rate
        n = max(8, min(w.N, int(n0 * 15.0 / max(timed(n0), 1e-3))))  # about 15 s
        t = timed(n)
        line["cpu_baseline"] = {"value": n / t, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                                "sample": f"fp64 oracle top-{w.K} cache of the first {n} of {w.N} positions "
                                          f"(full V={w.V}, d={w.d}), {t:.1f} s"}
    print(json.dumps(line), flush=True)
    return line


def main():
    args = parse()
    if args.topk:
        topk_bench(args)
        return 0
    if args.memory_sweep:
        if args.workload == DEFAULT_WORKLOAD:
            args.workload = "n262144_d3072_v128256"
        memory_sweep(args)
        return 0
    if args.positions:
        import dataclasses
        w = synthetic.WORKLOADS[args.workload]
        synthetic.WORKLOADS[args.workload] = dataclasses.replace(w, N=min(args.positions, w.N))
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
