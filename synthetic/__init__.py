"""Seeded synthetic inputs for the fused, chunked top-K KL distillation loss.

This module only draws random numbers. It holds none of the loss arithmetic, so
both the CUDA path's tests and the fp64 oracle can take their inputs from here
without sharing any of the method's code.

What the inputs stand for
-------------------------
* ``H [N, d]``: student hidden states fed to the output projection, one row per
  sequence position ("Hugging Face：让知识蒸馏廉价到可大规模运行", paragraph
  "Fused, chunked KL loss": the chunk's hidden states are projected to logits).
* ``W [V, d]``: the student's output projection (same paragraph).
* ``idx [N, K]`` int32 and ``logp [N, K]`` fp32: the offline teacher cache, the
  K most probable tokens of every position and their log-probabilities, kept
  without renormalising the truncated distribution ("Chunkovaná KL strata ...",
  section "Čo dopĺňajú podrobnejšie experimenty"; K = 100 in "Destilación de
  LLMs: Multiverse Computing reduce memoria 15× con 1 GPU", section "Dos
  innovaciones que cambian las reglas del juego").

No dataset, model or teacher is available, so every tensor is synthetic:

* ``H ~ N(0, 1)`` and ``W ~ N(0, 1/d)``, drawn in fp32; for bf16 workloads they
  are then rounded to bf16 (round to nearest even) and the oracle receives the
  rounded values, widened exactly.
* teacher, per row: K distinct token ids drawn uniformly from ``[0, V)``, ids in
  draw order, unsorted. When K*K <= V all rows are drawn with replacement and a row
  with a repeated id is drawn again whole (rare by the birthday bound); otherwise
  each row is drawn without replacement,
  scores ``t ~ N(0, 2^2)`` sorted descending, a kept mass ``S ~ U(0.85, 0.99)``
  and ``logp = log(S * softmax(t))`` computed in fp64 and stored as fp32.

Streams: ``numpy.random.Generator(PCG64(seed + j))`` with ``j = 0`` for H,
``1`` for W and ``2`` for the teacher cache. PCG64 gives the same numbers on
x86-64 and aarch64.
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = ["Workload", "WORKLOADS", "hidden_states", "output_projection",
           "teacher_cache", "make_inputs", "round_bf16", "round_tf32"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One problem shape: N positions, hidden size d, vocabulary V, top-K, chunk rows."""
    name: str
    N: int
    d: int
    V: int
    K: int
    chunk: int
    dtype: str  # "f32" or "bf16": storage type of H, W and dH

    def flops(self) -> float:
        """Tensor-core work of one forward+backward: four N x d x V products."""
        return 8.0 * self.N * self.d * self.V


# The five workloads. The pages measure a loss-only "toy output-projection
# network" at 32K and 256K positions ("扩展到长上下文") and distil at 8K
# ("这在实践中改变了什么"); they give no hidden size or vocabulary for the toy,
# so the Llama-3 vocabulary (128256, d=3072) and the gpt-oss vocabulary (201088,
# named in "为什么蒸馏恢复代价高昂") with d=2880 stand in.
WORKLOADS = {
    w.name: w for w in (
        Workload("tiny_n64_d256_v4096", 64, 256, 4096, 16, 16, "f32"),
        Workload("n8192_d3072_v128256", 8192, 3072, 128256, 100, 1024, "bf16"),
        Workload("n32768_d3072_v128256", 32768, 3072, 128256, 100, 2048, "bf16"),
        Workload("n65536_d2880_v201088", 65536, 2880, 201088, 100, 2048, "bf16"),
        Workload("n262144_d3072_v128256", 262144, 3072, 128256, 100, 4096, "bf16"),
    )
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def hidden_states(N: int, d: int, seed: int) -> np.ndarray:
    """H ~ N(0, 1), fp32, shape [N, d]."""
    return _rng(seed).standard_normal((N, d), dtype=np.float32)


def output_projection(V: int, d: int, seed: int) -> np.ndarray:
    """W ~ N(0, 1/d), fp32, shape [V, d]."""
    w = _rng(seed).standard_normal((V, d), dtype=np.float32)
    w *= np.float32(1.0 / np.sqrt(d))
    return w


def teacher_cache(N: int, V: int, K: int, seed: int,
                  s_lo: float = 0.85, s_hi: float = 0.99):
    """Top-K teacher cache: (idx int32 [N, K], logp fp32 [N, K]).

    Ids are distinct within a row and unsorted; logp is sorted descending and
    sums (after exp) to the row's kept mass S < 1.
    """
    if K > V:
        raise ValueError("K must not exceed V")
    rng = _rng(seed)
    if K * K <= V:
        idx = rng.integers(0, V, size=(N, K), dtype=np.int64)
        while True:
            s = np.sort(idx, axis=1)
            dup = (s[:, 1:] == s[:, :-1]).any(axis=1) if K > 1 else np.zeros(N, bool)
            n_dup = int(dup.sum())
            if n_dup == 0:
                break
            idx[dup] = rng.integers(0, V, size=(n_dup, K), dtype=np.int64)
    else:
        idx = np.stack([rng.choice(V, size=K, replace=False) for _ in range(N)]).astype(np.int64)
    t = rng.standard_normal((N, K)) * 2.0
    t = -np.sort(-t, axis=1)
    S = rng.uniform(s_lo, s_hi, size=(N, 1))
    t = t - t.max(axis=1, keepdims=True)
    log_soft = t - np.log(np.exp(t).sum(axis=1, keepdims=True))
    logp = np.log(S) + log_soft
    return idx.astype(np.int32), logp.astype(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even) and return them as fp32."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float32).numpy()


def round_tf32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to tf32 (10 explicit mantissa bits) to nearest, ties away from zero,
    and return them as fp32 with the low 13 bits zero: the values a tf32 product reads. Adding
    half a tf32 unit (bit 12) to the magnitude bits and clearing the 13 low bits rounds the
    magnitude; a carry into the exponent is the correct rounding up. Finite inputs."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x1000) & 0xFFFFE000).astype(np.uint32).view(np.float32)


def make_inputs(N: int, d: int, V: int, K: int, dtype: str = "bf16", seed: int = 0):
    """All inputs of one problem as numpy arrays.

    Returns a dict with ``H`` and ``W`` as fp32 arrays holding exactly the values
    the device will see (already rounded to bf16 when ``dtype == "bf16"``),
    ``idx`` int32 and ``logp`` fp32.
    """
    H = hidden_states(N, d, seed + 0)
    W = output_projection(V, d, seed + 1)
    idx, logp = teacher_cache(N, V, K, seed + 2)
    if dtype == "bf16":
        H = round_bf16(H)
        W = round_bf16(W)
    elif dtype != "f32":
        raise ValueError(f"unknown dtype {dtype!r}")
    return {"H": H, "W": W, "idx": idx, "logp": logp}
