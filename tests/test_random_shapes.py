"""A seeded sweep of random problem shapes, GPU against the fp64 oracle.

Each shape draws N, d (a multiple of 8), V, K <= V, the chunk and optional position weights
from a fixed seed, so every run checks the same cases: ragged tails in every dimension, chunks
smaller and larger than the 256-row tile, fewer vocabulary tiles than K, and so on.
"""
import numpy as np
import pytest
import torch

import synthetic
from oracle import fckl_oracle as orc

pytestmark = pytest.mark.gpu


def loss_shapes():
    rng = np.random.default_rng(2026)
    out = []
    for i in range(16):
        N = int(rng.integers(1, 700))
        d = 8 * int(rng.integers(1, 80))
        V = int(rng.integers(8, 6000))
        K = int(rng.integers(1, min(V, 120) + 1))
        chunk = int(rng.integers(1, 800))
        weighted = bool(rng.integers(0, 2))
        out.append((i, N, d, V, K, chunk, weighted))
    return out


@pytest.mark.parametrize("i,N,d,V,K,chunk,weighted", loss_shapes())
def test_random_shape_loss(fckl, i, N, d, V, K, chunk, weighted):
    x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=100 + i)
    wt = None
    if weighted:
        wt = np.random.default_rng(200 + i).uniform(0.0, 2.0, size=N).astype(np.float32)
        wt[::5] = 0.0
    dev = torch.device("cuda")
    H = torch.from_numpy(x["H"]).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(x["W"]).to(dev).to(torch.bfloat16)
    idx = torch.from_numpy(x["idx"]).to(dev)
    logp = torch.from_numpy(x["logp"]).to(dev)
    wd = torch.from_numpy(wt).to(dev) if weighted else None
    ws = fckl.Workspace(N, d, V, K, chunk, fckl.BF16)
    loss, lse, rl, dH, dW = fckl.forward_backward(H, W, idx, logp, chunk, grad_scale=0.5, ws=ws, weight=wd,
                                                  row_loss=True)
    assert fckl.check(ws) == fckl.OK
    r_loss, r_lse, r_rl = orc.forward(x["H"], x["W"], x["idx"], x["logp"], chunk, weight=wt)
    r_dH, r_dW = orc.backward(x["H"], x["W"], x["idx"], x["logp"], 0.5, chunk, weight=wt)
    assert abs(float(loss.item()) - r_loss) <= 1e-3 * max(abs(r_loss), 1e-6 * N)
    assert np.abs(lse.cpu().numpy() - r_lse).max() <= 1e-3 * (1 + np.abs(r_lse).max())
    assert np.abs(rl.cpu().numpy() - r_rl).max() <= 1e-3 * (1 + np.abs(r_rl).max())
    if np.abs(r_dH).max() > 0:
        assert np.abs(dH.float().cpu().numpy() - r_dH).max() <= 2e-2 * np.abs(r_dH).max()
        assert np.abs(dW.cpu().numpy() - r_dW).max() <= 2e-2 * np.abs(r_dW).max()


def topk_shapes():
    rng = np.random.default_rng(2027)
    out = []
    for i in range(6):
        N = int(rng.integers(1, 400))
        d = 8 * int(rng.integers(1, 50))
        V = int(rng.integers(16, 5000))
        K = int(rng.integers(1, min(V, 120) + 1))
        chunk = int(rng.integers(1, 500))
        out.append((i, N, d, V, K, chunk))
    return out


@pytest.mark.parametrize("i,N,d,V,K,chunk", topk_shapes())
def test_random_shape_topk(fckl, i, N, d, V, K, chunk):
    from test_topk import run_topk, assert_topk_parity
    rng = np.random.default_rng(300 + i)
    Ht = synthetic.round_bf16(rng.standard_normal((N, d), dtype=np.float32))
    Wt = synthetic.round_bf16(rng.standard_normal((V, d), dtype=np.float32) * 2.0 / np.sqrt(d))
    idx, logp = run_topk(fckl, Ht, Wt, K, chunk)
    assert_topk_parity(idx, logp, Ht, Wt, K)
