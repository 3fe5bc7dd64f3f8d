"""More than 2^31 elements: H and dH of 524,800 x 4096 (2,149,580,800 elements each).

The configured workloads stay below 2^31 elements per array; the interface accepts N up to
2^40. Here the rows from 524,288 on start past element 2^31 of H and dH, so any 32-bit
element offset on the way (host pointer arithmetic per chunk, the per-position arrays, the
loss sum) would show up as wrong rows there. The vocabulary is small (V = 256) to keep the
oracle's full dW affordable: it is summed over blocks of positions in fp64, each block's
contribution from the oracle's own backward. Sampled positions on both sides of the 2^31
boundary are checked one by one.
"""
import numpy as np
import pytest
import torch

import synthetic
from oracle import fckl_oracle as orc

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N, D, V, K, CHUNK = 524_800, 4096, 256, 8, 65536
BLOCK = 32768


def test_more_than_2_31_elements_in_H_and_dH(fckl):
    assert N * D > 2**31
    x = synthetic.make_inputs(N, D, V, K, dtype="f32", seed=51)
    dev = torch.device("cuda")
    H = torch.from_numpy(x["H"]).to(dev).to(torch.bfloat16)
    del x["H"]
    W = torch.from_numpy(x["W"]).to(dev).to(torch.bfloat16)
    idx = torch.from_numpy(x["idx"]).to(dev)
    logp = torch.from_numpy(x["logp"]).to(dev)
    ws = fckl.Workspace(N, D, V, K, CHUNK, fckl.BF16)
    loss, lse, rl, dH, dW = fckl.forward_backward(H, W, idx, logp, CHUNK, ws=ws, row_loss=True)
    assert fckl.check(ws) == fckl.OK

    Wq = W.double().cpu().numpy()
    first_past = 2**31 // D  # first row that starts at or past element 2^31
    rows = np.array([0, CHUNK - 1, CHUNK, first_past - 1, first_past, first_past + 1, N - CHUNK, N - 1])
    rows = np.unique(np.concatenate([rows, np.random.default_rng(52).integers(0, N, 8)]))
    sel = torch.from_numpy(rows).to(dev)
    Hs = H[sel].double().cpu().numpy()
    r_lse, r_rl, r_dH = orc.rows(Hs, Wq, x["idx"][rows], x["logp"][rows], np.arange(len(rows)))
    g_lse = lse[sel].double().cpu().numpy()
    g_rl = rl[sel].double().cpu().numpy()
    g_dH = dH[sel].double().cpu().numpy()
    assert np.abs(g_lse - r_lse).max() <= 1e-3 * (1 + np.abs(r_lse).max())
    assert np.abs(g_rl - r_rl).max() <= 1e-3 * (1 + np.abs(r_rl).max())
    assert np.abs(g_dH - r_dH).max() <= 2e-2 * np.abs(r_dH).max()

    total = rl.double().sum().item()
    assert abs(loss.item() - total) <= 1e-5 * abs(total)

    r_dW = np.zeros((V, D))
    for a in range(0, N, BLOCK):
        b = min(N, a + BLOCK)
        Hb = H[a:b].double().cpu().numpy()
        r_dW += orc.backward(Hb, Wq, x["idx"][a:b], x["logp"][a:b], 1.0)[1]
    g_dW = dW.double().cpu().numpy()
    assert np.abs(g_dW - r_dW).max() <= 2e-2 * np.abs(r_dW).max()
