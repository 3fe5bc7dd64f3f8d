"""GPU parity at the full workload sizes, in the launch configuration bench.py times (one
fckl_forward_backward call: each chunk's backward forms G from what its forward kept).

At these sizes the oracle cannot run the whole problem in a test, so it checks what it can
compute one position at a time — lse_n, the per-position loss and the dH row of sampled
positions, each depending only on its own logits row — and the rest through properties that
hold at any size: the vocabulary sum of dW vanishes (the rows of G sum to zero) and the
reported loss is the sum of the per-position losses. At the headline size the separate
forward and backward calls (logits recomputed) must give the same bits.
"""
import numpy as np
import pytest
import torch

import synthetic
from oracle import fckl_oracle as orc

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BF16_WORKLOADS = ["n8192_d3072_v128256", "n32768_d3072_v128256", "n65536_d2880_v201088",
                  "n262144_d3072_v128256"]


@pytest.mark.parametrize("name", BF16_WORKLOADS)
def test_full_size_sampled_rows_and_properties(fckl, name):
    w = synthetic.WORKLOADS[name]
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype="f32", seed=0)
    dev = torch.device("cuda")
    H = torch.from_numpy(x["H"]).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(x["W"]).to(dev).to(torch.bfloat16)
    idx = torch.from_numpy(x["idx"]).to(dev)
    logp = torch.from_numpy(x["logp"]).to(dev)
    ws = fckl.Workspace(w.N, w.d, w.V, w.K, w.chunk, fckl.BF16)
    loss, lse, rl, dH, dW = fckl.forward_backward(H, W, idx, logp, w.chunk, ws=ws, row_loss=True)
    assert fckl.check(ws) == fckl.OK
    if name == "n32768_d3072_v128256":
        ws2 = fckl.Workspace(w.N, w.d, w.V, w.K, w.chunk, fckl.BF16)
        loss2, lse2, rl2 = fckl.forward(H, W, idx, logp, w.chunk, ws=ws2, row_loss=True)
        dH2, dW2 = fckl.backward(H, W, idx, logp, lse2, w.chunk, ws=ws2)
        assert fckl.check(ws2) == fckl.OK
        for a, b in ((loss, loss2), (lse, lse2), (rl, rl2), (dH, dH2), (dW, dW2)):
            assert torch.equal(a, b)
        del ws2, loss2, lse2, rl2, dH2, dW2

    rng = np.random.default_rng(123)
    rows = np.unique(np.concatenate([[0, w.chunk - 1, w.chunk, w.N - 1], rng.integers(0, w.N, 4)]))
    Hs = H[torch.from_numpy(rows).to(dev)].float().cpu().numpy()
    Wq = W.float().cpu().numpy()
    r_lse, r_rl, r_dH = orc.rows(Hs, Wq, x["idx"][rows], x["logp"][rows], np.arange(len(rows)))
    g_lse = lse.cpu().numpy()[rows]
    g_rl = rl.cpu().numpy()[rows]
    g_dH = dH[torch.from_numpy(rows).to(dev)].float().cpu().numpy()
    assert np.abs(g_lse - r_lse).max() <= 1e-3 * (1 + np.abs(r_lse).max())
    assert np.abs(g_rl - r_rl).max() <= 1e-3 * (1 + np.abs(r_rl).max())
    assert np.abs(g_dH - r_dH).max() <= 2e-2 * np.abs(r_dH).max()

    total = rl.double().sum().item()
    assert abs(loss.item() - total) <= 1e-5 * abs(total)

    # sum_v dW[v, j] = sum_n H_nj sum_v G_nv = 0 up to the bf16 rounding of G. Rounding to
    # nearest with 8 significant bits leaves an unbiased relative error whose standard
    # deviation is at most 2^-8/sqrt(3) (a value at the bottom of its binade), so column j of
    # the vocabulary sum has standard deviation at most
    #   sigma_j = 2^-8/sqrt(3) sqrt(sum_n H_nj^2 |G_n|^2),  |G_n|^2 ~ sum_k p_nk^2
    # (the cached entries dominate the norm of G's rows).
    col = dW.double().sum(0).cpu().numpy()
    p2 = torch.from_numpy((np.exp(x["logp"].astype(np.float64)) ** 2).sum(1)).to(dev)
    sig = (2.0 ** -8 / np.sqrt(3.0)) * torch.sqrt((H.double() ** 2 * p2[:, None]).sum(0)).cpu().numpy()
    assert np.all(np.abs(col) <= 6.0 * sig + 1e-4 * dW.abs().max().item()), (np.abs(col) / sig).max()
