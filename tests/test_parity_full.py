"""GPU parity at the full workload sizes, in the launch configuration bench.py times (one
fckl_forward_backward call per step with the overlap workspace: the workload's chunk, every
chunk's forward, G pass (beside the next chunk's forward on the second stream), dH product and
dW reduce-add, the same dH split).

The oracle cannot redo a whole workload inside a test, so each workload is checked three ways:

* Unweighted run. Positions sampled across chunks are checked one by one (lse_n, the
  per-position loss and the dH row each depend on that position alone). The total loss and
  the sum of lse are checked against tests/golden/full_loss.json, which the fp64 oracle wrote
  over every position of the workload (tests/golden/make_full_loss.py, oracle and generators
  only). The vocabulary sum of dW must vanish, and the loss must equal the sum of the
  per-position losses.
* Weighted run, same launch configuration. Position weights are nonzero on a set of positions
  that includes the first and last row of every chunk plus random rows, and 0 elsewhere. The
  loss, dH and dW of that run involve only those positions, so the oracle computes them
  exactly: the weighted loss, every dH row (the zero-weight rows must be exactly 0) and all of
  dW [V, d], element by element. Every chunk's reduce-add into dW contributes to what is
  compared.
* At the headline size, the separate forward and backward calls (logits recomputed) and the
  one call with the minimum workspace (chunks in sequence) give the same bits as the
  overlapped one call.

The pages state that the dense, forward-chunked and fused variants compute the same loss
("Hugging Face：让知识蒸馏廉价到可大规模运行", paragraph "Fused, chunked KL loss"); these
tests hold the fused kernels to the dense definition at the sizes that are benchmarked.
Tolerances are those of the method for bf16 inputs: loss relative 1e-3, dH and dW max-abs
2e-2 x max|ref|.
"""
import json
import os

import numpy as np
import pytest
import torch

import synthetic
from oracle import fckl_oracle as orc

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BF16_WORKLOADS = ["n8192_d3072_v128256", "n32768_d3072_v128256", "n65536_d2880_v201088",
                  "n262144_d3072_v128256"]
LOSS_RTOL = 1e-3
GRAD_TOL = 2e-2
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "full_loss.json")


def _golden(name):
    with open(GOLDEN) as f:
        return json.load(f)[name]


def _fingerprint_matches(x, fp):
    """The inputs are the ones the golden file was written for (same generators, same seed)."""
    if int(x["idx"].astype(np.int64).sum()) != fp["idx_sum"]:
        return False
    for key, got in (("H_sum", x["H"].astype(np.float64).sum()),
                     ("H_abs_sum", np.abs(x["H"].astype(np.float64)).sum()),
                     ("W_abs_sum", np.abs(x["W"].astype(np.float64)).sum()),
                     ("logp_sum", x["logp"].astype(np.float64).sum())):
        if abs(float(got) - fp[key]) > 1e-9 * (1.0 + abs(fp[key])):
            return False
    return True


def _weighted_positions(w, rng):
    """First and last row of every chunk plus 48 random positions, with weights in [0.5, 2)."""
    starts = np.arange(0, w.N, w.chunk)
    ends = np.minimum(starts + w.chunk, w.N) - 1
    sel = np.unique(np.concatenate([starts, ends, rng.integers(0, w.N, 48)]))
    return sel, rng.uniform(0.5, 2.0, size=len(sel)).astype(np.float32)


def _max_abs_err_rows(got_dev, ref, block=8192):
    """max |got - ref| over a [rows, cols] device array against a host fp64 array, in row blocks
    (the full difference of a 201088 x 2880 dW would not fit comfortably on the host)."""
    err = 0.0
    for r0 in range(0, ref.shape[0], block):
        g = got_dev[r0:r0 + block].double().cpu().numpy()
        err = max(err, float(np.abs(g - ref[r0:r0 + block]).max()))
    return err


@pytest.mark.parametrize("name", BF16_WORKLOADS)
def test_full_size_against_oracle(fckl, name):
    w = synthetic.WORKLOADS[name]
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype="f32", seed=0)
    dev = torch.device("cuda")
    H = torch.from_numpy(x["H"]).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(x["W"]).to(dev).to(torch.bfloat16)
    idx = torch.from_numpy(x["idx"]).to(dev)
    logp = torch.from_numpy(x["logp"]).to(dev)
    Hq = synthetic.round_bf16(x["H"])  # the values the device sees, widened exactly
    Wq = synthetic.round_bf16(x["W"])
    ws = fckl.Workspace(w.N, w.d, w.V, w.K, w.chunk, fckl.BF16, kind="loss_overlap")

    # ---- unweighted run: sampled positions, golden total loss, properties
    loss, lse, rl, dH, dW = fckl.forward_backward(H, W, idx, logp, w.chunk, ws=ws, row_loss=True)
    assert fckl.check(ws) == fckl.OK
    if name == "n32768_d3072_v128256":
        ws2 = fckl.Workspace(w.N, w.d, w.V, w.K, w.chunk, fckl.BF16)
        loss2, lse2, rl2 = fckl.forward(H, W, idx, logp, w.chunk, ws=ws2, row_loss=True)
        dH2, dW2 = fckl.backward(H, W, idx, logp, lse2, w.chunk, ws=ws2)
        assert fckl.check(ws2) == fckl.OK
        for a, b in ((loss, loss2), (lse, lse2), (rl, rl2), (dH, dH2), (dW, dW2)):
            assert torch.equal(a, b)
        loss2, lse2, rl2, dH2, dW2 = fckl.forward_backward(H, W, idx, logp, w.chunk, ws=ws2, row_loss=True)
        assert fckl.check(ws2) == fckl.OK
        for a, b in ((loss, loss2), (lse, lse2), (rl, rl2), (dH, dH2), (dW, dW2)):
            assert torch.equal(a, b)
        del ws2, loss2, lse2, rl2, dH2, dW2

    rng = np.random.default_rng(123)
    rows = np.unique(np.concatenate([[0, w.chunk - 1, w.chunk, w.N - 1], rng.integers(0, w.N, 4)]))
    r_lse, r_rl, r_dH = orc.rows(Hq[rows], Wq, x["idx"][rows], x["logp"][rows], np.arange(len(rows)))
    g_lse = lse.cpu().numpy()[rows]
    g_rl = rl.cpu().numpy()[rows]
    g_dH = dH[torch.from_numpy(rows).to(dev)].float().cpu().numpy()
    assert np.abs(g_lse - r_lse).max() <= 1e-3 * (1 + np.abs(r_lse).max())
    assert np.abs(g_rl - r_rl).max() <= 1e-3 * (1 + np.abs(r_rl).max())
    assert np.abs(g_dH - r_dH).max() <= GRAD_TOL * np.abs(r_dH).max()

    gold = _golden(name)
    assert (gold["N"], gold["d"], gold["V"], gold["K"]) == (w.N, w.d, w.V, w.K)
    assert _fingerprint_matches({"H": Hq, "W": Wq, "idx": x["idx"], "logp": x["logp"]}, gold["inputs"]), \
        "the seeded generators gave other inputs than the ones the golden file was written for"
    got = float(loss.item())
    assert abs(got - gold["loss"]) <= LOSS_RTOL * abs(gold["loss"]), (got, gold["loss"])
    lse_sum = lse.double().sum().item()
    assert abs(lse_sum - gold["lse_sum"]) <= 1e-4 * abs(gold["lse_sum"]), (lse_sum, gold["lse_sum"])

    total = rl.double().sum().item()
    assert abs(got - total) <= 1e-5 * abs(total)

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
    del loss, lse, rl, dH, dW, col, p2, sig

    # ---- weighted run, same launch configuration: exact oracle for loss, dH and all of dW
    sel, wsel = _weighted_positions(w, np.random.default_rng(7))
    wt = np.zeros(w.N, dtype=np.float32)
    wt[sel] = wsel
    wt_dev = torch.from_numpy(wt).to(dev)
    loss, lse, dH, dW = fckl.forward_backward(H, W, idx, logp, w.chunk, ws=ws, weight=wt_dev)
    assert fckl.check(ws) == fckl.OK
    o_loss, o_lse, _ = orc.forward(Hq[sel], Wq, x["idx"][sel], x["logp"][sel], weight=wsel)
    o_dH, o_dW = orc.backward(Hq[sel], Wq, x["idx"][sel], x["logp"][sel], 1.0, weight=wsel)

    got = float(loss.item())
    assert abs(got - o_loss) <= LOSS_RTOL * abs(o_loss), (got, o_loss)
    g_lse = lse[torch.from_numpy(sel).to(dev)].cpu().numpy()
    assert np.abs(g_lse - o_lse).max() <= 1e-3 * (1 + np.abs(o_lse).max())

    sel_dev = torch.from_numpy(sel).to(dev)
    g_dH = dH[sel_dev].float().cpu().numpy()
    assert np.abs(g_dH - o_dH).max() <= GRAD_TOL * np.abs(o_dH).max()
    mask = torch.ones(w.N, dtype=torch.bool, device=dev)
    mask[sel_dev] = False
    assert int(torch.count_nonzero(dH[mask]).item()) == 0  # zero weight: exactly zero rows

    e_dW = _max_abs_err_rows(dW, o_dW)
    assert e_dW <= GRAD_TOL * np.abs(o_dW).max(), (e_dW, np.abs(o_dW).max())
