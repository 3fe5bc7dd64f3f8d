"""The one-call path that keeps each chunk's logits (fckl_forward_backward with a "fused"
workspace) against the oracle, and against the recomputing one-call path bit for bit.

Keeping the logits changes where z comes from (the forward's own fp32 tile, stored, instead
of the same product computed again), not what is computed from it, so every output must be
identical to the recomputing path's. The profile counters show which kernels ran, so the
comparison cannot pass by running the same path twice.
"""
import numpy as np
import pytest
import torch

import synthetic
from oracle import fckl_oracle as orc

pytestmark = pytest.mark.gpu

LOSS_RTOL = 1e-3
GRAD_TOL = 2e-2


def to_dev(x, dtype):
    dev = torch.device("cuda")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    H = torch.from_numpy(x["H"]).to(dev).to(tdt)
    W = torch.from_numpy(x["W"]).to(dev).to(tdt)
    idx = torch.from_numpy(np.ascontiguousarray(x["idx"], dtype=np.int32)).to(dev)
    logp = torch.from_numpy(np.ascontiguousarray(x["logp"], dtype=np.float32)).to(dev)
    return H, W, idx, logp


def run_both(fckl, x, chunk, dtype, grad_scale=1.0, weight=None):
    """(kept, recomputed) outputs of forward_backward, each with the kernels it launched."""
    H, W, idx, logp = to_dev(x, dtype)
    N, d = H.shape
    V, K = W.shape[0], idx.shape[1]
    dt = fckl.F32 if dtype == "f32" else fckl.BF16
    wd = torch.from_numpy(weight).cuda() if weight is not None else None
    out = []
    for kind in ("fused", "loss"):
        ws = fckl.Workspace(N, d, V, K, chunk, dt, kind=kind)
        fckl.profile_enable(True)
        fckl.profile_read()
        res = fckl.forward_backward(H, W, idx, logp, chunk, grad_scale=grad_scale, ws=ws, weight=wd,
                                    row_loss=True)
        prof = fckl.profile_read()
        fckl.profile_enable(False)
        assert fckl.check(ws) == fckl.OK
        launched = {k for k, (_, n) in prof.items() if n > 0}
        out.append((res, launched))
    (kept, l_keep), (rec, l_rec) = out
    assert "fwd_logits_keep" in l_keep and "bwd_grad_from_logits" in l_keep
    assert "bwd_logit_grad" not in l_keep and "fwd_logits_lse" not in l_keep
    assert "bwd_logit_grad" in l_rec and "fwd_logits_lse" in l_rec
    assert "bwd_grad_from_logits" not in l_rec and "fwd_logits_keep" not in l_rec
    return kept, rec


def assert_bitwise(kept, rec):
    for a, b in zip(kept, rec):
        assert a.dtype == b.dtype and a.shape == b.shape
        assert torch.equal(a, b)


def assert_oracle(kept, x, chunk, grad_scale=1.0, weight=None):
    loss, lse, rl, dH, dW = kept
    r_loss, r_lse, r_rl = orc.forward(x["H"], x["W"], x["idx"], x["logp"], chunk, weight=weight)
    r_dH, r_dW = orc.backward(x["H"], x["W"], x["idx"], x["logp"], grad_scale, chunk, weight=weight)
    assert abs(float(loss.item()) - r_loss) <= LOSS_RTOL * abs(r_loss)
    g = lse.cpu().numpy().astype(np.float64)
    assert np.abs(g - r_lse).max() <= 1e-3 * (1 + np.abs(r_lse).max())
    g = rl.cpu().numpy().astype(np.float64)
    assert np.abs(g - r_rl).max() <= 1e-3 * (1 + np.abs(r_rl).max())
    g = dH.float().cpu().numpy().astype(np.float64)
    assert np.abs(g - r_dH).max() <= GRAD_TOL * np.abs(r_dH).max()
    g = dW.cpu().numpy().astype(np.float64)
    assert np.abs(g - r_dW).max() <= GRAD_TOL * np.abs(r_dW).max()


@pytest.mark.parametrize("N,d,V,K,chunk", [
    (300, 256, 5000, 40, 128),     # ragged chunk (44 rows) and vocabulary tile
    (513, 320, 4097, 17, 256),     # V % 8 != 0: the last 8 columns of a row are a partial group
    (260, 128, 20000, 100, 260),   # three column segments of the G kernel per position
    (100, 64, 2048, 1024, 64),     # K = 1024: a cache slot in most groups of 8 columns
    (1, 64, 300, 5, 1),            # one position, one-row chunk
])
def test_kept_logits_bf16(fckl, N, d, V, K, chunk):
    x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=N + V)
    kept, rec = run_both(fckl, x, chunk, "bf16")
    assert_bitwise(kept, rec)
    assert_oracle(kept, x, chunk)


def test_kept_logits_fp32_inputs(fckl):
    w = synthetic.WORKLOADS["tiny_n64_d256_v4096"]
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype="f32", seed=41)
    kept, rec = run_both(fckl, x, w.chunk, "f32", grad_scale=0.25)
    assert_bitwise(kept, rec)
    xb = dict(x)
    xb["H"] = synthetic.round_bf16(x["H"])
    xb["W"] = synthetic.round_bf16(x["W"])
    assert_oracle(kept, xb, w.chunk, grad_scale=0.25)


def test_kept_logits_weights_repeats_and_empty_slots(fckl):
    N, d, V, K, chunk = 300, 192, 3000, 30, 128
    x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=42)
    idx = x["idx"].copy()
    logp = x["logp"].copy()
    idx[::3, 1] = idx[::3, 0]        # a repeated id: two slots, two subtractions
    logp[::4, -1] = -np.inf          # an empty slot
    idx[5, :] = idx[5, 0]            # one position whose slots all name one token
    x["idx"], x["logp"] = idx, logp
    wt = np.ones(N, dtype=np.float32)
    wt[::7] = 0.0
    wt[1::5] = 0.5
    kept, rec = run_both(fckl, x, chunk, "bf16", grad_scale=0.5, weight=wt)
    assert_bitwise(kept, rec)
    assert_oracle(kept, x, chunk, grad_scale=0.5, weight=wt)


def test_kept_logits_llama_vocab(fckl):
    """V = 128256 (16 column segments per position), d = 3072, K = 100, two chunks."""
    x = synthetic.make_inputs(320, 3072, 128256, 100, dtype="bf16", seed=43)
    kept, rec = run_both(fckl, x, 256, "bf16")
    assert_bitwise(kept, rec)
    assert_oracle(kept, x, 256)


def test_workspace_kind_decides_the_path(fckl):
    """A caller workspace of the "fused" size keeps the logits; keep_logits=False hands the
    library only the smaller size and it recomputes; outputs equal."""
    x = synthetic.make_inputs(200, 128, 2500, 10, dtype="bf16", seed=44)
    H, W, idx, logp = to_dev(x, "bf16")
    ws = fckl.Workspace(200, 128, 2500, 10, 64, fckl.BF16, kind="fused")
    assert ws.nbytes == fckl.forward_backward_workspace_bytes(200, 128, 2500, 10, 64, fckl.BF16)
    fckl.profile_enable(True)
    fckl.profile_read()
    a = fckl.forward_backward(H, W, idx, logp, 64, ws=ws)
    pa = fckl.profile_read()
    b = fckl.forward_backward(H, W, idx, logp, 64, ws=ws, keep_logits=False)
    pb = fckl.profile_read()
    fckl.profile_enable(False)
    assert fckl.check(ws) == fckl.OK
    assert pa["bwd_grad_from_logits"][1] == 4 and pa["bwd_logit_grad"][1] == 0
    assert pb["bwd_grad_from_logits"][1] == 0 and pb["bwd_logit_grad"][1] == 4
    assert_bitwise(a, b)
