"""The one call (fckl_forward_backward), whose backward forms G in place from what each
chunk's forward kept in the gradient slab (fp16 exp(z - tile max)), against the oracle, and
against the separate calls (fckl_forward, then fckl_backward recomputing the logits) bit for
bit.

Both paths take the same steps from the same logits (tile maximum, fp16 e, the same products
and roundings); only where the logits come from differs (the forward's own tile, kept, or the
same product computed again), so every output must be identical. The profile counters show
which kernels ran, so the comparison cannot pass by running the same path twice.
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
    """(kept, recomputed) outputs: the one call, and the separate calls; each with the kernels
    it launched."""
    H, W, idx, logp = to_dev(x, dtype)
    N, d = H.shape
    V, K = W.shape[0], idx.shape[1]
    dt = fckl.F32 if dtype == "f32" else fckl.BF16
    wd = torch.from_numpy(weight).cuda() if weight is not None else None
    out = []
    for one_call in (True, False):
        ws = fckl.Workspace(N, d, V, K, chunk, dt)
        fckl.profile_enable(True)
        fckl.profile_read()
        if one_call:
            res = fckl.forward_backward(H, W, idx, logp, chunk, grad_scale=grad_scale, ws=ws, weight=wd,
                                        row_loss=True)
        else:
            loss, lse, rl = fckl.forward(H, W, idx, logp, chunk, ws=ws, weight=wd, row_loss=True)
            dH, dW = fckl.backward(H, W, idx, logp, lse, chunk, grad_scale=grad_scale, ws=ws, weight=wd)
            res = (loss, lse, rl, dH, dW)
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
    (40, 8, 16, 16, 16),           # smallest d, V below one tile and one 16-column step, K = V
    (33, 64, 8, 8, 16),            # V = K = 8: the whole vocabulary cached
    (64, 8192, 2048, 16, 64),      # wide d: 128 K-blocks per logits tile, 32 N-tiles in dH and dW
])
def test_kept_logits_bf16(fckl, N, d, V, K, chunk):
    x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=N + V)
    kept, rec = run_both(fckl, x, chunk, "bf16")
    assert_bitwise(kept, rec)
    assert_oracle(kept, x, chunk)


@pytest.mark.parametrize("weighted", [False, True])
def test_kept_logits_fp32_inputs(fckl, weighted):
    w = synthetic.WORKLOADS["tiny_n64_d256_v4096"]
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype="f32", seed=41)
    wt = None
    if weighted:
        wt = np.linspace(0.0, 2.0, w.N).astype(np.float32)
        wt[::9] = 0.0
    kept, rec = run_both(fckl, x, w.chunk, "f32", grad_scale=0.25, weight=wt)
    assert_bitwise(kept, rec)
    xb = dict(x)
    xb["H"] = synthetic.round_bf16(x["H"])
    xb["W"] = synthetic.round_bf16(x["W"])
    assert_oracle(kept, xb, w.chunk, grad_scale=0.25, weight=wt)


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


def test_one_call_needs_no_workspace_beyond_the_slab(fckl):
    """The kept values live in the gradient slab: a workspace of fckl_workspace_bytes runs the
    one call, and one byte less is refused before anything is launched."""
    x = synthetic.make_inputs(200, 128, 2500, 10, dtype="bf16", seed=44)
    H, W, idx, logp = to_dev(x, "bf16")
    ws = fckl.Workspace(200, 128, 2500, 10, 64, fckl.BF16)
    assert ws.nbytes == fckl.workspace_bytes(200, 128, 2500, 10, 64, fckl.BF16)
    fckl.profile_enable(True)
    fckl.profile_read()
    fckl.forward_backward(H, W, idx, logp, 64, ws=ws)
    prof = fckl.profile_read()
    fckl.profile_enable(False)
    assert fckl.check(ws) == fckl.OK
    assert prof["bwd_grad_from_logits"][1] == 4 and prof["bwd_logit_grad"][1] == 0

    class Short:
        tensor = ws.tensor
        nbytes = ws.nbytes - 1
        ptr = ws.ptr
    n0 = fckl.launch_count()
    with pytest.raises(fckl.FcklError):
        fckl.forward_backward(H, W, idx, logp, 64, ws=Short())
    assert fckl.launch_count() == n0


def test_one_token_vocabulary(fckl):
    """V = K = 1: the softmax is 1, S = p, so the loss is sum_n p_n logp_n and G vanishes. On the
    device exp(m - lse) is 1 only to within its rounding (~1e-7), so the gradients are bounded
    absolutely rather than relative to an all-zero reference; the two paths still agree bit for
    bit."""
    x = synthetic.make_inputs(8, 64, 1, 1, dtype="bf16", seed=9)
    kept, rec = run_both(fckl, x, 8, "bf16")
    assert_bitwise(kept, rec)
    loss, lse, rl, dH, dW = kept
    r_loss, r_lse, r_rl = orc.forward(x["H"], x["W"], x["idx"], x["logp"], 8)
    assert abs(float(loss.item()) - r_loss) <= LOSS_RTOL * abs(r_loss)
    assert np.abs(lse.cpu().numpy() - r_lse).max() <= 1e-3 * (1 + np.abs(r_lse).max())
    assert dH.float().abs().max().item() <= 1e-5 and dW.abs().max().item() <= 1e-5
