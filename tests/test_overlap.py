"""The one call with the overlap workspace (fckl_overlap_workspace_bytes): each chunk's G is
formed on a second stream while the next chunk's forward runs on the caller's stream.

Every kernel computes what it does in the sequential order from the same inputs, so the
outputs must be bitwise those of the minimum workspace (chunks one after another), which the
other parity tests pin to the oracle; one case is also compared with the oracle directly. The
profile counters show that the second buffer set was used (the G pass ran once per chunk, one
block per SM beside the next forward for all but the last chunk: the side instance's counter).
The library overlaps only where it pays (a long enough projection per chunk, d >= 2048); the
small shapes here force it with FCKL_OVERLAP=1, and test_overlap_rule checks the automatic
choice.
"""
import numpy as np
import pytest
import torch

import synthetic
from oracle import fckl_oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def forced_overlap(monkeypatch):
    monkeypatch.setenv("FCKL_OVERLAP", "1")


def to_dev(x, dtype):
    dev = torch.device("cuda")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    H = torch.from_numpy(x["H"]).to(dev).to(tdt)
    W = torch.from_numpy(x["W"]).to(dev).to(tdt)
    idx = torch.from_numpy(np.ascontiguousarray(x["idx"], dtype=np.int32)).to(dev)
    logp = torch.from_numpy(np.ascontiguousarray(x["logp"], dtype=np.float32)).to(dev)
    return H, W, idx, logp


def one_call(fckl, t, chunk, kind, dt, weight=None, grad_scale=1.0):
    H, W, idx, logp = t
    N, d = H.shape
    V, K = W.shape[0], idx.shape[1]
    ws = fckl.Workspace(N, d, V, K, chunk, dt, kind=kind)
    fckl.profile_enable(True)
    fckl.profile_read()
    out = fckl.forward_backward(H, W, idx, logp, chunk, grad_scale=grad_scale, ws=ws, weight=weight,
                                row_loss=True)
    torch.cuda.synchronize()
    prof = fckl.profile_read()
    fckl.profile_enable(False)
    assert fckl.check(ws) == fckl.OK
    return [o.clone() for o in out], prof, ws.nbytes


@pytest.mark.parametrize("N,d,V,K,chunk,dtype", [
    (600, 256, 5000, 40, 128, "bf16"),    # 5 chunks, the last one ragged (88 rows)
    (1000, 128, 3001, 17, 256, "bf16"),   # V % 8 != 0, 4 chunks
    (513, 64, 777, 5, 512, "bf16"),       # two chunks: 512 rows and 1
    (300, 256, 4096, 16, 64, "f32"),      # fp32 inputs: tf32 logits, a bf16 H copy per buffer set
    (2048, 512, 8192, 64, 1024, "bf16"),  # two full chunks of 4 M-blocks
    (1100, 64, 300, 5, 100, "bf16"),      # 11 chunks, V below two vocabulary tiles
    (100, 64, 1000, 8, 100, "bf16"),      # one chunk: no second set, the same workspace
    (5, 64, 300, 5, 1, "bf16"),           # five one-row chunks: the buffer sets alternate every row
    (33, 8, 100, 100, 16, "bf16"),        # d = 8, V below one tile, K = V; last chunk one row
    (257, 128, 2049, 1024, 128, "bf16"),  # K = 1024 slots; last chunk one row; V % 8 = 1
    (700, 264, 3000, 30, 300, "f32"),     # fp32, d not a multiple of 64, ragged chunks of 300
])
def test_overlap_is_bitwise_the_sequential_one_call(fckl, N, d, V, K, chunk, dtype):
    x = synthetic.make_inputs(N, d, V, K, dtype=dtype, seed=N + 7 * V)
    t = to_dev(x, dtype)
    dt = fckl.F32 if dtype == "f32" else fckl.BF16
    weight = torch.from_numpy(np.random.default_rng(N).random(N).astype(np.float32)).cuda()
    seq, p_seq, n_seq = one_call(fckl, t, chunk, "loss", dt, weight, 0.25)
    ovl, p_ovl, n_ovl = one_call(fckl, t, chunk, "loss_overlap", dt, weight, 0.25)
    for a, b in zip(seq, ovl):
        assert a.dtype == b.dtype and a.shape == b.shape
        assert torch.equal(a, b)
    chunks = -(-N // chunk)
    assert p_seq["bwd_grad_from_logits"][1] == chunks and p_seq["bwd_grad_from_logits_side"][1] == 0
    assert p_ovl["bwd_grad_from_logits"][1] == 1 and p_ovl["bwd_grad_from_logits_side"][1] == chunks - 1
    assert p_ovl["fwd_logits_keep"][1] == chunks and p_ovl["bwd_dW_gemm"][1] == chunks
    if chunks > 1:
        assert n_ovl > n_seq
    else:
        assert n_ovl == n_seq


def test_overlap_against_the_oracle(fckl):
    """Five chunks with position weights and grad_scale 1/N, against the fp64 oracle at the
    tests' tolerances (loss 1e-3 relative; dH, dW 2e-2 of the largest entry)."""
    N, d, V, K, chunk = 600, 256, 5000, 40, 128
    x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=5)
    wt = np.random.default_rng(5).random(N).astype(np.float32)
    wt[::7] = 0.0  # padding positions
    (loss, lse, rl, dH, dW), _, _ = one_call(fckl, to_dev(x, "bf16"), chunk, "loss_overlap", fckl.BF16,
                                             torch.from_numpy(wt).cuda(), 1.0 / N)
    r_loss, r_lse, r_rl = orc.forward(x["H"], x["W"], x["idx"], x["logp"], chunk, weight=wt)
    r_dH, r_dW = orc.backward(x["H"], x["W"], x["idx"], x["logp"], 1.0 / N, chunk, weight=wt)
    assert abs(float(loss.item()) - r_loss) <= 1e-3 * abs(r_loss)
    assert np.abs(lse.cpu().numpy() - r_lse).max() <= 1e-3 * (1 + np.abs(r_lse).max())
    assert np.abs(rl.cpu().numpy() - r_rl).max() <= 1e-3 * (1 + np.abs(r_rl).max())
    assert np.abs(dH.float().cpu().numpy() - r_dH).max() <= 2e-2 * np.abs(r_dH).max()
    assert np.abs(dW.cpu().numpy() - r_dW).max() <= 2e-2 * np.abs(r_dW).max()
    assert np.all(rl.cpu().numpy()[::7] == 0.0) and np.all(dH.float().cpu().numpy()[::7] == 0.0)


def test_overlap_captured_in_a_cuda_graph(fckl):
    """The overlapped one call records into a CUDA graph: the second stream joins the capture
    through the fork event and rejoins the caller's stream before the call returns, so replays
    give the eager call's bits."""
    N, d, V, K, chunk = 600, 256, 5000, 40, 128
    x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=63)
    H, W, idx, logp = to_dev(x, "bf16")
    ws = fckl.Workspace(N, d, V, K, chunk, fckl.BF16, kind="loss_overlap")
    ref = [t.clone() for t in fckl.forward_backward(H, W, idx, logp, chunk, ws=ws, grad_scale=0.5)]
    assert fckl.check(ws) == fckl.OK
    dH = torch.empty_like(H)
    dW = torch.empty(V, d, dtype=torch.float32, device=H.device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        loss, lse = fckl.forward_backward(H, W, idx, logp, chunk, ws=ws, grad_scale=0.5, dH=dH, dW=dW)[:2]
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert fckl.check(ws) == fckl.OK
        for u, v in zip((loss, lse, dH, dW), ref):
            assert torch.equal(u, v)


def test_overlap_rule(fckl, monkeypatch):
    """Without FCKL_OVERLAP the library overlaps only where it pays: at d = 3072, V = 128256,
    chunk 2048 (a 1.6e12-FLOP projection per chunk) the G pass of the first chunk runs beside
    the second chunk's forward; at d = 256 it does not, even with the overlap workspace; and
    FCKL_OVERLAP=0 turns it off. The outputs are the same bits in every case."""
    res = {}
    for name, (N, d, V, K, chunk), env in (("big", (4096, 3072, 128256, 100, 2048), None),
                                           ("big_off", (4096, 3072, 128256, 100, 2048), "0"),
                                           ("small", (600, 256, 5000, 40, 128), None)):
        if env is None:
            monkeypatch.delenv("FCKL_OVERLAP", raising=False)
        else:
            monkeypatch.setenv("FCKL_OVERLAP", env)
        x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=9)
        out, prof, _ = one_call(fckl, to_dev(x, "bf16"), chunk, "loss_overlap", fckl.BF16)
        res[name] = (out, prof)
    assert res["big"][1]["bwd_grad_from_logits_side"][1] == 1
    assert res["big_off"][1]["bwd_grad_from_logits_side"][1] == 0
    assert res["small"][1]["bwd_grad_from_logits_side"][1] == 0
    for a, b in zip(res["big"][0], res["big_off"][0]):
        assert torch.equal(a, b)
