"""GPU parity of the teacher top-K cache builder against the fp64 oracle.

Where two logits are closer than the fp32 products can resolve, either token is a correct
K-th entry, so the comparison takes what is unique and checks the rest for validity:
  * every row's K log-probabilities, sorted, match the oracle's (max-abs <= 1e-3);
  * every returned id is distinct, in range, and its log-probability matches the oracle's
    log-softmax at that id (max-abs <= 1e-3);
  * an id returned by one side but not the other lies within 1e-3 of the oracle's K-th logit;
  * rows are ordered by log-probability, and exactly tied logits (duplicated rows of Wt)
    come out smaller id first, as the oracle orders them.
"""
import numpy as np
import pytest
import scipy.special
import torch

import synthetic
from oracle import fckl_oracle as orc

pytestmark = pytest.mark.gpu
TOL = 1e-3


def run_topk(fckl, Ht, Wt, K, chunk, dtype="bf16"):
    dev = torch.device("cuda")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    H = torch.from_numpy(np.ascontiguousarray(Ht, dtype=np.float32)).to(dev).to(tdt)
    W = torch.from_numpy(np.ascontiguousarray(Wt, dtype=np.float32)).to(dev).to(tdt)
    ws = fckl.Workspace(H.shape[0], H.shape[1], W.shape[0], K, chunk, fckl.BF16 if dtype == "bf16" else fckl.F32,
                        kind="topk")
    idx, logp = fckl.teacher_topk(H, W, K, chunk, ws=ws)
    assert fckl.check(ws) == fckl.OK
    return idx.cpu().numpy().astype(np.int64), logp.cpu().numpy().astype(np.float64)


def assert_topk_parity(idx, logp, Ht, Wt, K):
    V = np.shape(Wt)[0]
    r_idx, r_logp = orc.teacher_topk(Ht, Wt, K)
    lq = scipy.special.log_softmax(orc.logits(Ht, Wt), axis=1)
    assert idx.shape == r_idx.shape
    assert idx.min() >= 0 and idx.max() < V
    for n in range(idx.shape[0]):
        assert len(set(idx[n].tolist())) == K
    assert np.abs(np.sort(logp, axis=1) - np.sort(r_logp, axis=1)).max() <= TOL
    assert np.abs(logp - np.take_along_axis(lq, idx, axis=1)).max() <= TOL
    assert np.all(np.diff(logp, axis=1) <= TOL)
    kth = r_logp[:, -1]
    for n in range(idx.shape[0]):
        g, o = set(idx[n].tolist()), set(r_idx[n].tolist())
        for v in g ^ o:
            assert abs(lq[n, v] - kth[n]) <= TOL, (n, v)
    return r_idx


@pytest.mark.parametrize("N,d,V,K,chunk", [
    (300, 256, 5000, 40, 128),   # ragged chunk and vocabulary tails
    (64, 128, 1000, 20, 64),     # fewer vocabulary tiles (4) than K: every token a candidate
    (130, 320, 2056, 100, 200),  # K = 100 over 9 tiles; d not a multiple of 64
])
def test_topk_small(fckl, N, d, V, K, chunk):
    rng = np.random.default_rng(N + V)
    Ht = synthetic.round_bf16(rng.standard_normal((N, d), dtype=np.float32))
    Wt = synthetic.round_bf16(rng.standard_normal((V, d), dtype=np.float32) * 3.0 / np.sqrt(d))
    idx, logp = run_topk(fckl, Ht, Wt, K, chunk)
    assert_topk_parity(idx, logp, Ht, Wt, K)


def test_topk_llama_vocab(fckl):
    """K = 100 over V = 128256 at d = 3072 (the cache of the 8K-256K workloads)."""
    x = synthetic.make_inputs(192, 3072, 128256, 1, dtype="bf16", seed=21)
    idx, logp = run_topk(fckl, x["H"], x["W"], 100, 128)
    assert_topk_parity(idx, logp, x["H"], x["W"], 100)


def test_topk_exact_ties_take_the_smaller_id(fckl):
    rng = np.random.default_rng(22)
    Ht = synthetic.round_bf16(rng.standard_normal((50, 64), dtype=np.float32))
    base = synthetic.round_bf16(rng.standard_normal((600, 64), dtype=np.float32) / 8)
    Wt = np.repeat(base, 2, axis=0)          # tokens 2i and 2i+1 have identical logits
    idx, logp = run_topk(fckl, Ht, Wt, 30, 64)
    r_idx = assert_topk_parity(idx, logp, Ht, Wt, 30)
    # tied pairs are adjacent, smaller id first, and a pair cut by K keeps its smaller id
    for n in range(50):
        for k in range(30):
            if idx[n, k] % 2 == 1:
                assert k > 0 and idx[n, k - 1] == idx[n, k] - 1


def test_topk_fp32_inputs_and_round_trip(fckl):
    """fp32 teacher inputs (logits products in tf32 on rounded copies) against the oracle on the
    tf32-rounded values; and a cache built from the student's own H and W gives a loss of
    (almost) zero through the loss path, which rounds the same values the same way."""
    w = synthetic.WORKLOADS["tiny_n64_d256_v4096"]
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype="f32", seed=23)
    idx, logp = run_topk(fckl, x["H"], x["W"], w.K, w.chunk, dtype="f32")
    # the exact reference of a tf32 product is the oracle on the tf32-rounded values, as the
    # bf16 tests take the oracle on bf16-rounded values
    assert_topk_parity(idx, logp, synthetic.round_tf32(x["H"]), synthetic.round_tf32(x["W"]), w.K)
    dev = torch.device("cuda")
    H = torch.from_numpy(x["H"]).to(dev)
    W = torch.from_numpy(x["W"]).to(dev)
    loss, _, rl = fckl.forward(H, W, torch.from_numpy(idx.astype(np.int32)).to(dev),
                               torch.from_numpy(logp.astype(np.float32)).to(dev), w.chunk, row_loss=True)
    fckl.check()
    assert np.abs(rl.cpu().numpy()).max() < 1e-4


def test_topk_is_deterministic(fckl):
    rng = np.random.default_rng(24)
    Ht = synthetic.round_bf16(rng.standard_normal((200, 128), dtype=np.float32))
    Wt = synthetic.round_bf16(rng.standard_normal((3000, 128), dtype=np.float32) / 4)
    a = run_topk(fckl, Ht, Wt, 50, 100)
    b = run_topk(fckl, Ht, Wt, 50, 100)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("N,d,V,K,chunk", [
    (300, 256, 5000, 40, 128),
    (64, 128, 1000, 20, 64),      # every token a candidate
    (130, 320, 2057, 100, 200),   # V % 8 == 1: a partial group of 8 columns per position
])
def test_topk_kept_and_recomputed_logits_agree(fckl, N, d, V, K, chunk):
    """Pass 2 reading the logits pass 1 kept gives the cache that projecting again gives, bit
    for bit; the profile counters show which kernels ran."""
    rng = np.random.default_rng(N + V + K)
    Ht = synthetic.round_bf16(rng.standard_normal((N, d), dtype=np.float32))
    Wt = synthetic.round_bf16(rng.standard_normal((V, d), dtype=np.float32) * 3.0 / np.sqrt(d))
    dev = torch.device("cuda")
    H = torch.from_numpy(Ht).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(Wt).to(dev).to(torch.bfloat16)
    out = {}
    for keep in (True, False):
        fckl.profile_enable(True)
        fckl.profile_read()
        out[keep] = fckl.teacher_topk(H, W, K, chunk, keep_logits=keep)
        prof = fckl.profile_read()
        fckl.profile_enable(False)
        assert fckl.check() == fckl.OK
        ran = {k for k, (_, n) in prof.items() if n > 0}
        if keep:
            assert {"topk_logits_keep", "topk_collect_from_logits"} <= ran
            assert not ran & {"topk_logits_stats", "topk_collect"}
        else:
            assert {"topk_logits_stats", "topk_collect"} <= ran
            assert not ran & {"topk_logits_keep", "topk_collect_from_logits"}
    assert torch.equal(out[True][0], out[False][0])
    assert torch.equal(out[True][1], out[False][1])
    idx, logp = (t.cpu().numpy() for t in out[True])
    assert_topk_parity(idx.astype(np.int64), logp.astype(np.float64), Ht, Wt, K)


@pytest.mark.parametrize("keep", [True, False])
def test_topk_candidate_overflow_is_reported(fckl, keep):
    """Every token ties (identical rows of Wt), so all V = 5000 logits of a position reach the
    threshold and overflow the 2048-slot candidate buffer: the status reports FCKL_ERR_CAPACITY,
    nothing is written out of bounds (the K outputs are still distinct tokens with the right
    log-probability, -log V, since any K tied tokens are a top-K), and the next call on the same
    context is exact again."""
    rng = np.random.default_rng(25)
    N, d, V, K = 64, 128, 5000, 10
    Ht = synthetic.round_bf16(rng.standard_normal((N, d), dtype=np.float32))
    row = synthetic.round_bf16(rng.standard_normal((1, d), dtype=np.float32) / 8)
    Wt = np.repeat(row, V, axis=0)
    dev = torch.device("cuda")
    H = torch.from_numpy(Ht).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(Wt).to(dev).to(torch.bfloat16)
    idx, logp = fckl.teacher_topk(H, W, K, 64, keep_logits=keep)
    assert fckl.check(raise_on_error=False) == fckl.ERR_CAPACITY
    idx, logp = idx.cpu().numpy(), logp.cpu().numpy()
    assert idx.min() >= 0 and idx.max() < V
    for n in range(N):
        assert len(set(idx[n].tolist())) == K
    assert np.abs(logp + np.log(V)).max() <= 1e-3
    # the context and the library state are intact
    rng2 = np.random.default_rng(26)
    Ht2 = synthetic.round_bf16(rng2.standard_normal((N, d), dtype=np.float32))
    Wt2 = synthetic.round_bf16(rng2.standard_normal((V, d), dtype=np.float32) / 4)
    i2, l2 = run_topk(fckl, Ht2, Wt2, K, 64)
    assert_topk_parity(i2, l2, Ht2, Wt2, K)


def test_topk_zero_logits(fckl):
    """All-zero teacher hidden states: every logit is zero, the threshold is zero, and every
    tile is live. Both pass-2 paths return tokens 0..K-1 (equal logits: smaller id first) with
    log-probability -log V, bit for bit alike."""
    N, d, V, K = 40, 64, 1000, 10
    rng = np.random.default_rng(27)
    Wt = synthetic.round_bf16(rng.standard_normal((V, d), dtype=np.float32))
    dev = torch.device("cuda")
    H = torch.zeros(N, d, dtype=torch.bfloat16, device=dev)
    W = torch.from_numpy(Wt).to(dev).to(torch.bfloat16)
    out = {}
    for keep in (True, False):
        out[keep] = fckl.teacher_topk(H, W, K, 16, keep_logits=keep)
        assert fckl.check() == fckl.OK
    assert torch.equal(out[True][0], out[False][0]) and torch.equal(out[True][1], out[False][1])
    idx, logp = (t.cpu().numpy() for t in out[True])
    assert np.array_equal(idx, np.tile(np.arange(K, dtype=np.int32), (N, 1)))
    assert np.abs(logp + np.log(V)).max() <= 1e-5


@pytest.mark.parametrize("N,d,V,K,chunk,dtype", [
    (300, 256, 5000, 40, 128, "bf16"),   # 3 chunks, the last ragged
    (64, 128, 1000, 20, 16, "bf16"),     # every token a candidate; 4 chunks of 16
    (130, 320, 2057, 100, 40, "bf16"),   # V % 8 == 1; 4 chunks, the last 10 rows
    (200, 128, 3000, 50, 64, "f32"),     # fp32 inputs (tf32 passes)
    (100, 64, 1000, 8, 100, "bf16"),     # one chunk: no second set, the same workspace
])
def test_topk_overlap_is_bitwise_the_sequential_build(fckl, N, d, V, K, chunk, dtype, monkeypatch):
    """With the overlap workspace each chunk's collect and select run on the second stream
    beside the next chunk's pass 1 (buffer sets alternating by chunk; forced with FCKL_OVERLAP=1,
    since these projections are too short for the library to choose it): the cache is bitwise
    the one of the kept-logits workspace, and every chunk ran each step once."""
    monkeypatch.setenv("FCKL_OVERLAP", "1")
    rng = np.random.default_rng(N + 3 * V)
    Ht = synthetic.round_bf16(rng.standard_normal((N, d), dtype=np.float32))
    Wt = synthetic.round_bf16(rng.standard_normal((V, d), dtype=np.float32) * 3.0 / np.sqrt(d))
    dev = torch.device("cuda")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    H = torch.from_numpy(Ht).to(dev).to(tdt)
    W = torch.from_numpy(Wt).to(dev).to(tdt)
    code = fckl.BF16 if dtype == "bf16" else fckl.F32
    out, nbytes = {}, {}
    for kind in ("topk", "topk_overlap"):
        ws = fckl.Workspace(N, d, V, K, chunk, code, kind=kind)
        fckl.profile_enable(True)
        fckl.profile_read()
        out[kind] = [t.clone() for t in fckl.teacher_topk(H, W, K, chunk, ws=ws)]
        torch.cuda.synchronize()
        prof = fckl.profile_read()
        fckl.profile_enable(False)
        assert fckl.check(ws) == fckl.OK
        nbytes[kind] = ws.nbytes
        chunks = -(-N // chunk)
        for k in ("topk_logits_keep", "topk_threshold"):
            assert prof[k][1] == chunks, (kind, k)
        side = kind == "topk_overlap" and N > chunk
        for k in ("topk_collect_from_logits", "topk_select"):
            assert prof[k][1] == (0 if side else chunks), (kind, k)
            assert prof[k + "_side"][1] == (chunks if side else 0), (kind, k)
    assert torch.equal(out["topk"][0], out["topk_overlap"][0])
    assert torch.equal(out["topk"][1], out["topk_overlap"][1])
    assert (nbytes["topk_overlap"] > nbytes["topk"]) == (N > chunk)
    if dtype == "bf16":
        idx, logp = (t.cpu().numpy() for t in out["topk_overlap"])
        assert_topk_parity(idx.astype(np.int64), logp.astype(np.float64), Ht, Wt, K)
