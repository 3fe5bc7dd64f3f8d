"""Pins for the fp64 oracle: each check ties it to something other than itself.

CPU only. The checks and what each would catch:

* full-vocabulary KL against ``scipy.stats.entropy`` (a library KL): a wrong
  sign, a dropped lse, a transposed projection;
* student equal to teacher, full and truncated: zero loss, and a gradient that
  is either zero (K = V) or the closed form (S - 1) q on the cached ids and S q
  elsewhere (K < V);
* the log-sum inequality loss_n >= S_n log(S_n / Q_n), with equality when the
  teacher is proportional to the student on its ids;
* gradient rows summing to zero, hence vocabulary-summed dW equal to zero;
* central finite differences of the loss against dH and dW;
* the "Dense KL" variant built from ``torch.nn.functional.kl_div`` + autograd;
* chunk invariance ("mathematically equivalent" variants);
* -inf cache entries and repeated ids, as reductions to other problems;
* a stored fixture written by ``tests/golden/make_golden.py`` from the oracle.
"""
import json
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

from oracle import fckl_oracle as orc
from oracle.dense_kl import dense_kl
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(N, d, V, K, seed=0, dtype="f32"):
    return synthetic.make_inputs(N, d, V, K, dtype=dtype, seed=seed)


def test_generator_recipe():
    x = _problem(32, 16, 500, 20, seed=3)
    idx, logp = x["idx"], x["logp"]
    assert idx.dtype == np.int32 and logp.dtype == np.float32
    assert all(len(set(r)) == 20 for r in idx.tolist())
    assert idx.min() >= 0 and idx.max() < 500
    assert np.all(np.diff(logp, axis=1) <= 0)
    S = np.exp(logp.astype(np.float64)).sum(1)
    assert np.all(S > 0.85 - 1e-6) and np.all(S < 0.99 + 1e-6)
    # not sorted by id: draw order is kept
    assert not np.all(np.diff(idx, axis=1) > 0)
    # bf16 rounding leaves values representable in bf16
    y = _problem(4, 16, 64, 4, dtype="bf16")
    bits = y["W"].view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)


def test_full_vocab_kl_matches_library():
    rng = np.random.default_rng(1)
    N, d, V = 6, 12, 40
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) / np.sqrt(d)
    t = rng.standard_normal((N, V)) * 2.0
    p_dense = scipy.special.softmax(t, axis=1)
    idx = np.stack([rng.permutation(V) for _ in range(N)])
    logp = np.log(np.take_along_axis(p_dense, idx, axis=1))
    loss, lse, rl = orc.forward(H, W, idx, logp)
    q = scipy.special.softmax(H @ W.T, axis=1)
    want = np.array([scipy.stats.entropy(p_dense[n], q[n]) for n in range(N)])
    np.testing.assert_allclose(rl, want, rtol=1e-12, atol=1e-14)
    assert loss == pytest.approx(want.sum(), rel=1e-12)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(H @ W.T, axis=1), rtol=1e-14)


def test_student_equals_teacher_full_vocab():
    rng = np.random.default_rng(2)
    N, d, V = 5, 10, 30
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d))
    logq = scipy.special.log_softmax(H @ W.T, axis=1)
    idx = np.stack([rng.permutation(V) for _ in range(N)])
    logp = np.take_along_axis(logq, idx, axis=1)
    loss, _, rl = orc.forward(H, W, idx, logp)
    assert abs(loss) < 1e-12
    dH, dW = orc.backward(H, W, idx, logp)
    assert np.abs(dH).max() < 1e-12 and np.abs(dW).max() < 1e-12


def test_student_equals_teacher_truncated():
    rng = np.random.default_rng(3)
    N, d, V, K = 4, 9, 50, 7
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d))
    z = H @ W.T
    logq = scipy.special.log_softmax(z, axis=1)
    idx = np.argsort(-z, axis=1)[:, :K]
    logp = np.take_along_axis(logq, idx, axis=1)
    loss, lse, rl = orc.forward(H, W, idx, logp)
    assert np.abs(rl).max() < 1e-13
    # K < V: S < 1, and the gradient is (S-1) q on the cached ids, S q off them.
    q = np.exp(logq)
    S = np.take_along_axis(q, idx, axis=1).sum(1)
    want = S[:, None] * q
    for n in range(N):
        want[n, idx[n]] = (S[n] - 1.0) * q[n, idx[n]]
    G = orc.logit_grad(z, lse, idx, logp)
    np.testing.assert_allclose(G, want, rtol=1e-11, atol=1e-15)
    dH, dW = orc.backward(H, W, idx, logp)
    np.testing.assert_allclose(dH, want @ W, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dW, want.T @ H, rtol=1e-10, atol=1e-13)


def test_log_sum_bound_and_equality():
    x = _problem(48, 32, 700, 25, seed=4)
    loss, lse, rl = orc.forward(x["H"], x["W"], x["idx"], x["logp"])
    z = orc.logits(x["H"], x["W"])
    q = scipy.special.softmax(z, axis=1)
    Q = np.take_along_axis(q, x["idx"].astype(np.int64), axis=1).sum(1)
    S = np.exp(x["logp"].astype(np.float64)).sum(1)
    bound = S * np.log(S / Q)
    assert np.all(rl >= bound - 1e-12)
    assert np.any(rl > bound + 1e-3)
    # equality when the teacher is proportional to the student on its ids
    qk = np.take_along_axis(q, x["idx"].astype(np.int64), axis=1)
    logp_eq = np.log(S[:, None] * qk / Q[:, None])
    _, _, rl_eq = orc.forward(x["H"], x["W"], x["idx"], logp_eq)
    np.testing.assert_allclose(rl_eq, bound, rtol=1e-10, atol=1e-12)


def test_gradient_rows_and_dW_sum_to_zero():
    x = _problem(40, 24, 300, 10, seed=5)
    z = orc.logits(x["H"], x["W"])
    lse = orc.log_partition(z)
    G = orc.logit_grad(z, lse, x["idx"], x["logp"])
    assert np.abs(G.sum(1)).max() < 1e-14 * 300
    _, dW = orc.backward(x["H"], x["W"], x["idx"], x["logp"])
    assert np.abs(dW.sum(0)).max() < 1e-12 * np.abs(dW).max() * 300


def test_finite_differences():
    rng = np.random.default_rng(6)
    N, d, V, K = 4, 8, 32, 5
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) / np.sqrt(d)
    idx, logp = synthetic.teacher_cache(N, V, K, seed=7)
    scale = 1.7
    dH, dW = orc.backward(H, W, idx, logp, grad_scale=scale)
    h = 1e-6

    def f(Hx, Wx):
        return scale * orc.forward(Hx, Wx, idx, logp)[0]

    for _ in range(10):
        i, j = rng.integers(N), rng.integers(d)
        Hp, Hm = H.copy(), H.copy()
        Hp[i, j] += h
        Hm[i, j] -= h
        fd = (f(Hp, W) - f(Hm, W)) / (2 * h)
        assert fd == pytest.approx(dH[i, j], rel=1e-6, abs=1e-8)
        v, j = rng.integers(V), rng.integers(d)
        Wp, Wm = W.copy(), W.copy()
        Wp[v, j] += h
        Wm[v, j] -= h
        fd = (f(H, Wp) - f(H, Wm)) / (2 * h)
        assert fd == pytest.approx(dW[v, j], rel=1e-6, abs=1e-8)


def test_dense_kl_variant_agrees():
    x = _problem(64, 256, 4096, 16, seed=0)
    loss, lse, dH, dW = orc.forward_backward(x["H"], x["W"], x["idx"], x["logp"], grad_scale=0.5)
    dl, dHd, dWd = dense_kl(x["H"], x["W"], x["idx"], x["logp"], grad_scale=0.5)
    assert loss == pytest.approx(dl, rel=1e-12)
    assert np.abs(dH - dHd).max() <= 1e-10 * np.abs(dHd).max()
    assert np.abs(dW - dWd).max() <= 1e-10 * np.abs(dWd).max()


def test_chunk_invariance():
    x = _problem(23, 16, 200, 9, seed=8)
    ref = orc.forward_backward(x["H"], x["W"], x["idx"], x["logp"], chunk=None)
    for chunk in (1, 7, 16, 23, 64):
        got = orc.forward_backward(x["H"], x["W"], x["idx"], x["logp"], chunk=chunk)
        assert got[0] == pytest.approx(ref[0], rel=1e-12)
        for a, b in zip(got[1:], ref[1:]):
            np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-14)


def test_neg_inf_slots_drop_out():
    x = _problem(12, 16, 128, 6, seed=9)
    logp = x["logp"].copy()
    logp[:, -1] = -np.inf
    full = orc.forward_backward(x["H"], x["W"], x["idx"], logp)
    cut = orc.forward_backward(x["H"], x["W"], x["idx"][:, :-1], x["logp"][:, :-1])
    assert np.isfinite(full[0])
    assert full[0] == pytest.approx(cut[0], rel=1e-13)
    for a, b in zip(full[1:], cut[1:]):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)


def test_repeated_ids_split_slot():
    x = _problem(10, 16, 128, 6, seed=10)
    idx, logp = x["idx"], x["logp"].astype(np.float64)
    # slot 0 split into two slots with the same id and half the probability each
    idx2 = np.concatenate([idx[:, :1], idx], axis=1)
    logp2 = np.concatenate([logp[:, :1] - np.log(2.0), logp[:, :1] - np.log(2.0), logp[:, 1:]], axis=1)
    base = orc.forward_backward(x["H"], x["W"], idx, logp)
    split = orc.forward_backward(x["H"], x["W"], idx2, logp2)
    shift = -(np.exp(logp[:, 0]) * np.log(2.0)).sum()
    assert split[0] == pytest.approx(base[0] + shift, rel=1e-12)
    for a, b in zip(split[1:], base[1:]):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)
    # gradients equal the dense variant's, which merges the repeated slots
    _, dHd, dWd = dense_kl(x["H"], x["W"], idx2, logp2)
    np.testing.assert_allclose(split[2], dHd, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(split[3], dWd, rtol=1e-10, atol=1e-13)


def test_grad_scale_is_linear():
    x = _problem(9, 16, 100, 5, seed=11)
    a = orc.backward(x["H"], x["W"], x["idx"], x["logp"], grad_scale=1.0)
    b = orc.backward(x["H"], x["W"], x["idx"], x["logp"], grad_scale=-2.5)
    np.testing.assert_allclose(b[0], -2.5 * a[0], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(b[1], -2.5 * a[1], rtol=1e-12, atol=1e-15)


def test_rows_match_full_pass():
    x = _problem(30, 32, 256, 8, seed=12)
    loss, lse, rl = orc.forward(x["H"], x["W"], x["idx"], x["logp"])
    dH, _ = orc.backward(x["H"], x["W"], x["idx"], x["logp"], grad_scale=0.25)
    which = [0, 7, 29]
    l2, r2, h2 = orc.rows(x["H"], x["W"], x["idx"], x["logp"], which, grad_scale=0.25)
    np.testing.assert_allclose(l2, lse[which], rtol=1e-14)
    np.testing.assert_allclose(r2, rl[which], rtol=1e-13)
    np.testing.assert_allclose(h2, dH[which], rtol=1e-12, atol=1e-15)


def test_bad_index_rejected():
    x = _problem(4, 8, 32, 3, seed=13)
    idx = x["idx"].copy()
    idx[1, 2] = 32
    with pytest.raises(IndexError):
        orc.forward(x["H"], x["W"], idx, x["logp"])


def test_lse_statistics_sanity():
    """Not a pin: with z ~ N(0, 1), E[exp z] = e^(1/2), so lse is near ln V + 1/2."""
    x = _problem(64, 256, 4096, 16, seed=0)
    _, lse, _ = orc.forward(x["H"], x["W"], x["idx"], x["logp"])
    assert abs(lse.mean() - (np.log(4096) + 0.5)) < 0.05


def test_golden_fixture():
    """Values stored by tests/golden/make_golden.py from the oracle itself: catch
    unintended changes of the oracle or of the generators on another machine."""
    with open(os.path.join(GOLDEN, "tiny_oracle.json")) as f:
        g = json.load(f)
    w = synthetic.WORKLOADS[g["workload"]]
    x = synthetic.make_inputs(w.N, w.d, w.V, w.K, dtype=w.dtype, seed=g["seed"])
    assert x["idx"][0, :8].tolist() == g["idx_row0"]
    np.testing.assert_array_equal(x["logp"][0, :4], np.array(g["logp_row0"], np.float32))
    np.testing.assert_array_equal(x["H"][0, :4], np.array(g["H_row0"], np.float32))
    loss, lse, dH, dW = orc.forward_backward(x["H"], x["W"], x["idx"], x["logp"],
                                             grad_scale=g["grad_scale"], chunk=w.chunk)
    assert loss == pytest.approx(g["loss"], rel=1e-12)
    np.testing.assert_allclose(lse[:8], g["lse_head"], rtol=1e-12)
    np.testing.assert_allclose(dH[0, :8], g["dH_row0"], rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(dW[x["idx"][0, 0], :8], g["dW_hit_row"], rtol=1e-10, atol=1e-14)


def test_weight_zero_drops_a_position_and_two_duplicates_it():
    x = _problem(12, 16, 128, 6, seed=14)
    w = np.ones(12)
    w[[2, 7]] = 0.0
    w[5] = 2.0
    got = orc.forward_backward(x["H"], x["W"], x["idx"], x["logp"], grad_scale=0.5, chunk=5, weight=w)
    keep = [i for i in range(12) if w[i] != 0] + [5]          # drop 2 and 7, repeat 5
    ref = orc.forward_backward(x["H"][keep], x["W"], x["idx"][keep], x["logp"][keep], grad_scale=0.5)
    assert got[0] == pytest.approx(ref[0], rel=1e-12)
    np.testing.assert_allclose(got[3], ref[3], rtol=1e-11, atol=1e-14)          # dW
    assert np.abs(got[2][[2, 7]]).max() == 0.0                                  # dropped rows
    np.testing.assert_allclose(got[2][5], 2 * ref[2][keep.index(5)], rtol=1e-12)
    np.testing.assert_allclose(got[1], orc.forward(x["H"], x["W"], x["idx"], x["logp"])[1], rtol=1e-14)


def test_weighted_finite_differences():
    rng = np.random.default_rng(15)
    N, d, V, K = 3, 6, 20, 4
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) / np.sqrt(d)
    idx, logp = synthetic.teacher_cache(N, V, K, seed=16)
    w = np.array([0.3, 0.0, 1.7])
    dH, dW = orc.backward(H, W, idx, logp, grad_scale=1.0, weight=w)
    h = 1e-6
    for _ in range(6):
        i, j = rng.integers(N), rng.integers(d)
        Hp, Hm = H.copy(), H.copy()
        Hp[i, j] += h
        Hm[i, j] -= h
        fd = (orc.forward(Hp, W, idx, logp, weight=w)[0] - orc.forward(Hm, W, idx, logp, weight=w)[0]) / (2 * h)
        assert fd == pytest.approx(dH[i, j], rel=1e-6, abs=1e-9)
        v, j = rng.integers(V), rng.integers(d)
        Wp, Wm = W.copy(), W.copy()
        Wp[v, j] += h
        Wm[v, j] -= h
        fd = (orc.forward(H, Wp, idx, logp, weight=w)[0] - orc.forward(H, Wm, idx, logp, weight=w)[0]) / (2 * h)
        assert fd == pytest.approx(dW[v, j], rel=1e-6, abs=1e-9)


def test_teacher_topk_matches_library_topk():
    rng = np.random.default_rng(17)
    Ht = rng.standard_normal((20, 16))
    Wt = rng.standard_normal((300, 16)) / 4
    idx, logp = orc.teacher_topk(Ht, Wt, 12, chunk=7)
    import torch
    z = torch.tensor(Ht @ Wt.T)
    vals, ids = torch.topk(z, 12, dim=1, largest=True, sorted=True)
    np.testing.assert_array_equal(idx, ids.numpy())
    lq = torch.log_softmax(z, dim=1)
    np.testing.assert_allclose(logp, torch.gather(lq, 1, ids).numpy(), rtol=1e-13, atol=1e-13)


def test_teacher_topk_invariants():
    rng = np.random.default_rng(18)
    Ht = rng.standard_normal((9, 8))
    Wt = rng.standard_normal((40, 8))
    # K = V: the whole distribution, so the kept probabilities sum to 1
    idx, logp = orc.teacher_topk(Ht, Wt, 40)
    assert np.all(np.sort(idx, axis=1) == np.arange(40))
    np.testing.assert_allclose(scipy.special.logsumexp(logp, axis=1), 0.0, atol=1e-13)
    # K < V: not renormalised (mass < 1), descending, and nothing left out beats the K-th
    idx, logp = orc.teacher_topk(Ht, Wt, 6)
    assert np.all(np.exp(logp).sum(1) < 1.0)
    assert np.all(np.diff(logp, axis=1) <= 0)
    lq = scipy.special.log_softmax(Ht @ Wt.T, axis=1)
    for n in range(9):
        rest = np.setdiff1d(np.arange(40), idx[n])
        assert lq[n, rest].max() <= logp[n, -1]
    # equal logits: the smaller id first
    Wd = np.repeat(Wt[:5], 2, axis=0)
    idx, _ = orc.teacher_topk(Ht, Wd, 10)
    for n in range(9):
        for a, b in zip(idx[n][0::2], idx[n][1::2]):
            assert a // 2 == b // 2 and a < b


def test_cache_built_from_the_student_gives_zero_loss():
    """A cache built by the teacher-side routine from the student's own H and W makes the
    student equal to the teacher on the cached ids: the loss vanishes."""
    x = _problem(16, 24, 500, 30, seed=19)
    idx, logp = orc.teacher_topk(x["H"], x["W"], 30)
    loss, _, rl = orc.forward(x["H"], x["W"], idx, logp)
    assert np.abs(rl).max() < 1e-12


def test_teacher_generator_terminates_when_K_is_close_to_V():
    import time
    t0 = time.time()
    for N, V, K in [(40, 16, 16), (96, 2048, 1024), (513, 256, 7), (8, 100, 99)]:
        idx, logp = synthetic.teacher_cache(N, V, K, seed=1)
        assert all(len(set(r)) == K for r in idx.tolist()) and idx.max() < V
    assert time.time() - t0 < 10


def test_empty_row_and_one_hot_row_closed_forms():
    """A position whose slots are all empty carries no teacher mass: no loss and no gradient.
    A position whose mass is one token (p = 1) has the cross-entropy -log q_i = lse - z_i as
    its loss and G = softmax(z) - e_i, checked against scipy's log-softmax."""
    rng = np.random.default_rng(17)
    N, d, V, K = 6, 16, 50, 4
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) / 4
    idx = np.stack([rng.choice(V, K, replace=False) for _ in range(N)]).astype(np.int32)
    logp = np.full((N, K), -np.inf)
    logp[1, 2] = 0.0   # row 1: one-hot on idx[1, 2]; row 0 and the others: empty
    logp[3, 0] = 0.0
    loss, lse, rl = orc.forward(H, W, idx, logp)
    dH, dW = orc.backward(H, W, idx, logp)
    z = H @ W.T
    lq = scipy.special.log_softmax(z, axis=1)
    for n in (0, 2, 4, 5):
        assert rl[n] == 0.0 and np.all(dH[n] == 0.0)
    for n, k in ((1, 2), (3, 0)):
        assert rl[n] == pytest.approx(-lq[n, idx[n, k]], rel=1e-12)
        G = np.exp(lq[n])
        G[idx[n, k]] -= 1.0
        np.testing.assert_allclose(dH[n], G @ W, rtol=1e-10, atol=1e-12)
    assert loss == pytest.approx(rl.sum(), rel=1e-12)
    G_all = np.zeros((N, V))
    for n, k in ((1, 2), (3, 0)):
        G_all[n] = np.exp(lq[n])
        G_all[n, idx[n, k]] -= 1.0
    np.testing.assert_allclose(dW, G_all.T @ H, rtol=1e-10, atol=1e-12)


def test_tf32_rounding_of_inputs():
    """synthetic.round_tf32 against a frexp restatement: nearest value with 11 significant bits,
    ties away from zero."""
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 10 ** rng.uniform(-6, 6, 10000),
                        np.float32([0.0, -0.0, 1.0, -1.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                                    -(1.0 + 2.0 ** -11), 2.0 - 2.0 ** -12])]).astype(np.float32)
    m, e = np.frexp(x.astype(np.float64))            # |m| in [0.5, 1): 11 bits are m * 2^11
    q = np.floor(np.abs(m) * 2.0 ** 11 + 0.5) * np.sign(m)
    ref = np.ldexp(q / 2.0 ** 11, e)
    got = synthetic.round_tf32(x).astype(np.float64)
    assert np.array_equal(got, ref)
    # exact ties round away from zero; the largest value below 2 rounds up to 2
    assert synthetic.round_tf32(np.float32([1.0 + 2.0 ** -11]))[0] == np.float32(1.0 + 2.0 ** -10)
    assert synthetic.round_tf32(np.float32([2.0 - 2.0 ** -12]))[0] == np.float32(2.0)
