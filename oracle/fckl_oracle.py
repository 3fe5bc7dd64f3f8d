"""fp64 CPU oracle for the fused, chunked top-K KL distillation loss.

TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and the
benchmark's CPU-baseline leg may import this module. The product path never
calls it and shares no code with it.

What it computes, and where the pages say so
--------------------------------------------
The pages ("Hugging Face：让知识蒸馏廉价到可大规模运行", paragraphs
"离线蒸馏" and "Fused, chunked KL loss"; "Chunkovaná KL strata umožnila
destilovať LLM s 32-tisícovým kontextom na jednom H200", sections "Dva odlišné
zdroje úspory" and "Čo dopĺňajú podrobnejšie experimenty") describe a KL
distillation loss between a teacher cache holding, per position, the K most
probable token ids and their values (kept WITHOUT renormalisation) and the
student's softmax over the whole vocabulary. The student's logits come from
projecting the hidden states through the output matrix, one chunk of positions
at a time; the backward pass recomputes each chunk's logits. The pages state
that the dense, the forward-chunked and the fused variants give the same loss
up to rounding (the first page above, section "Fused, chunked KL loss";
"Knowledge distillation barata ... (vazinovacao.com.br)", section "Duas
Inovações que Mudam o Jogo"), so the oracle writes out the plain definition.

Notation (per position n, vocabulary entry v, cache slot k):

    z_nv    = sum_j H_nj W_vj                     student logits
    lse_n   = log sum_v exp(z_nv)                 log-partition function
    log q_nv = z_nv - lse_n                       student log-probabilities
    p_nk    = exp(logp_nk)                        cached teacher probabilities
    S_n     = sum_k p_nk      (< 1: not renormalised)
    loss    = sum_n sum_k p_nk (logp_nk - log q_{n, idx_nk})

with 0 * log 0 taken as 0 (an entry whose logp is -inf adds nothing). Each
cache slot is its own term: a token id repeated within a row contributes once
per slot. The loss is a SUM over positions; a caller divides for a mean.

Optional position weights w_n (default 1) make the loss sum_n w_n loss_n: a
weight of 0 drops a padded position, the plain reading of the sequence packing
the article lists among its ablations (same page, section "得到的 student").

Differentiating, with p_sparse_nv = sum_{k: idx_nk = v} p_nk,

    G_nv  = d loss / d z_nv = S_n softmax(z_n)_v - p_sparse_nv
    dH    = G W,   dW = G^T H

(The article names a closed-form gradient without printing it: "Hugging
Face：让知识蒸馏廉价到可大规模运行", closing paragraph of section "得到的
student". This is the derivative of the loss above; the tests pin it by finite
differences and by autograd of the dense variant.)

Precision: inputs are widened exactly to fp64; every step runs in fp64. The
matrix products are numpy's fp64 matmul (a library primitive). Rows are
processed in chunks, exactly as the pages' fused loss walks the sequence; the
chunk changes only the memory held, not the result.
"""
from __future__ import annotations

import numpy as np

__all__ = ["teacher_mass", "logits", "log_partition", "row_loss", "logit_grad",
           "forward", "backward", "forward_backward", "rows", "teacher_topk"]


def teacher_mass(logp):
    """p = exp(logp), S_n = sum_k p_nk, and T_n = sum_k p_nk logp_nk (0 log 0 = 0).

    The cached values are the teacher's log-probabilities of its top-K tokens,
    not renormalised ("Čo dopĺňajú podrobnejšie experimenty"), so S_n < 1.
    """
    logp = np.asarray(logp, dtype=np.float64)
    p = np.exp(logp)
    plogp = np.where(p > 0.0, p * np.where(p > 0.0, logp, 0.0), 0.0)
    return p, p.sum(axis=1), plogp.sum(axis=1)


def logits(Hc, W):
    """z = Hc W^T in fp64: the output projection of one chunk of positions
    ("Fused, chunked KL loss": project the chunk's hidden states to logits)."""
    return np.asarray(Hc, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def log_partition(z):
    """lse_n = log sum_v exp(z_nv), with the row maximum taken out first."""
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def row_loss(z, lse, idx, logp):
    """Per-position loss sum_k p_nk (logp_nk - (z_{n,idx_nk} - lse_n))."""
    p, _, _ = teacher_mass(logp)
    logq = np.take_along_axis(z, np.asarray(idx, dtype=np.int64), axis=1) - lse[:, None]
    logp64 = np.asarray(logp, dtype=np.float64)
    term = np.where(p > 0.0, p * (np.where(p > 0.0, logp64, 0.0) - logq), 0.0)
    return term.sum(axis=1)


def logit_grad(z, lse, idx, logp):
    """G_nv = S_n softmax(z_n)_v - sum_{k: idx_nk = v} p_nk."""
    p, S, _ = teacher_mass(logp)
    G = S[:, None] * np.exp(z - lse[:, None])
    rows_ = np.repeat(np.arange(z.shape[0]), p.shape[1])
    np.add.at(G, (rows_, np.asarray(idx, dtype=np.int64).ravel()), -p.ravel())
    return G


def _check(H, W, idx, logp):
    H = np.asarray(H)
    W = np.asarray(W)
    idx = np.asarray(idx)
    if H.ndim != 2 or W.ndim != 2 or H.shape[1] != W.shape[1]:
        raise ValueError("H [N,d] and W [V,d] must share d")
    if idx.shape != np.shape(logp) or idx.shape[0] != H.shape[0]:
        raise ValueError("idx and logp must be [N,K]")
    if idx.size and (idx.min() < 0 or idx.max() >= W.shape[0]):
        raise IndexError("teacher index outside [0, V)")


def _weights(weight, N):
    if weight is None:
        return np.ones(N)
    w = np.asarray(weight, dtype=np.float64)
    if w.shape != (N,):
        raise ValueError("weight must be [N]")
    return w


def forward(H, W, idx, logp, chunk=None, weight=None):
    """Loss (weighted sum over positions), lse [N] and per-position weighted loss [N],
    chunk by chunk.

    "Fused, chunked KL loss": each chunk's logits are formed, folded into the
    accumulated loss and dropped before the next chunk.
    """
    _check(H, W, idx, logp)
    N = np.shape(H)[0]
    w = _weights(weight, N)
    chunk = N if not chunk else int(chunk)
    lse = np.empty(N)
    rl = np.empty(N)
    for s in range(0, N, max(chunk, 1)):
        e = min(N, s + chunk)
        z = logits(H[s:e], W)
        lse[s:e] = log_partition(z)
        rl[s:e] = w[s:e] * row_loss(z, lse[s:e], idx[s:e], logp[s:e])
    return float(rl.sum()), lse, rl


def backward(H, W, idx, logp, grad_scale=1.0, chunk=None, weight=None):
    """dH [N,d] and dW [V,d] (fp64), each chunk's logits recomputed.

    "Fused, chunked KL loss": the backward pass recomputes each chunk instead of
    keeping it. ``grad_scale`` is the upstream derivative of the caller's
    objective with respect to the loss; it multiplies both gradients.
    """
    _check(H, W, idx, logp)
    N, d = np.shape(H)
    w = _weights(weight, N)
    W64 = np.asarray(W, dtype=np.float64)
    chunk = N if not chunk else int(chunk)
    dH = np.empty((N, d))
    dW = np.zeros_like(W64)
    for s in range(0, N, max(chunk, 1)):
        e = min(N, s + chunk)
        H64 = np.asarray(H[s:e], dtype=np.float64)
        z = H64 @ W64.T
        lse = log_partition(z)
        G = logit_grad(z, lse, idx[s:e], logp[s:e]) * (grad_scale * w[s:e])[:, None]
        dH[s:e] = G @ W64
        dW += G.T @ H64
    return dH, dW


def forward_backward(H, W, idx, logp, grad_scale=1.0, chunk=None, weight=None):
    """(loss, lse, dH, dW) in one pass over the chunks."""
    loss, lse, _ = forward(H, W, idx, logp, chunk, weight)
    dH, dW = backward(H, W, idx, logp, grad_scale, chunk, weight)
    return loss, lse, dH, dW


def rows(H, W, idx, logp, which, grad_scale=1.0, weight=None):
    """lse_n, loss_n and dH_n for selected positions only.

    Every one of these depends on its own position alone (its logits row and its
    cache row), so they can be checked one by one at any problem size.
    """
    which = np.asarray(which, dtype=np.int64)
    w = _weights(weight, np.shape(H)[0])[which]
    Hs = np.asarray(H)[which]
    W64 = np.asarray(W, dtype=np.float64)
    z = np.asarray(Hs, dtype=np.float64) @ W64.T
    lse = log_partition(z)
    rl = w * row_loss(z, lse, np.asarray(idx)[which], np.asarray(logp)[which])
    G = logit_grad(z, lse, np.asarray(idx)[which], np.asarray(logp)[which]) * (grad_scale * w)[:, None]
    return lse, rl, G @ W64


def teacher_topk(Ht, Wt, K, chunk=None):
    """The offline teacher cache: per position, the K tokens of largest teacher logit and
    their log-probabilities under the teacher's full softmax, not renormalised over the K.

    "Hugging Face：让知识蒸馏廉价到可大规模运行", paragraph "离线蒸馏": the teacher runs
    once and the 100 most probable tokens of every position are cached; "Chunkovaná KL
    strata ...", section "Čo dopĺňajú podrobnejšie experimenty": the truncated distribution
    is kept without renormalisation. Returns (idx int64 [N, K], logp fp64 [N, K]), each row
    ordered by logp descending, equal logits by smaller token id.
    """
    Ht = np.asarray(Ht)
    N = Ht.shape[0]
    V = np.shape(Wt)[0]
    if not 1 <= K <= V:
        raise ValueError("need 1 <= K <= V")
    chunk = N if not chunk else int(chunk)
    idx = np.empty((N, K), dtype=np.int64)
    logp = np.empty((N, K))
    ids = np.arange(V)
    for s in range(0, N, max(chunk, 1)):
        e = min(N, s + chunk)
        z = logits(Ht[s:e], Wt)
        lse = log_partition(z)
        for r in range(e - s):
            order = np.lexsort((ids, -z[r]))[:K]   # primary key -z, then id
            idx[s + r] = order
            logp[s + r] = z[r, order] - lse[r]
    return idx, logp
