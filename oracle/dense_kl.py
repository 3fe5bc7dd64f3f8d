"""The "Dense KL" variant, in fp64 PyTorch on the CPU: a second, independent oracle.

TEST INFRASTRUCTURE. Only the test suite may import this module.

"Hugging Face：让知识蒸馏廉价到可大规模运行", paragraph "Dense KL": the
textbook form rebuilds a full dense teacher-probability grid from the cached
top-K values and compares it with the student's dense log-probability grid; the
article uses it as its correctness baseline. Here the grid is built by a
scatter-add of exp(logp) into zeros, the comparison is
``torch.nn.functional.kl_div`` (summed, which takes 0 * log 0 as 0) and the
gradients come from autograd, so no line of it repeats the closed form used by
``fckl_oracle``.

For a row whose cache ids are distinct this equals the per-slot loss of
``fckl_oracle`` exactly; with a repeated id the dense grid merges the slots, so
the two losses differ by a constant of the teacher alone while the gradients
stay equal.
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = ["dense_kl"]


def dense_kl(H, W, idx, logp, grad_scale=1.0):
    """Returns (loss, dH, dW) as fp64 numpy values."""
    Ht = torch.tensor(np.asarray(H, dtype=np.float64), requires_grad=True)
    Wt = torch.tensor(np.asarray(W, dtype=np.float64), requires_grad=True)
    idx_t = torch.tensor(np.asarray(idx, dtype=np.int64))
    p = torch.exp(torch.tensor(np.asarray(logp, dtype=np.float64)))
    teacher = torch.zeros(Ht.shape[0], Wt.shape[0], dtype=torch.float64)
    teacher.scatter_add_(1, idx_t, p)
    student_logq = torch.log_softmax(Ht @ Wt.T, dim=1)
    loss = torch.nn.functional.kl_div(student_logq, teacher, reduction="sum")
    (loss * grad_scale).backward()
    return float(loss.detach()), Ht.grad.numpy(), Wt.grad.numpy()
