"""Fused, chunked top-K KL distillation loss on GB300: Python binding of ``include/fckl.h``.

Argument marshalling only. Every step of the loss and its gradients runs in the CUDA
library ``_build/libfckl.so``; PyTorch supplies device memory and the stream. There is
no CPU fallback: if the library is missing, ``load()`` raises.

Typical use (tensors on the current CUDA device)::

    import chunked_kl_loss_gb300 as fckl
    loss, lse, dH, dW = fckl.forward_backward(H, W, idx, logp, chunk=2048)   # one call
    fckl.check()            # raises on a device-detected error (bad teacher id, timeout)
    loss, lse = fckl.forward(H, W, idx, logp, chunk=2048)                    # or separately:
    dH, dW = fckl.backward(H, W, idx, logp, lse, chunk=2048)                 # recomputes the logits
    loss = fckl.fused_chunked_kl(H, W, idx, logp, 2048); loss.backward()     # autograd

``H [N, d]`` and ``W [V, d]`` are bf16 or fp32, ``idx [N, K]`` int32 teacher token ids,
``logp [N, K]`` fp32 teacher log-probabilities (not renormalised). The loss is a sum over
positions; ``grad_scale`` carries an upstream derivative (e.g. ``1/N`` for a mean).
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["LIB_PATH", "FcklError", "load", "workspace_bytes", "overlap_workspace_bytes", "Workspace", "forward", "backward",
           "forward_backward", "fused_chunked_kl", "teacher_topk", "check", "shard_range",
           "allreduce_loss_and_dW", "data_parallel_forward_backward", "launch_count", "profile_enable", "profile_read",
           "kernel_names", "OK", "ERR_ARG", "ERR_INDEX", "ERR_CUDA", "ERR_TIMEOUT",
           "ERR_WORKSPACE", "ERR_UNSUPPORTED", "ERR_CAPACITY"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfckl.so")

OK, ERR_ARG, ERR_INDEX, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CAPACITY = range(8)
BF16, F32 = 0, 1

_lib = None


class FcklError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = load().fckl_status_string(status).decode()
        extra = load().fckl_last_error().decode() if status == ERR_CUDA else ""
        super().__init__(f"{where}: {msg}" + (f" ({extra})" if extra else ""))


def load():
    """Loads the CUDA library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
    lib = ctypes.CDLL(LIB_PATH)
    c = ctypes
    vp, i64, i32, sz, f32 = c.c_void_p, c.c_int64, c.c_int, c.c_size_t, c.c_float
    lib.fckl_workspace_bytes.restype = sz
    lib.fckl_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i32]
    lib.fckl_overlap_workspace_bytes.restype = sz
    lib.fckl_overlap_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i32]
    lib.fckl_forward.restype = i32
    lib.fckl_forward.argtypes = [vp, vp, i32, vp, vp, vp, i64, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.fckl_backward.restype = i32
    lib.fckl_backward.argtypes = [vp, vp, i32, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32, vp, vp, vp, sz, vp]
    lib.fckl_forward_backward.restype = i32
    lib.fckl_forward_backward.argtypes = [vp, vp, i32, vp, vp, vp, i64, i32, i32, i32, i32, f32, vp, vp, vp, vp,
                                          vp, vp, sz, vp]
    lib.fckl_selftest_wait_timeout.restype = i32
    lib.fckl_selftest_wait_timeout.argtypes = [vp, sz, vp]
    lib.fckl_topk_workspace_bytes.restype = sz
    lib.fckl_topk_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i32]
    lib.fckl_topk_kept_logits_workspace_bytes.restype = sz
    lib.fckl_topk_kept_logits_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i32]
    lib.fckl_topk_overlap_workspace_bytes.restype = sz
    lib.fckl_topk_overlap_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i32]
    lib.fckl_teacher_topk.restype = i32
    lib.fckl_teacher_topk.argtypes = [vp, vp, i32, i64, i32, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.fckl_check.restype = i32
    lib.fckl_check.argtypes = [vp, vp]
    lib.fckl_status_string.restype = c.c_char_p
    lib.fckl_status_string.argtypes = [i32]
    lib.fckl_last_error.restype = c.c_char_p
    lib.fckl_last_error.argtypes = []
    lib.fckl_launch_count.restype = i64
    lib.fckl_launch_count.argtypes = []
    lib.fckl_profile_enable.restype = i32
    lib.fckl_profile_enable.argtypes = [i32]
    lib.fckl_profile_read.restype = i32
    lib.fckl_profile_read.argtypes = [c.POINTER(c.c_double), c.POINTER(c.c_int64), i32]
    lib.fckl_kernel_name.restype = c.c_char_p
    lib.fckl_kernel_name.argtypes = [i32]
    _lib = lib
    return lib


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"H and W must be bfloat16 or float32, got {t.dtype}")


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def workspace_bytes(N: int, d: int, V: int, K: int, chunk: int, dtype: int = BF16) -> int:
    return int(load().fckl_workspace_bytes(N, d, V, K, chunk, dtype))


def overlap_workspace_bytes(N: int, d: int, V: int, K: int, chunk: int, dtype: int = BF16) -> int:
    return int(load().fckl_overlap_workspace_bytes(N, d, V, K, chunk, dtype))


class Workspace:
    """A device workspace sized for one problem shape (a torch uint8 tensor); ``kind`` is
    "loss" (forward, backward, forward_backward), "loss_overlap" (the same, plus a second set
    of one chunk's buffers with which forward_backward overlaps consecutive chunks), "topk"
    (teacher cache builder keeping each chunk's logits), "topk_overlap" (the same plus a second
    set of one chunk's buffers, with which the builder overlaps consecutive chunks) or
    "topk_min" (the builder's minimum, which projects each chunk twice)."""

    def __init__(self, N, d, V, K, chunk, dtype=BF16, device=None, kind="loss"):
        import torch
        if kind == "topk":
            n = int(load().fckl_topk_kept_logits_workspace_bytes(N, d, V, K, chunk, dtype))
        elif kind == "topk_overlap":
            n = int(load().fckl_topk_overlap_workspace_bytes(N, d, V, K, chunk, dtype))
        elif kind == "topk_min":
            n = int(load().fckl_topk_workspace_bytes(N, d, V, K, chunk, dtype))
        elif kind == "loss":
            n = workspace_bytes(N, d, V, K, chunk, dtype)
        elif kind == "loss_overlap":
            n = overlap_workspace_bytes(N, d, V, K, chunk, dtype)
        else:
            raise ValueError(f"unknown workspace kind {kind!r}")
        if n == 0:
            raise FcklError(ERR_UNSUPPORTED, "workspace_bytes")
        self.nbytes = n
        self.tensor = torch.empty(n, dtype=torch.uint8, device=device or "cuda")

    @property
    def ptr(self):
        return ctypes.c_void_p(self.tensor.data_ptr())


# Workspace of the last call, for check(): held strongly when the binding created it (the
# caller has no other handle), weakly when the caller passed it in (the caller owns it).
_last_ws = None


def _weight(weight, N):
    if weight is None:
        return None
    import torch
    if tuple(weight.shape) != (N,) or not weight.is_cuda or not weight.is_contiguous():
        raise ValueError("weight must be a contiguous CUDA tensor of shape [N]")
    if weight.dtype != torch.float32:
        raise TypeError("weight must be float32")
    return weight


def _shape(H, W, idx, logp):
    N, d = H.shape
    V = W.shape[0]
    K = idx.shape[1]
    if W.shape[1] != d or idx.shape[0] != N or tuple(logp.shape) != tuple(idx.shape):
        raise ValueError("expected H [N,d], W [V,d], idx [N,K], logp [N,K]")
    if H.dtype != W.dtype:
        raise TypeError("H and W must share a dtype")
    for t in (H, W, idx, logp):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    return N, d, V, K


def _ws_for(ws, N, d, V, K, chunk, dt, device, kind="loss"):
    global _last_ws
    import weakref
    if ws is None:
        ws = Workspace(N, d, V, K, chunk, dt, device, kind=kind)
        _last_ws = ws
    else:
        _last_ws = weakref.ref(ws)
    return ws


def forward(H, W, idx, logp, chunk, ws=None, stream=None, row_loss=False, weight=None):
    """Returns (loss [1] fp32, lse [N] fp32) or, with ``row_loss=True``, also the
    per-position losses [N]. ``weight`` [N] fp32 scales each position's loss (0 = padding)."""
    import torch
    N, d, V, K = _shape(H, W, idx, logp)
    weight = _weight(weight, N)
    dt = _dtype_code(H)
    ws = _ws_for(ws, N, d, V, K, chunk, dt, H.device)
    loss = torch.empty(1, dtype=torch.float32, device=H.device)
    lse = torch.empty(N, dtype=torch.float32, device=H.device)
    rl = torch.empty(N, dtype=torch.float32, device=H.device) if row_loss else None
    st = load().fckl_forward(_ptr(H), _ptr(W), dt, _ptr(idx), _ptr(logp), _ptr(weight), N, d, V, K, chunk,
                             _ptr(loss), _ptr(lse), _ptr(rl), ws.ptr, ws.nbytes, _stream_ptr(stream))
    if st != OK:
        raise FcklError(st, "fckl_forward")
    return (loss, lse, rl) if row_loss else (loss, lse)


def backward(H, W, idx, logp, lse, chunk, grad_scale=1.0, ws=None, stream=None, dH=None, dW=None,
             weight=None):
    """Returns (dH [N,d] in H's dtype, dW [V,d] fp32)."""
    import torch
    N, d, V, K = _shape(H, W, idx, logp)
    weight = _weight(weight, N)
    dt = _dtype_code(H)
    ws = _ws_for(ws, N, d, V, K, chunk, dt, H.device)
    if dH is None:
        dH = torch.empty_like(H)
    if dW is None:
        dW = torch.empty(V, d, dtype=torch.float32, device=H.device)
    st = load().fckl_backward(_ptr(H), _ptr(W), dt, _ptr(idx), _ptr(logp), _ptr(weight), _ptr(lse), N, d, V, K,
                              chunk, float(grad_scale), _ptr(dH), _ptr(dW), ws.ptr, ws.nbytes, _stream_ptr(stream))
    if st != OK:
        raise FcklError(st, "fckl_backward")
    return dH, dW


def forward_backward(H, W, idx, logp, chunk, grad_scale=1.0, ws=None, stream=None, weight=None,
                     row_loss=False, dH=None, dW=None):
    """(loss, lse, dH, dW) — or (loss, lse, row_loss, dH, dW) with ``row_loss=True`` — from
    one fckl_forward_backward call: each chunk's backward right after its forward, from what
    the forward kept in the gradient slab (no logits recomputed). Bitwise the outputs of
    forward() then backward(). Without ``ws`` it allocates the "loss_overlap" workspace, with
    which consecutive chunks overlap (one more chunk's buffers); pass a "loss" workspace for
    the minimum memory."""
    import torch
    N, d, V, K = _shape(H, W, idx, logp)
    weight = _weight(weight, N)
    dt = _dtype_code(H)
    ws = _ws_for(ws, N, d, V, K, chunk, dt, H.device, kind="loss_overlap")
    loss = torch.empty(1, dtype=torch.float32, device=H.device)
    lse = torch.empty(N, dtype=torch.float32, device=H.device)
    rl = torch.empty(N, dtype=torch.float32, device=H.device) if row_loss else None
    if dH is None:
        dH = torch.empty_like(H)
    if dW is None:
        dW = torch.empty(V, d, dtype=torch.float32, device=H.device)
    st = load().fckl_forward_backward(_ptr(H), _ptr(W), dt, _ptr(idx), _ptr(logp), _ptr(weight), N, d, V, K,
                                      chunk, float(grad_scale), _ptr(loss), _ptr(lse), _ptr(rl), _ptr(dH),
                                      _ptr(dW), ws.ptr, ws.nbytes, _stream_ptr(stream))
    if st != OK:
        raise FcklError(st, "fckl_forward_backward")
    return (loss, lse, rl, dH, dW) if row_loss else (loss, lse, dH, dW)


def _autograd_function():
    import torch

    class FusedChunkedKL(torch.autograd.Function):
        """Autograd wrapper of scale * loss. When H or W needs a gradient, the forward runs the
        one call (fckl_forward_backward with grad_scale = scale) and holds dH and dW; the
        backward multiplies them by the upstream gradient g on the device (fp32 product, one
        rounding to H's dtype; no host synchronisation). For g = 1 (``out.backward()`` on the
        scalar itself) the held gradients are returned as the library wrote them, so a caller
        that folds its reduction (e.g. scale = 1/N for a mean) into ``scale`` gets dH rounded
        once. Without gradients the forward runs fckl_forward alone."""

        @staticmethod
        def forward(ctx, H, W, idx, logp, chunk, weight, scale):
            if ctx.needs_input_grad[0] or ctx.needs_input_grad[1]:
                loss, _, dH, dW = forward_backward(H, W, idx, logp, chunk, grad_scale=scale, weight=weight)
                ctx.grads = (dH, dW)
            else:
                loss, _ = forward(H, W, idx, logp, chunk, weight=weight)
                ctx.grads = None
            return loss[0] if scale == 1.0 else loss[0] * scale

        @staticmethod
        def backward(ctx, g):
            dH, dW = ctx.grads
            ctx.grads = None
            g32 = g.float()
            gH = (dH.float() * g32).to(dH.dtype) if ctx.needs_input_grad[0] else None
            gW = dW * g32 if ctx.needs_input_grad[1] else None
            return gH, gW, None, None, None, None, None

    return FusedChunkedKL


_FusedChunkedKL = None


def fused_chunked_kl(H, W, idx, logp, chunk, weight=None, scale=1.0):
    """``scale`` times the loss as a differentiable scalar: gradients reach H and W through
    autograd (W's fp32 gradient is cast to W's dtype by autograd). Fold a known reduction into
    ``scale`` (1/N for a mean over positions) rather than dividing the result: the library then
    applies it before dH's one rounding."""
    global _FusedChunkedKL
    if _FusedChunkedKL is None:
        _FusedChunkedKL = _autograd_function()
    return _FusedChunkedKL.apply(H, W, idx, logp, chunk, weight, float(scale))


def shard_range(N: int, rank: int, world: int):
    """Contiguous positions [start, end) of rank ``rank`` out of ``world`` for a global batch of
    N positions: the first N % world ranks take one position more. Every position belongs to
    exactly one rank and the ranks' ranges are in rank order."""
    if world < 1 or not 0 <= rank < world or N < 0:
        raise ValueError("need 0 <= rank < world and N >= 0")
    base, extra = divmod(N, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def allreduce_loss_and_dW(loss, dW, group=None):
    """Sums the loss [1] and dW [V, d] (fp32) over the ranks of ``group`` in place: the one
    exchange step of the data-parallel loss (the positions are independent except through
    dW, whose gradient is a sum over positions, and the loss, a sum too). With the NCCL
    backend the device tensors are reduced directly; with gloo (CPU ranks, or GPU ranks that
    exchange through the host) device tensors are staged through host memory."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return loss, dW
    via_host = dW.is_cuda and dist.get_backend(group) != "nccl"
    for t in (dW, loss):
        if via_host:
            h = t.cpu()
            dist.all_reduce(h, op=dist.ReduceOp.SUM, group=group)
            t.copy_(h)
        else:
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    if via_host:
        torch.cuda.current_stream(dW.device).synchronize()
    return loss, dW


def data_parallel_forward_backward(H, W, idx, logp, chunk, grad_scale=1.0, ws=None, stream=None, weight=None,
                                   dH=None, dW=None, group=None):
    """One data-parallel step: ``H``, ``idx``, ``logp`` (and ``weight``) hold this rank's
    contiguous range of positions (``shard_range``), ``W`` is replicated. The rank runs the one
    call on its positions, then the loss and dW are summed over the ranks; lse and dH stay with
    the rank's positions. Returns (loss of all ranks, lse, dH, dW of all ranks). A rank with no
    positions contributes zeros to both sums."""
    if H.shape[0] == 0:
        import torch
        loss = torch.zeros(1, dtype=torch.float32, device=H.device)
        lse = torch.empty(0, dtype=torch.float32, device=H.device)
        dH = torch.empty_like(H) if dH is None else dH
        if dW is None:
            dW = torch.empty(W.shape[0], W.shape[1], dtype=torch.float32, device=H.device)
        dW.zero_()
        allreduce_loss_and_dW(loss, dW, group)
        return loss, lse, dH, dW
    loss, lse, dH, dW = forward_backward(H, W, idx, logp, chunk, grad_scale=grad_scale, ws=ws, stream=stream,
                                         weight=weight, dH=dH, dW=dW)
    allreduce_loss_and_dW(loss, dW, group)
    return loss, lse, dH, dW


def teacher_topk(Ht, Wt, K, chunk, ws=None, stream=None, keep_logits=True):
    """Offline teacher cache: (idx int32 [N, K], logp fp32 [N, K]) — the K tokens of largest
    teacher logit per position, by logit descending, with full-softmax log-probabilities.
    ``keep_logits=False`` hands the library only the minimum workspace, so it projects each
    chunk twice instead of keeping its logits; the outputs are the same. Without ``ws`` the
    "topk_overlap" workspace is allocated (consecutive chunks overlap)."""
    import torch
    N, d = Ht.shape
    V = Wt.shape[0]
    if Wt.shape[1] != d or Ht.dtype != Wt.dtype:
        raise ValueError("expected Ht [N,d] and Wt [V,d] of one dtype")
    for t in (Ht, Wt):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    dt = _dtype_code(Ht)
    global _last_ws
    import weakref
    if ws is None:
        ws = Workspace(N, d, V, K, chunk, dt, Ht.device, kind="topk_overlap" if keep_logits else "topk_min")
        _last_ws = ws
    else:
        _last_ws = weakref.ref(ws)
    nbytes = ws.nbytes if keep_logits else min(ws.nbytes, int(load().fckl_topk_workspace_bytes(N, d, V, K, chunk,
                                                                                                 dt)))
    idx = torch.empty(N, K, dtype=torch.int32, device=Ht.device)
    logp = torch.empty(N, K, dtype=torch.float32, device=Ht.device)
    st = load().fckl_teacher_topk(_ptr(Ht), _ptr(Wt), dt, N, d, V, K, chunk, _ptr(idx), _ptr(logp), ws.ptr,
                                  nbytes, _stream_ptr(stream))
    if st != OK:
        raise FcklError(st, "fckl_teacher_topk")
    return idx, logp


def check(ws=None, stream=None, raise_on_error=True) -> int:
    """Synchronises and reads the device status word of ``ws`` (default: the workspace
    of the last call); raises FcklError on a device-detected error."""
    if ws is None and _last_ws is not None:
        import weakref
        ws = _last_ws() if isinstance(_last_ws, weakref.ref) else _last_ws
    if ws is None:
        return OK
    st = load().fckl_check(ws.ptr, _stream_ptr(stream))
    if st != OK and raise_on_error:
        raise FcklError(st, "device status")
    return st


def launch_count() -> int:
    return int(load().fckl_launch_count())


def profile_enable(on: bool = True) -> None:
    load().fckl_profile_enable(1 if on else 0)


def kernel_names():
    lib = load()
    out = []
    while True:
        n = lib.fckl_kernel_name(len(out))
        if n is None:
            return out
        out.append(n.decode())


def profile_read():
    """{kernel name: (total ms, launches)} since the last read."""
    names = kernel_names()
    ms = (ctypes.c_double * len(names))()
    ln = (ctypes.c_int64 * len(names))()
    st = load().fckl_profile_read(ms, ln, len(names))
    if st != OK:
        raise FcklError(st, "fckl_profile_read")
    return {n: (ms[i], int(ln[i])) for i, n in enumerate(names)}
