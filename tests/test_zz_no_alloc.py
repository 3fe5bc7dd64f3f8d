"""fckl_forward_static: the forward pass for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: for example a custom operator inside a
framework or inference server whose pooling allocator owns all device memory (a raw
cudaMalloc there bypasses the pool), or a step loop that must not pay for cudaMalloc and
cudaFree. For them the library keeps its own scratch in a static device array, and this
entry point takes only inputs and outputs. These tests call it through the C ABI and check
that it returns what the workspace-based fckl_forward returns, on two calls in a row (the
second call reuses the array the first one left behind), and that a shape whose scratch
exceeds the array is refused before anything runs.

Collected last on purpose (file name), so a run that stops at the first failure has run
every other test before this one.
"""
import ctypes

import numpy as np
import pytest

import synthetic

LOSS_RTOL = 1e-3


def _bind(lib):
    f = lib.fckl_forward_static
    vp = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, ctypes.c_int, vp, vp, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, vp, vp, vp, vp, vp]
    return f


def test_oversized_shape_is_refused_before_any_launch(fckl):
    lib = fckl.load()
    f = _bind(lib)
    before = lib.fckl_launch_count()
    p = ctypes.c_void_p(256)  # never dereferenced: the size check fails first
    # chunk 8192 at K=100, V=128256 needs ~56 MB of scratch, above the 32 MiB array
    st = f(p, p, 0, p, p, 65536, 3072, 128256, 100, 8192, p, p, p, p, ctypes.c_void_p(0))
    assert st == fckl.ERR_WORKSPACE
    assert b"maximum" in lib.fckl_last_error()
    # fp32 inputs are not taken by this entry point
    assert f(p, p, 1, p, p, 64, 256, 4096, 16, 16, p, p, p, p, ctypes.c_void_p(0)) == fckl.ERR_UNSUPPORTED
    assert lib.fckl_launch_count() == before


@pytest.mark.gpu
def test_static_scratch_forward_matches_workspace_forward(fckl):
    import torch

    lib = fckl.load()
    f = _bind(lib)
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    cases = [(300, 320, 5000, 40, 128, 21), (256, 3072, 128256, 100, 128, 22)]
    for N, d, V, K, chunk, seed in cases:  # two calls in a row on the same static array
        x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=seed)
        H = torch.from_numpy(x["H"]).to(dev).to(torch.bfloat16)
        W = torch.from_numpy(x["W"]).to(dev).to(torch.bfloat16)
        idx = torch.from_numpy(x["idx"]).to(dev)
        logp = torch.from_numpy(x["logp"]).to(dev)

        ref_loss, ref_lse, ref_rl = fckl.forward(H, W, idx, logp, chunk, row_loss=True)
        fckl.check()

        loss = torch.full((1,), float("nan"), dtype=torch.float32, device=dev)
        lse = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
        rl = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
        status = torch.full((1,), 0x7FFFFFFF, dtype=torch.int32, device=dev)
        st = f(H.data_ptr(), W.data_ptr(), 0, idx.data_ptr(), logp.data_ptr(), N, d, V, K, chunk,
               loss.data_ptr(), lse.data_ptr(), rl.data_ptr(), status.data_ptr(),
               ctypes.c_void_p(stream.cuda_stream))
        assert st == fckl.OK, lib.fckl_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0

        a, b = float(loss.item()), float(ref_loss.item())
        assert abs(a - b) <= LOSS_RTOL * abs(b)
        g, r = lse.cpu().numpy(), ref_lse.cpu().numpy()
        assert np.abs(g - r).max() <= 1e-3 * (1 + np.abs(r).max())
        g, r = rl.cpu().numpy(), ref_rl.cpu().numpy()
        assert np.abs(g - r).max() <= 1e-3 * (1 + np.abs(r).max())
