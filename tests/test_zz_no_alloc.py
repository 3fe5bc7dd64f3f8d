"""fckl_forward_static: the forward pass for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: for example a custom operator inside a
framework or inference server whose pooling allocator owns all device memory (a raw
cudaMalloc there bypasses the pool), or a step loop that must not pay for cudaMalloc and
cudaFree. For them the library keeps its own scratch in a static device array, and this
entry point takes only inputs and outputs. These tests call it through the C ABI and check
that it returns, bit for bit, what the workspace-based fckl_forward returns, on two calls in
a row (the second call reuses the array the first one left behind), and the oracle's values;
that a bad teacher id is reported in its status output and that the following call starts
from a cleared status word; and that a shape whose scratch exceeds the array is refused
before anything runs.

Collected last on purpose (file name), so a run that stops at the first failure has run
every other test before this one.
"""
import ctypes

import numpy as np
import pytest

import synthetic

LOSS_RTOL = 1e-3  # loss relative error against the fp64 oracle


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


def _device_inputs(N, d, V, K, seed):
    import torch
    x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=seed)
    dev = torch.device("cuda")
    t = {"H": torch.from_numpy(x["H"]).to(dev).to(torch.bfloat16),
         "W": torch.from_numpy(x["W"]).to(dev).to(torch.bfloat16),
         "idx": torch.from_numpy(x["idx"]).to(dev),
         "logp": torch.from_numpy(x["logp"]).to(dev)}
    return x, t


def _call_static(f, t, N, d, V, K, chunk):
    """One fckl_forward_static call on poisoned outputs; returns (rc, loss, lse, rl, status)."""
    import torch
    dev = t["H"].device
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    rl = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    status = torch.full((1,), 0x7FFFFFFF, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    st = f(t["H"].data_ptr(), t["W"].data_ptr(), 0, t["idx"].data_ptr(), t["logp"].data_ptr(), N, d, V, K,
           chunk, loss.data_ptr(), lse.data_ptr(), rl.data_ptr(), status.data_ptr(),
           ctypes.c_void_p(stream.cuda_stream))
    torch.cuda.synchronize()
    return st, loss, lse, rl, int(status.item())


@pytest.mark.gpu
def test_static_scratch_forward_matches_workspace_forward(fckl):
    """Two calls in a row on the one static array, each bitwise equal to fckl_forward (same
    kernels in the same order, only the scratch differs), the first also against the oracle."""
    import torch
    from oracle import fckl_oracle as orc

    lib = fckl.load()
    f = _bind(lib)
    cases = [(300, 320, 5000, 40, 128, 21), (256, 3072, 128256, 100, 128, 22)]
    for i, (N, d, V, K, chunk, seed) in enumerate(cases):
        x, t = _device_inputs(N, d, V, K, seed)
        ref_loss, ref_lse, ref_rl = fckl.forward(t["H"], t["W"], t["idx"], t["logp"], chunk, row_loss=True)
        assert fckl.check() == fckl.OK

        st, loss, lse, rl, status = _call_static(f, t, N, d, V, K, chunk)
        assert st == fckl.OK, lib.fckl_last_error()
        assert status == 0
        assert torch.equal(loss, ref_loss)
        assert torch.equal(lse, ref_lse)
        assert torch.equal(rl, ref_rl)

        if i == 0:
            o_loss, o_lse, o_rl = orc.forward(x["H"], x["W"], x["idx"], x["logp"], chunk)
            assert abs(float(loss.item()) - o_loss) <= LOSS_RTOL * abs(o_loss)
            g = lse.cpu().numpy()
            assert np.abs(g - o_lse).max() <= 1e-3 * (1 + np.abs(o_lse).max())
            g = rl.cpu().numpy()
            assert np.abs(g - o_rl).max() <= 1e-3 * (1 + np.abs(o_rl).max())


@pytest.mark.gpu
def test_static_scratch_status_is_reported_then_cleared(fckl):
    """A teacher id outside [0, V) sets bit 0 of the status output; the next call on the same
    array, with clean inputs, starts from a cleared status word and matches fckl_forward."""
    import torch

    lib = fckl.load()
    f = _bind(lib)
    N, d, V, K, chunk = 200, 256, 3000, 24, 64
    _, t = _device_inputs(N, d, V, K, 31)
    bad = dict(t)
    bad["idx"] = t["idx"].clone()
    bad["idx"][7, 3] = V  # one id past the vocabulary
    st, _, _, _, status = _call_static(f, bad, N, d, V, K, chunk)
    assert st == fckl.OK, lib.fckl_last_error()
    assert status & 1 == 1

    ref_loss, ref_lse, ref_rl = fckl.forward(t["H"], t["W"], t["idx"], t["logp"], chunk, row_loss=True)
    assert fckl.check() == fckl.OK
    st, loss, lse, rl, status = _call_static(f, t, N, d, V, K, chunk)
    assert st == fckl.OK, lib.fckl_last_error()
    assert status == 0
    assert torch.equal(loss, ref_loss) and torch.equal(lse, ref_lse) and torch.equal(rl, ref_rl)
