"""Data-parallel mode: positions split into contiguous ranges over ranks, W replicated, one
all-reduce of dW and of the loss.

The positions of the loss are independent except through dW, a sum over positions, and the
loss, a sum too, so the exchange step is exactly those two sums. The CPU tests run the host
logic on world-size-2 and -3 gloo ranks: each rank takes its range, computes its share with
the fp64 oracle, and the reduced loss and dW must equal the oracle's on the whole problem. The
GPU test runs two ranks on the one GPU, each through the CUDA library on its own range, with the
exchange staged through the host (gloo); the reduced results must match the single-process one
call and the oracle.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import synthetic


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _init(rank, world, port):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    return dist


def test_shards_cover_every_position_once():
    import chunked_kl_loss_gb300 as fckl
    for N in (0, 1, 7, 64, 1001):
        for world in (1, 2, 3, 8):
            ranges = [fckl.shard_range(N, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == N
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [e - s for s, e in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        fckl.shard_range(10, 2, 2)


def _cpu_worker(rank, world, port, out):
    dist = _init(rank, world, port)
    import chunked_kl_loss_gb300 as fckl
    from oracle import fckl_oracle as orc
    N, d, V, K, chunk = 37, 16, 64, 5, 8
    x = synthetic.make_inputs(N, d, V, K, dtype="f32", seed=3)
    s, e = fckl.shard_range(N, rank, world)
    loss, lse, _ = orc.forward(x["H"][s:e], x["W"], x["idx"][s:e], x["logp"][s:e], chunk)
    dH, dW = orc.backward(x["H"][s:e], x["W"], x["idx"][s:e], x["logp"][s:e], 0.5, chunk)
    local = float(np.abs(dW).sum())
    loss_t = torch.tensor([loss], dtype=torch.float64)
    dW_t = torch.from_numpy(dW.copy())
    fckl.allreduce_loss_and_dW(loss_t, dW_t)
    out[rank] = (float(loss_t.item()), dW_t.numpy(), (s, e), dH, local)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_reduced_shards_equal_the_whole_problem(world):
    from oracle import fckl_oracle as orc
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_cpu_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    N, d, V, K, chunk = 37, 16, 64, 5, 8
    x = synthetic.make_inputs(N, d, V, K, dtype="f32", seed=3)
    ref_loss, _, ref_dH, ref_dW = orc.forward_backward(x["H"], x["W"], x["idx"], x["logp"], 0.5, chunk)
    for r in range(world):
        loss, dW, (s, e), dH, local = out[r]
        assert abs(loss - ref_loss) <= 1e-12 * abs(ref_loss)
        assert np.abs(dW - ref_dW).max() <= 1e-12 * np.abs(ref_dW).max()
        assert np.abs(dH - ref_dH[s:e]).max() <= 1e-12 * np.abs(ref_dH).max()
        # one rank's own share is not the whole gradient: the exchange is what completes it
        assert abs(local - np.abs(ref_dW).sum()) > 1e-6 * np.abs(ref_dW).sum()


def _gpu_worker(rank, world, port, out):
    dist = _init(rank, world, port)
    torch.cuda.set_device(0)
    import chunked_kl_loss_gb300 as fckl
    N, d, V, K, chunk = 700, 256, 3000, 24, 128
    x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=5)
    s, e = fckl.shard_range(N, rank, world)
    dev = torch.device("cuda", 0)
    H = torch.from_numpy(x["H"][s:e]).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(x["W"]).to(dev).to(torch.bfloat16)
    idx = torch.from_numpy(x["idx"][s:e]).to(dev)
    logp = torch.from_numpy(x["logp"][s:e]).to(dev)
    loss, lse, dH, dW = fckl.data_parallel_forward_backward(H, W, idx, logp, chunk, grad_scale=0.25)
    fckl.check()
    out[rank] = (float(loss.item()), dW.cpu().numpy(), lse.cpu().numpy(), dH.float().cpu().numpy(), (s, e))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.gpu
def test_two_ranks_on_one_gpu_match_the_one_call(fckl):
    from oracle import fckl_oracle as orc
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_gpu_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    N, d, V, K, chunk = 700, 256, 3000, 24, 128
    x = synthetic.make_inputs(N, d, V, K, dtype="bf16", seed=5)
    dev = torch.device("cuda")
    t = [torch.from_numpy(x[k]).to(dev) for k in ("H", "W", "idx", "logp")]
    loss, lse, dH, dW = fckl.forward_backward(t[0].to(torch.bfloat16), t[1].to(torch.bfloat16), t[2], t[3],
                                              chunk, grad_scale=0.25)
    fckl.check()
    ref_loss, ref_lse, ref_dH, ref_dW = orc.forward_backward(x["H"], x["W"], x["idx"], x["logp"], 0.25, chunk)
    one_dW = dW.cpu().numpy()
    for r in range(world):
        g_loss, g_dW, g_lse, g_dH, (s, e) = out[r]
        assert abs(g_loss - float(loss.item())) <= 1e-6 * abs(ref_loss)
        assert abs(g_loss - ref_loss) <= 1e-3 * abs(ref_loss)
        assert np.abs(g_dW - one_dW).max() <= 1e-5 * np.abs(ref_dW).max()
        assert np.abs(g_dW - ref_dW).max() <= 2e-2 * np.abs(ref_dW).max()
        assert np.array_equal(g_lse, lse.cpu().numpy()[s:e])
        assert np.abs(g_dH - ref_dH[s:e]).max() <= 2e-2 * np.abs(ref_dH).max()
