"""Data-parallel invariant on two CPU ranks (gloo, no GPU).

Splitting the batch across ranks and averaging the per-rank gradients of the
per-rank mean loss gives the full-batch gradient, because every rank holds
the same number of positions. This is the exchange a data-parallel version
of the step would perform once per step (llm.c "State of the Union",
"Multi-GPU training"). The library itself runs one GPU per process and
never exchanges anything; this pins the oracle-side arithmetic of the shard.
"""
import os

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import gpt2_ref as R
from step_gpt_train_gb300 import data

CFG = R.Config(n_layer=1, n_embd=32, n_head=2, vocab=64, vocab_padded=64, max_T=16)


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    params = R.init_params(CFG, 99)
    tok, tgt = data.batches("uniform", 4, 16, 1, 21, vocab=64)
    b = 4 // world
    _, cache = R.forward(CFG, params, tok[0, rank * b:(rank + 1) * b], tgt[0, rank * b:(rank + 1) * b])
    grads = R.backward(CFG, cache)
    names = sorted(grads)
    flat = torch.tensor(np.concatenate([grads[n].reshape(-1) for n in names]))
    dist.all_reduce(flat, op=dist.ReduceOp.SUM)
    flat /= world
    if rank == 0:
        np.save(os.path.join(out_dir, "avg.npy"), flat.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_dp_average_equals_full_batch(tmp_path):
    port = 29500 + os.getpid() % 1000
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    avg = np.load(tmp_path / "avg.npy")
    params = R.init_params(CFG, 99)
    tok, tgt = data.batches("uniform", 4, 16, 1, 21, vocab=64)
    _, cache = R.forward(CFG, params, tok[0], tgt[0])
    grads = R.backward(CFG, cache)
    full = np.concatenate([grads[n].reshape(-1) for n in sorted(grads)])
    assert np.allclose(avg, full, rtol=1e-12, atol=1e-15)


def _zero1_worker(rank, world, port, out_dir):
    """ZeRO-1 on CPU ranks: each rank holds the full parameters, computes the
    gradient of its share of the batch, takes the average gradient of its own
    shard of the flat layout (an all-reduce here; a reduce-scatter moves only
    the shard), applies AdamW to that shard of the masters and moments, and the
    updated shards are all-gathered."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    params = R.init_params(CFG, 99)
    names = sorted(params)
    theta = np.concatenate([params[n].reshape(-1).astype(np.float64) for n in names])
    wd_flat = np.concatenate([np.full(params[n].size, 0.1 if R.decays(n, params[n]) else 0.0) for n in names])
    tok, tgt = data.batches("uniform", 4, 16, 1, 21, vocab=64)
    b = 4 // world
    _, cache = R.forward(CFG, params, tok[0, rank * b:(rank + 1) * b], tgt[0, rank * b:(rank + 1) * b])
    grads = R.backward(CFG, cache)
    flat = torch.tensor(np.concatenate([grads[n].reshape(-1) for n in names]).astype(np.float64))
    dist.all_reduce(flat, op=dist.ReduceOp.SUM)
    g = flat.numpy() / world
    n = theta.size
    lo, hi = rank * n // world, (rank + 1) * n // world
    th, _, _ = R.adamw_update(theta[lo:hi], g[lo:hi], np.zeros(hi - lo), np.zeros(hi - lo), 1e-3, 0.9, 0.95, 1e-8,
                              wd_flat[lo:hi], 1)
    parts = [torch.zeros(((r + 1) * n // world) - r * n // world, dtype=torch.float64) for r in range(world)]
    dist.all_gather(parts, torch.tensor(th))
    if rank == 0:
        np.save(os.path.join(out_dir, "theta.npy"), torch.cat(parts).numpy())
        np.save(os.path.join(out_dir, "grad.npy"), g)
    dist.barrier()
    dist.destroy_process_group()


def test_zero1_sharded_adamw_equals_full_update(tmp_path):
    """The all-gathered ZeRO-1 update equals one AdamW step of the whole flat
    parameter vector with the same averaged gradient (exactly: the update is
    elementwise), and that gradient is the full batch's."""
    port = 30500 + os.getpid() % 1000
    mp.start_processes(_zero1_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    got = np.load(tmp_path / "theta.npy")
    g = np.load(tmp_path / "grad.npy")
    params = R.init_params(CFG, 99)
    names = sorted(params)
    theta = np.concatenate([params[n].reshape(-1).astype(np.float64) for n in names])
    wd_flat = np.concatenate([np.full(params[n].size, 0.1 if R.decays(n, params[n]) else 0.0) for n in names])
    ref, _, _ = R.adamw_update(theta, g, np.zeros_like(theta), np.zeros_like(theta), 1e-3, 0.9, 0.95, 1e-8,
                               wd_flat, 1)
    assert np.array_equal(got, ref)
    tok, tgt = data.batches("uniform", 4, 16, 1, 21, vocab=64)
    _, cache = R.forward(CFG, params, tok[0], tgt[0])
    full = R.backward(CFG, cache)
    assert np.allclose(g, np.concatenate([full[n].reshape(-1) for n in names]), rtol=1e-12, atol=1e-15)
