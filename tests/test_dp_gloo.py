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
