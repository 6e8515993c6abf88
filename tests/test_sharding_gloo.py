"""Host logic of the data-parallel split, run as two gloo ranks on the CPU.

Each rank takes its batch slice; together the slices cover every batch entry
exactly once, and the bench's max-over-ranks reduction of step times returns
the slowest rank's time.  No rank exchanges any data of the forward itself.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from differential_attention_03_gb300.sharding import batch_slice, weak_scaling_seed


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, global_batch, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    start, stop = batch_slice(global_batch, world, rank)
    mine = torch.zeros(global_batch, dtype=torch.int64)
    mine[start:stop] = 1
    dist.all_reduce(mine)  # coverage count per batch entry
    t = torch.tensor([10.0 + rank], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    seeds = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(seeds, torch.tensor([weak_scaling_seed(4, rank)]))
    if rank == 0:
        out.put((mine.tolist(), float(t.item()), [int(s.item()) for s in seeds]))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("global_batch", [8, 7, 1])
def test_two_gloo_ranks_cover_the_batch_once(global_batch):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, global_batch, q)) for r in range(2)]
    for p in procs:
        p.start()
    cover, tmax, seeds = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert cover == [1] * global_batch
    assert tmax == 11.0
    assert len(set(seeds)) == 2


def test_batch_slice_edges():
    assert batch_slice(5, 3, 0) == (0, 2)
    assert batch_slice(5, 3, 2) == (4, 5)
    assert batch_slice(1, 2, 1) == (1, 1)
    with pytest.raises(ValueError):
        batch_slice(4, 2, 2)


def _bwd_worker(rank, world, port, out):
    # Every rank draws the same global batch, takes its slice, computes the
    # backward of its entries (the oracle stands in for the kernels on the
    # CPU) and sums the shared parameters' gradients over the ranks.
    import numpy as np

    import oracle
    from differential_attention_03_gb300.sharding import allreduce_shared_grads

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r = np.random.default_rng(5)
    B, n, H, d = 5, 6, 2, 4
    x = {k: r.normal(size=(B, n, H, d)) for k in ("q1", "q2", "k1", "k2")}
    x["v"], x["dy"] = r.normal(size=(B, n, H, 2 * d)), r.normal(size=(B, n, H, 2 * d))
    gamma = r.uniform(0.5, 1.5, size=2 * d)
    start, stop = batch_slice(B, world, rank)
    mine = oracle.diff_attn_v1_backward(*(x[k][start:stop] for k in ("q1", "q2", "k1", "k2", "v")), 0.4, 0.3,
                                        gamma, 1e-5, True, x["dy"][start:stop])
    shared = [torch.tensor([mine["dlam"]], dtype=torch.float64), torch.tensor(mine["dgamma"])]
    allreduce_shared_grads(shared)
    full = oracle.diff_attn_v1_backward(*(x[k] for k in ("q1", "q2", "k1", "k2", "v")), 0.4, 0.3, gamma, 1e-5,
                                        True, x["dy"])
    ok_shared = (abs(float(shared[0]) - full["dlam"]) < 1e-10
                 and float(np.max(np.abs(shared[1].numpy() - full["dgamma"]))) < 1e-10)
    ok_local = all(float(np.max(np.abs(mine[k] - full[k][start:stop]))) < 1e-12 for k in ("dq1", "dk2", "dv"))
    flags = torch.tensor([int(ok_shared), int(ok_local)])
    dist.all_reduce(flags, op=dist.ReduceOp.MIN)
    if rank == 0:
        out.put(flags.tolist())
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_sum_the_shared_gradients():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bwd_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    flags = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert flags == [1, 1]  # shared gradients summed to the full batch's; per-entry gradients need no exchange


def test_allreduce_shared_grads_rejects_mixed_dtypes():
    from differential_attention_03_gb300.sharding import allreduce_shared_grads
    with pytest.raises(ValueError):
        allreduce_shared_grads([torch.zeros(1, dtype=torch.float32), torch.zeros(2, dtype=torch.float64)])
