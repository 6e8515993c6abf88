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
