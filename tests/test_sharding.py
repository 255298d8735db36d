"""Head sharding across ranks (gloo, world size 2, CPU): the ranks' blocks
partition the (b, h) sequences, and the gathered per-rank results equal the
unsharded result (computed by the fp64 oracle, standing in for the device
path on a machine without GPUs)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mlstm_matrix_memory_gb300 import shard, workloads as W


def test_head_ranges_partition():
    for n in (0, 1, 7, 32, 1024):
        for world in (1, 2, 3, 8):
            spans = [shard.head_range(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            for a, b in zip(spans, spans[1:]):
                assert a[1] == b[0]
            sizes = [e - s for s, e in spans]
            assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = W.sequence_inputs(2, 3, 24, 8, 8, torch.float32, seed=5)
    mine = shard.shard_sequences(x, rank, world)
    h, _, _ = oracle.parallel_stabilized(mine["q"], mine["k"], mine["v"], mine["igate_pre"], mine["fgate_pre"],
                                         nthreads=1)
    local = torch.from_numpy(h[0])
    sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(sizes, torch.tensor([local.shape[0]]))
    pad = torch.zeros((max(int(s) for s in sizes),) + tuple(local.shape[1:]), dtype=local.dtype)
    pad[: local.shape[0]] = local
    parts = [torch.zeros_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad)
    if rank == 0:
        full = torch.cat([p[: int(s)] for p, s in zip(parts, sizes)])
        torch.save(full, result_path)
    dist.destroy_process_group()


def test_sharded_forward_equals_unsharded(tmp_path):
    import oracle
    world, port, path = 2, _free_port(), str(tmp_path / "gathered.pt")
    mp.start_processes(_worker, args=(world, port, path), nprocs=world, start_method="spawn", join=True)
    x = W.sequence_inputs(2, 3, 24, 8, 8, torch.float32, seed=5)
    h, _, _ = oracle.parallel_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    gathered = torch.load(path).numpy()
    assert np.array_equal(gathered, h.reshape(6, 24, 8))
