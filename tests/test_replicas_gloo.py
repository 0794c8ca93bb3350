"""The multi-rank path of the bench, on CPU with the gloo backend (world size 2):
ranks draw distinct, reproducible batches, and the timing reduction gives every
rank the slowest rank's time and the whole-job rate."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import kpool_inputs as KI
from dsa_indexer_sparse_kpool_b300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        spec = KI.named("tiny")
        spec.seed = replicas.rank_seed(spec.seed, rank)
        wl = KI.make(spec)
        local_ms = [1.0 + rank, 5.0 - rank]          # rank 0 slower on the second entry
        replicas.barrier()
        mx = replicas.max_over_ranks(local_ms)
        rate = replicas.job_rate(wl.NQ, world, mx[0] * 1e-3)
        np.save(os.path.join(out_dir, f"r{rank}.npy"),
                np.array([spec.seed, mx[0], mx[1], rate, float(KI.bits(wl.keys)[:64].astype(np.int64).sum())]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    r0, r1 = (np.load(tmp_path / f"r{r}.npy") for r in range(world))
    assert r0[0] != r1[0]                              # distinct seeds ...
    assert r0[4] != r1[4]                              # ... give distinct batches
    assert r0[1] == r1[1] == 2.0 and r0[2] == r1[2] == 5.0   # max over ranks, on every rank
    assert r0[3] == r1[3] == pytest.approx(4 * 2 / 2.0e-3)   # 4 queries x 2 ranks / 2 ms


def test_single_process_is_identity():
    assert replicas.max_over_ranks([3.0, 1.5]) == [3.0, 1.5]
    assert replicas.rank_seed(1, 0) == 1 and replicas.rank_seed(1, 3) == 3001
