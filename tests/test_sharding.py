"""Batch sharding over ranks (CPU, gloo, world size 2).

Each rank verifies its shard with the oracle, offsetting the sequence index of
the random draws, and the gathered outputs equal the unsharded run.  A second
case checks that a rank which fails before the collective is reported on the
other rank by the process-group timeout instead of hanging it.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_draft_online_gb300.sharding import gather_rows, shard_bounds


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    import workloads as wl
    from oracle import verify as ov
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = wl.gaussian_pair(7, 3, 500, wl.BF16, 0.9, seed=41, sigma_t=3.0, sigma_d=1.0)
    a, b = shard_bounds(w.B, rank, world)
    r = ov.verify_stochastic(w.target[a:b], w.draft[a:b], w.tokens[a:b], w.dtype, 0.9, seed=5, seq_offset=a)
    out = gather_rows(torch.from_numpy(r.out_tokens), w.B, world)
    n = gather_rows(torch.from_numpy(r.n_accepted), w.B, world)
    if rank == 0:
        full = ov.verify_stochastic(w.target, w.draft, w.tokens, w.dtype, 0.9, seed=5)
        ok = np.array_equal(out.numpy(), full.out_tokens) and np.array_equal(n.numpy(), full.n_accepted)
        with open(result_path, "w") as f:
            f.write("ok" if ok else "mismatch")
    dist.barrier()
    dist.destroy_process_group()


def test_shard_bounds_cover_the_batch():
    for B in (1, 2, 7, 64):
        for world in (1, 2, 3, 8):
            spans = [shard_bounds(B, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1
    with pytest.raises(ValueError):
        shard_bounds(4, 2, 2)


def test_two_rank_sharded_verification_equals_unsharded(tmp_path):
    path = str(tmp_path / "result")
    mp.start_processes(_worker, args=(2, _free_port(), path), nprocs=2, start_method="spawn", join=True)
    assert open(path).read() == "ok"


def _failing_worker(rank, world, port, result_path):
    import datetime
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=5))
    if rank == 1:
        os._exit(0)                       # leaves between steps, before the collective
    try:
        gather_rows(torch.zeros((2, 4), dtype=torch.int32), 4, world)
        msg = "no error"
    except Exception as e:                # noqa: BLE001 -- any collective failure is the expected outcome
        msg = "error: " + type(e).__name__
    with open(result_path, "w") as f:
        f.write(msg)
    os._exit(0)


def test_lost_rank_surfaces_as_an_error(tmp_path):
    path = str(tmp_path / "result")
    ctx = mp.start_processes(_failing_worker, args=(2, _free_port(), path), nprocs=2, start_method="spawn",
                             join=False)
    import time
    deadline = time.time() + 120
    while not ctx.join(timeout=5) and time.time() < deadline:   # join returns once any process exits
        pass
    assert open(path).read().startswith("error")
