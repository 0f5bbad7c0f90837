"""The several-rank path on CPU: two gloo ranks, each serving its own share of a step's
requests with the oracle, and the benchmark's cross-rank timing helpers.  Requests never
exchange data, so the shards put together equal the whole step exactly."""
import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp

import oracle
from continuous_batching_paged_step_gb300 import replicas
from continuous_batching_paged_step_gb300 import workloads as wl


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist = replicas.init("gloo")
    assert replicas.dist_env() == (rank, world, rank)
    inp = wl.make_inputs(wl.small_mixed_step(n_decode=6, chunks=((40, 9), (33, 0)), ctx_range=(1, 200),
                                             num_blocks=256))
    reqs = replicas.shard_requests(inp.spec.num_reqs, rank, world)
    sub, rows = replicas.sub_step(inp, reqs)
    out = oracle.step_reference(sub)                     # this rank's requests only
    np.save(os.path.join(out_dir, f"rank{rank}_out.npy"), out)
    np.save(os.path.join(out_dir, f"rank{rank}_rows.npy"), rows)
    replicas.barrier(dist)
    slowest = replicas.max_over_ranks(dist, 10.0 * (rank + 1))
    with open(os.path.join(out_dir, f"rank{rank}_max.txt"), "w") as f:
        f.write(repr(slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_a_step(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    inp = wl.make_inputs(wl.small_mixed_step(n_decode=6, chunks=((40, 9), (33, 0)), ctx_range=(1, 200),
                                             num_blocks=256))
    whole = oracle.step_reference(inp)
    got = np.full_like(whole, np.nan)
    seen = []
    for r in range(world):
        rows = np.load(tmp_path / f"rank{r}_rows.npy")
        got[rows] = np.load(tmp_path / f"rank{r}_out.npy")
        seen.append(rows)
        assert float(open(tmp_path / f"rank{r}_max.txt").read()) == 20.0   # the slowest rank's time
    assert sorted(np.concatenate(seen).tolist()) == list(range(inp.spec.num_tokens))
    assert np.array_equal(got, whole)


def test_shards_cover_requests_once():
    for n in (1, 7, 66, 256):
        for world in (1, 2, 3, 8):
            parts = [replicas.shard_requests(n, r, world) for r in range(world)]
            assert sum(parts, []) == list(range(n))
            assert max(map(len, parts)) - min(map(len, parts)) <= 1


def test_aggregate_rate_is_all_units_over_slowest_time():
    assert replicas.aggregate_rate(1000, 4, 500.0) == 8000.0
