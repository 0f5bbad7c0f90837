"""Several GPUs: the step shards by request, with no exchange on the data path.

Requests of one step never read each other's keys (the block-diagonal mask of page
"Continuous Batching" on k4i.top, section "防止跨请求 attention"), so every rank can serve
its own requests with its own pool: each rank runs independent steps (weak scaling) and
only the benchmark's timing is combined across ranks (a barrier and a max).  One process
per GPU, launched by torchrun; the same helpers run on CPU with the gloo backend.
"""
from __future__ import annotations

import os

import numpy as np


def dist_env():
    """(rank, world size, local rank) from the torchrun environment (1 process: 0, 1, 0)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(backend: str = "nccl", device=None):
    """Join the process group when there is more than one rank; returns the dist module or None."""
    _, world, _ = dist_env()
    if world <= 1:
        return None
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        if backend == "nccl":
            dist.init_process_group("nccl", device_id=device)
        else:
            dist.init_process_group(backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """The largest value over all ranks (the slowest rank's time)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: float, world: int, max_ms: float) -> float:
    """Units per second for the whole job: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (max_ms / 1e3)


def shard_requests(num_reqs: int, rank: int, world: int):
    """Contiguous share of a step's requests for one rank (sizes differ by at most one)."""
    lo = (num_reqs * rank) // world
    hi = (num_reqs * (rank + 1)) // world
    return list(range(lo, hi))


def sub_step(inp, reqs):
    """The step restricted to `reqs` (a StepInputs with re-packed rows and metadata, same
    bits): what one rank serves when a step's requests are split across ranks."""
    from .workloads import StepInputs, StepSpec
    spec = inp.spec
    cu = inp.cu_seqlens_q
    rows = np.concatenate([np.arange(cu[r], cu[r + 1]) for r in reqs]) if reqs else np.zeros(0, np.int64)
    q_lens = [spec.q_lens[r] for r in reqs]
    sub = StepSpec(f"{spec.name}-shard", q_lens=q_lens, ctx_lens=[spec.ctx_lens[r] for r in reqs],
                   num_blocks=spec.num_blocks, seed=spec.seed)
    new_cu = np.zeros(len(reqs) + 1, np.int32)
    new_cu[1:] = np.cumsum(q_lens)
    return StepInputs(spec=sub, q=inp.q[rows], k_new=inp.k_new[rows], v_new=inp.v_new[rows],
                      k_prior=[inp.k_prior[r] for r in reqs], v_prior=[inp.v_prior[r] for r in reqs],
                      cu_seqlens_q=new_cu, context_lens=inp.context_lens[reqs].astype(np.int32),
                      block_tables=inp.block_tables[reqs], block_order=inp.block_order), rows
