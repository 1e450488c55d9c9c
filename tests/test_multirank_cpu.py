"""Two ranks on CPU (gloo): each rank plans its own independent batch; timing is the max over ranks.

The decode path shards by request with no exchange on the data path; the only cross-rank
operations are the benchmark's barrier and max-reduction of the elapsed time, run here.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    from beam_search_shared_gb300 import bsp, synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(4)
    case = synth.make_case(wl, 1000 + 97 * rank, full_step=True)           # the bench's per-rank seed
    g = bsp.geometry(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, case.num_pages, wl.dtype)
    plan, _ = bsp.plan_build(g, wl.batch, wl.beam_width, case.prefix_len, case.tail_len, case.prefix_pages, 8, 152)
    elapsed = 1.0 + rank                                                    # a slower rank 1
    bench.barrier(world)
    mx = bench.reduce_max(elapsed, world)
    out[rank] = (int(case.prefix_len.sum()), plan.num_units, mx)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_shard_and_take_max_time():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    (s0, u0, m0), (s1, u1, m1) = out[0], out[1]
    assert s0 != s1                      # independent batches
    assert u0 % 8 == 0 and u1 % 8 == 0 and u0 >= 32 and u1 >= 32   # (request, split) x 8 kv heads
    assert m0 == m1 == 2.0               # both ranks report the slowest rank's time


def _prefill_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    from beam_search_shared_gb300 import bsp, synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = synth.PREFILL_WORKLOADS["prefill_text_b8"]
    case = synth.make_prefill_case(wl, 2000 + 97 * rank)                  # the bench's per-rank seed
    g = bsp.geometry(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, case.num_pages, wl.dtype)
    plan, _ = bsp.plan_prefill_build(g, wl.batch, case.cached_len, case.prompt_len, case.pages, wl.causal, 152)
    tokens = world * case.rows
    mx = bench.reduce_max(0.5 * (rank + 1), world)
    out[rank] = (case.rows, plan.total_rows, plan.kind, mx, tokens)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_prefill_plans_are_independent():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_prefill_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    (r0, t0, k0, m0, _), (r1, t1, k1, m1, _) = out[0], out[1]
    assert r0 == t0 and r1 == t1 and k0 == k1 == 1       # each rank plans all of its own prompt tokens
    assert r0 != r1                                      # independent batches
    assert m0 == m1 == 1.0
