"""Multi-rank plumbing of bench.py on CPU: two gloo ranks, each an independent
replica with its own seed; the step time reported is the maximum over ranks and
nothing else crosses ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from mla_decode_attention_absorbed_gb300.workloads import CONFIGS, make_inputs


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, lr = bench.dist_env()
    active = bench.init_dist(w, "gloo")
    cfg = CONFIGS["tiny"]
    seed = bench.replica_seed(cfg.seed, r)
    inp = make_inputs(cfg.with_(seed=seed))
    local_ms = 1.0 + 2.0 * r
    m = bench.reduce_max(local_ms, active)
    bench.barrier(active)
    q.put((r, w, lr, seed, float(inp["q_nope"].float().sum()), m))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, s0, sum0, m0), (r1, w1, l1, s1, sum1, m1) = res
    assert (r0, r1) == (0, 1) and w0 == w1 == 2 and (l0, l1) == (0, 1)
    assert s0 != s1 and sum0 != sum1          # independent replicas
    assert m0 == m1 == 3.0                    # max over ranks


def test_single_rank_needs_no_process_group():
    assert bench.init_dist(1, "gloo") is False
    assert bench.reduce_max(2.5, False) == 2.5
