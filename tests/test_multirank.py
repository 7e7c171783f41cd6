"""The N > 1 host path of bench.py, run as two gloo ranks on the CPU: the
barrier, the max-over-ranks timing, and the per-rank independent problems
(weak scaling: same shape, different seed, no data-path collective)."""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world),
                       "LOCAL_RANK": str(rank), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    import bench
    from exact_attention_24_gb300.workloads import C3, Workload, make_inputs
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    assert bench.init_dist(w, "gloo")
    bench.barrier(w)
    t = bench.reduce_max(1.5 + rank, w)
    seed = bench.rank_seed(C3.seed, r)
    small = Workload("s", 1, 1, 8, 64, "bf16", True, seed)
    q, _, _ = make_inputs(small)
    out[rank] = (t, seed, float(q.float().sum()))
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_gloo_bench_host_path():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    (t0, s0, q0), (t1, s1, q1) = out[0], out[1]
    assert t0 == t1 == 2.5          # the slowest rank sets the job time
    assert s0 != s1 and q0 != q1    # independent problems of the same shape


def _split_worker(rank, world, port, out):
    """Each rank attends to its own contiguous shard of the keys (positions
    kept absolute for the causal mask), exchanges (O_g, L_g) with an
    all-gather, and merges with the STAGE 3 rescale: the split-key exchange
    a multi-GPU split would do, on gloo."""
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import numpy as np
    import torch.distributed as dist
    from oracle import attention_ref, attention_rows, merge_partials
    dist.init_process_group("gloo")
    r = np.random.default_rng(0)
    n, d = 300, 16
    q, k, v = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, d))
    lo, hi = rank * n // world, (rank + 1) * n // world
    o_g, l_g = attention_rows(q, k, v, 0.25, True, np.arange(n), lo, hi)
    o_all = [torch.zeros(n, d, dtype=torch.float64) for _ in range(world)]
    l_all = [torch.zeros(n, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(o_all, torch.from_numpy(o_g))
    dist.all_gather(l_all, torch.from_numpy(l_g))
    o, l = merge_partials(np.stack([x.numpy() for x in o_all]), np.stack([x.numpy() for x in l_all]))
    of, lf = attention_ref(q, k, v, 0.25, True)
    out[rank] = (float(np.max(np.abs(o - of))), float(np.max(np.abs(l - lf))))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_split_key_exchange():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_split_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    for rank in range(2):
        eo, el = out[rank]
        assert eo < 1e-12 and el < 1e-12
