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


def _run_bench(rank, world, *args):
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=300)


@pytest.mark.timeout(300)
def test_reference_arm_prints_on_rank_zero_only():
    """Under torchrun the reference arm (the float64 oracle on the host) runs
    and prints on rank 0 alone; the other ranks exit 0 without output."""
    import json
    args = ("--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
            "--workload", "B1_H1_N256_D64_f32", "--ref-seconds", "1")
    r1 = _run_bench(1, 2, *args)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_bench(0, 2, *args)
    assert r0.returncode == 0, r0.stderr[-500:]
    rec = json.loads(r0.stdout.strip().splitlines()[-1])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["steps"] == 2
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["cpu_baseline"]["value"] == rec["value"]
