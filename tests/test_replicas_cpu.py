"""The replica path of bench.py (one process per GPU, no data exchange) on the CPU.

Two gloo ranks exercise the rank helpers the GPU run uses over NCCL: the
barrier, and the maximum over ranks that turns per-rank times into the job's
time.  Each rank's replica is its own shard of seeded inputs, and its result
(computed here on the oracle) is what one process gets alone.  The reference
arm's ranks other than 0 exit at once, without output.
"""

from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        r = bench.Ranks(dist)
        r.barrier()
        t = r.max_over_ranks(10.0 + 5.0 * rank)   # per-rank "ms"; the slowest rank wins
        r.barrier()
        out.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    assert got == {0: 15.0, 1: 15.0}


def test_single_process_helpers_are_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks()
    r.barrier()
    assert r.max_over_ranks(3.25) == 3.25


def test_reference_arm_other_ranks_exit_without_output():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip() == ""


def test_torchrun_two_ranks_reference_arm_prints_one_line():
    """The N > 1 launch of bench.py (torchrun, two local ranks, rendezvous on
    127.0.0.1): rank 0 alone times the oracle on the host cores and prints the
    one JSON line (n_gpus 0: no GPU in that arm), rank 1 exits at once, and
    both exit 0.  Runs here without a GPU."""
    import json
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "small", "--ref-seconds", "0.5", "--only", "chunk"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["steps"] == 1 and rec["n_gpus"] == 0
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"


def _shard_main(rank: int, world: int, port: int, out):
    import numpy as np
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from oracle import gla_oracle
    from synth import CHUNK_CONFIGS
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        cfg = CHUNK_CONFIGS["small"]
        q, k, v, a, h0 = bench.replica_inputs(cfg, rank, "cpu")
        o, hT = gla_oracle.forward_torch(q, k, v, a, cfg.scale, h0, nthreads=1)
        tokens = [None] * world
        dist.all_gather_object(tokens, int(q.shape[0] * q.shape[1] * q.shape[2]))
        out.put((rank, np.asarray(o), np.asarray(hT), tokens, bench.job_tokens(cfg, world)))
    finally:
        dist.destroy_process_group()


def test_replica_shards_are_independent_workloads():
    """Two gloo ranks, each with its replica of the small workload, computed on
    the oracle: the ranks hold distinct shards, each rank's result is what one
    process computes alone on that rank's inputs (no data crosses ranks), and
    the job's token count is the sum over the ranks' shards."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from oracle import gla_oracle
    from synth import CHUNK_CONFIGS
    gla_oracle.build()   # once, before the ranks load it
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        r, o, hT, tokens, job = q.get(timeout=300)
        got[r] = (o, hT, tokens, job)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    cfg = CHUNK_CONFIGS["small"]
    for r in range(world):
        qi, ki, vi, ai, h0 = bench.replica_inputs(cfg, r, "cpu")
        o, hT = gla_oracle.forward_torch(qi, ki, vi, ai, cfg.scale, h0, nthreads=1)
        np.testing.assert_array_equal(got[r][0], o)
        np.testing.assert_array_equal(got[r][1], hT)
        assert got[r][2] == [cfg.tokens] * world
        assert got[r][3] == sum(got[r][2])
    assert not np.allclose(got[0][0], got[1][0])
