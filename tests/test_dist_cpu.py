"""The multi-process timing logic of bench.py on CPU (gloo, two ranks).

Under torchrun every rank of the benchmark runs T tokens of its own (weak scaling), and
the job's time is the slowest rank's.  These tests run that host logic (the max over
ranks and the whole-job rate) with two gloo ranks, and launch the reference arm under
torchrun with two processes (rank 0 alone works and prints one line), and check that the
ranks' inputs share W and differ in their rows.  The token-sharded loss itself, with its
all-reduces, is covered by test_dist_sharded_cpu.py."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, ws = bench.dist_env()
        t = bench.max_over_ranks(10.0 + 5.0 * rank, dist)
        out[rank] = (r, lr, ws, t, bench.job_rate(1000, ws, t / 1e3))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_two_gloo_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(2):
        rank, local_rank, world, t, rate = res[r]
        assert (rank, local_rank, world) == (r, r, 2)
        assert t == 15.0  # both ranks see the slowest rank's time
        assert rate == pytest.approx(2 * 1000 / 0.015)


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--config", "tiny_fp32",
           "--ref-rows", "4"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_ranks_share_W_and_own_their_rows():
    """Each rank of the benchmark's token-sharded step holds the same lm_head W and its own
    rows; rank 0's inputs are the single-GPU workload's."""
    import numpy as np

    sys.path.insert(0, ROOT)
    import bench
    from gen import CONFIGS, make_inputs

    cfg = CONFIGS["tiny_fp32"]
    r0, r1 = bench.rank_inputs(cfg, 0), bench.rank_inputs(cfg, 1)
    one = make_inputs(cfg)
    assert np.array_equal(r0["W"], r1["W"])
    assert not np.array_equal(r0["H"], r1["H"]) and not np.array_equal(r0["topk_idx"], r1["topk_idx"])
    for k in ("H", "W", "topk_idx", "topk_logits", "valid"):
        assert np.array_equal(r0[k], one[k]), k
