"""Token-sharded data parallelism on one GPU: the shards of a batch run one after the
other in one process through chunked_kl_loss_head_b300.dist, with the sums over ranks
done in-process (the partials and dW of the shards added up), and the result is
compared with the oracle on the whole batch: the loss on every shard, dH row by row,
and dW summed over the shards.  The collectives themselves (gloo on CPU) are covered by
test_dist_sharded_cpu.py."""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch

from chunked_kl_loss_head_b300 import FusedChunkedKLLoss
from chunked_kl_loss_head_b300.dist import ShardedFusedChunkedKLLoss, ShardedKL
from gen import make_small
from helpers import TOL, oracle_of, rel, rel_max, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("cuts", [(1700,), (700, 1900), (300,)])
def test_shards_add_up_to_the_whole_batch(dtype, cuts):
    x = make_small(T=3000, d=64, V=9000, K=9, tau=1.4, dtype=dtype, seed=41, mask="random", mask_frac=0.1)
    if cuts == (300,):
        x["valid"][:300] = 0  # the first shard has no valid row
    g = to_device(x)
    bounds = list(zip((0,) + cuts, cuts + (3000,)))
    shards = [ShardedKL(tau=1.4, chunk=1024) for _ in bounds]
    parts = [sh.forward_local(g["H"][a:b], g["W"], g["topk_idx"][a:b], g["topk_logits"][a:b], g["valid"][a:b])
             for sh, (a, b) in zip(shards, bounds)]
    total = torch.stack(parts).sum(0)  # the sum over ranks
    losses = [sh.finish(total).item() for sh in shards]
    grads = [sh.backward_local(2.0) for sh in shards]
    dH = torch.cat([gr[0] for gr in grads]).float().cpu().numpy()
    dW = torch.stack([gr[1] for gr in grads]).sum(0).cpu().numpy()  # the sum over ranks
    ref = oracle_of(x, grad=2.0)
    tol = TOL[dtype]
    errs = dict(loss=max(rel(l, ref["loss"]) for l in losses), dH=rel_max(dH, ref["dH"]), dW=rel_max(dW, ref["dW"]))
    print(dtype, cuts, {k: f"{v:.2e}" for k, v in errs.items()})
    assert len(set(losses)) == 1
    assert errs["loss"] <= tol["loss"] and errs["dH"] <= tol["grad"] and errs["dW"] <= tol["grad"], errs
    assert np.all(dH[~np.asarray(x["valid"]).astype(bool)] == 0.0)


def test_sharded_module_of_one_rank_is_the_module():
    """With one rank (the sum over ranks is the identity) the sharded module gives what
    FusedChunkedKLLoss gives, gradients included, through autograd."""
    x = make_small(T=900, d=96, V=3000, K=9, tau=1.2, dtype="bf16", seed=42, mask="random", mask_frac=0.1)
    d = to_device(x)
    out = []
    for mod in (FusedChunkedKLLoss(tau=1.2, chunk=256),
                ShardedFusedChunkedKLLoss(tau=1.2, chunk=256, reduce=lambda t: None)):
        H = d["H"].clone().requires_grad_(True)
        W = d["W"].clone().requires_grad_(True)
        loss = mod(H, W, d["topk_idx"], d["topk_logits"], d["valid"])
        (0.5 * loss).backward()
        out.append((loss.item(), H.grad.float().cpu().numpy(), W.grad.float().cpu().numpy()))
    (l0, h0, w0), (l1, h1, w1) = out
    assert rel(l1, l0) <= 1e-6
    assert rel_max(h1, h0) <= 1e-2 and rel_max(w1, w0) <= 1e-2
    ref = oracle_of(x, grad=0.5)
    assert rel(l1, ref["loss"]) <= TOL["bf16"]["loss"]
    assert rel_max(h1, ref["dH"]) <= TOL["bf16"]["grad"] and rel_max(w1, ref["dW"]) <= TOL["bf16"]["grad"]


def _free_port():
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def _bench_line(args, torchrun=False):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable]
    if torchrun:
        cmd += ["-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "1", "--master-addr", "127.0.0.1",
                "--master-port", str(_free_port())]
    cmd += [os.path.join(root, "bench.py")] + args
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_sharded_path_under_torchrun():
    """bench.py's token-sharded step on the GPU: an NCCL process group (one rank here) with
    the loss partials and dW all-reduced inside the timed step, against the direct path
    on the same workload: the same loss."""
    args = ["--shape", "8192,2880,201088,100", "--steps", "2", "--warmup", "3", "--no-e2e", "--no-cpu"]
    dp = _bench_line(args + ["--dp"], torchrun=True)
    one = _bench_line(args)
    print(dp["config"]["parallelism"], dp["value"], one["value"], dp["loss"], one["loss"])
    assert dp["config"]["parallelism"].startswith("dp1")
    assert dp["value"] > 0 and dp["gpu_launches"] > one["gpu_launches"]  # + partials and finish
    assert dp["loss"] == one["loss"]
