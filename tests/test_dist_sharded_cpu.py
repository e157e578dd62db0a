"""Token-sharded data parallelism (chunked_kl_loss_head_b300.dist) with two and three gloo
ranks on CPU.

The per-rank steps of the library need a GPU, so here a stand-in runs them with the fp64
oracle on each rank's own rows, with the library's semantics: the forward returns the
rank's partials (loss sum, N), the finish turns the partials summed over ranks into the
mean loss and the gradient scale N_local / N_total, and the backward scales by
grad_loss * grad_scale / (tau N_local).  What is under test is the wrapper's collective
logic: which values cross ranks, in which order, and how they combine.  The result on
every rank must equal the oracle on the whole batch: the same loss, dH of the rank's own
rows, dW of all rows."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The per-rank steps of the loss, done by the oracle on CPU tensors (test stand-in)."""

    def __init__(self, tau):
        self.tau = tau

    def forward_local(self, H, W, topk_idx, topk_logits, valid):
        from oracle import fwd_bwd

        o = fwd_bwd(H.numpy(), W.numpy(), topk_idx.numpy(), topk_logits.numpy(), valid.numpy(), self.tau,
                    want_grads=False)
        return torch.from_numpy(o["lse"]), torch.tensor([o["row_loss"].sum(), float(o["N"])], dtype=torch.float64)

    def finish(self, total, local):
        n = float(total[1])
        loss = torch.tensor(float(total[0]) / n if n > 0 else 0.0, dtype=torch.float64)
        scale = torch.tensor(float(local[1]) / n if n > 0 else 0.0, dtype=torch.float64)
        return loss, scale

    def backward_local(self, H, W, topk_idx, topk_logits, valid, lse, grad_loss, grad_scale):
        from oracle import fwd_bwd

        o = fwd_bwd(H.numpy(), W.numpy(), topk_idx.numpy(), topk_logits.numpy(), valid.numpy(), self.tau,
                    grad=grad_loss * float(grad_scale))
        return torch.from_numpy(o["dH"]), torch.from_numpy(o["dW"])


def _inputs(all_ignored_rank):
    sys.path.insert(0, ROOT)
    from gen import make_small

    x = make_small(T=41, d=12, V=37, K=5, tau=1.7, dtype="f32", seed=3, mask="random", mask_frac=0.2)
    if all_ignored_rank:
        x["valid"][:9] = 0  # rank 0's rows: no valid row on that rank
    return x


def _bounds(T, world):
    """Row ranges of the ranks: uneven shards, rank 0 always rows [0, 9)."""
    cuts = [0, 9, 25, T] if world == 3 else [0, 9, T]
    return list(zip(cuts[:-1], cuts[1:]))


def _worker(rank, world, port, all_ignored_rank, use_module, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from chunked_kl_loss_head_b300.dist import ShardedKL, _ShardedFn

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = _inputs(all_ignored_rank)
        a, b = _bounds(x["H"].shape[0], world)[rank]
        H = torch.from_numpy(x["H"][a:b].astype(np.float64))
        W = torch.from_numpy(x["W"].astype(np.float64))
        idx = torch.from_numpy(x["topk_idx"][a:b])
        lg = torch.from_numpy(x["topk_logits"][a:b])
        va = torch.from_numpy(np.ascontiguousarray(x["valid"][a:b]))
        sharded = ShardedKL(ops=OracleOps(x["cfg"].tau))
        if use_module:
            Hg = H.clone().requires_grad_(True)
            Wg = W.clone().requires_grad_(True)
            loss = _ShardedFn.apply(Hg, Wg, idx, lg, va, sharded)
            (2.5 * loss).backward()
            out[rank] = (float(loss), Hg.grad.numpy().copy(), Wg.grad.numpy().copy())
        else:
            loss = sharded.forward(H, W, idx, lg, va)
            dH, dW = sharded.backward(2.5)
            out[rank] = (float(loss), dH.numpy().copy(), dW.numpy().copy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,all_ignored_rank,use_module", [(2, False, False), (2, True, False), (3, False, False),
                                                               (2, False, True)])
def test_sharded_loss_matches_whole_batch(world, all_ignored_rank, use_module):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, all_ignored_rank, use_module, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(180)
            assert p.exitcode == 0
        res = dict(out)
    sys.path.insert(0, ROOT)
    from oracle import fwd_bwd

    x = _inputs(all_ignored_rank)
    ref = fwd_bwd(x["H"], x["W"], x["topk_idx"], x["topk_logits"], x["valid"], x["cfg"].tau, grad=2.5)
    for r, (a, b) in enumerate(_bounds(x["H"].shape[0], world)):
        loss, dH, dW = res[r]
        assert loss == pytest.approx(ref["loss"], rel=1e-12, abs=0)
        np.testing.assert_allclose(dH, ref["dH"][a:b], rtol=1e-10, atol=1e-15)
        np.testing.assert_allclose(dW, ref["dW"], rtol=1e-10, atol=1e-15)


def test_phases_out_of_order_are_refused():
    sys.path.insert(0, ROOT)
    from chunked_kl_loss_head_b300.dist import ShardedKL

    sh = ShardedKL(ops=OracleOps(1.0), reduce=lambda t: None)
    with pytest.raises(RuntimeError):
        sh.backward_local()
    with pytest.raises(RuntimeError):
        sh.finish(torch.zeros(2, dtype=torch.float64))


def test_two_micro_batches_before_one_backward():
    """Two forwards through one sharded object, then one backward of their sum: each call's
    gradient uses its own rows (one rank; the sum over ranks is the identity)."""
    sys.path.insert(0, ROOT)
    from chunked_kl_loss_head_b300.dist import ShardedKL, _ShardedFn
    from gen import make_small
    from oracle import fwd_bwd

    sh = ShardedKL(ops=OracleOps(1.2), reduce=lambda t: None)
    W = torch.from_numpy(make_small(T=3, d=6, V=29, K=4, tau=1.2, dtype="f32", seed=9)["W"].astype(np.float64))
    Wg = W.clone().requires_grad_(True)
    xs, Hs, total = [], [], 0.0
    for seed in (10, 11):
        x = make_small(T=13, d=6, V=29, K=4, tau=1.2, dtype="f32", seed=seed, mask="random", mask_frac=0.2)
        H = torch.from_numpy(x["H"].astype(np.float64)).requires_grad_(True)
        total = total + _ShardedFn.apply(H, Wg, torch.from_numpy(x["topk_idx"]), torch.from_numpy(x["topk_logits"]),
                                         torch.from_numpy(np.ascontiguousarray(x["valid"])), sh)
        xs.append(x)
        Hs.append(H)
    total.backward()
    dW = 0.0
    for x, H in zip(xs, Hs):
        ref = fwd_bwd(x["H"], W.numpy(), x["topk_idx"], x["topk_logits"], x["valid"], 1.2)
        np.testing.assert_allclose(H.grad.numpy(), ref["dH"], rtol=1e-10, atol=1e-15)
        dW = dW + ref["dW"]
    np.testing.assert_allclose(Wg.grad.numpy(), dW, rtol=1e-10, atol=1e-15)
