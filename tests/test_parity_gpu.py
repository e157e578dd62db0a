"""CUDA path vs the fp64 oracle, element by element, on seeded inputs that span
several tiles, several chunks and vocab stripes, and ragged tails, plus the
degenerate cases of the loss.  Everything goes through the C-ABI."""

import numpy as np
import pytest
import torch

from chunked_kl_loss_head_b300 import api
from gen import CONFIGS, make_inputs, make_small
from helpers import TOL, oracle_of, rel, rel_max, to_device

pytestmark = pytest.mark.gpu


def run_gpu(x, chunk, grad_loss=1.0):
    cfg = x["cfg"]
    d = to_device(x)
    T, dd = d["H"].shape
    V, K = d["W"].shape[0], d["topk_idx"].shape[1]
    ws = api.workspace(T, dd, V, K, chunk, d["H"].dtype)
    loss, lse, rl = api.forward(d["H"], d["W"], d["topk_idx"], d["topk_logits"], d["valid"], cfg.tau, chunk, ws=ws,
                                want_row_loss=True)
    dH, dW = api.backward(d["H"], d["W"], d["topk_idx"], d["topk_logits"], d["valid"], lse, cfg.tau, chunk,
                          grad_loss=grad_loss, ws=ws)
    status = api.fckl_get_error(ws)
    torch.cuda.synchronize()
    return dict(loss=loss.item(), lse=lse.cpu().numpy(), row_loss=rl.cpu().numpy(),
                dH=dH.float().cpu().numpy(), dW=dW.cpu().numpy(), status=status)


def check(x, got, grad_loss=1.0, label=""):
    tol = TOL[x["cfg"].dtype]
    ref = oracle_of(x, grad=grad_loss)
    assert got["status"] == 0, api.fckl_status_string(got["status"])
    errs = dict(loss=rel(got["loss"], ref["loss"]), lse=rel_max(got["lse"], ref["lse"]),
                row_loss=rel_max(got["row_loss"], ref["row_loss"]), dH=rel_max(got["dH"], ref["dH"]),
                dW=rel_max(got["dW"], ref["dW"]))
    print(label, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["loss"] <= tol["loss"], errs
    assert errs["lse"] <= tol["loss"], errs
    assert errs["row_loss"] <= tol["loss"], errs
    assert errs["dH"] <= tol["grad"], errs
    assert errs["dW"] <= tol["grad"], errs
    valid = np.asarray(x["valid"]).astype(bool)
    assert np.all(got["dH"][~valid] == 0.0), "ignored rows must have dH exactly 0"
    assert np.all(got["row_loss"][~valid] == 0.0)
    return errs


# ------------------------------------------------------------------------------ GEMM engine


@pytest.mark.parametrize("a_mn,b_mn,pair", [(0, 0, 1), (1, 0, 1), (0, 0, 0), (0, 1, 0), (1, 0, 0), (1, 1, 0)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (304, 520, 200), (1000, 2880, 136), (8, 8, 8), (520, 224, 4104)])
def test_engine_gemm_layouts(a_mn, b_mn, pair, M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N + K)
    A = torch.randn((K, M) if a_mn else (M, K), generator=g).to(torch.bfloat16)
    B = torch.randn((K, N) if b_mn else (N, K), generator=g).to(torch.bfloat16)
    A64 = A.double().T if a_mn else A.double()
    B64 = B.double() if b_mn else B.double().T
    ref = (A64 @ B64).numpy()
    D = torch.full((M, N), float("nan"), device="cuda")
    api.fckl_debug_gemm_bf16(A.cuda(), B.cuda(), D, M, N, K, a_mn, b_mn, pair)
    torch.cuda.synchronize()
    err = rel_max(D.cpu().numpy(), ref)
    assert err <= 1e-5, err


# ------------------------------------------------------------------------------ loss parity


@pytest.mark.parametrize("chunk", [64, 16, 7])
def test_tiny_fp32_config(chunk):
    x = make_inputs(CONFIGS["tiny_fp32"])
    check(x, run_gpu(x, chunk), label=f"tiny_fp32 chunk={chunk}")


def test_fp32_several_chunks_and_stripes():
    x = make_small(T=4200, d=40, V=10000, K=5, tau=1.3, dtype="f32", seed=3, mask="random", mask_frac=0.1)
    check(x, run_gpu(x, 4096), label="f32 multi-chunk/stripe")


def test_bf16_several_chunks_and_stripes():
    # stripes of 16384 vocab columns: 5 stripes, the last ragged (4464 columns), so the three
    # gradient buffers rotate; two backward blocks (4096 + 904 rows)
    x = make_small(T=5000, d=64, V=70000, K=13, tau=1.5, dtype="bf16", seed=1, mask="random", mask_frac=0.1)
    check(x, run_gpu(x, 4096), label="bf16 multi-chunk/stripe")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chunk_above_the_backward_block(dtype):
    # chunk 6000: forward chunks of 6000 + 3000 rows, backward blocks of 4096 + 4096 + 808
    x = make_small(T=9000, d=64, V=20000, K=11, tau=1.2, dtype=dtype, seed=15, mask="random", mask_frac=0.1)
    a = run_gpu(x, 6000)
    check(x, a, label=f"{dtype} chunk 6000")
    b = run_gpu(x, 4096)
    # the backward blocks are the same as chunk 4096's.  dW is bit for bit equal: each block
    # writes each dW element once, in block order.  dH's fp32 accumulator takes one
    # reduce-add per vocab stripe, and tiles of consecutive stripes overlap in time, so the
    # order of those adds (dH's last bits) may differ from run to run.
    assert a["loss"] == b["loss"]
    np.testing.assert_array_equal(a["lse"], b["lse"])
    np.testing.assert_array_equal(a["dW"], b["dW"])
    assert rel_max(a["dH"], b["dH"]) <= TOL[dtype]["grad"]


@pytest.mark.parametrize("chunk", [128, 100, 1000])
def test_bf16_ragged_tiles(chunk):
    x = make_small(T=300, d=200, V=1000, K=7, tau=0.8, dtype="bf16", seed=2, mask="random", mask_frac=0.2)
    check(x, run_gpu(x, chunk), label=f"bf16 ragged chunk={chunk}")


def test_bf16_uniform_ids_onehot_teacher():
    x = make_small(T=700, d=128, V=3000, K=10, tau=1.0, dtype="bf16", seed=4, ids="uniform", onehot_frac=0.1,
                   logit_offset=10.0)
    check(x, run_gpu(x, 512), label="bf16 uniform ids / one-hot")


def test_bf16_chunk_invariance_of_loss():
    x = make_small(T=5000, d=64, V=20000, K=13, tau=1.5, dtype="bf16", seed=1, mask="random", mask_frac=0.1)
    runs = [run_gpu(x, c) for c in (4096, 1000, 5000, 333)]
    for r in runs[1:]:
        assert r["loss"] == runs[0]["loss"], "loss depends on the chunk size"
        np.testing.assert_array_equal(r["lse"], runs[0]["lse"])
        np.testing.assert_array_equal(r["row_loss"], runs[0]["row_loss"])
        assert rel_max(r["dW"], runs[0]["dW"]) <= 1e-3
        assert rel_max(r["dH"], runs[0]["dH"]) <= 1e-2


# ------------------------------------------------------------------------------ edge cases


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_no_valid_rows(dtype):
    x = make_small(T=200, d=64, V=600, K=4, tau=1.0, dtype=dtype, seed=6)
    x["valid"] = np.zeros(200, np.uint8)
    got = run_gpu(x, 128)
    assert got["status"] == 0
    assert got["loss"] == 0.0
    assert not got["dH"].any() and not got["dW"].any()
    ref = oracle_of(x, want_grads=False)
    assert rel_max(got["lse"], ref["lse"]) <= TOL[dtype]["loss"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 5, 129])
def test_short_inputs(dtype, T):
    x = make_small(T=T, d=32, V=300, K=3, tau=2.0, dtype=dtype, seed=7 + T)
    check(x, run_gpu(x, 64), label=f"{dtype} T={T}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_k_equals_one_and_v(dtype):
    x = make_small(T=50, d=16, V=64, K=1, tau=1.0, dtype=dtype, seed=8)
    check(x, run_gpu(x, 32), label=f"{dtype} K=1")
    x = make_small(T=50, d=16, V=64, K=64, tau=1.7, dtype=dtype, seed=9, ids="uniform")
    check(x, run_gpu(x, 32), label=f"{dtype} K=V")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_duplicate_ids_add_up(dtype):
    x = make_small(T=40, d=24, V=500, K=6, tau=1.0, dtype=dtype, seed=10)
    x["topk_idx"][:, 1] = x["topk_idx"][:, 0]
    x["topk_idx"][3, :] = 7
    check(x, run_gpu(x, 16), label=f"{dtype} duplicate ids")


@pytest.mark.parametrize("V", [(1 << 24) - 2, (1 << 24) + 5])
@pytest.mark.parametrize("K", [10, 100])
def test_vocabulary_at_the_24_bit_edge(V, K):
    """Teacher preparation packs (id, position) into 32-bit sort keys below V = 2^24 - 1 and
    into 64-bit keys from there on: both sides of the edge, with ids planted at the top of
    the vocabulary and duplicated, through the whole loss."""
    x = make_small(T=24, d=8, V=V, K=K, tau=1.3, dtype="bf16", seed=33, ids="uniform", mask="random", mask_frac=0.2)
    x["topk_idx"][:, 0] = V - 1
    x["topk_idx"][:, 1] = V - 2
    x["topk_idx"][3, 2] = V - 1  # a duplicate
    x["topk_idx"][5, 4] = x["topk_idx"][5, 3]
    ref = oracle_of(x, row_block=4)
    got = run_gpu(x, 16)
    tol = TOL["bf16"]
    assert got["status"] == 0
    errs = dict(loss=rel(got["loss"], ref["loss"]), lse=rel_max(got["lse"], ref["lse"]),
                row_loss=rel_max(got["row_loss"], ref["row_loss"]), dH=rel_max(got["dH"], ref["dH"]),
                dW=rel_max(got["dW"], ref["dW"]))
    print(V, K, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["loss"] <= tol["loss"] and errs["lse"] <= tol["loss"] and errs["row_loss"] <= tol["loss"], errs
    assert errs["dH"] <= tol["grad"] and errs["dW"] <= tol["grad"], errs


def test_grad_scale_and_grad_loss():
    x = make_small(T=256, d=64, V=800, K=5, tau=1.0, dtype="bf16", seed=11, mask="random", mask_frac=0.1)
    a = run_gpu(x, 128, grad_loss=2.5)
    check(x, a, grad_loss=2.5, label="grad_loss=2.5")
    d = to_device(x)
    ws = api.workspace(256, 64, 800, 5, 128, torch.bfloat16)
    loss, lse = api.forward(d["H"], d["W"], d["topk_idx"], d["topk_logits"], d["valid"], 1.0, 128, ws=ws)
    gs = torch.tensor(2.5, device="cuda")
    dH, dW = api.backward(d["H"], d["W"], d["topk_idx"], d["topk_logits"], d["valid"], lse, 1.0, 128, 1.0, ws=ws,
                          grad_scale=gs)
    # the same scale given two ways gives the same bits; V = 800 is one vocab stripe, so each
    # dH element takes a single reduce-add and dH is bit-reproducible too
    np.testing.assert_array_equal(dW.cpu().numpy(), a["dW"])
    np.testing.assert_array_equal(dH.float().cpu().numpy(), a["dH"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bad_index_reports_status(dtype):
    x = make_small(T=100, d=32, V=400, K=4, tau=1.0, dtype=dtype, seed=12)
    x["topk_idx"][5, 2] = 400
    x["topk_idx"][9, 0] = -3
    got = run_gpu(x, 64)
    assert got["status"] == 5
    assert np.isfinite(got["lse"]).all()
    # the status word is cleared by the read
    d = to_device(x)
    ws = api.workspace(100, 32, 400, 4, 64, d["H"].dtype)
    assert api.fckl_get_error(ws) == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_negative_grad_loss(dtype):
    """A negative gradient of the loss (g = -1.5): the gradient tiles carry the sign."""
    x = make_small(T=700, d=64, V=5000, K=9, tau=1.1, dtype=dtype, seed=34, mask="random", mask_frac=0.1)
    check(x, run_gpu(x, 256, grad_loss=-1.5), grad_loss=-1.5, label=f"{dtype} g=-1.5")


@pytest.mark.parametrize("dtype,tau", [("bf16", 0.05), ("bf16", 30.0), ("f32", 0.2), ("f32", 30.0)])
def test_extreme_temperatures(dtype, tau):
    """Sharp and flat distributions.  At tau = 0.05 the scaled student logits z/tau reach
    about 100 (most of a row's exponentials underflow next to its max, so the online max
    must be right tile by tile) and both softmaxes are near one-hot; at
    tau = 30 both are near uniform, so q - p is small everywhere and dz is a difference of
    close numbers.  Teacher logits sit at an offset of 40."""
    x = make_small(T=700, d=64, V=3000, K=17, tau=tau, dtype=dtype, seed=61, mask="random", mask_frac=0.1,
                   logit_offset=40.0)
    check(x, run_gpu(x, 256), label=f"{dtype} tau={tau}")


@pytest.mark.parametrize("dtype,K", [("f32", 13), ("bf16", 13), ("bf16", 200)])
def test_absent_entries(dtype, K):
    """Rows with fewer than K cached pairs, padded with logit -inf: such a pair has p = 0
    and adds nothing (0 log 0 = 0); the oracle is the definition over p's support.  K = 200
    takes the teacher prep that ranks ids instead of sorting them in registers."""
    x = make_small(T=3000, d=64, V=9000, K=K, tau=1.1, dtype=dtype, seed=67, mask="random", mask_frac=0.1)
    rng = np.random.default_rng(67)
    rows = rng.choice(3000, 1200, replace=False)
    for t, n in zip(rows, rng.integers(1, K, size=1200)):  # keep at least one finite logit
        x["topk_logits"][t, K - n:] = -np.inf
    got = run_gpu(x, 1024)
    assert np.isfinite(got["loss"]) and np.all(np.isfinite(got["row_loss"]))
    check(x, got, label=f"{dtype} K={K} -inf padded rows")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ignored_rows_hold_anything(dtype):
    """NaN and infinite teacher logits in ignored rows change no output: the same loss,
    lse, per-row losses and dW bit for bit as with finite ones, and dH within the order
    of its reduce-adds (its ignored rows exactly 0)."""
    x = make_small(T=5000, d=64, V=20000, K=9, tau=1.3, dtype=dtype, seed=71, mask="random", mask_frac=0.2)
    a = run_gpu(x, 4096)
    ign = ~np.asarray(x["valid"]).astype(bool)
    junk = np.array([np.nan, np.inf, -np.inf], np.float32)
    x["topk_logits"][ign] = junk[np.arange(int(ign.sum()) * 9).reshape(-1, 9) % 3]
    x["topk_logits"][np.nonzero(ign)[0][:5]] = np.nan
    b = run_gpu(x, 4096)
    assert b["loss"] == a["loss"]
    np.testing.assert_array_equal(b["lse"], a["lse"])
    np.testing.assert_array_equal(b["row_loss"], a["row_loss"])
    np.testing.assert_array_equal(b["dW"], a["dW"])
    assert np.all(np.isfinite(b["dH"])) and rel_max(b["dH"], a["dH"]) <= TOL[dtype]["grad"]
    check(x, b, label=f"{dtype} ignored rows with NaN / inf logits")


def test_autograd_module_matches_abi():
    from chunked_kl_loss_head_b300 import FusedChunkedKLLoss

    x = make_small(T=300, d=64, V=900, K=6, tau=1.5, dtype="f32", seed=13, mask="random", mask_frac=0.1)
    d = to_device(x)
    H = d["H"].clone().requires_grad_(True)
    W = d["W"].clone().requires_grad_(True)
    loss = FusedChunkedKLLoss(tau=1.5, chunk=128)(H, W, d["topk_idx"], d["topk_logits"], d["valid"])
    (3.0 * loss).backward()
    ref = oracle_of(x, grad=3.0)
    assert rel(loss.item(), ref["loss"]) <= 1e-5
    assert rel_max(H.grad.cpu().numpy(), ref["dH"]) <= 1e-4
    assert rel_max(W.grad.cpu().numpy(), ref["dW"]) <= 1e-4


def test_autograd_module_bf16():
    from chunked_kl_loss_head_b300 import FusedChunkedKLLoss

    x = make_small(T=600, d=96, V=3000, K=9, tau=1.2, dtype="bf16", seed=14, mask="random", mask_frac=0.1)
    d = to_device(x)
    H = d["H"].clone().requires_grad_(True)
    W = d["W"].clone().requires_grad_(True)
    loss = FusedChunkedKLLoss(tau=1.2, chunk=256)(H, W, d["topk_idx"], d["topk_logits"], d["valid"])
    (0.5 * loss).backward()
    ref = oracle_of(x, grad=0.5)
    assert H.grad.dtype == torch.bfloat16 and W.grad.dtype == torch.bfloat16
    assert rel(loss.item(), ref["loss"]) <= TOL["bf16"]["loss"]
    assert rel_max(H.grad.float().cpu().numpy(), ref["dH"]) <= TOL["bf16"]["grad"]
    assert rel_max(W.grad.float().cpu().numpy(), ref["dW"]) <= TOL["bf16"]["grad"]


def test_cast_matches_round_to_nearest_even():
    """The library's float32 -> bfloat16 cast against torch's (round to nearest, ties to even),
    bit for bit, on values that include exact ties, subnormals, infinities and signed zeros
    (NaNs, which some random tie patterns are, are left out: their payloads may differ)."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn(4096, generator=g) * torch.exp2(torch.randint(-130, 40, (4096,), generator=g).float())
    ties = (torch.randint(0, 1 << 16, (256,), generator=g, dtype=torch.int32) << 16) | 0x8000
    x[:256] = ties.view(torch.float32)
    x[256:260] = torch.tensor([float("inf"), -float("inf"), 0.0, -0.0])
    x = x.cuda()
    out = torch.empty(4096, dtype=torch.bfloat16, device="cuda")
    api.fckl_cast_f32_to_bf16(x, out)
    ref = x.to(torch.bfloat16)
    finite = torch.isfinite(x) | torch.isinf(x)
    assert torch.equal(out.view(torch.int16)[finite], ref.view(torch.int16)[finite])


def test_autograd_module_two_micro_batches():
    """Two calls of one module instance (different sizes, so its workspace is made anew for
    the second), then one backward of their sum: each call's gradients against the oracle."""
    from chunked_kl_loss_head_b300 import FusedChunkedKLLoss

    mod = FusedChunkedKLLoss(tau=1.1, chunk=192)
    xa = make_small(T=500, d=64, V=2000, K=7, tau=1.1, dtype="bf16", seed=16, mask="random", mask_frac=0.1)
    xb = make_small(T=333, d=64, V=2000, K=7, tau=1.1, dtype="bf16", seed=17, mask="random", mask_frac=0.1)
    xb["W"] = xa["W"]
    da, db = to_device(xa), to_device(xb)
    W = da["W"].clone().requires_grad_(True)
    Ha = da["H"].clone().requires_grad_(True)
    Hb = db["H"].clone().requires_grad_(True)
    la = mod(Ha, W, da["topk_idx"], da["topk_logits"], da["valid"])
    lb = mod(Hb, W, db["topk_idx"], db["topk_logits"], db["valid"])
    (la + 2.0 * lb).backward()
    ra, rb = oracle_of(xa), oracle_of(xb, grad=2.0)
    tol = TOL["bf16"]
    assert rel(la.item(), ra["loss"]) <= tol["loss"] and rel(lb.item(), rb["loss"]) <= tol["loss"]
    assert rel_max(Ha.grad.float().cpu().numpy(), ra["dH"]) <= tol["grad"]
    assert rel_max(Hb.grad.float().cpu().numpy(), rb["dH"]) <= tol["grad"]
    assert rel_max(W.grad.float().cpu().numpy(), ra["dW"] + rb["dW"]) <= tol["grad"]


def test_bounded_wait_reports_timeout():
    """A pipeline wait that never completes gives up after its bound and reports
    FCKL_ERR_TIMEOUT through the workspace; the device stays usable afterwards."""
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    api.fckl_debug_wait_timeout(ws)
    assert api.fckl_get_error(ws) == 6  # FCKL_ERR_TIMEOUT
    assert api.fckl_get_error(ws) == 0  # the read cleared it
    x = make_small(T=64, d=32, V=300, K=3, tau=1.0, dtype="bf16", seed=31)
    check(x, run_gpu(x, 64), label="after a timeout")


@pytest.mark.parametrize("K", [31, 32, 33, 64, 65, 127, 128, 129])
def test_teacher_prep_k_edges(K):
    """K at the edges of the teacher-prep kernels: one, two or four sort keys per lane (up
    to 32, 64, 128 ids) and the ranking kernel above 128; duplicates planted."""
    x = make_small(T=90, d=32, V=3000, K=K, tau=1.3, dtype="bf16", seed=40 + K, ids="uniform", mask="random",
                   mask_frac=0.1)
    x["topk_idx"][7, K - 1] = x["topk_idx"][7, 0]
    check(x, run_gpu(x, 64), label=f"K={K}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_largest_k(dtype):
    x = make_small(T=70, d=64, V=5000, K=1024, tau=1.3, dtype=dtype, seed=32, ids="uniform")
    check(x, run_gpu(x, 64), label=f"{dtype} K=1024")


@pytest.mark.parametrize("case", range(24))
def test_random_shapes(case):
    """Seeded random small shapes across both paths: ragged T, d (a multiple of 8 for
    bf16), V, K, tau and chunk, random masks, some near-one-hot teachers."""
    rng = np.random.default_rng(1000 + case)
    dtype = "bf16" if case % 3 else "f32"
    T = int(rng.integers(1, 1500))
    d = int(rng.integers(1, 48)) * 8
    V = int(rng.integers(16, 9000))
    K = int(min(V, rng.choice([1, 2, 5, 17, 64])))
    tau = float(rng.choice([0.5, 1.0, 1.7, 3.0]))
    chunk = int(rng.choice([1, 7, 64, 128, 300, 1000, 4096]))
    x = make_small(T=T, d=d, V=V, K=K, tau=tau, dtype=dtype, seed=case, ids="uniform" if case % 2 else "zipf",
                   mask="random", mask_frac=float(rng.choice([0.0, 0.1, 0.5])),
                   onehot_frac=float(rng.choice([0.0, 0.2])), logit_offset=10.0)
    check(x, run_gpu(x, chunk), label=f"random {case}: {dtype} T={T} d={d} V={V} K={K} tau={tau} chunk={chunk}")
