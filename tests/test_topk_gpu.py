"""Teacher top-K extraction through the C-ABI against the oracle, bit for bit: the
order (value descending, id ascending) makes the answer unique, so ids and values must
match exactly.  The cases reach every path of the kernel: rows short enough to keep
whole, the sampled threshold on long rows, the exact radix-select path (forced by heavy
ties and by rows whose entries are all equal), rows whose start is 16-byte aligned (read
with 16-byte vector loads, four in flight per thread, plus a short tail of fewer than one
vector) and rows whose start is not (read entry by entry), rows of every length around
the vector width, K = 1 and K = V, signed zeros and infinities."""

import numpy as np
import pytest
import torch

from chunked_kl_loss_head_b300 import api
from gen import bf16_bits_to_f32, f32_to_bf16_bits, make_teacher_logits
from oracle import topk_rows

pytestmark = pytest.mark.gpu


def run(x_host, K, dtype):
    """x_host: float32 values (for bf16 they must be bf16-representable)."""
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x_host)
        x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
        ref_in = bf16_bits_to_f32(bits)
    else:
        x = torch.from_numpy(np.ascontiguousarray(x_host, dtype=np.float32)).cuda()
        ref_in = x_host.astype(np.float32)
    idx, val = api.topk_extract(x, K)
    torch.cuda.synchronize()
    ref_idx, ref_val = topk_rows(ref_in, K)
    got_idx, got_val = idx.cpu().numpy(), val.cpu().numpy()
    assert np.array_equal(got_idx, ref_idx), np.argwhere(got_idx != ref_idx)[:5]
    assert np.array_equal(got_val.view(np.uint32), ref_val.view(np.uint32))
    return got_idx, got_val


def bf16_grid(a):
    return bf16_bits_to_f32(f32_to_bf16_bits(a.astype(np.float32)))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,V,K", [(7, 300, 17), (3, 8192, 64), (3, 8193, 64), (4, 50000, 1024), (2, 40001, 1),
                                   (5, 201088, 100)])
def test_random_rows(dtype, T, V, K):
    rng = np.random.default_rng(T * 1000 + V + K)
    x = rng.standard_normal((T, V)).astype(np.float32) * 3
    run(bf16_grid(x) if dtype == "bf16" else x, K, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gumbel_zipf_teacher_rows(dtype):
    # the extraction workload: top-K ids are Zipf(1.1) draws without replacement
    x = make_teacher_logits(6, 201088, seed=3, dtype=dtype)
    xf = bf16_bits_to_f32(x) if dtype == "bf16" else x
    idx, _ = run(xf, 100, dtype)
    assert np.median(idx) < 2000  # small ids dominate, as Zipf(1.1) weights say


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_heavy_ties_take_the_exact_path(dtype):
    rng = np.random.default_rng(5)
    # 200k entries from 6 values: far more than the candidate list can hold tie at the K-th
    x = rng.integers(0, 6, size=(3, 200000)).astype(np.float32)
    run(x, 100, dtype)
    # every entry equal: the answer is ids 0..K-1
    y = np.full((2, 30000), 1.5, np.float32)
    idx, _ = run(y, 300, dtype)
    assert np.array_equal(idx, np.tile(np.arange(300, dtype=np.int32), (2, 1)))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_unaligned_rows_and_k_equals_v(dtype):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((5, 20001)).astype(np.float32)  # odd V: rows start off 16-byte boundaries
    run(bf16_grid(x) if dtype == "bf16" else x, 33, dtype)
    y = rng.standard_normal((4, 37)).astype(np.float32)
    run(bf16_grid(y) if dtype == "bf16" else y, 37, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [1, 3, 5, 8, 9, 15, 16, 17, 31, 4097, 8191, 16385])
def test_short_rows_every_alignment(dtype, V):
    # 9 rows of V entries: row starts fall on every 2- (bf16) or 4-byte (f32) offset, so rows
    # with no 16-byte block, with only a head and tail, and with a body ending mid-chunk occur
    rng = np.random.default_rng(V)
    x = rng.standard_normal((9, V)).astype(np.float32)
    run(bf16_grid(x) if dtype == "bf16" else x, min(V, 3), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_signed_zeros_and_infinities(dtype):
    x = np.zeros((2, 9000), np.float32)
    x[:, ::3] = -0.0
    x[0, 17] = np.inf
    x[0, 23] = -np.inf
    x[1, 4000:4010] = 7.0
    run(x, 20, dtype)


def test_empty_and_bad_arguments():
    x = torch.zeros((0, 100), dtype=torch.bfloat16, device="cuda")
    idx, val = api.topk_extract(x, 10)
    assert idx.shape == (0, 10)
    y = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.FcklError):
        api.topk_extract(y, 101)  # K > V
    with pytest.raises(api.FcklError):
        api.topk_extract(y, 0)


def test_extracted_cache_feeds_the_loss():
    """The extraction's output is the loss's teacher input as is (ids and float32 logits)."""
    T, V, d, K = 64, 4096, 128, 20
    logits = make_teacher_logits(T, V, seed=7, dtype="bf16")
    g = torch.from_numpy(logits.view(np.int16)).view(torch.bfloat16).cuda()
    idx, val = api.topk_extract(g, K)
    rng = np.random.default_rng(2)
    H = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).cuda()
    W = torch.from_numpy((rng.standard_normal((V, d)) / np.sqrt(d)).astype(np.float32)).cuda()
    valid = torch.ones(T, dtype=torch.uint8, device="cuda")
    loss, lse = api.forward(H, W, idx, val, valid, 1.0, 64)
    torch.cuda.synchronize()
    assert np.isfinite(loss.item()) and loss.item() > 0
