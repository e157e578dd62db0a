"""Seeded synthetic workloads for the fused chunked KL distillation loss.

The five workloads mirror the shapes the pages discuss: the gpt-oss
vocabulary of 201,088 ids at 32K context and batch 4 (axbrief.com, "The
250GB VRAM Wall"), a Llama-3.1-8B -> 3.2B student (axbrief.com, "Breaking the
Bottleneck"), a top-100 teacher cache (calcaas.com, "What actually changed?")
and K=10 (getaibook.com, "Preparing Offline Top-K Logits").

Recipe (all draws from NumPy PCG64, seed 0 unless stated otherwise):

* H ~ N(0, 1) and W ~ N(0, 1/d), drawn in float32, then rounded to bfloat16
  (round to nearest even) for the bf16 workloads.
* teacher ids: K distinct ids per row.  "Zipf(1.1) without replacement" is
  read as weights w_i proportional to (i+1)^-1.1 over ids 0..V-1 (rank = id),
  sampled sequentially without replacement; this equals drawing i.i.d. by
  inverse CDF and keeping the first K distinct draws, which is how it is
  done here.  "uniform" draws ids uniformly, again keeping the first K
  distinct.
* teacher logits: K Gumbel(0, 1) draws sorted in descending order plus a
  constant offset, in float32; the k-th drawn id gets the k-th largest logit.
* masks: "random" ignores round(frac*T) rows chosen uniformly without
  replacement; "tail" ignores the last floor(frac*seq_len) rows of every
  sequence; "none" keeps every row.
* one-hot rows: round(frac*T) rows chosen uniformly without replacement get
  +boost added to their top logit (a near-one-hot teacher).

Every per-row quantity is drawn from a stream keyed by (seed, tag, block of
1024 rows), so any subset of rows can be regenerated without the rest, and
blocks are generated in parallel threads.  This module holds none of the
loss arithmetic.
"""

from __future__ import annotations

import concurrent.futures as _fut
import dataclasses
import functools
import os

import numpy as np

ROWS_PER_BLOCK = 1024

_TAG_H, _TAG_W, _TAG_IDS, _TAG_GUMBEL, _TAG_MASK, _TAG_ONEHOT, _TAG_FALLBACK, _TAG_TEACHER = range(1, 9)


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    T: int
    d: int
    V: int
    K: int
    tau: float
    dtype: str  # "f32" or "bf16": storage type of H, W and dH
    ids: str = "zipf"  # "zipf" or "uniform"
    zipf_a: float = 1.1
    logit_offset: float = 12.0
    seq_len: int = 0  # 0 means one sequence of length T
    mask: str = "none"  # "none", "random" or "tail"
    mask_frac: float = 0.0
    onehot_frac: float = 0.0
    onehot_boost: float = 30.0
    chunks: tuple = (4096,)
    seed: int = 0

    @property
    def batch(self) -> int:
        return self.T // (self.seq_len or self.T) if self.T else 0

    def with_(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    # T=64 tokens, d=256, V=4096, K=10, tau=1, fp32, all rows valid.
    "tiny_fp32": Config("tiny_fp32", T=64, d=256, V=4096, K=10, tau=1.0, dtype="f32",
                        logit_offset=8.0, chunks=(64,)),
    # Llama-8B -> 3B shaped: batch 1 x seq 8192, 5% random rows ignored.
    "llama_bf16": Config("llama_bf16", T=8192, d=3072, V=128256, K=100, tau=1.0, dtype="bf16",
                         logit_offset=12.0, seq_len=8192, mask="random", mask_frac=0.05,
                         chunks=(4096,)),
    # gpt-oss shaped: batch 4 x seq 32768, last 2% of each sequence ignored.
    "gptoss_bf16": Config("gptoss_bf16", T=131072, d=2880, V=201088, K=100, tau=1.0,
                          dtype="bf16", logit_offset=12.0, seq_len=32768, mask="tail",
                          mask_frac=0.02, chunks=(4096,)),
    # long context: batch 1 x seq 262144, tau=2, chunk swept.
    "longctx_bf16": Config("longctx_bf16", T=262144, d=2880, V=201088, K=100, tau=2.0,
                           dtype="bf16", logit_offset=12.0, seq_len=262144, mask="tail",
                           mask_frac=0.02, chunks=(1024, 4096, 16384)),
    # small-K / wide-vocab stress: uniform ids, 10% near-one-hot teachers.
    "stress_bf16": Config("stress_bf16", T=65536, d=4096, V=256000, K=10, tau=1.0,
                          dtype="bf16", ids="uniform", logit_offset=10.0, onehot_frac=0.1,
                          onehot_boost=30.0, chunks=(4096,)),
}


# ----------------------------------------------------------------------------------------
# storage conversions (bfloat16 as raw uint16 bit patterns)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even (torch's cast)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float32, exact."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------------------
# streams


def _rng(seed: int, tag: int, block: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(tag, block))))


def _pool_map(fn, items):
    items = list(items)
    if len(items) <= 1:
        return [fn(i) for i in items]
    workers = min(len(items), max(1, len(os.sched_getaffinity(0))))
    with _fut.ThreadPoolExecutor(workers) as ex:
        return list(ex.map(fn, items))


def _blocks_of(rows: np.ndarray):
    """Map block index -> positions (into `rows`) of the rows that fall in it."""
    blk = rows // ROWS_PER_BLOCK
    out = {}
    for b in np.unique(blk):
        out[int(b)] = np.nonzero(blk == b)[0]
    return out


def _block_rows(n_total: int, b: int) -> int:
    return min(ROWS_PER_BLOCK, n_total - b * ROWS_PER_BLOCK)


# ----------------------------------------------------------------------------------------
# dense operands


def _normal_block(seed, tag, b, n_total, d, scale, dtype):
    n = _block_rows(n_total, b)
    x = _rng(seed, tag, b).standard_normal((n, d), dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def _dense_rows(cfg: Config, tag: int, n_total: int, scale: float, rows=None):
    if rows is None:
        nb = (n_total + ROWS_PER_BLOCK - 1) // ROWS_PER_BLOCK
        parts = _pool_map(lambda b: _normal_block(cfg.seed, tag, b, n_total, cfg.d, scale, cfg.dtype),
                          range(nb))
        if not parts:
            return np.zeros((0, cfg.d), np.uint16 if cfg.dtype == "bf16" else np.float32)
        return np.concatenate(parts, axis=0)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((len(rows), cfg.d), np.uint16 if cfg.dtype == "bf16" else np.float32)
    blocks = _blocks_of(rows)

    def fill(item):
        b, pos = item
        blk = _normal_block(cfg.seed, tag, b, n_total, cfg.d, scale, cfg.dtype)
        out[pos] = blk[rows[pos] - b * ROWS_PER_BLOCK]

    _pool_map(fill, blocks.items())
    return out


def make_H(cfg: Config, rows=None) -> np.ndarray:
    """H[T, d] ~ N(0, 1) (bf16 bit patterns for bf16 workloads, else float32)."""
    return _dense_rows(cfg, _TAG_H, cfg.T, 1.0, rows)


def make_W(cfg: Config, rows=None) -> np.ndarray:
    """W[V, d] ~ N(0, 1/d) (bf16 bit patterns for bf16 workloads, else float32)."""
    return _dense_rows(cfg, _TAG_W, cfg.V, 1.0 / np.sqrt(cfg.d), rows)


# ----------------------------------------------------------------------------------------
# teacher top-K cache


@functools.lru_cache(maxsize=8)
def _zipf_cdf(V: int, a: float) -> np.ndarray:
    w = (np.arange(V, dtype=np.float64) + 1.0) ** (-a)
    c = np.cumsum(w)
    c /= c[-1]
    c[-1] = 1.0
    return c


def _first_k_distinct(cand: np.ndarray, K: int):
    """First K distinct values of each row of `cand`, in draw order.

    Returns (values[B, K], ok[B]); ok is False where a row had fewer than K distinct.
    """
    B, M = cand.shape
    order = np.argsort(cand, axis=1, kind="stable")
    sv = np.take_along_axis(cand, order, axis=1)
    first = np.ones((B, M), dtype=bool)
    first[:, 1:] = sv[:, 1:] != sv[:, :-1]
    pos = np.where(first, order, M)
    pos.sort(axis=1)
    ok = pos[:, K - 1] < M
    vals = np.take_along_axis(cand, np.minimum(pos[:, :K], M - 1), axis=1)
    return vals, ok


def _draw_ids(cfg: Config, rng: np.random.Generator, n: int) -> np.ndarray:
    if cfg.ids == "zipf":
        cdf = _zipf_cdf(cfg.V, cfg.zipf_a)
        return np.minimum(np.searchsorted(cdf, rng.random(n), side="right"), cfg.V - 1)
    if cfg.ids == "uniform":
        return rng.integers(0, cfg.V, size=n)
    raise ValueError(f"unknown id distribution {cfg.ids!r}")


def _ids_block(cfg: Config, b: int) -> np.ndarray:
    n = _block_rows(cfg.T, b)
    K = cfg.K
    if K > cfg.V:
        raise ValueError("K > V: no K distinct ids exist")
    # enough draws that nearly every row reaches K distinct ids
    M = max(4 * K + 32, 256) if cfg.ids == "zipf" else 2 * K + 16
    if K == cfg.V:
        M = max(M, 64 * cfg.V)
    rng = _rng(cfg.seed, _TAG_IDS, b)
    cand = _draw_ids(cfg, rng, n * M).reshape(n, M)
    vals, ok = _first_k_distinct(cand, K)
    for r in np.nonzero(~ok)[0]:
        # rare: keep drawing from this row's own stream until K distinct ids
        frng = _rng(cfg.seed, _TAG_FALLBACK, b * ROWS_PER_BLOCK + int(r))
        seen, got = set(), []
        for v in cand[r]:
            if int(v) not in seen:
                seen.add(int(v))
                got.append(int(v))
        while len(got) < K:
            for v in _draw_ids(cfg, frng, 4 * M):
                if int(v) not in seen:
                    seen.add(int(v))
                    got.append(int(v))
                    if len(got) == K:
                        break
        vals[r] = got[:K]
    return vals.astype(np.int32)


def _logits_block(cfg: Config, b: int) -> np.ndarray:
    n = _block_rows(cfg.T, b)
    g = _rng(cfg.seed, _TAG_GUMBEL, b).gumbel(0.0, 1.0, size=(n, cfg.K))
    g = -np.sort(-g, axis=1)  # descending
    return (g + cfg.logit_offset).astype(np.float32)


@functools.lru_cache(maxsize=16)
def _onehot_rows(cfg: Config) -> np.ndarray:
    n = int(round(cfg.onehot_frac * cfg.T))
    if n <= 0:
        return np.zeros(0, np.int64)
    return np.sort(_rng(cfg.seed, _TAG_ONEHOT).choice(cfg.T, n, replace=False))


def _topk_rows(cfg: Config, rows=None):
    if rows is None:
        rows = np.arange(cfg.T, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    idx = np.empty((len(rows), cfg.K), np.int32)
    lg = np.empty((len(rows), cfg.K), np.float32)
    blocks = _blocks_of(rows) if len(rows) else {}

    def fill(item):
        b, pos = item
        loc = rows[pos] - b * ROWS_PER_BLOCK
        idx[pos] = _ids_block(cfg, b)[loc]
        lg[pos] = _logits_block(cfg, b)[loc]

    _pool_map(fill, blocks.items())
    hot = _onehot_rows(cfg)
    if len(hot):
        sel = np.isin(rows, hot)
        lg[sel, 0] += np.float32(cfg.onehot_boost)
    return idx, lg


@functools.lru_cache(maxsize=16)
def valid_mask(cfg: Config) -> np.ndarray:
    """valid[T] uint8: 1 = the row takes part in the loss, 0 = ignored."""
    v = np.ones(cfg.T, np.uint8)
    if cfg.mask == "none" or cfg.T == 0:
        pass
    elif cfg.mask == "random":
        n = int(round(cfg.mask_frac * cfg.T))
        v[_rng(cfg.seed, _TAG_MASK).choice(cfg.T, n, replace=False)] = 0
    elif cfg.mask == "tail":
        S = cfg.seq_len or cfg.T
        cut = int(np.floor(cfg.mask_frac * S))
        for s0 in range(0, cfg.T, S):
            if cut:
                v[s0 + S - cut: s0 + S] = 0
    else:
        raise ValueError(f"unknown mask {cfg.mask!r}")
    v.setflags(write=False)
    return v


# ----------------------------------------------------------------------------------------
# public entry points


def make_inputs(cfg: Config, with_W: bool = True) -> dict:
    """All inputs of a workload: H[T,d], W[V,d], topk_idx[T,K] int32,
    topk_logits[T,K] float32, valid[T] uint8 (H/W as bf16 bits or float32)."""
    idx, lg = _topk_rows(cfg)
    out = dict(cfg=cfg, H=make_H(cfg), topk_idx=idx, topk_logits=lg,
               valid=np.array(valid_mask(cfg)))
    if with_W:
        out["W"] = make_W(cfg)
    return out


def make_rows(cfg: Config, rows) -> dict:
    """The per-row inputs (H, topk_idx, topk_logits, valid) of selected rows only."""
    rows = np.asarray(rows, dtype=np.int64)
    idx, lg = _topk_rows(cfg, rows)
    return dict(cfg=cfg, rows=rows, H=make_H(cfg, rows), topk_idx=idx, topk_logits=lg,
                valid=np.array(valid_mask(cfg))[rows])


def make_small(T, d, V, K, tau=1.0, dtype="bf16", seed=0, ids="zipf", mask="none",
               mask_frac=0.0, seq_len=0, onehot_frac=0.0, logit_offset=12.0, name="custom"):
    """A small workload of any shape from the same generators."""
    cfg = Config(name, T=T, d=d, V=V, K=K, tau=tau, dtype=dtype, ids=ids, seq_len=seq_len,
                 mask=mask, mask_frac=mask_frac, onehot_frac=onehot_frac,
                 logit_offset=logit_offset, seed=seed)
    return make_inputs(cfg)


# ----------------------------------------------------------------------------------------
# full teacher logits (the input of the top-K extraction that builds the cache)


_TEACHER_ROWS = 64  # rows per random stream of the teacher logits (V-wide rows are large)


def _teacher_block(seed, b, n_total, V, zipf_a, offset, dtype):
    n = min(_TEACHER_ROWS, n_total - b * _TEACHER_ROWS)
    bias = (offset - zipf_a * np.log1p(np.arange(V, dtype=np.float64))).astype(np.float32)
    # Gumbel(0, 1) = -ln(-ln u), u uniform on (0, 1), in float32 (u kept off 0 and 1)
    u = _rng(seed, _TAG_TEACHER, b).random((n, V), dtype=np.float32)
    u *= np.float32(1.0 - 2.0 ** -23)
    u += np.float32(2.0 ** -24)
    np.log(u, out=u)
    np.negative(u, out=u)
    np.log(u, out=u)
    x = bias - u
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def make_teacher_logits(T, V, seed=0, dtype="bf16", zipf_a=1.1, offset=12.0):
    """Full teacher logits [T, V]: offset - zipf_a * ln(v + 1) + Gumbel(0, 1) per entry
    (bf16 bit patterns or float32).  With this bias the K largest entries of a row are a
    sample of K distinct ids from Zipf(zipf_a) drawn without replacement (the Gumbel top-k
    property), the distribution of the cached ids of the loss workloads."""
    nb = (T + _TEACHER_ROWS - 1) // _TEACHER_ROWS
    parts = _pool_map(lambda b: _teacher_block(seed, b, T, V, zipf_a, offset, dtype), range(nb))
    if not parts:
        return np.zeros((0, V), np.uint16 if dtype == "bf16" else np.float32)
    return np.concatenate(parts, axis=0)
