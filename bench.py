"""Benchmark of the fused chunked KL loss (forward + backward) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config gptoss_bf16] [--chunk 4096]
    python bench.py --impl reference ...      # the fp64 oracle on the host cores

One step = fckl_forward + fckl_backward over one batch of the workload (all
T tokens): loss, per-row logsumexp, dH and dW.  Inputs are synthetic (seeded
generators, shapes of the pages' workloads) and larger than the 126 MB L2.
Prints one JSON line (rank 0).  Under torchrun the batch is token-sharded: each
rank holds T tokens of its own (weak scaling) and the whole lm_head weight, and
every step sums the loss partials (loss sum, N) over ranks before the backward and
dW after it (chunked_kl_loss_head_b300.dist, NCCL all-reduces inside the timed
step); the time is the max over ranks.

    python bench.py --path module ...   # the FusedChunkedKLLoss autograd module
    python bench.py --path topk ...     # teacher top-K extraction
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "top-K KL fwd+bwd tokens/s; % of BF16 tensor peak; peak device GiB"
DEFAULT_CONFIG = "gptoss_bf16"
FALLBACK_PEAKS = dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


def algorithmic_flops(T, d, V, n_valid):
    """Forward logits for every row (2dV); backward recompute + dH + dW for valid rows (6dV)."""
    return 8.0 * d * V * n_valid + 2.0 * d * V * (T - n_valid)


def dist_env():
    """(rank, local_rank, world_size) from the launcher's environment (1 process: 0, 0, 1)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest of every rank's x: a job's time is that of its slowest rank.  `dist` is
    torch.distributed with an initialized group (None: one process)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, seconds):
    """Whole-job throughput when every rank processes its own batch of `units_per_rank`
    (token-sharded, weak scaling)."""
    return world * units_per_rank / seconds


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def __enter__(self):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.f.flush()

    def summary(self):
        rows = []
        try:
            for line in open(self.f.name):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        finally:
            os.unlink(self.f.name)
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["unsampled"])
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        load = [s for s in sm if s > 0.5 * (max(mx) if mx else 1)] or sm
        return dict(sm_mhz=float(np.median(load)) if load else None, sm_max_mhz=max(mx) if mx else None,
                    power_w_max=max(pw) if pw else None, samples=len(rows), reasons=reasons)


def host_info():
    """The host the CPU legs run on: CPU model, and the BLAS library numpy calls with the
    threads it runs (the oracle's matrix products are its only multi-threaded part)."""
    info = dict(cores=len(os.sched_getaffinity(0)))
    try:
        with open("/proc/cpuinfo") as f:
            info["cpu_model"] = next((ln.split(":", 1)[1].strip() for ln in f if ln.startswith("model name")), None)
    except OSError:
        pass
    try:
        from threadpoolctl import threadpool_info

        blas = [p for p in threadpool_info() if p.get("user_api") == "blas"]
        if blas:
            info["blas"] = f"{blas[0].get('internal_api')} {blas[0].get('version')}"
            info["cores"] = int(blas[0].get("num_threads") or info["cores"])
            return info
    except ImportError:
        pass
    # without threadpoolctl: numpy's build record names the library; OpenBLAS runs one
    # thread per available core unless OPENBLAS_NUM_THREADS says otherwise
    try:
        blas = np.show_config(mode="dicts")["Build Dependencies"]["blas"]
        info["blas"] = f"{blas.get('name')} {blas.get('version')}"
        env = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
        if env and env.isdigit() and "openblas" in str(blas.get("name")):
            info["cores"] = min(info["cores"], int(env))
    except (KeyError, TypeError, AttributeError):
        pass
    return info


def rank_inputs(cfg, rank):
    """One rank's inputs for the token-sharded step: its own batch of rows (the workload's
    seed + rank) and the same W on every rank (the lm_head is replicated).  Rank 0's
    inputs are the single-GPU workload's."""
    from gen import make_inputs, make_W

    x = make_inputs(cfg.with_(seed=cfg.seed + rank), with_W=False)
    x["W"] = make_W(cfg)
    return x


def cpu_oracle_rate(cfg, W_bits, rows, reps=1):
    """Oracle fwd+bwd (fp64, full-vocab logit rows, analytic dH / dW) on `rows` rows of
    the workload; returns (tokens/s, seconds)."""
    from gen import bf16_bits_to_f32, make_rows, valid_mask
    from oracle import fwd_bwd

    x = make_rows(cfg, np.arange(rows))
    H = bf16_bits_to_f32(x["H"]).astype(np.float64) if x["H"].dtype == np.uint16 else x["H"].astype(np.float64)
    W = bf16_bits_to_f32(W_bits) if W_bits.dtype == np.uint16 else W_bits
    n_all = int(np.asarray(valid_mask(cfg)).sum())
    t0 = time.perf_counter()
    for _ in range(reps):
        fwd_bwd(H, W, x["topk_idx"], x["topk_logits"], x["valid"], cfg.tau, N=n_all)
    dt = time.perf_counter() - t0
    return rows * reps / dt, dt


def run_reference(args, cfg):
    """The oracle as the reference arm: each step is a bounded row sample of the workload."""
    rank, _, world = dist_env()
    if world > 1 and rank != 0:
        return
    from gen import make_W

    W_bits = make_W(cfg)
    rows = min(args.ref_rows, cfg.T)
    for _ in range(args.warmup):
        cpu_oracle_rate(cfg, W_bits, rows)
    t = 0.0
    for _ in range(args.steps):
        t += cpu_oracle_rate(cfg, W_bits, rows)[1]
    rate = rows * args.steps / t
    host = host_info()
    sample = f"oracle fwd+bwd on rows 0..{rows - 1} of {cfg.name} per step (fp64 numpy/BLAS)"
    line = dict(impl="reference", metric=METRIC, value=rate, unit="tokens/s", n_gpus=args.gpus, steps=args.steps,
                warmup=args.warmup, ms_per_step=1e3 * t / args.steps, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64", data="synthetic",
                config=dict(workload=cfg.name, T=cfg.T, d=cfg.d, V=cfg.V, K=cfg.K, tau=cfg.tau),
                cpu_baseline=dict(value=rate, unit="tokens/s", cores=host["cores"], kind="oracle", sample=sample,
                                  cpu_model=host.get("cpu_model"), blas=host.get("blas")),
                e2e=dict(value=rate, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def dense_torch_step(H, W, idx, tl, valid, tau):
    """The loss the plain way, for comparison only: build the [T, V] student logits with one
    bf16 matmul, log-softmax them in fp32, gather at the teacher's ids and let autograd
    produce dH and dW.  Plain PyTorch ops on the GPU, none of this library's kernels.
    Returns (loss, dH, dW)."""
    import torch

    Hl = H.detach().requires_grad_(True)
    Wl = W.detach().requires_grad_(True)
    z = Hl @ Wl.t()
    logq = torch.log_softmax(z.float() / tau, dim=-1)
    logp = torch.log_softmax(tl.float() / tau, dim=-1)
    row = (logp.exp() * (logp - logq.gather(1, idx.long()))).sum(1)
    v = valid.float()
    loss = (row * v).sum() / v.sum().clamp(min=1.0)
    loss.backward()
    return loss.detach(), Hl.grad, Wl.grad


# Bytes per [T x V] element the dense path holds at its peak, rounded up: at 8K and 32K
# tokens of the gpt-oss vocabulary its measured peak is 14 bytes per logit (the fp32
# log-softmax kept for backward plus, in backward, fp32 gradients and a bf16 cast).
DENSE_BYTES_PER_ELEM = 16


def linear_bytes(T, d, K, elem):
    """Bytes of one fwd+bwd that grow with the token count: H and dH (elem bytes each), the
    teacher cache (ids and logits, 4 bytes each), the valid mask, lse and the per-row losses
    the workspace holds."""
    return T * (2 * d * elem + 2 * K * 4 + 1 + 4 + 4)


def memory_point(c, chunk, dense=True, timing=True):
    """One point of the memory curve: the peak device memory of one fused fwd+bwd of
    workload `c` (inputs, outputs and workspace included), optionally its time, and, where
    it fits, the same step done the dense way in plain PyTorch (peak memory, time, loss).  A
    dense point whose predicted peak exceeds 80% of the free device memory is not run (no
    out-of-memory attempts); its prediction is reported instead."""
    import torch

    from chunked_kl_loss_head_b300 import api
    from chunked_kl_loss_head_b300.memory import dense_logit_bytes
    from gen import make_inputs

    dev = torch.device("cuda", torch.cuda.current_device())
    T = c.T
    x = make_inputs(c)
    tdt = torch.bfloat16 if c.dtype == "bf16" else torch.float32

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats(dev)
    free0, _ = torch.cuda.mem_get_info(dev)
    g = {k: to_dev(x[k]) for k in ("H", "W", "topk_idx", "topk_logits", "valid")}
    del x
    ws = api.workspace(T, c.d, c.V, c.K, chunk, tdt, dev)
    loss, lse = api.forward(g["H"], g["W"], g["topk_idx"], g["topk_logits"], g["valid"], c.tau, chunk, ws=ws)
    dH, dW = api.backward(g["H"], g["W"], g["topk_idx"], g["topk_logits"], g["valid"], lse, c.tau, chunk, ws=ws)
    torch.cuda.synchronize(dev)
    status = api.fckl_get_error(ws)
    if status != 0:
        raise RuntimeError(f"device status: {api.fckl_status_string(status)}")
    peak = torch.cuda.max_memory_allocated(dev)
    free1, _ = torch.cuda.mem_get_info(dev)
    elem = 2 if c.dtype == "bf16" else 4
    pt = dict(T=T, peak_device_gib=peak / 2 ** 30,
              nontorch_device_gib=max(0.0, (free0 - free1 - peak) / 2 ** 30),
              workspace_gib=ws.numel() / 2 ** 30, loss=float(loss.item()),
              linear_gib=linear_bytes(T, c.d, c.K, elem) / 2 ** 30,
              W_and_dW_gib=c.V * c.d * (elem + 4) / 2 ** 30,
              dense_TxV_bf16_gib=dense_logit_bytes(T, c.V) / 2 ** 30)
    if timing:
        pt["fused_ms"] = time_ms(lambda: (api.forward(g["H"], g["W"], g["topk_idx"], g["topk_logits"], g["valid"],
                                                      c.tau, chunk, ws=ws)[1],
                                          api.backward(g["H"], g["W"], g["topk_idx"], g["topk_logits"], g["valid"],
                                                       lse, c.tau, chunk, ws=ws)), dev)
    del ws, loss, lse, dH, dW
    if dense:
        base = torch.cuda.memory_allocated(dev)
        predicted = base + DENSE_BYTES_PER_ELEM * T * c.V
        torch.cuda.empty_cache()
        free2, _ = torch.cuda.mem_get_info(dev)
        pt["dense_predicted_gib"] = predicted / 2 ** 30
        if predicted - base > 0.8 * free2:
            pt["dense"] = "not run: predicted peak above 80% of free device memory"
        else:
            torch.cuda.reset_peak_memory_stats(dev)
            dl, _, _ = dense_torch_step(g["H"], g["W"], g["topk_idx"], g["topk_logits"], g["valid"], c.tau)
            torch.cuda.synchronize(dev)
            pt["dense_peak_device_gib"] = torch.cuda.max_memory_allocated(dev) / 2 ** 30
            pt["dense_loss"] = float(dl.item())
            if timing:
                pt["dense_ms"] = time_ms(lambda: dense_torch_step(g["H"], g["W"], g["topk_idx"], g["topk_logits"],
                                                                  g["valid"], c.tau), dev)
    del g
    torch.cuda.empty_cache()
    return pt


def run_memory_curve(args, cfg):
    """Peak device memory of one fused fwd+bwd (inputs, outputs and workspace included) as
    the token count grows, next to the size of the one dense [T x V] bf16 tensor the
    method never builds, and the same step done the dense way in plain PyTorch (peak
    memory, time, loss) where it fits: the pages' isolated loss benchmark compares the two
    this way (axbrief.com, "Quantifying the Efficiency Gain: 15.6x VRAM Reduction")."""
    import torch

    torch.cuda.set_device(0)
    chunk = args.chunk or cfg.chunks[0]
    points = []
    for T in (int(v) for v in args.memory_curve.split(",")):
        c = cfg.with_(name=f"{cfg.name}[T={T}]", T=T, seq_len=min(cfg.seq_len or T, T))
        points.append(memory_point(c, chunk, dense=not args.no_dense))
    print(json.dumps(dict(metric="peak device GiB of one fused fwd+bwd vs tokens", unit="GiB",
                          config=dict(workload=cfg.name, d=cfg.d, V=cfg.V, K=cfg.K, chunk=chunk),
                          points=points)), flush=True)


def time_ms(fn, dev, reps=3):
    """Mean device time of fn() over `reps` runs after one warm-up, with CUDA events on the
    current stream."""
    import torch

    fn()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps


def run_topk(args, cfg):
    """Teacher top-K extraction (the offline step that builds the cache): the K largest
    logits and their ids per row of a [T, V] bf16 teacher logit matrix of the workload's
    vocabulary (offset - 1.1 ln(v+1) + Gumbel noise, whose per-row top-K ids are Zipf(1.1)
    draws without replacement).  HBM-bound: the roofline is the measured copy bandwidth."""
    import torch

    from chunked_kl_loss_head_b300 import api
    from gen import bf16_bits_to_f32, make_teacher_logits

    if args.warmup < 3:
        args.warmup = 3
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    T = args.topk_rows
    V, K = cfg.V, cfg.K
    host = make_teacher_logits(T, V, seed=cfg.seed, dtype="bf16")
    x = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    val = torch.empty((T, K), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        api.fckl_topk_extract(x, K, idx, val, stream)
    torch.cuda.synchronize(dev)
    launches0 = api.fckl_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler("0") as clk:
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            api.fckl_topk_extract(x, K, idx, val, stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    launches = api.fckl_launch_count() - launches0
    algo_bytes = T * V * 2 + T * K * 8
    gbs = algo_bytes / (ms / 1e3) / 1e9
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    cpu = None
    if not args.no_cpu:
        from oracle import topk_rows

        rows = 8
        t0 = time.perf_counter()
        topk_rows(bf16_bits_to_f32(host[:rows]), K)
        secs = time.perf_counter() - t0
        # numpy's sort runs on one thread
        cpu = dict(value=rows / secs, unit="rows/s", cores=1, kind="oracle", cpu_model=host_info().get("cpu_model"),
                   sample=f"oracle top-K (numpy lexsort per row, one thread) on rows 0..{rows - 1}; {secs:.2f} s")
    # DRAM bytes per launch from the committed ncu capture of this workload, while the kernel
    # source is the one that capture ran
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        try:
            tj = json.load(open(tpath)).get("topk_bf16", {})
            if tj.get("rows") == T and tj.get("V") == V and tj.get("K") == K and \
                    tj.get("src_sha") == _src_sha(("fckl_topk.cu",)):
                traffic = tj["bytes_per_launch"]
        except (ValueError, KeyError):
            traffic = None
    line = dict(metric="teacher top-K extraction rows/s", value=T / (ms / 1e3), unit="rows/s", n_gpus=1,
                steps=args.steps, warmup=args.warmup, ms_per_step=ms, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="bf16", data="synthetic",
                config=dict(workload=f"teacher logits [T={T}, V={V}] bf16, K={K}",
                            l2=f"input larger than L2 ({T * V * 2 / 1e9:.2f} GB)"),
                roofline=dict(bound="hbm", achieved=gbs, peak=hbm, unit="GB/s", frac=gbs / hbm, traffic=traffic,
                              peak_note=f"HBM copy ({peaks['source']})"),
                cpu_baseline=cpu, gpu_launches=int(launches), clocks=clk.summary())
    print(json.dumps(line), flush=True)


def run_module(args, cfg):
    """The user's entry point, the FusedChunkedKLLoss autograd module: forward and backward
    through autograd (hidden states and lm_head weight as leaf tensors of the workload's
    dtype), gradients landing in .grad in that dtype.  Reports tokens/s and the peak device
    memory of the timed steps (inputs, gradients, the module's workspace and its float32
    dW before the cast)."""
    import torch

    from chunked_kl_loss_head_b300 import FusedChunkedKLLoss, api
    from gen import make_inputs

    if args.warmup < 3:
        args.warmup = 3
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    chunk = args.chunk or cfg.chunks[0]
    peaks = load_peaks()
    x = make_inputs(cfg)
    n_valid = int(x["valid"].sum())

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    g = {k: to_dev(x[k]) for k in ("H", "W", "topk_idx", "topk_logits", "valid")}
    del x
    H = g["H"].requires_grad_(True)
    W = g["W"].requires_grad_(True)
    mod = FusedChunkedKLLoss(tau=cfg.tau, chunk=chunk)

    def step():
        H.grad = None
        W.grad = None
        loss = mod(H, W, g["topk_idx"], g["topk_logits"], g["valid"])
        loss.backward()
        return loss

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    H.grad = None
    W.grad = None
    torch.cuda.reset_peak_memory_stats(dev)
    launches0 = api.fckl_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler("0") as clk:
        torch.cuda.synchronize(dev)
        e0.record()
        for _ in range(args.steps):
            loss = step()
        e1.record()
        torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    launches = api.fckl_launch_count() - launches0
    peak = torch.cuda.max_memory_allocated(dev)
    T, d, V = cfg.T, cfg.d, cfg.V
    flops = algorithmic_flops(T, d, V, n_valid)
    tflops = flops / (ms / 1e3) / 1e12
    peak_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    elem = 2 if cfg.dtype == "bf16" else 4
    line = dict(metric="FusedChunkedKLLoss module fwd+bwd tokens/s", value=T / (ms / 1e3), unit="tokens/s", n_gpus=1,
                steps=args.steps, warmup=args.warmup, ms_per_step=ms, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype=cfg.dtype, data="synthetic",
                config=dict(workload=cfg.name, T=T, d=d, V=V, K=cfg.K, tau=cfg.tau, chunk=chunk,
                            l2="inputs larger than L2"),
                tflops=tflops, frac_bf16_peak=tflops / peak_burst, peak_device_gib=peak / 2 ** 30,
                memory_parts_gib=dict(inputs=sum(t.numel() * t.element_size() for t in g.values()) / 2 ** 30,
                                      grads=(T * d + V * d) * elem / 2 ** 30,
                                      dW_float32=V * d * 4 / 2 ** 30,
                                      workspace=api.fckl_workspace_size(T, d, V, cfg.K, chunk, H.dtype) / 2 ** 30,
                                      dense_TxV_bf16=T * V * 2 / 2 ** 30),
                loss=float(loss.item()), gpu_launches=int(launches), clocks=clk.summary())
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="fckl", choices=["fckl", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--chunk", type=int, default=0, help="chunk size (default: the workload's first)")
    ap.add_argument("--cpu-rows", type=int, default=256, help="rows of the oracle CPU-baseline sample")
    ap.add_argument("--ref-rows", type=int, default=128, help="rows per reference-arm step")
    ap.add_argument("--shape", default="", help="override T,d,V,K of the workload (e.g. a small ncu case)")
    ap.add_argument("--dp", action="store_true",
                    help="take the token-sharded path (NCCL process group, loss partials and dW all-reduced in "
                         "the step) even with one process; under torchrun with N > 1 it is always taken")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--topk-rows", type=int, default=4096, help="rows of the --path topk workload")
    ap.add_argument("--path", default="loss", choices=["loss", "topk", "module"],
                    help="topk: time the teacher top-K extraction instead; module: the FusedChunkedKLLoss "
                         "autograd module (one JSON line)")
    ap.add_argument("--no-dense", action="store_true", help="--memory-curve without the dense PyTorch arm")
    ap.add_argument("--memory-curve", default="",
                    help="comma-separated token counts: peak device memory of one fwd+bwd of the workload's "
                         "shape at each T (one JSON line), instead of the timing run")
    args = ap.parse_args()

    from gen import CONFIGS

    cfg = CONFIGS[args.config]
    if args.shape:
        T_, d_, V_, K_ = (int(v) for v in args.shape.split(","))
        cfg = cfg.with_(name=f"{cfg.name}[T={T_},d={d_},V={V_},K={K_}]", T=T_, d=d_, V=V_, K=K_,
                        seq_len=min(cfg.seq_len or T_, T_))
    if args.impl == "reference":
        run_reference(args, cfg)
        return
    if args.memory_curve:
        run_memory_curve(args, cfg)
        return
    if args.path == "topk":
        run_topk(args, cfg)
        return
    if args.path == "module":
        run_module(args, cfg)
        return
    if args.warmup < 3:
        args.warmup = 3  # timing rule: at least three warm-up steps

    import torch

    from chunked_kl_loss_head_b300 import api
    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dist = None
    sharded_path = world > 1 or args.dp
    if sharded_path:
        import torch.distributed as dist

        # no NVLink multicast objects (NVLS) on shared GPUs: a plain ring all-reduce of dW
        os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
        if "MASTER_ADDR" not in os.environ:  # one process, not under a launcher
            os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=os.environ.get("MASTER_PORT", "29533"),
                              RANK="0", WORLD_SIZE="1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    chunk = args.chunk or cfg.chunks[0]
    peaks = load_peaks()

    # ---- inputs, resident in HBM
    x = rank_inputs(cfg, rank)
    n_valid = int(x["valid"].sum())
    T, d, V, K = cfg.T, cfg.d, cfg.V, cfg.K
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32

    def host(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a))

    h = dict(H=host(x["H"]), W=host(x["W"]), topk_idx=host(x["topk_idx"]), topk_logits=host(x["topk_logits"]),
             valid=host(x["valid"]))
    del x
    torch.cuda.reset_peak_memory_stats(dev)
    free0, _ = torch.cuda.mem_get_info(dev)
    g = {k: v.to(dev) for k, v in h.items()}
    ws = api.workspace(T, d, V, K, chunk, tdt, dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    dH = torch.empty((T, d), dtype=tdt, device=dev)
    dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    if sharded_path:
        # token-sharded: the loss partials and dW are summed over ranks inside the step
        from chunked_kl_loss_head_b300.dist import ShardedKL

        del ws, lse, dH, dW
        sharded = ShardedKL(cfg.tau, chunk)

        def step(src):
            out = sharded.forward(src["H"], src["W"], src["topk_idx"], src["topk_logits"], src["valid"])
            sharded.backward(1.0)
            return out
    else:
        def step(src):
            api.fckl_forward(src["H"], src["W"], src["topk_idx"], src["topk_logits"], src["valid"], cfg.tau, chunk,
                             loss, lse, None, ws, stream)
            api.fckl_backward(src["H"], src["W"], src["topk_idx"], src["topk_logits"], src["valid"], cfg.tau, chunk,
                              lse, 1.0, dH, dW, ws, None, stream)
            return loss

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step(g)
    if sharded_path:
        ws = sharded.ops.ws
    status = api.fckl_get_error(ws)
    if status != 0:
        raise SystemExit(f"device status after warm-up: {api.fckl_status_string(status)}")

    # ---- timed region: K steps, device-resident inputs, per-class kernel events
    for c in api.KERNEL_CLASSES:
        api.fckl_profile_read(c, reset=True)
    api.fckl_profile_enable(True)
    launches0 = api.fckl_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_id = vis.split(",")[local_rank] if vis else str(local_rank)
    with ClockSampler(smi_id) as clk:
        barrier()
        e0.record(stream)
        for _ in range(args.steps):
            last = step(g)
        e1.record(stream)
        barrier()
    api.fckl_profile_enable(False)
    launches = api.fckl_launch_count() - launches0
    ms = e0.elapsed_time(e1)
    per_class = {c: api.fckl_profile_read(c) for c in api.KERNEL_CLASSES}
    status = api.fckl_get_error(ws)
    if status != 0:
        raise SystemExit(f"device status after the timed region: {api.fckl_status_string(status)}")
    t_max = max_over_ranks(ms, dist, dev)
    peak_alloc = torch.cuda.max_memory_allocated(dev)
    free1, _ = torch.cuda.mem_get_info(dev)
    loss_val = float(last.item())

    sec_per_step = t_max / 1e3 / args.steps
    tokens_per_s = job_rate(T, world, sec_per_step)
    flops = algorithmic_flops(T, d, V, n_valid)
    tflops = flops / sec_per_step / 1e12

    # ---- roofline of the dominant kernel class (device time from its own events)
    fused_bwd = per_class["grad_gemm"][0] == 0  # bf16: one launch per chunk runs G, dW and dH

    def class_flops(c):
        if c == "fwd_tiles":
            return 2.0 * d * V * T * args.steps
        if c == "bwd_tiles":
            return (6.0 if fused_bwd else 2.0) * d * V * n_valid * args.steps
        if c == "grad_gemm":
            return 4.0 * d * V * n_valid * args.steps
        return 0.0

    tc_classes = [c for c in ("fwd_tiles", "bwd_tiles", "grad_gemm") if per_class[c][0] > 0]
    total_ms = sum(v[1] for v in per_class.values())
    dom = max(tc_classes, key=lambda c: per_class[c][1])
    dom_launches, dom_ms = per_class[dom]
    achieved = class_flops(dom) / (dom_ms / 1e3) / 1e12
    peak_sust = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        try:
            tj = json.load(open(tpath)).get(cfg.name, {}).get(dom)
            if tj and tj.get("src_sha") == _kernel_src_sha():
                traffic = tj["bytes_per_launch"]
        except (ValueError, KeyError):
            traffic = None
    if cfg.dtype == "f32":
        # fp32 work runs on the CUDA cores (FFMA): 148 SMs x 128 fp32 lanes x 2 FLOP per clock
        peak_r, bound, note = 148 * 128 * 2 * peaks.get("sm_max_mhz", 2032.0) / 1e6, "alu", \
            "fp32 FFMA: 148 SMs x 128 lanes x 2 FLOP x max SM clock"
    else:
        peak_r, bound, note = peak_sust, "tensor", \
            f"sustained bf16 ({peaks['source']}): kernel timed inside a long step"
    roofline = dict(bound=bound, kernel=dom, achieved=achieved, peak=peak_r, unit="TFLOP/s",
                    frac=achieved / peak_r, traffic=traffic,
                    peak_note=note,
                    launches=dom_launches, avg_launch_ms=dom_ms / max(1, dom_launches),
                    share_of_device_time=dom_ms / total_ms if total_ms else None,
                    classes={c: dict(launches=v[0], ms=v[1]) for c, v in per_class.items()})

    # ---- end to end through the public API with host buffers (pinned), loss read back.
    # Every step copies all of its inputs (H, W and the teacher cache) from pinned host
    # memory and reads its loss back.  The copies run on a second stream into one of two
    # device buffer sets, so step i + 1's inputs travel while step i computes, as a training
    # loop that prefetches its next batch would; the first step's copy is not hidden.
    e2e = None
    if not args.no_e2e:
        pinned = {k: v.pin_memory() for k, v in h.items()}
        bufs = [{k: torch.empty_like(v, device=dev) for k, v in h.items()} for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in pinned.values())
        n_e2e = max(1, min(args.steps, 10))
        loss_host = torch.empty(n_e2e, dtype=torch.float32).pin_memory()
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        used = [torch.cuda.Event() for _ in range(2)]

        def upload(j):
            copy_stream.wait_event(used[j])  # the step that last read buffer set j is done
            with torch.cuda.stream(copy_stream):
                for k in bufs[j]:
                    bufs[j][k].copy_(pinned[k], non_blocking=True)
            copied[j].record(copy_stream)

        barrier()
        t0 = time.perf_counter()
        upload(0)
        for i in range(n_e2e):
            j = i % 2
            if i + 1 < n_e2e:
                upload(1 - j)
            stream.wait_event(copied[j])
            out = step(bufs[j])
            used[j].record(stream)
            loss_host[i].copy_(out, non_blocking=True)
        stream.synchronize()
        barrier()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, dist, dev)
        e2e = dict(value=job_rate(T, world, e2e_s), unit="tokens/s", h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=4,
                   ms_per_step=1e3 * e2e_s, steps=n_e2e, overlap="next step's input copy under this step's compute",
                   outputs="the loss is read back each step; dH and dW stay on the device for the training "
                           "step that consumes them")
        del bufs, pinned

    # ---- CPU baseline: the oracle on a bounded sample, rank 0 at N = 1 only
    cpu = None
    if not args.no_cpu and world == 1 and rank == 0:
        cpu_rows = min(args.cpu_rows, T)
        rate, secs = cpu_oracle_rate(cfg, h["W"].view(torch.int16).numpy().view(np.uint16)
                                     if tdt == torch.bfloat16 else h["W"].numpy(), cpu_rows)
        host = host_info()
        cpu = dict(value=rate, unit="tokens/s", cores=host["cores"], kind="oracle",
                   cpu_model=host.get("cpu_model"), blas=host.get("blas"),
                   sample=f"oracle fwd+bwd (fp64, full-vocab logit rows, analytic dH/dW) on rows 0..{cpu_rows - 1}"
                          f" of {cfg.name}; {secs:.1f} s")

    if rank == 0:
        line = dict(metric=METRIC, value=tokens_per_s, unit="tokens/s", n_gpus=world, steps=args.steps,
                    warmup=args.warmup, ms_per_step=1e3 * sec_per_step, higher_is_better=True, scaling="weak",
                    vs_baseline=None, dtype=cfg.dtype, data="synthetic",
                    config=dict(workload=cfg.name, T=T, d=d, V=V, K=K, tau=cfg.tau, chunk=chunk, valid_rows=n_valid,
                                batch=cfg.batch, seq_len=cfg.seq_len or T,
                                l2="inputs larger than L2 (H %.2f GB, W %.2f GB)" % (T * d * 2 / 1e9, V * d * 2 / 1e9),
                                parallelism=(f"dp{world}: token-sharded, loss partials and dW all-reduced "
                                             "(NCCL) inside the step" if sharded_path else "one GPU")),
                    tflops=tflops, frac_bf16_peak=tflops / peak_burst,
                    frac_bf16_peak_sustained=tflops / peak_sust, peak_source=peaks["source"],
                    peak_device_gib=peak_alloc / 2 ** 30, nontorch_device_gib=max(0.0, (free0 - free1 - peak_alloc) / 2 ** 30),
                    loss=loss_val, roofline=roofline, cpu_baseline=cpu, e2e=e2e, gpu_launches=int(launches),
                    clocks=clk.summary())
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def _kernel_src_sha():
    return _src_sha(("fckl_tc.cu", "fckl_ptx.cuh", "fckl_api.cu"))


def _src_sha(files):
    import hashlib

    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "chunked_kl_loss_head_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    main()
