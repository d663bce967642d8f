#!/usr/bin/env python3
"""Throughput of the gated sparse attention decode step at 128K context.

One step = one sparse_attn_decode call for a batch of 32 sequences, each with
131072 cached rows: indexer scan over every cached indexer key, exact Top-K
(K=2048), gathered attention over the kept rows with the sigmoid gate, split-K
combine. Prints one JSON line (rank 0). Also reports, in the same line, the
prefill throughput of the 8K and 128K workloads with the tensor-core rate of
their indexers, the dominant kernel's roofline, an end-to-end number through
host buffers, the fp64 oracle timed on the host, and at the 8K prefill shapes
the gradients over the kept set (fp32 CUDA-core rate), the block-granular
selection, the local-branch fusion, and dense causal attention against the
sparse layer across lengths (the break-even).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own batch of 32 sequences (weak scaling, no
collective on the data path; the only collectives are the timing barrier and
the max over ranks).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse-attn decode tok/s @128K ctx K=2048; prefill tok/s; % of roofline"
WORKLOAD = "decode_128k"
PREFILL_WORKLOAD = "prefill_8k"
SCAN_KERNEL_SRC = os.path.join(ROOT, "indexer_top_sparse_03_b300", "csrc", "decode_scan.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ---------------------------------------------------------------------------
# process group helpers (also exercised by the gloo tests on CPU)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[int(str(device).split(":")[1])])
        else:
            dist.barrier()


def aggregate_throughput(units_per_rank: int, world: int, max_seconds: float) -> float:
    """Whole-job units per second: all ranks' units over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML, read-only)
# ---------------------------------------------------------------------------

class ClockSampler:
    """SM clock and clock-event reasons during a timed region, read-only: NVML
    when importable, else `nvidia-smi --query-gpu ... -lms` in the background."""
    REASONS = {0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle",
               0x2: "applications_clocks_setting", 0x10: "sync_boost", 0x100: "display_clock_setting"}

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.error = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self.nvml = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.handle = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.handle, pynvml.NVML_CLOCK_SM)
            self.nvml = pynvml
            self.source = "nvml"
        except Exception as e:
            self.error = f"nvml: {e!r}"

    def _add_reasons(self, bits):
        for b, name in self.REASONS.items():
            if bits & b:
                self.reasons.add(name)

    def sample(self):
        nv = self.nvml
        try:
            self.samples.append(nv.nvmlDeviceGetClockInfo(self.handle, nv.NVML_CLOCK_SM))
            try:
                bits = nv.nvmlDeviceGetCurrentClocksEventReasons(self.handle)
            except AttributeError:
                bits = nv.nvmlDeviceGetCurrentClocksThrottleReasons(self.handle)
            self._add_reasons(bits)
            return True
        except Exception as e:                              # report, do not fail the bench
            self.error = repr(e)
            return False

    def _run(self):
        while not self._stop.is_set() and self.sample():
            time.sleep(0.001)

    def __enter__(self):
        if self.nvml is not None:
            self.sample()                                   # at least one sample per region
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        else:
            import subprocess
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                time.sleep(0.3)                             # let the first sample land
            except Exception as e:
                self.error = (self.error or "") + f"; nvidia-smi: {e!r}"
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self.sample()
        self._stop.set()
        if self._thread is not None:
            self._thread.join()
        if self._proc is not None:
            time.sleep(0.05)
            self._proc.terminate()
            out, _ = self._proc.communicate(timeout=10)
            for line in out.splitlines():
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 3:
                    continue
                try:
                    mhz, mx, bits = float(parts[0]), float(parts[1]), int(parts[2], 16)
                except ValueError:
                    continue
                self.max_mhz = mx
                if bits & 0x1:                              # idle sample (before/after the work)
                    continue
                self.samples.append(mhz)
                self._add_reasons(bits)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": self.source, "error": self.error}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons - {"gpu_idle"}), "samples": len(self.samples),
                "source": self.source}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


def queue_ahead(torch, seconds: float):
    """Hold the current stream on the device for about `seconds` (a bounded
    spin), so that the launches enqueued meanwhile run back to back."""
    torch.cuda._sleep(int(seconds * 2.0e9))


def file_sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def recorded_traffic(kernel: str, src: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel's source
    is unchanged since the capture."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    d = json.load(open(TRAFFIC_FILE)).get(kernel)
    if not d or d.get("source_sha") != file_sha(src):
        return None
    return d.get("dram_bytes_per_launch")


def decode_bytes(cfg, lens):
    """Algorithmic bytes of one decode step and of its indexer scan."""
    import torch
    n = sum(lens)
    fp8 = cfg.idx_dtype == torch.float8_e4m3fn
    es = 1 if fp8 else 2                     # FP8 keys: one code byte per element + a 4-byte row scale
    scan = n * (cfg.di * es + (4 if fp8 else 0)) + cfg.B * cfg.Hi * (cfg.di * es + 4 + (4 if fp8 else 0))
    kept = sum(min(cfg.K, x) for x in lens)
    row = (cfg.dqk * 2 + cfg.dv * 2) if not cfg.latent else cfg.dqk * 2
    gather = kept * row
    small = cfg.B * (cfg.Hq * cfg.dqk * 2 + cfg.Hq * 4 + cfg.Hq * cfg.dv * 2 + 12)
    return scan + gather + small, scan


def oracle_sample_decode(cfg, seed, nseq, nthreads=0, min_seconds=0.0):
    """Time the fp64 oracle on nseq sequences of the workload (CPU): the same
    sample is evaluated repeatedly until min_seconds have passed (at least
    once). Returns (seconds per pass, threads used, passes)."""
    import oracle
    from workloads import get_config, make_decode
    small = get_config(cfg.name, B=nseq)
    inp = make_decode(small, seed=seed)
    passes = 0
    t0 = time.perf_counter()
    while True:
        oracle.decode_layer(inp, small.K, small.dv, 1 / math.sqrt(small.dqk), nthreads=nthreads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return dt / passes, oracle.threads_used(nthreads, nseq), passes


# ---------------------------------------------------------------------------
# the reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    from workloads import get_config
    cfg = get_config(WORKLOAD)
    ncores = os.cpu_count() or 1
    nseq = max(1, min(cfg.B, ncores))
    times = []
    cores = 1
    for i in range(args.warmup + args.steps):
        dt, cores, _ = oracle_sample_decode(cfg, args.seed + i, nseq)
        if i >= args.warmup:
            times.append(dt)
    step = sum(times) / len(times)
    value = nseq / step
    sample = (f"{nseq} of the {cfg.B} sequences of one decode step (ctx {cfg.ctx}, K {cfg.K}) "
              f"per step, full layer in fp64")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(cfg),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(cfg):
    return {"workload": cfg.name, "batch_per_gpu": cfg.B, "ctx": cfg.ctx, "K": cfg.K, "Hq": cfg.Hq,
            "dqk": cfg.dqk, "dv": cfg.dv, "Hi": cfg.Hi, "di": cfg.di, "attn_dtype": "bf16",
            "indexer_dtype": "bf16",
            "l2": "inputs larger than L2: every step streams the 537 MB indexer-key cache",
            "parallelism": "replicas, one batch per GPU, no data-path collective"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def indexer_roofline(sa, torch, dev, cfg, inp, iters):
    """The tensor-core indexer alone over every causal row of the workload, in
    the same <= 1 GiB row passes the prefill uses; FLOPs = 2*Hi*di per causal
    (query, key) pair."""
    L = cfg.L
    rows = max(1, min(L, (1 << 30) // (4 * ((L + 3) // 4 * 4))))
    ld = (L + 3) // 4 * 4
    scores = torch.empty((rows, ld), dtype=torch.float32, device=dev)

    def sweep():
        for t0 in range(0, L, rows):
            t1 = min(L, t0 + rows)
            qs = None if inp["q_scale"] is None else inp["q_scale"][t0:t1]
            sa.indexer_score(inp["q_idx"][t0:t1], inp["w"][t0:t1], inp["k_idx"], qs, inp["k_scale"],
                             causal_offset=t0, scores=scores[: t1 - t0])
    sweep()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        sweep()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    flops = 2 * cfg.Hi * cfg.di * (L * (L + 1) // 2)
    peaks = measured_peaks()
    tflops = flops / (ms * 1e-3) / 1e12
    del scores
    return {"kernel": "indexer_tc_kernel", "bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"],
            "peak_source": peaks["source"] + " burst bf16 (the reference for both dtypes: the target is stated against bf16)",
            "algorithmic_flops": flops, "ms": ms, "dtype": str(inp["q_idx"].dtype).replace("torch.", "")}


FP32_ALU_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12   # SMs x fp32 lanes x FMA x max SM clock


def bench_backward(sa, torch, dev, seed, iters=3):
    """Gradients over the index set the prefill selects, at the 8K prefill
    shapes: tok/s and the rate of 14 * Hq * d FLOP per kept (query, key) pair
    (the forward recomputed, then q.k, do.v, dq, dk, dv) against the bf16
    tensor peak (and, for reference, the fp32 CUDA-core peak)."""
    from workloads import get_config, make_prefill
    cfg = get_config(PREFILL_WORKLOAD)
    inp = make_prefill(cfg, seed=seed, device=dev)
    scale = 1 / math.sqrt(cfg.dqk)
    idx = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device=dev)
    sa.sparse_attn_prefill(inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"], inp["w"], inp["gate"],
                           cfg.K, scale, idx_out=idx)
    g = torch.Generator(device=dev)
    g.manual_seed(seed + 1)
    dout = torch.randn((cfg.L, cfg.Hq, cfg.dv), generator=g, device=dev).to(cfg.attn_dtype)

    def step():
        return sa.sparse_attn_backward(inp["q"], inp["k"], inp["v"], idx, inp["gate"], dout, scale)
    step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    pairs = sum(min(cfg.K, t + 1) for t in range(cfg.L))
    flops = 14 * cfg.Hq * cfg.dqk * pairs
    tf = flops / (ms * 1e-3) / 1e12
    peaks = measured_peaks()
    return {"workload": cfg.name, "L": cfg.L, "K": cfg.K, "ms": ms, "tok_s": cfg.L / (ms * 1e-3),
            "roofline": {"kernel": "attn_bwd_tc_kernel", "bound": "tensor", "achieved": tf,
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                         "peak_source": peaks["source"] + " burst bf16",
                         "algorithmic_flops": flops,
                         "fp32_alu_frac": tf / FP32_ALU_PEAK_TFLOPS}}


def bench_decode_config(sa, torch, dev, seed, name, iters=200, **over):
    """Decode throughput of another decode workload (graph replay of one step)
    and its whole-step fraction of the HBM roofline (the same byte count as the
    headline workload: indexer keys scanned + kept rows + small tensors)."""
    from workloads import get_config, make_decode
    cfg = get_config(name, **over)
    inp = make_decode(cfg, seed=seed, device=dev)
    lens = inp["lens"]
    scale = 1 / math.sqrt(cfg.dqk)
    out = torch.empty((cfg.B, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device=dev)
    idx = torch.empty((cfg.B, cfg.K), dtype=torch.int32, device=dev)

    def step():
        sa.sparse_attn_decode(inp["q"], inp["q_idx"], inp["w"], inp["gate"], inp["k_cache"], inp["v_cache"],
                              inp["k_idx_cache"], inp["seq_start"], inp["ctx_len"], max(lens), cfg.K, scale,
                              dv=cfg.dv, q_scale=inp["q_scale"], k_idx_scale=inp["k_idx_scale"],
                              ld_k=inp["ld_k"], ld_v=inp["ld_v"], out=out, idx_out=idx)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    step_bytes, _ = decode_bytes(cfg, lens)
    peak = measured_peaks()["hbm_gbs"]
    res = {"workload": cfg.name, "indexer_dtype": str(cfg.idx_dtype).replace("torch.", ""), "B": cfg.B,
           "ctx_sum": int(sum(lens)), "ms": ms, "tok_s": cfg.B / (ms * 1e-3),
           "step_bytes": step_bytes, "hbm_frac": step_bytes / (ms * 1e-3) / 1e9 / peak}
    del graph, inp
    torch.cuda.empty_cache()
    return res


def bench_variants(sa, torch, dev, seed, iters=5):
    """The block-granular and the local-branch prefill at the 8K prefill shapes
    (tok/s; selection and attention split by events for the block variant)."""
    from workloads import get_config, make_prefill
    cfg = get_config(PREFILL_WORKLOAD)
    inp = make_prefill(cfg, seed=seed, device=dev)
    scale = 1 / math.sqrt(cfg.dqk)
    out = torch.empty((cfg.L, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device=dev)
    res = {}

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / iters
    for bs in (64, 16):
        ms = timed(lambda: sa.sparse_attn_prefill_blocks(inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"],
                                                         inp["w"], inp["gate"], cfg.K, scale, bs, out=out))
        res[f"blocks_{bs}"] = {"workload": cfg.name, "block_size": bs, "K": cfg.K, "ms": ms,
                               "tok_s": cfg.L / (ms * 1e-3)}
    for win in (512,):
        ms = timed(lambda: sa.sparse_attn_prefill_local(inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"],
                                                        inp["w"], inp["gate"], cfg.K, scale, win, out=out))
        res[f"local_{win}"] = {"workload": cfg.name, "window": win, "K": cfg.K, "ms": ms, "tok_s": cfg.L / (ms * 1e-3)}
    # the attention stage under each kernel choice for the gathered rows, at
    # the 8K prefill's shapes and L = 16384 (rows below 4K = 8192 go to the
    # dense kernel whatever the choice, the other half is gathered)
    del out, inp
    cfg = get_config(PREFILL_WORKLOAD, L=16384)
    inp = make_prefill(cfg, seed=seed, device=dev)
    out = torch.empty((cfg.L, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    kernels = {}
    for name, which in (("mma_sync", sa.ATTN_AUTO), ("tcgen05", sa.ATTN_TCGEN05)):
        prev = sa.set_prefill_attention_kernel(which)
        try:
            times = []
            for _ in range(iters + 1):
                sa.sparse_attn_prefill(inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"], inp["w"],
                                       inp["gate"], cfg.K, scale, q_scale=inp["q_scale"], k_scale=inp["k_scale"],
                                       out=out, stage_events=ev)
                torch.cuda.synchronize()
                times.append(ev[0].elapsed_time(ev[1]))
        finally:
            sa.set_prefill_attention_kernel(prev)
        kernels[name] = statistics.median(times[1:])
    res["prefill_attention_kernels"] = {"workload": cfg.name, "L": cfg.L, "attention_ms": kernels}
    return res


def bench_break_even(sa, torch, dev, seed, lengths=(4096, 8192, 16384, 32768, 65536), iters=3):
    """Full attention against the sparse layer across lengths, at the 8K
    prefill's shapes (K = 2048): dense causal attention time, and the sparse
    prefill split into selection (indexer + Top-K) and sparse attention;
    saving = full - sparse attention - selection (> 0: the sparse layer wins)."""
    from workloads import get_config, make_prefill
    rows = []
    for L in lengths:
        cfg = get_config(PREFILL_WORKLOAD, L=L)
        inp = make_prefill(cfg, seed=seed, device=dev)
        scale = 1 / math.sqrt(cfg.dqk)
        out = torch.empty((cfg.L, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device=dev)

        def dense():
            sa.attention_dense_causal(inp["q"], inp["k"], inp["v"], inp["gate"], scale, out=out)

        def sparse(ev=None):
            sa.sparse_attn_prefill(inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"], inp["w"], inp["gate"],
                                   cfg.K, scale, out=out, stage_events=ev)
        dense()
        sparse()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            dense()
        e1.record()
        torch.cuda.synchronize()
        dense_ms = e0.elapsed_time(e1) / iters
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(iters)]
        queue_ahead(torch, 0.02)
        for i in range(iters):
            ev[i][0].record()
            sparse(ev[i][1:])
        torch.cuda.synchronize()
        sel = statistics.median(ev[i][0].elapsed_time(ev[i][1]) for i in range(iters))
        att = statistics.median(ev[i][1].elapsed_time(ev[i][2]) for i in range(iters))
        flops = 4 * cfg.Hq * cfg.dqk * (L * (L + 1) // 2)
        rows.append({"L": L, "K": cfg.K, "dense_ms": dense_ms, "dense_tflops": flops / (dense_ms * 1e-3) / 1e12,
                     "selection_ms": sel, "sparse_attention_ms": att, "saving_ms": dense_ms - att - sel})
        del inp, out
        torch.cuda.empty_cache()
    return rows


def bench_prefill(sa, torch, dev, seed, name, iters):
    """Prefill tok/s of one workload (stage split by events), plus the tensor
    rate of its indexer."""
    from workloads import get_config, make_prefill
    cfg = get_config(name)
    inp = make_prefill(cfg, seed=seed, device=dev)
    scale = 1 / math.sqrt(cfg.dqk)
    out = torch.empty((cfg.L, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device=dev)
    idx = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(iters)]

    def step(e=None):
        if e is not None:
            e[0].record()
        sa.sparse_attn_prefill(inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"], inp["w"],
                               inp["gate"], cfg.K, scale, q_scale=inp["q_scale"], k_scale=inp["k_scale"],
                               out=out, idx_out=idx, stage_events=None if e is None else e[1:])
    step()
    torch.cuda.synchronize()
    queue_ahead(torch, 0.02)
    for i in range(iters):
        step(ev[i])
    torch.cuda.synchronize()
    tot = [ev[i][0].elapsed_time(ev[i][2]) for i in range(iters)]
    sel = [ev[i][0].elapsed_time(ev[i][1]) for i in range(iters)]
    ms = statistics.median(tot)
    del out, idx
    roof = indexer_roofline(sa, torch, dev, cfg, inp, iters)
    return {"workload": cfg.name, "L": cfg.L, "K": cfg.K, "tok_s": cfg.L / (ms * 1e-3), "ms": ms,
            "selection_ms": statistics.median(sel), "attention_ms": ms - statistics.median(sel),
            "indexer_roofline": roof}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import indexer_top_sparse_03_b300 as sa
    from indexer_top_sparse_03_b300.binding import DecodeArgs  # noqa: F401
    from workloads import get_config, make_decode

    rank, local_rank, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device(dev))
    sa.load_library()

    cfg = get_config(WORKLOAD)
    inp = make_decode(cfg, seed=args.seed + rank, device=dev)
    lens = inp["lens"]
    scale = 1 / math.sqrt(cfg.dqk)
    out = torch.empty((cfg.B, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device=dev)
    idx = torch.empty((cfg.B, cfg.K), dtype=torch.int32, device=dev)
    max_ctx = max(lens)

    def step(events=None):
        sa.sparse_attn_decode(inp["q"], inp["q_idx"], inp["w"], inp["gate"], inp["k_cache"],
                              inp["v_cache"], inp["k_idx_cache"], inp["seq_start"], inp["ctx_len"],
                              max_ctx, cfg.K, scale, out=out, idx_out=idx, stage_events=events)

    K, W = args.steps, args.warmup
    for _ in range(W):
        step()
    torch.cuda.synchronize()

    # The timed region replays a CUDA graph of one step (its five launches,
    # chained by programmatic dependent launch), so that the host's launch
    # cost, which varies from host to host, stays out of the device-timed
    # throughput; the end-to-end number below goes through the API per step.
    replay, launch_mode = step, "eager"
    try:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        with torch.cuda.graph(graph):
            step()
        for _ in range(W):
            graph.replay()
        torch.cuda.synchronize()
        replay, launch_mode = graph.replay, "cuda_graph"
    except RuntimeError:
        torch.cuda.synchronize()

    # the timed region: K back-to-back steps, no events between the stages
    clocks = ClockSampler(local_rank)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dev)
    torch.cuda.synchronize()
    with clocks:
        t_start.record()
        for i in range(K):
            replay()
        t_end.record()
        torch.cuda.synchronize()
    barrier(dev)
    ms_step = t_start.elapsed_time(t_end) / K
    ms_step_max = reduce_max(ms_step, dev)
    value = aggregate_throughput(cfg.B, world, ms_step_max * 1e-3)

    # stage breakdown, measured separately (events between the stages break the
    # programmatic launch chain, so these steps run a little slower). The steps
    # are queued behind a device-side delay, so that the host's launch time
    # never shows up as idle time between two events.
    KS = min(K, 50)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(KS)]
    queue_ahead(torch, KS * 5e-4)
    for i in range(KS):
        ev[i][0].record()
        step(ev[i][1:])
    torch.cuda.synchronize()
    stage = {
        "indexer_scan_ms": statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(KS)),
        "topk_ms": statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for i in range(KS)),
        "attention_ms": statistics.mean(ev[i][2].elapsed_time(ev[i][3]) for i in range(KS)),
    }
    step_bytes, scan_bytes = decode_bytes(cfg, lens)
    peaks = measured_peaks()
    # the scan stage's duration (zeroing kernel + scan kernel), from events on
    # the stream the kernels run on: a conservative duration for the scan
    scan_s = stage["indexer_scan_ms"] * 1e-3
    achieved = scan_bytes / scan_s / 1e9
    traffic = recorded_traffic("decode_scan_kernel", SCAN_KERNEL_SRC)
    roofline = {"kernel": "decode_scan_kernel", "bound": "hbm", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "peak_source": peaks["source"], "algorithmic_bytes": scan_bytes,
                "traffic": traffic,
                "step_frac": step_bytes / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"]}

    # end to end through host buffers, as a serving loop runs it: every step
    # goes through the C-ABI call with host buffers (sparse_attn_decode_host):
    # the step's q, q_idx, w and gate are copied in from pinned host memory
    # (one copy: they sit packed in one device buffer, each part at a 16-byte
    # offset), the step runs, and its output is copied back to pinned host
    # memory. The host waits for step i - 1's output while step i is queued
    # (outputs double-buffered), so its own call overhead overlaps the
    # device work instead of adding to it.
    names = ("q", "q_idx", "w", "gate")
    sizes = [inp[k].numel() * inp[k].element_size() for k in names]
    offs = [sum(sizes[:i]) for i in range(len(sizes))]
    assert all(o % 16 == 0 for o in offs)
    dbuf = torch.empty(sum(sizes), dtype=torch.uint8, device=dev)
    hbuf = torch.empty(sum(sizes), dtype=torch.uint8).pin_memory()
    staged = {}
    for k_, o, n_ in zip(names, offs, sizes):
        staged[k_] = dbuf[o:o + n_].view(inp[k_].dtype).view(inp[k_].shape)
        hbuf[o:o + n_].copy_(inp[k_].cpu().contiguous().view(-1).view(torch.uint8))
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = hbuf.numel()
    d2h = out_h[0].numel() * out_h[0].element_size()
    stream = torch.cuda.current_stream()
    done = [torch.cuda.Event() for _ in range(2)]
    call = sa.DecodeStep(staged["q"], staged["q_idx"], staged["w"], staged["gate"], inp["k_cache"], inp["v_cache"],
                         inp["k_idx_cache"], inp["seq_start"], inp["ctx_len"], max_ctx, cfg.K, scale, out=out,
                         idx_out=idx, stream=stream)

    def e2e_run(n):
        for i in range(n):
            call.run_host(hbuf, dbuf, out_h[i & 1])
            done[i & 1].record(stream)
            if i > 0:
                done[(i - 1) & 1].synchronize()      # the host has step i - 1's output
        done[(n - 1) & 1].synchronize()              # and the last step's
    e2e_run(max(W, 20))                      # untimed: the host path settles over the first steps
    barrier(dev)
    t0 = time.perf_counter()
    e2e_run(K)
    e2e_s = reduce_max((time.perf_counter() - t0) / K, dev)
    e2e = {"value": aggregate_throughput(cfg.B, world, e2e_s), "unit": "tok/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    del call

    prefill = backward = variants = other_decode = None
    if not args.no_prefill:
        del inp, staged, dbuf, hbuf, out_h
        torch.cuda.empty_cache()
        prefill = [bench_prefill(sa, torch, dev, args.seed + rank, PREFILL_WORKLOAD, 10),
                   bench_prefill(sa, torch, dev, args.seed + rank, "prefill_128k", 2)]
        backward = bench_backward(sa, torch, dev, args.seed + rank)
        other_decode = [bench_decode_config(sa, torch, dev, args.seed + rank, n)
                        for n in ("decode_mla", "decode_ragged")]
        # the 128K point with FP8-e4m3 indexer keys (one fp32 scale per cached row)
        other_decode.append(bench_decode_config(sa, torch, dev, args.seed + rank, WORKLOAD,
                                                idx_dtype=torch.float8_e4m3fn))
        variants = bench_variants(sa, torch, dev, args.seed + rank)
        variants["break_even"] = bench_break_even(sa, torch, dev, args.seed + rank)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ncores = os.cpu_count() or 1
        nseq = max(1, min(cfg.B, ncores))
        dt, cores, passes = oracle_sample_decode(cfg, args.seed, nseq, min_seconds=12.0)
        cpu = {"value": nseq / dt, "unit": "tok/s", "cores": cores, "kind": "oracle",
               "sample": f"{nseq} of the {cfg.B} sequences of one decode step (ctx {cfg.ctx}, "
                         f"K {cfg.K}), full layer in fp64, evaluated {passes} times "
                         f"({dt * passes:.1f} s of CPU work)"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": K,
                "warmup": W, "ms_per_step": ms_step_max, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": dict(workload_config(cfg), launch=launch_mode), "roofline": roofline,
                "stages_ms": stage,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 5 * K,
                "clocks": clocks.summary(), "prefill": prefill, "backward": backward,
                "variants": variants, "decode_other": other_decode}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    p.add_argument("--gpus", type=int, default=int(os.environ.get("WORLD_SIZE", "1")))
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile-prefill", type=int, default=0, metavar="L",
                   help="for profiler captures only: run the FP8 128K-prefill shapes at length L\n"
                        "(--steps calls, no timing, no JSON line) and exit")
    p.add_argument("--prefill-attention", choices=("auto", "tcgen05"), default="auto",
                   help="with --profile-prefill: the kernel for the gathered attention of prefill rows")
    args = p.parse_args(argv)
    if args.profile_prefill:
        return profile_prefill(args)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


def profile_prefill(args):
    """A plain sequence of sparse_attn_prefill calls for ncu: the prefill_128k
    shapes at length args.profile_prefill, args.steps calls."""
    import torch

    import indexer_top_sparse_03_b300 as sa
    from workloads import get_config, make_prefill
    sa.load_library()
    sa.set_prefill_attention_kernel(sa.ATTN_TCGEN05 if args.prefill_attention == "tcgen05" else sa.ATTN_AUTO)
    cfg = get_config("prefill_128k", L=args.profile_prefill)
    inp = make_prefill(cfg, seed=args.seed, device="cuda")
    out = torch.empty((cfg.L, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device="cuda")
    for _ in range(args.steps):
        sa.sparse_attn_prefill(inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"], inp["w"], inp["gate"],
                               cfg.K, 1 / math.sqrt(cfg.dqk), q_scale=inp["q_scale"], k_scale=inp["k_scale"],
                               out=out, idx_out=idx)
    torch.cuda.synchronize()
    return 0


if __name__ == "__main__":
    sys.exit(main())
