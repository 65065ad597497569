#!/usr/bin/env python
"""Benchmark of the tiled GEMM C = A x B on GB300.

A step is one pass of the whole path: one tg_gemm call (one kernel launch)
on one batch of synthetic fp16 operands already resident in HBM.  The
default workload is the 8192^3 fp16 GEMM (U(-1,1) inputs, fp32 accumulation,
fp16 output), the compute-bound shape of the tensor-core roofline.  Two operand
sets rotate between steps so every step streams 384 MB of fresh A/B/C, more
than the 129 MB L2.

Prints ONE JSON line (rank 0):
  value      whole-job TFLOP/s (2*M*N*K per step) over the timed steps;
  e2e        the same metric through the C ABI from pinned HOST buffers,
             with the host->device copies of A and B and the device->host
             copy of C inside the timed region;
  roofline   achieved TFLOP/s of the GEMM kernel (CUDA events around each
             launch on the launching stream) against the measured peak;
  cpu_baseline  the CPU oracle timed on a bounded row sample of the same
             product, on the host's cores (N=1 only).
`--impl reference` times the oracle itself as the reference arm.

Multi-GPU (torchrun): every rank runs an independent replica of the same
workload on its own GPU; there is no data exchange.  value = all ranks'
FLOPs / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s and % of GB300 dense FP16 tensor peak (1 GPU), vs CPU oracle"
# GB300 dense fp16/bf16 tensor peak, the vendor's figure (2:4 sparsity not
# counted): the "spec" denominator beside the measured one
SPEC_FP16_DENSE_TFLOPS = 2500.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic (read + write bytes per launch) of a workload's kernel from
# one ncu capture, with the hash of the kernel's sources it was taken on.  A
# stale hash means the kernel changed since: traffic is then null.
PAIR_SOURCES = ["tiled_gemm_tg_gb300/csrc/gemm_tc2.cu", "tiled_gemm_tg_gb300/csrc/ptx.cuh",
                "tiled_gemm_tg_gb300/csrc/tc_common.cuh", "tiled_gemm_tg_gb300/csrc/tg_internal.h"]
MAIN_SOURCES = ["tiled_gemm_tg_gb300/csrc/gemm_tc.cu", "tiled_gemm_tg_gb300/csrc/ptx.cuh",
                "tiled_gemm_tg_gb300/csrc/tc_common.cuh", "tiled_gemm_tg_gb300/csrc/tg_internal.h",
                "tiled_gemm_tg_gb300/csrc/l2_prefetch.cuh"]
KERNEL_SOURCES = PAIR_SOURCES
ATTN_KERNEL_SOURCES = ["tiled_gemm_tg_gb300/csrc/attention_fwd2.cu", "tiled_gemm_tg_gb300/csrc/ptx.cuh",
                       "tiled_gemm_tg_gb300/csrc/tc_common.cuh", "tiled_gemm_tg_gb300/csrc/tg_internal.h"]

NCU_TRAFFIC = {
    # the pair kernel's ncu summary under profiles/: 774.6 MB read + 124.7 MB written
    "square_8192": {"bytes": 899289088, "kernel_hash": "8d1ea02ab18e6368",
                    "sources": PAIR_SOURCES},
    # the one-CTA kernel on the tiling example: 3.23 MB read, C still in L2 at exit
    "tile_1024x2048x512": {"bytes": 3236096, "kernel_hash": "95357b09aa000fae",
                           "sources": MAIN_SOURCES},
    # the one-CTA kernel on 256 products of 256^3: 67.2 MB read + 3.5 MB written
    "batched_256x256x256x256": {"bytes": 70665728, "kernel_hash": "95357b09aa000fae",
                                "sources": MAIN_SOURCES},
}

# DRAM traffic per launch of the attention kernel that keeps P in tensor
# memory, from one ncu capture, valid while its sources hash the same
ATTN_NCU_TRAFFIC = {
    # the kernel's ncu summary under profiles/: 50.4 MB read + 0.9 MB written
    "attn_16x4096x128": {"bytes": 51291136, "kernel_hash": "93f45a4ce8dd9af5",
                         "sources": ATTN_KERNEL_SOURCES},
}


def traffic_of(table, name):
    """The recorded DRAM bytes per launch for a workload, or None if there is
    no record or the kernel's sources have changed since it was taken."""
    rec = table.get(name)
    if rec and rec.get("kernel_hash") == kernel_hash(rec.get("sources")):
        return rec["bytes"]
    return None


def kernel_hash(sources=None) -> str:
    h = hashlib.sha256()
    for p in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------- clocks

class NvmlPoller:
    """In-process NVML reads of the SM clock, its maximum, the clock-event
    reasons and the power draw every `period_s`, so that a timed region of a
    few milliseconds still holds samples (nvidia-smi's floor is 100 ms).
    Only reads: nvmlDeviceGetClockInfo, nvmlDeviceGetMaxClockInfo,
    nvmlDeviceGetCurrentClocksEventReasons, nvmlDeviceGetPowerUsage."""

    NVML_CLOCK_SM = 1
    # clock-event reason bits of the public NVML API
    REASON_BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown",
                   0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, uuid: str | None, period_s: float = 0.002):
        self.samples = []
        self.period_s = period_s
        self.ok = False
        self._stop = threading.Event()
        self.thread = None
        if not uuid:
            return
        try:
            import ctypes

            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            dev = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(dev)) != 0:
                return
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self._ct, self._lib, self._dev, self._reasons = ctypes, lib, dev, reasons
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _one(self):
        ct, lib, dev = self._ct, self._lib, self._dev
        mhz, mx, mw = ct.c_uint(), ct.c_uint(), ct.c_uint()
        mask = ct.c_ulonglong()
        if lib.nvmlDeviceGetClockInfo(dev, self.NVML_CLOCK_SM, ct.byref(mhz)) != 0:
            return None
        lib.nvmlDeviceGetMaxClockInfo(dev, self.NVML_CLOCK_SM, ct.byref(mx))
        self._reasons(dev, ct.byref(mask))
        lib.nvmlDeviceGetPowerUsage(dev, ct.byref(mw))
        return (float(mhz.value), float(mx.value), int(mask.value), mw.value / 1000.0)

    def _loop(self):
        while not self._stop.is_set():
            r = self._one()
            if r is not None:
                self.samples.append((time.time(),) + r)
            time.sleep(self.period_s)

    def start(self):
        if self.ok:
            self._stop.clear()
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()

    def stop(self):
        self._stop.set()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        if not inside:
            return None
        sm = sorted(x[1] for x in inside)
        reasons = sorted({name for x in inside for bit, name in self.REASON_BITS.items()
                          if x[3] & bit})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(x[2] for x in inside),
                "sm_mhz_min": sm[0], "reasons": reasons, "samples": len(inside),
                "window": f"timed (NVML every {self.period_s * 1e3:.0f} ms)",
                "power_w_max": max(x[4] for x in inside)}


class ClockSampler:
    """Clock/throttle samples while running: NVML polled in-process every
    2 ms (the timed region is often shorter than nvidia-smi's 100 ms period),
    with nvidia-smi every 100 ms beside it as the fallback."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id
        self.thread = None
        self.nvml = NvmlPoller(gpu_id)

    def start(self):
        self.nvml.start()
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        self.nvml.stop()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        fine = self.nvml.summary(t0, t1)
        if fine is not None:
            return fine
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed"
        if len(inside) < 3:
            inside = [p for (_, p) in self.samples]
            window = "whole run (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = sorted(v for v in (num(p[1]) for p in inside) if v is not None)
        smax = max((v for v in (num(p[2]) for p in inside) if v is not None), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower().startswith("active")})
        power = [v for v in (num(p[3]) for p in inside) if v is not None]
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------- CPU oracle leg

def host_array(t):
    """A CPU tensor as the NumPy array the oracle takes (E4M3 as its bytes)."""
    import torch

    return t.view(torch.uint8).numpy() if t.dtype == torch.float8_e4m3fn else t.numpy()


def oracle_rows_sample(w, a_cpu, b_cpu, target_s: float):
    """Time the oracle on whole rows of C, growing the row count until one
    timed call takes about target_s.  Returns (TFLOP/s, rows, seconds, threads)."""
    import oracle

    nt = oracle.num_threads()
    a_np = host_array(a_cpu)
    b_np = host_array(b_cpu)
    rows = max(1, min(nt, w.M))
    while True:
        t = time.perf_counter()
        oracle.gemm(a_np[:rows], b_np)
        dt = time.perf_counter() - t
        if dt >= 0.6 * target_s or rows >= w.M:
            break
        rows = min(w.M, rows * max(2, int(0.9 * target_s / max(dt, 1e-3))))
    return 2.0 * rows * w.N * w.K / dt / 1e12, rows, dt, nt


# ------------------------------------------------------------------- main

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device) -> float:
    """The largest x over all ranks of the process group (x itself on one
    rank): the job is as slow as its slowest replica."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, ws: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput in tera-units per second: the units every rank
    processed over `steps` steps, divided by the slowest rank's time."""
    return ws * units_per_rank_step * steps / (elapsed_ms * 1e-3) / 1e12


def run_reference(args, w):
    """The reference arm: the CPU oracle, timed on the host's cores."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from tiled_gemm_tg_gb300 import inputs

    a, b = inputs.operands(w)
    if w.batch > 1:  # rows of the first product of the batch
        a, b = a[0], b[0]
    nt = oracle.num_threads()
    a_np, b_np = host_array(a), host_array(b)
    # size one step so that warmup + steps stay within ~2-3 minutes
    budget = 150.0 / max(1, args.steps + args.warmup)
    rows = max(1, min(nt, w.M))
    t = time.perf_counter()
    oracle.gemm(a_np[:rows], b_np)
    dt = time.perf_counter() - t
    if dt < budget:
        rows = min(w.M, rows * max(1, int(budget / max(dt, 1e-3))))
    for _ in range(args.warmup):
        oracle.gemm(a_np[:rows], b_np)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm(a_np[:rows], b_np)
    el = time.perf_counter() - t0
    value = 2.0 * rows * w.N * w.K * args.steps / el / 1e12
    sample = f"{rows} of {w.M} rows of C per step (full N={w.N}, K={w.K})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "in_dtype": w.in_dtype,
                   "out_dtype": w.out_dtype, "dist": w.dist},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# Fused epilogues the bench can time (tg_gemm_ex): C = act(alpha*AB + beta*D + bias).
EPILOGUES = {
    "none": None,
    "bias_relu": dict(alpha=1.0, beta=0.0, bias=True, act=1),
    "axpby_bias": dict(alpha=0.5, beta=1.0, bias=True, act=0),
    "axpby_bias_gelu": dict(alpha=0.5, beta=1.0, bias=True, act=2),
}


def _attn_oracle_sample(w, q, k, v, heads: int, rows: int) -> float:
    """Run the oracle on the first `rows` query rows of heads 0..heads-1 (each
    against its own keys and values); return the elapsed seconds."""
    import oracle

    t = time.perf_counter()
    for h in range(heads):
        kv = h if k.shape[0] > 1 else 0
        oracle.attention(q[h].numpy()[:rows], k[kv].numpy(), v[kv].numpy(), w.scale)
    return time.perf_counter() - t


def attn_cpu_sample(w, q, k, v, target_s: float):
    """Time the oracle on whole query rows of head 0, growing the row count
    until one call takes about target_s, then on whole heads if a full head
    is quicker than that.  Returns (TFLOP/s, heads, rows, s, threads)."""
    import oracle

    nt = oracle.num_threads()
    rows = max(1, min(nt, w.Nq))
    while True:
        dt = _attn_oracle_sample(w, q, k, v, 1, rows)
        if dt >= 0.6 * target_s or rows >= w.Nq:
            break
        rows = min(w.Nq, rows * max(2, int(0.9 * target_s / max(dt, 1e-3))))
    heads = 1
    if rows >= w.Nq and dt < 0.6 * target_s and w.batch > 1:
        heads = min(w.batch, max(2, int(0.9 * target_s / max(dt, 1e-3))))
        dt = _attn_oracle_sample(w, q, k, v, heads, rows)
    return 2.0 * heads * rows * w.Nk * (w.d + w.dv) / dt / 1e12, heads, rows, dt, nt


def _attn_sample_text(w, heads, rows):
    if heads > 1:
        return f"{heads} of {w.batch} heads, all {w.Nq} query rows"
    return f"{rows} of {w.Nq} query rows of head 0"


def run_reference_attention(args, w):
    """The reference arm for an attention workload: the oracle on host cores."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from tiled_gemm_tg_gb300 import inputs

    q, k, v = inputs.attn_operands(w)
    budget = 150.0 / max(1, args.steps + args.warmup)
    v0, heads, rows, dt, nt = attn_cpu_sample(w, q, k, v, min(budget, 5.0))
    for _ in range(args.warmup):
        _attn_oracle_sample(w, q, k, v, heads, rows)
    el = 0.0
    for _ in range(args.steps):
        el += _attn_oracle_sample(w, q, k, v, heads, rows)
    value = 2.0 * heads * rows * w.Nk * (w.d + w.dv) * args.steps / el / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "dv": w.dv, "scale": w.scale},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
                         "sample": _attn_sample_text(w, heads, rows) + " per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main_attention(args, w):
    """Attention forward, O = softmax(scale * Q K^T) V, timed like the GEMM:
    device-resident inputs rotated past L2, CUDA events per launch, clocks
    sampled, an end-to-end leg through the C ABI from pinned host buffers."""
    import torch

    import tiled_gemm_tg_gb300 as tg
    from tiled_gemm_tg_gb300 import inputs

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    tg.lib()
    q_cpu, k_cpu, v_cpu = inputs.attn_operands(w)
    out_dt = torch.float16 if w.out_dtype == "f16" else torch.float32
    oc = tg.F16 if w.out_dtype == "f16" else tg.F32
    set_bytes = w.algorithmic_bytes()
    n_sets = max(2, min(64, -(-3 * 129 * 2**20 // set_bytes)))
    sets = []
    for i in range(n_sets):
        sets.append((q_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev),
                     torch.empty((w.batch, w.Nq, w.dv), dtype=out_dt, device=dev)))
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    B, Nq, Nk, d, dv = w.batch, w.Nq, w.Nk, w.d, w.dv
    # a workspace lets calls with few CTAs split the keys, and calls whose
    # last wave of tiles is short split that wave's tiles (the library says
    # how much)
    ws_bytes = tg.tg_attention_workspace_size(B, Nq, Nk, d, dv)
    workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    forced = {"auto": 0, "general": 1, "tmem_p": 3}[args.attn_kernel]
    if tg.tg_attention_force_kernel(forced) != tg.TG_OK:
        raise RuntimeError("attention kernel override refused")
    kern = tg.tg_attention_kernel(B, Nq, Nk, d, dv, split_allowed=bool(ws_bytes))
    kern_name = {1: "attention_fwd_kernel", 2: "attention_fwd_kernel (+ attention_combine_kernel)",
                 3: "attention_fwd2_kernel" + (" (+ tail_zero_kernel)" if ws_bytes else "")
                 }.get(kern, "none")
    # kernels per call: the combine kernel after a key split; the counters'
    # zeroing kernel before a split of the last wave
    per_call = 2 if kern == 2 or (kern == 3 and ws_bytes) else 1

    def call(q, k, v, o, handle):
        st = tg.tg_attention_ws(B, Nq, Nk, d, dv, q.data_ptr(), d, Nq * d, k.data_ptr(), d,
                                Nk * d, v.data_ptr(), dv, Nk * dv, o.data_ptr(), dv, Nq * dv,
                                w.scale, tg.F16, oc, workspace.data_ptr() if ws_bytes else 0,
                                ws_bytes,
                                handle)
        if st != tg.TG_OK:
            raise tg.TgError(st, "tg_attention")

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    for i in range(args.warmup):
        call(*sets[i % n_sets], sh)
    tg.check(stream)
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            h = torch.cuda.current_stream().cuda_stream
            for i in range(args.steps):
                call(*sets[i % n_sets], h)
        graph.replay()  # warm replay
        tg.check(stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    host_t0 = time.time()
    t_start.record(stream)
    if graph is not None:
        # all K calls replayed from one CUDA graph: no host gaps between them
        graph.replay()
    else:
        for i in range(args.steps):
            evs[i][0].record(stream)
            call(*sets[i % n_sets], sh)
            evs[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    host_t1 = time.time()
    if ws > 1:
        torch.distributed.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    if graph is not None:
        per_launch = []  # one graph replay: only the mean per call is known
        kern_ms = elapsed_ms / args.steps
    else:
        per_launch = sorted(a.elapsed_time(b) for a, b in evs)
        kern_ms = sum(per_launch) / args.steps
    if tg.tg_gemm_check(sh) != tg.TG_OK:
        raise RuntimeError("a kernel abandoned a bounded wait during the timed region")
    elapsed_ms = max_over_ranks(elapsed_ms, ws, dev)
    flops = float(w.flops)
    value = job_throughput(flops, ws, args.steps, elapsed_ms)

    # end to end: Q, K, V in from pinned host memory, O out, every step;
    # steps are pipelined over three streams (H2D, attention, D2H) and two
    # device buffer sets, so step i's transfers overlap the kernels of steps
    # i-1 and i+1
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 20))
    qh, kh, vh = q_cpu.pin_memory(), k_cpu.pin_memory(), v_cpu.pin_memory()
    oh = [torch.empty((B, Nq, dv), dtype=out_dt).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "mm", "out")}
    started = [False, False]

    def e2e_step(i):
        slot = i % 2
        qd, kd, vd, od = sets[slot]
        if started[slot]:
            s_in.wait_event(ev["mm"][slot])  # the slot's previous call has read Q, K, V
        with torch.cuda.stream(s_in):
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
        ev["in"][slot].record(s_in)
        stream.wait_event(ev["in"][slot])
        if started[slot]:
            stream.wait_event(ev["out"][slot])  # the slot's previous O has been read out
        call(qd, kd, vd, od, sh)
        ev["mm"][slot].record(stream)
        s_out.wait_event(ev["mm"][slot])
        with torch.cuda.stream(s_out):
            oh[slot].copy_(od, non_blocking=True)
        ev["out"][slot].record(s_out)
        started[slot] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)  # after the last D2H, which follows every earlier step's work
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if tg.tg_gemm_check(sh) != tg.TG_OK:
        raise RuntimeError("a kernel abandoned a bounded wait during the e2e region")
    e2e_ms = max_over_ranks(e2e_ms, ws, dev)
    e2e_value = job_throughput(flops, ws, e2e_steps, e2e_ms)
    sampler.stop()
    clocks = sampler.summary(host_t0, host_t1)

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (kern_ms * 1e-3) / 1e12
    alg_bytes = w.algorithmic_bytes()
    attn_traffic = traffic_of(ATTN_NCU_TRAFFIC, w.name) if kern == 3 else None
    roofline = {
        "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
        "frac": achieved / peak, "traffic": attn_traffic, "kernel": kern_name,
        "kernel_ms": kern_ms,
        "kernel_ms_median": per_launch[len(per_launch) // 2] if per_launch else None,
        "kernel_ms_best": per_launch[0] if per_launch else None,
        "peak_source": f"{peak_src} bf16 burst (torch.matmul 8192^3) x 1.0 fp16/bf16 nominal ratio",
        "flop_per_byte": flops / alg_bytes, "algorithmic_bytes": alg_bytes,
        "achieved_gbs": alg_bytes / (kern_ms * 1e-3) / 1e9,
        "tensor_flops_executed": 2.0 * B * Nq * Nk * (d * -(-dv // 256) + dv),
    }
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v0, heads, rows, secs, nt = attn_cpu_sample(w, q_cpu, k_cpu, v_cpu, args.cpu_seconds)
        cpu = {"value": v0, "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
               "sample": f"{_attn_sample_text(w, heads, rows)}, {secs:.1f} s"}
    if rank == 0:
        line = {
            "metric": "attention forward TFLOP/s (4 Nq Nk d per head) and % of GB300 dense "
                      "FP16 tensor peak (1 GPU)",
            "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": w.name, "batch": B, "Nq": Nq, "Nk": Nk, "d": d, "dv": dv,
                       "scale": w.scale, "out_dtype": w.out_dtype, "accum": "f32",
                       "workspace_bytes": ws_bytes,
                       "workspace_use": ("key split" if kern == 2 else
                                         "last-wave split" if ws_bytes else "none"),
                       "timing": "CUDA graph replay" if graph is not None else "stream launches",
                       "kernel": {1: "general, P in shared memory", 2: "general, keys split",
                                  3: "P in tensor memory"}.get(kern, "none"),
                       "l2": f"{n_sets} rotating Q/K/V/O sets, "
                             f"{n_sets * set_bytes / 2**20:.0f} MB per pass",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": B * (Nq * d + Nk * (d + dv)) * 2,
                    "d2h_bytes_per_step": B * Nq * dv * oh[0].element_size(), "steps": e2e_steps,
                    "pipeline": "H2D / tg_attention / D2H on three streams, two device buffer sets"},
            "gpu_launches": args.steps * per_call,
            "roofline": roofline,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


# The specified workloads besides the headline 8192^3 square, measured in
# the same run as the headline: (group, workload name).
SPEC_WORKLOADS = [
    ("fp32 example", "f32_128x128x128"),
    ("edge set", "edge_4x4x4"), ("edge set", "edge_128x256x512"),
    ("edge set", "edge_127x255x512"), ("edge set", "edge_1x255x17"),
    ("tiling example", "tile_1024x2048x512"),
    ("skinny", "skinny_16x4096x4096"),
    ("wide", "wide_4096x16384x4096"),
]

KERNEL_OF_PATH = {1: "epilogue_only_kernel", 2: "gemm_simt_f32_kernel", 3: "gemm_tc_main_kernel",
                  4: "gemm_tc_boundary_kernel", 5: "gemm_skinny_kernel", 6: "gemm_tc_pair_kernel"}


def roofline_of(flops: float, alg_bytes: float, seconds: float, peak_tflops: float,
                hbm_gbs: float, alu_tflops: float | None = None):
    """(bound, fraction of roofline): the roofline time is the larger of the
    FLOPs at the compute peak and the algorithmic bytes at the copy
    bandwidth; the fraction is that time over the measured one."""
    compute = flops / ((alu_tflops if alu_tflops else peak_tflops) * 1e12)
    memory = alg_bytes / (hbm_gbs * 1e9)
    bound = "hbm" if memory > compute else ("alu" if alu_tflops else "tensor")
    return bound, max(compute, memory) / seconds


def measure_config(label, w, dev, launches, sampler, peaks, cpu_s, num_sms):
    """One specified workload: per-launch time stream-launched (launches
    back to back from the host, CUDA events around the whole loop) and
    replayed from one CUDA graph (no host gaps),
    operand sets rotated so one pass over them is at least 3x the L2; the
    roofline fraction of each; the clocks sampled meanwhile; the oracle's
    time on the host cores."""
    import torch

    import tiled_gemm_tg_gb300 as tg
    from tiled_gemm_tg_gb300 import inputs

    a_cpu, b_cpu = inputs.operands(w)
    out_dt = torch.float16 if w.out_dtype == "f16" else torch.float32
    in_code = {"f16": tg.F16, "e4m3": tg.E4M3}.get(w.in_dtype, tg.F32)
    out_code = tg.F16 if w.out_dtype == "f16" else tg.F32
    set_bytes = w.algorithmic_bytes()
    n_sets = max(2, min(4096, -(-3 * 129 * 2**20 // set_bytes)))
    sets = [(a_cpu.to(dev), b_cpu.to(dev), torch.empty((w.M, w.N), dtype=out_dt, device=dev))
            for _ in range(n_sets)]
    M, N, K = w.M, w.N, w.K
    stream = torch.cuda.current_stream()

    def call(i, h):
        a, b, c = sets[i % n_sets]
        st = tg.tg_gemm(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, in_code,
                        out_code, h)
        if st != tg.TG_OK:
            raise tg.TgError(st, w.name)

    path = tg.tg_gemm_path(M, N, K, sets[0][0].data_ptr(), K, sets[0][1].data_ptr(), N,
                           sets[0][2].data_ptr(), N, in_code, out_code)
    sh = stream.cuda_stream
    for i in range(10):
        call(i, sh)
    tg.check(stream)
    t0 = time.time()
    # stream-launched: back-to-back launches between two events (events
    # around every launch would add their own host time to each gap)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s0.record(stream)
    for i in range(launches):
        call(i, sh)
    s1.record(stream)
    torch.cuda.synchronize()
    us_stream = s0.elapsed_time(s1) * 1e3 / launches
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        h = torch.cuda.current_stream().cuda_stream
        for i in range(launches):
            call(i, h)
    graph.replay()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if tg.tg_gemm_check(sh) != tg.TG_OK:
        raise RuntimeError(f"{w.name}: a kernel abandoned a bounded wait")
    us_graph = g0.elapsed_time(g1) * 1e3 / launches
    del graph

    flops = float(w.flops)
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    alu = None
    if w.in_dtype == "f32":
        # fp32 FMA units: 128 lanes per SM, 2 FLOP each per clock, at the
        # largest SM clock the clock sampler reports
        mhz = float(peaks.get("sm_max_mhz", 2070.0))
        alu = num_sms * 128 * 2 * mhz * 1e6 / 1e12
    bound, frac_graph = roofline_of(flops, set_bytes, us_graph * 1e-6, peak, hbm, alu)
    _, frac_stream = roofline_of(flops, set_bytes, us_stream * 1e-6, peak, hbm, alu)
    rec = {
        "group": label, "workload": w.name, "M": M, "N": N, "K": K,
        "in_dtype": w.in_dtype, "out_dtype": w.out_dtype, "dist": w.dist,
        "path": tg.PATHS.get(path, str(path)), "kernel": KERNEL_OF_PATH.get(path, str(path)),
        "launches": launches,
        "us_stream": us_stream, "us_graph": us_graph,
        "tflops_graph": flops / (us_graph * 1e-6) / 1e12,
        "tflops_stream": flops / (us_stream * 1e-6) / 1e12,
        "gbs_graph": set_bytes / (us_graph * 1e-6) / 1e9,
        "gbs_stream": set_bytes / (us_stream * 1e-6) / 1e9,
        "algorithmic_bytes": set_bytes, "flop_per_byte": flops / set_bytes,
        "bound": bound,
        "peak": alu if bound == "alu" else (hbm if bound == "hbm" else peak),
        "peak_unit": "GB/s" if bound == "hbm" else "TFLOP/s",
        "peak_source": ("fp32 FMA lanes x 2 x SMs x max SM clock" if bound == "alu" else
                        "measured copy bandwidth" if bound == "hbm" else
                        "measured bf16 burst (fp16 has the same nominal rate)"),
        "frac_graph": frac_graph, "frac_stream": frac_stream,
        "l2": f"{n_sets} rotating A/B/C sets, {n_sets * set_bytes / 2**20:.0f} MB per pass",
        "traffic": traffic_of(NCU_TRAFFIC, w.name),
        "clocks": sampler.summary(t0, t1),
    }
    if cpu_s > 0:
        import oracle
        a_np, b_np = host_array(a_cpu), host_array(b_cpu)
        if flops <= 4.4e9:
            t = time.perf_counter()
            oracle.gemm(a_np, b_np)
            dt = time.perf_counter() - t
            rec["cpu_oracle"] = {"seconds": dt, "tflops": flops / dt / 1e12,
                                 "cores": oracle.num_threads(), "sample": "all of C"}
        else:
            v, rows, secs, nt = oracle_rows_sample(w, a_cpu, b_cpu, cpu_s)
            rec["cpu_oracle"] = {"seconds_full_estimate": flops / (v * 1e12), "tflops": v,
                                 "cores": nt, "sample": f"{rows} of {M} rows of C, {secs:.1f} s"}
    del sets
    torch.cuda.empty_cache()
    return rec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="square_8192")
    ap.add_argument("--e2e-steps", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--epilogue", default="none", choices=sorted(EPILOGUES),
                    help="time tg_gemm_ex with this fused epilogue instead of tg_gemm")
    ap.add_argument("--attn-kernel", default="auto", choices=["auto", "general", "tmem_p"],
                    help="attention workloads: the library's choice of forward kernel, or one "
                         "forced (tmem_p serves d <= 128, dv <= 128)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload records (fp32 example, edge set, tiling "
                         "example, skinny, wide)")
    ap.add_argument("--config-launches", type=int, default=200,
                    help="launches per specified workload, stream-launched and in a graph")
    ap.add_argument("--group-m", type=int, default=0,
                    help="grouped tile-order height of the GEMM kernels (tg_gemm_force_tiling); "
                         "0 = each kernel's default")
    ap.add_argument("--graph", action="store_true",
                    help="replay the timed launches from one CUDA graph (for us-scale shapes)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    from tiled_gemm_tg_gb300 import inputs
    if args.workload in inputs.ATTN_WORKLOADS:
        wa = inputs.ATTN_WORKLOADS[args.workload]
        if args.impl == "reference":
            return run_reference_attention(args, wa)
        return main_attention(args, wa)
    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)

    import torch

    import tiled_gemm_tg_gb300 as tg

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    tg.lib()  # fail loudly if the library is missing
    if args.group_m and tg.tg_gemm_force_tiling(0, args.group_m) != tg.TG_OK:
        ap.error("--group-m must be 0..64")

    # operands: drawn on the host from the workload's seeds, copied to HBM
    a_cpu, b_cpu = inputs.operands(w)
    out_dt = torch.float16 if w.out_dtype == "f16" else torch.float32
    in_code = {"f16": tg.F16, "e4m3": tg.E4M3}.get(w.in_dtype, tg.F32)
    out_code = tg.F16 if w.out_dtype == "f16" else tg.F32
    # Rotate enough operand sets that one pass over them is at least three
    # times the 129 MB L2 (two sets for the large shapes).
    epi = EPILOGUES[args.epilogue]
    use_d = epi is not None and epi["beta"] != 0.0
    use_bias = epi is not None and epi["bias"]
    out_es = 2 if w.out_dtype == "f16" else 4
    NB = w.batch
    if NB > 1 and epi is not None:
        ap.error("--epilogue applies to single products, not to a strided batch")
    set_bytes = NB * ((w.M * w.K + w.K * w.N) * a_cpu.element_size() + w.M * w.N * out_es * (
        2 if use_d else 1))
    # D and bias for a fused epilogue, drawn on the host like the operands
    d_cpu = inputs.draw((w.M, w.N), "normal", w.seed_base + 7, w.out_dtype) if use_d else None
    bias_cpu = inputs.draw((1, w.N), "normal", w.seed_base + 8, "f32")[0] if use_bias else None
    n_sets = max(2, min(64, -(-3 * 129 * 2**20 // set_bytes)))
    sets = []
    for i in range(n_sets):
        a = a_cpu.to(dev)
        b = b_cpu.to(dev)
        if i:  # distinct buffers with the same values (rotated for L2)
            a = a.clone()
            b = b.clone()
        c = torch.empty(((NB,) if NB > 1 else ()) + (w.M, w.N), dtype=out_dt, device=dev)
        d = d_cpu.to(dev) if use_d else None
        bias = bias_cpu.to(dev) if use_bias else None
        sets.append((a, b, c, d, bias))
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    M, N, K = w.M, w.N, w.K

    def call(a, b, c, d, bias, handle):
        if NB > 1:
            st = tg.tg_gemm_batched(NB, M, N, K, a.data_ptr(), K, M * K, b.data_ptr(), N, K * N,
                                    c.data_ptr(), N, M * N, in_code, out_code, handle)
        elif epi is None:
            st = tg.tg_gemm(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, in_code,
                            out_code, handle)
        else:
            st = tg.tg_gemm_ex(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N,
                               in_code, out_code, epi["alpha"], epi["beta"],
                               d.data_ptr() if use_d else 0, N,
                               bias.data_ptr() if use_bias else 0, epi["act"], handle)
        if st != tg.TG_OK:
            raise tg.TgError(st)

    def step(i, handle=None):
        call(*sets[i % n_sets], sh if handle is None else handle)

    path = tg.tg_gemm_batched_path(NB, M, N, K, sets[0][0].data_ptr(), K, M * K,
                                   sets[0][1].data_ptr(), N, K * N, sets[0][2].data_ptr(), N,
                                   M * N, in_code, out_code)

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)

    for i in range(args.warmup):
        step(i)
    tg.check(stream)
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            h = torch.cuda.current_stream().cuda_stream
            for i in range(args.steps):
                step(i, h)
        graph.replay()  # warm replay
        tg.check(stream)

    # --- timed region: K steps, an event pair around every launch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    host_t0 = time.time()
    if graph is not None:
        # all K launches replayed from one CUDA graph: no host gaps between them
        t_start.record(stream)
        graph.replay()
        t_end.record(stream)
    else:
        t_start.record(stream)
        for i in range(args.steps):
            evs[i][0].record(stream)
            step(i)
            evs[i][1].record(stream)
        t_end.record(stream)
    torch.cuda.synchronize()
    host_t1 = time.time()
    if ws > 1:
        torch.distributed.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    if graph is not None:
        kern_ms = elapsed_ms / args.steps
        per_launch = []  # one graph replay: only the mean per launch is known
    else:
        per_launch = sorted(s.elapsed_time(e) for s, e in evs)
        kern_ms = sum(per_launch) / args.steps
    if tg.tg_gemm_check(sh) != tg.TG_OK:
        raise RuntimeError("a kernel abandoned a bounded wait during the timed region")

    elapsed_ms = max_over_ranks(elapsed_ms, ws, dev)
    flops = 2.0 * NB * M * N * K
    value = job_throughput(flops, ws, args.steps, elapsed_ms)

    # --- end to end through the C ABI from pinned host buffers.  Every step
    # copies its A and B in, runs tg_gemm and copies C out; steps are
    # pipelined over three streams (H2D, GEMM, D2H) and two device buffer
    # sets, so step i's transfers overlap the GEMMs of steps i-1 and i+1.
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 20))
    a_h = a_cpu.pin_memory()
    b_h = b_cpu.pin_memory()
    c_h = [torch.empty(((NB,) if NB > 1 else ()) + (M, N), dtype=out_dt).pin_memory()
           for _ in range(2)]
    d_h = d_cpu.pin_memory() if use_d else None
    bias_h = bias_cpu.pin_memory() if use_bias else None
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_mm = stream
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "mm", "out")}
    started = [False, False]

    def e2e_step(i):
        slot = i % 2
        a_d, b_d, c_d, d_d, bias_d = sets[slot]
        if started[slot]:
            s_in.wait_event(ev["mm"][slot])  # the slot's previous GEMM has read A, B
        with torch.cuda.stream(s_in):
            a_d.copy_(a_h, non_blocking=True)
            b_d.copy_(b_h, non_blocking=True)
            if use_d:
                d_d.copy_(d_h, non_blocking=True)
            if use_bias:
                bias_d.copy_(bias_h, non_blocking=True)
        ev["in"][slot].record(s_in)
        s_mm.wait_event(ev["in"][slot])
        if started[slot]:
            s_mm.wait_event(ev["out"][slot])  # the slot's previous C has been read out
        call(a_d, b_d, c_d, d_d, bias_d, s_mm.cuda_stream)
        ev["mm"][slot].record(s_mm)
        s_out.wait_event(ev["mm"][slot])
        with torch.cuda.stream(s_out):
            c_h[slot].copy_(c_d, non_blocking=True)
        ev["out"][slot].record(s_out)
        started[slot] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)  # after the last D2H, which follows every earlier step's work
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if tg.tg_gemm_check(s_mm.cuda_stream) != tg.TG_OK:
        raise RuntimeError("a kernel abandoned a bounded wait during the e2e region")
    e2e_ms = max_over_ranks(e2e_ms, ws, dev)
    e2e_value = job_throughput(flops, ws, e2e_steps, e2e_ms)
    ein = a_cpu.element_size()
    h2d = NB * (M * K + K * N) * ein + (M * N * out_es if use_d else 0) + (
        N * 4 if use_bias else 0)
    d2h = NB * M * N * c_h[0].element_size()

    sampler.stop()
    clocks = sampler.summary(host_t0, host_t1)

    peaks, peak_src = load_peaks()
    # fp8 (E4M3) tensor-core work has twice the dense rate of bf16/fp16
    # (nominal 4.5 against 2.25 PFLOP/s on GB300): scale the measured bf16 peak
    ratio = 2.0 if w.in_dtype == "e4m3" else 1.0
    peak = ratio * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (kern_ms * 1e-3) / 1e12
    alg_bytes = w.algorithmic_bytes() + (M * N * out_es if use_d else 0) + (
        N * 4 if use_bias else 0)
    traffic = traffic_of(NCU_TRAFFIC, w.name) if epi is None else None
    # The bound is the roofline's: a workload whose FLOP per algorithmic byte
    # lies below the ridge (measured tensor peak / measured HBM bandwidth) is
    # bound by HBM and is reported in GB/s against the copy bandwidth.
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved_gbs = alg_bytes / (kern_ms * 1e-3) / 1e9
    ridge = peak * 1e12 / (hbm * 1e9)
    hbm_bound = flops / alg_bytes < ridge
    roofline = {
        "bound": "hbm" if hbm_bound else "tensor",
        "achieved": achieved_gbs if hbm_bound else achieved,
        "peak": hbm if hbm_bound else peak,
        "unit": "GB/s" if hbm_bound else "TFLOP/s",
        "frac": achieved_gbs / hbm if hbm_bound else achieved / peak,
        "traffic": traffic,
        "kernel": {3: "gemm_tc_main_kernel", 4: "gemm_tc_boundary_kernel",
                   2: "gemm_simt_f32_kernel", 5: "gemm_skinny_kernel",
                   6: "gemm_tc_pair_kernel"}.get(path, str(path)),
        "kernel_ms": kern_ms,
        "kernel_ms_median": per_launch[len(per_launch) // 2] if per_launch else None,
        "kernel_ms_best": per_launch[0] if per_launch else None,
        "peak_source": (f"{peak_src} STREAM-style copy bandwidth" if hbm_bound else
                        f"{peak_src} bf16 burst (torch.matmul 8192^3) x {ratio} "
                        f"{'fp8' if ratio == 2.0 else 'fp16'}/bf16 nominal ratio"),
        "flop_per_byte": flops / alg_bytes, "ridge_flop_per_byte": ridge,
        "achieved_tflops": achieved,
        "spec_tflops": ratio * SPEC_FP16_DENSE_TFLOPS,
        "frac_of_spec": achieved / (ratio * SPEC_FP16_DENSE_TFLOPS),
        "algorithmic_bytes": alg_bytes,
        "achieved_gbs": achieved_gbs,
    }

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, rows, secs, nt = oracle_rows_sample(w, a_cpu[0] if NB > 1 else a_cpu,
                                               b_cpu[0] if NB > 1 else b_cpu, args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
               "sample": f"{rows} of {M} rows of C (full N={N}, K={K}), {secs:.1f} s"}
        # small products: the whole product on one core as well
        if 2.0 * M * N * K <= 4.4e9:
            import oracle
            a1 = host_array(a_cpu[0] if NB > 1 else a_cpu)
            b1 = host_array(b_cpu[0] if NB > 1 else b_cpu)
            t1 = time.perf_counter()
            oracle.gemm(a1, b1, nthreads=1)
            s1 = time.perf_counter() - t1
            cpu["single_thread"] = {"value": 2.0 * M * N * K / s1 / 1e12, "unit": "TFLOP/s",
                                    "sample": f"all of C, one thread, {s1:.2f} s"}

    configs = None
    if (rank == 0 and ws == 1 and not args.no_configs and w.name == "square_8192"
            and epi is None):
        num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
        sampler.start()
        time.sleep(0.3)
        configs = [measure_config(label, inputs.WORKLOADS[name], dev, args.config_launches,
                                  sampler, peaks, 0.0 if args.no_cpu_baseline else 2.0, num_sms)
                   for label, name in SPEC_WORKLOADS]
        sampler.stop()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.in_dtype,
            "data": "synthetic",
            "config": {"workload": w.name, "batch": NB, "M": M, "N": N, "K": K,
                       "in_dtype": w.in_dtype,
                       "accum": "f32", "out_dtype": w.out_dtype, "dist": w.dist,
                       "path": tg.PATHS.get(path, str(path)),
                       "epilogue": args.epilogue if epi is None else
                       f"{args.epilogue}: C = act(alpha*AB + beta*D + bias), {epi}",
                       "l2": f"{n_sets} rotating A/B/C sets, {n_sets * set_bytes / 2**20:.0f} MB "
                             "per pass (> L2)",
                       "timing": "CUDA graph replay" if graph is not None else "stream launches",
                       "group_m": args.group_m or "default",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "pipeline": "H2D / tg_gemm{} / D2H on three streams, two device buffer "
                                "sets".format("" if epi is None else "_ex")},
            "gpu_launches": args.steps,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
