#!/usr/bin/env python3
"""Benchmark of the paged-KV MLA hot path on GB300.

Default workload (one step = one call of mla_decompress_k_paged): the DeepSeek-V3-shaped
bf16 decompress (16 requests, lengths ~U[512, 4096], cache_offsets ~U[0, len/4],
page_size 128, kv_lora_rank 512 + rope 64, W_k [16384, 512]), seeded synthetic data.
The headline value is decompress TFLOP/s (2 * rows * 512 * 16384 per step); the same line
carries rows/s, the roofline of the kernel, the FP8 decompress, the long-context
decompress and kv_matmul (TFLOP/s and GB/s), an end-to-end number with host buffers, and
the CPU oracle timed on this host.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 is launched by torchrun: each rank runs its own replica of the workload (weak
scaling, no collective on the data path); timing is the max over ranks.
--impl reference times the CPU oracle (the only other implementation of this method) on a
bounded sample per step, on every host core (one process per core, each the unchanged
single-thread oracle on its own rows).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA K-decompress TFLOP/s & rows/s (% of GB300 tensor peak); kv_matmul GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "decompress_bf16_kernel": ["decompress_bf16.cu"],
    "decompress_fp8_gemm_kernel": ["decompress_fp8.cu"],
    "decompress_fp8_wide_kernel": ["decompress_fp8_wide.cu"],
    "fp8_gather_quantize_kernel": ["decompress_fp8.cu"],
    "kv_matmul_kernel": ["kv_matmul.cu"],
    "cache_write_kernel": ["cache_write.cu"],
    "cache_write_q_kernel": ["cache_write.cu"],   # the quantising instantiation
    "fp8_gather_qcache_kernel": ["decompress_fp8.cu"],
    "kv_matmul_fp8_kernel": ["kv_matmul_fp8.cu"],
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources a kernel is built from (its .cu file plus the shared headers)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_mla_gb300", "csrc")
    names = KERNEL_SOURCES[kernel] + ["pkm_device.cuh", "pkm_internal.h"]
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json), if it
    was taken on the kernel's current sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    entry = t.get(kernel)
    if not entry or entry.get("source_hash") != kernel_source_hash(kernel):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock / throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        inside = [r for r in rows if self.window and self.window[0] <= r[0] <= self.window[1]]
        note = None
        if not inside:
            inside = rows
            note = "timed region shorter than the sampling interval: samples span the run"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3])
                          if v.lower().startswith("active")})
        out = {"sm_mhz": statistics.median(r[1] for r in inside),
               "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
               "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# ----------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------

def max_over_ranks(local_seconds: float, dist=None, device=None) -> float:
    """The timed region's length as the max over ranks (the slowest replica sets the time)."""
    if dist is None:
        return local_seconds
    import torch
    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units processed by all ranks (each runs its own replica) per second of the slowest."""
    return units_per_rank * world / seconds


def bf16_algorithmic_bytes(d) -> int:
    """Per covered row: the latent row read (2C bytes) and copied (2C), one bf16 output row
    per up-projection (2 N, + 2 N_v with V); the weights once."""
    rows = min(int(d.buffer_row_offsets[-1]), d.buffer_length)
    n = d.n_out + d.n_out_v
    return rows * (4 * d.latent_cols + 2 * n) + n * d.kv_lora_rank * 2


def fp8_algorithmic_bytes(d) -> int:
    """As bf16_algorithmic_bytes, plus the quantised row the entry point writes to its
    workspace (R e4m3 codes and R/128 fp32 scales); e4m3 weights."""
    rows = min(int(d.buffer_row_offsets[-1]), d.buffer_length)
    n = d.n_out + d.n_out_v
    R = d.kv_lora_rank
    return rows * (4 * d.latent_cols + 2 * n + R + 4 * (R // 128)) + n * R


def qcache_algorithmic_bytes(d) -> int:
    """FP8 decompress from a quantised cache, per covered row: the slot payload read
    (R + 2P + 4R/128 bytes), the dequantised bf16 latent row written (2C), the codes and
    scales written to the workspace (R + 4R/128), one bf16 output row (2N); the e4m3
    weight once."""
    rows = min(int(d.buffer_row_offsets[-1]), d.buffer_length)
    R, P = d.kv_lora_rank, d.rope_dim
    payload = R + 2 * P + 4 * (R // 128)
    return rows * (payload + 2 * d.latent_cols + R + 4 * (R // 128) + 2 * d.n_out) + d.n_out * R


def _device_problem(d, fp8=False):
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from gpu_util import DeviceDecompress
    return DeviceDecompress(d, fp8=fp8)


def _time_steps(step, steps, warmup, flush, stream, event_pairs=None):
    """Runs warmup untimed steps, then `steps` timed ones with an L2 flush before each;
    returns (summed device time of the timed steps, median step time), in seconds."""
    import torch
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    per = [s.elapsed_time(e) / 1e3 for s, e in zip(starts, ends)]
    return sum(per), statistics.median(per)


def _time_row(step, steps, warmup, flush, stream):
    """Median device time (s) of one step of a secondary row."""
    return _time_steps(step, steps, warmup, flush, stream)[1]


def measure_fp8_peak(dev, seconds=2.0):
    """Dense e4m3 GEMM throughput of the vendor library on this GPU (torch._scaled_mm,
    8192^3, bf16 output, per-tensor scales; fast accumulation on and off, the better kept):
    best single call after warm-up (burst) and back-to-back calls for `seconds`
    (sustained).  The FP8 rows' tensor fractions are taken against it."""
    import torch
    n = 8192
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    one = torch.ones((), device=dev, dtype=torch.float32)
    flop = 2.0 * n ** 3
    out = {}
    for fast in (False, True):
        def mm():
            return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16,
                                    use_fast_accum=fast)
        for _ in range(3):
            mm()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record()
            mm()
            s1.record()
            s1.synchronize()
            best = min(best, s0.elapsed_time(s1) / 1e3)
        reps = max(10, int(seconds / best))
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(reps):
            mm()
        s1.record()
        s1.synchronize()
        out["fast_accum" if fast else "fp32_accum"] = {
            "burst_tflops": flop / best / 1e12,
            "sustained_tflops": flop * reps / (s0.elapsed_time(s1) / 1e3) / 1e12}
    best_key = max(out, key=lambda k: out[k]["burst_tflops"])
    del a, b
    torch.cuda.empty_cache()
    return {"burst_tflops": out[best_key]["burst_tflops"],
            "sustained_tflops": out[best_key]["sustained_tflops"], "mode": best_key,
            "how": "torch._scaled_mm e4m3 8192^3 (bf16 out, per-tensor scales), best of 10 "
                   "after warm-up (burst) and back to back for ~2 s (sustained)",
            "modes": out}


def roofline_row(kernels, t, flop, nbytes, peaks, tensor_peak, tensor_peak_kind, traffic=None):
    """The roofline of one secondary row, recomputable from its own fields: the bound is the
    slower of the FLOPs at the tensor peak and the algorithmic bytes at the HBM peak;
    `achieved` and `frac` are in that bound's unit (per step, device time t)."""
    t_tensor = flop / (tensor_peak * 1e12) if flop else 0.0
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    achieved = flop / t / 1e12 if bound == "tensor" else nbytes / t / 1e9
    peak = tensor_peak if bound == "tensor" else peaks["hbm_gbs"]
    return {"kernels": kernels, "ms": t * 1e3, "flop": flop, "algorithmic_bytes": nbytes,
            "bound": bound, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s" if bound == "tensor" else "GB/s", "frac": achieved / peak,
            "tensor_tflops": flop / t / 1e12 if flop else None,
            "tensor_peak": tensor_peak if flop else None,
            "tensor_peak_kind": tensor_peak_kind if flop else None,
            "tensor_frac": (flop / t / 1e12 / tensor_peak) if flop else None,
            "hbm_gbs": nbytes / t / 1e9, "hbm_peak": peaks["hbm_gbs"],
            "hbm_frac": nbytes / t / 1e9 / peaks["hbm_gbs"], "traffic": traffic}


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import workloads
    import paged_kv_mla_gb300 as pkm

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    peaks, peak_kind = load_peaks()
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush():
        # write a buffer larger than L2, then read another one: the timed step starts with
        # no line of its inputs in L2 and no dirty line of the flush left to write back
        flush_buf.fill_(1)
        flush_read.max()

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", rank=rank, world_size=world, device_id=dev)

    # ---------------- headline: DeepSeek-V3-shaped bf16 decompress ----------------
    d = workloads.WORKLOADS["deepseek_v3_bf16_decompress"]()
    g = _device_problem(d)
    rows = min(int(d.buffer_row_offsets[-1]), d.buffer_length)
    flop = d.flops
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for _ in range(args.warmup):
        g.run()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t_dev, t_med = _time_steps(g.run, args.steps, 0, flush, stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall1 = time.time()
    if sampler:
        sampler.mark(wall0, wall1)
    t_max = max_over_ranks(t_dev, dist, dev)
    assert int(g.status.item()) == 0, "device status reported an error"
    per_step = t_max / args.steps
    value = whole_job_rate(flop * args.steps, world, t_max) / 1e12
    achieved = flop / per_step / 1e12

    if sampler:
        time.sleep(0.25)
        sampler.stop()
    if rank != 0:
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return

    # ---------------- secondary rows (rank 0 only, fewer steps) ----------------
    # the FP8 denominator: the vendor library's dense e4m3 GEMM on this GPU, measured here
    fp8_peak = measure_fp8_peak(dev)
    fp8_tf = fp8_peak["burst_tflops"]
    fp8_kind = "measured in this run (torch._scaled_mm e4m3 8192^3, burst)"
    bf16_tf = peaks["bf16_tflops"]
    bf16_kind = peak_kind + " bf16 burst (MEASURED_PEAKS.json)"
    extra = {"fp8_peak": fp8_peak}
    sec_steps = max(5, min(args.steps, 50))
    d8 = workloads.WORKLOADS["deepseek_v3_fp8_decompress"]()
    g8 = _device_problem(d8, fp8=True)
    t8 = _time_row(g8.run, sec_steps, 3, flush, stream)
    assert int(g8.status.item()) == 0
    b8 = fp8_algorithmic_bytes(d8)
    extra["fp8_decompress"] = {
        "workload": d8.name, "rows": d8.buffer_length, "ms": t8 * 1e3,
        "tflops": d8.flops / t8 / 1e12, "rows_per_s": d8.buffer_length / t8,
        "hbm_gbs": b8 / t8 / 1e9, "hbm_frac_of_measured": b8 / t8 / 1e9 / peaks["hbm_gbs"],
        "launches_per_step": 2,
        "roofline": roofline_row(["fp8_gather_quantize_kernel", "decompress_fp8_wide_kernel"],
                                 t8, d8.flops, b8, peaks, fp8_tf, fp8_kind,
                                 profiled_traffic("decompress_fp8_wide_kernel"))}
    del g8
    dl = workloads.WORKLOADS["long_context_decompress"]()
    gl = _device_problem(dl)
    tl = _time_row(gl.run, max(3, sec_steps // 4), 2, flush, stream)
    assert int(gl.status.item()) == 0
    extra["long_context_decompress"] = {
        "workload": dl.name, "rows": dl.buffer_length, "ms": tl * 1e3,
        "tflops": dl.flops / tl / 1e12, "rows_per_s": dl.buffer_length / tl,
        "frac_of_measured_bf16": dl.flops / tl / 1e12 / bf16_tf,
        "roofline": roofline_row(["decompress_bf16_kernel"], tl, dl.flops,
                                 bf16_algorithmic_bytes(dl), peaks, bf16_tf, bf16_kind)}
    del gl
    # K and V from one gather (w_uv up-projection rides along; same rows and weights shape)
    for key, wl, fp8 in [("kv_decompress_bf16", "deepseek_v3_bf16_decompress_kv", False),
                         ("kv_decompress_fp8", "deepseek_v3_fp8_decompress_kv", True)]:
        dv = workloads.WORKLOADS[wl]()
        gv = _device_problem(dv, fp8=fp8)
        tv = _time_row(gv.run, sec_steps, 3, flush, stream)
        assert int(gv.status.item()) == 0
        lv = dv.buffer_length
        bv = fp8_algorithmic_bytes(dv) if fp8 else bf16_algorithmic_bytes(dv)
        kernels = (["fp8_gather_quantize_kernel", "decompress_fp8_wide_kernel"] if fp8
                   else ["decompress_bf16_kernel"])
        extra[key] = {
            "workload": dv.name, "rows": lv, "n_out_k": dv.n_out, "n_out_v": dv.n_out_v,
            "ms": tv * 1e3, "tflops": dv.flops / tv / 1e12, "rows_per_s": lv / tv,
            "hbm_gbs": bv / tv / 1e9, "launches_per_step": 2 if fp8 else 1,
            "roofline": roofline_row(kernels, tv, dv.flops, bv, peaks,
                                     fp8_tf if fp8 else bf16_tf, fp8_kind if fp8 else bf16_kind)}
        del gv, dv
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from gpu_util import DeviceKvMatmul
    km = workloads.WORKLOADS["kv_matmul_write_path"]()
    gk = DeviceKvMatmul(km)
    tk = _time_row(gk.run, sec_steps, 3, flush, stream)
    assert int(gk.status.item()) == 0
    extra["kv_matmul"] = {
        "workload": km.name, "rows": km.total_rows, "ms": tk * 1e3,
        "tflops": km.flops / tk / 1e12, "gbs": km.bytes_moved / tk / 1e9,
        "roofline": roofline_row(["kv_matmul_kernel"], tk, km.flops, km.bytes_moved, peaks,
                                 bf16_tf, bf16_kind, profiled_traffic("kv_matmul_kernel"))}
    del gk
    kf = workloads.WORKLOADS["kv_matmul_fp8_write_path"]()
    gf = DeviceKvMatmul(kf)
    tf = _time_row(gf.run, sec_steps, 3, flush, stream)
    assert int(gf.status.item()) == 0
    extra["kv_matmul_fp8"] = {
        "workload": kf.name, "rows": kf.total_rows, "ms": tf * 1e3,
        "tflops": kf.flops / tf / 1e12, "gbs": kf.bytes_moved / tf / 1e9,
        "launches_per_step": 2,
        "roofline": roofline_row(["fp8_quantize_rows_kernel", "kv_matmul_fp8_kernel"], tf,
                                 kf.flops, kf.bytes_moved, peaks, fp8_tf, fp8_kind,
                                 profiled_traffic("kv_matmul_fp8_kernel"))}
    del gf, kf
    from gpu_util import DeviceCacheWrite
    for key, wl in [("cache_write", "cache_write_path"), ("cache_write_q", "cache_write_q_path")]:
        cw = workloads.WORKLOADS[wl]()
        gc = DeviceCacheWrite(cw)
        tc = _time_row(gc.run, sec_steps, 3, flush, stream)
        assert int(gc.status.item()) == 0
        kname = "cache_write_kernel" if key == "cache_write" else "cache_write_q_kernel"
        extra[key] = {
            "workload": cw.name, "rows": cw.total_rows, "ms": tc * 1e3,
            "rows_per_s": cw.total_rows / tc, "gbs": cw.bytes_moved / tc / 1e9,
            "hbm_frac_of_measured": cw.bytes_moved / tc / 1e9 / peaks["hbm_gbs"],
            "launches_per_step": 1,
            "roofline": roofline_row([kname], tc, 0, cw.bytes_moved, peaks, bf16_tf, bf16_kind,
                                     profiled_traffic(kname))}
        del gc, cw
    # FP8 decompress from a quantised cache (codes and scales gathered as they are)
    dq = workloads.WORKLOADS["deepseek_v3_fp8_qcache_decompress"]()
    gq = _device_problem(dq, fp8=True)
    tq = _time_row(gq.run, sec_steps, 3, flush, stream)
    assert int(gq.status.item()) == 0
    bq = qcache_algorithmic_bytes(dq)
    extra["fp8_qcache_decompress"] = {
        "workload": dq.name, "rows": dq.buffer_length, "ms": tq * 1e3,
        "tflops": dq.flops / tq / 1e12, "rows_per_s": dq.buffer_length / tq,
        "hbm_gbs": bq / tq / 1e9, "hbm_frac_of_measured": bq / tq / 1e9 / peaks["hbm_gbs"],
        "launches_per_step": 2,
        "roofline": roofline_row(["fp8_gather_qcache_kernel", "decompress_fp8_wide_kernel"], tq,
                                 dq.flops, bq, peaks, fp8_tf, fp8_kind)}
    del gq, dq

    # ---------------- end to end: host buffers through the C ABI ----------------
    e2e = run_e2e(d, max(3, min(args.steps, 10)))

    # ---------------- CPU oracle on a bounded sample ----------------
    cpu = cpu_baseline_sample(d, args.cpu_rows, args.cpu_rows_per_core)

    algo_bytes = bf16_algorithmic_bytes(d)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "ms_per_step_median": t_med * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded)",
        "config": {"workload": d.name, "batch": d.batch, "buffer_length": d.buffer_length,
                   "kv_lora_rank": d.kv_lora_rank, "qk_rope_head_dim": d.rope_dim,
                   "n_out": d.n_out, "page_size": d.page_size, "num_pages": d.num_pages,
                   "l2": "flushed before every timed step (256 MiB write, then 256 MiB read; untimed)",
                   "parallelism": f"replica x{world}" if world > 1 else "single GPU"},
        "rows_per_s": whole_job_rate(rows * args.steps, world, t_max),
        "pct_tensor_peak": 100.0 * achieved / peaks["bf16_tflops"],
        "roofline": {"bound": "tensor", "kernel": "decompress_bf16_kernel",
                     "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "peak_kind": peak_kind + " burst",
                     "traffic": profiled_traffic("decompress_bf16_kernel"),
                     "algorithmic_bytes": algo_bytes,
                     "hbm_gbs_algorithmic": algo_bytes / per_step / 1e9},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": sampler.summary() if sampler else None,
        "gpu_launches": args.steps,
        "extra": extra,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_e2e(d, steps):
    """TFLOP/s through the public call with the step's inputs in pinned host memory: H2D of
    cache, page table, offsets and W_k, the decompress, D2H of k_latent_buffer and k_buffer,
    all inside CUDA events on the stream."""
    import numpy as np
    import torch
    from gpu_util import DeviceDecompress

    g = DeviceDecompress(d)
    host_in = [torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if a.dtype == np.uint16 else np.int32)).pin_memory()
               for a in (d.cache, d.page_table, d.buffer_row_offsets, d.cache_offsets, d.w_k)]
    dev_in = [g.cache, g.pt, g.bro, g.co, g.w]
    host_out = [torch.empty(g.k_latent.shape, dtype=torch.int16).pin_memory(),
                torch.empty(g.k_buffer.shape, dtype=torch.int16).pin_memory()]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    stream = torch.cuda.current_stream()

    def step():
        for h, dv in zip(host_in, dev_in):
            dv.copy_(h, non_blocking=True)
        g.run()
        host_out[0].copy_(g.k_latent, non_blocking=True)
        host_out[1].copy_(g.k_buffer, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    t = s.elapsed_time(e) / 1e3 / steps
    return {"value": d.flops / t / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": t * 1e3}


def _sub_problem(d, start, rows):
    """Rows [start, start + rows) of a decompress workload as a problem of its own: the same
    cache, page table and requests, with buffer_row_offsets shifted and clipped to the window
    and each request's cache_offset advanced past the rows the window skips."""
    import numpy as np
    bro = d.buffer_row_offsets.astype(np.int64)
    sub_bro = (bro.clip(start, start + rows) - start).astype(np.uint32)
    sub_co = d.cache_offsets.astype(np.int64).copy()
    for b in range(d.batch):
        sub_co[b] += max(0, start - int(bro[b]))
    return sub_bro, sub_co.astype(np.uint32)


# The oracle worker of the all-cores leg: each process attaches the workload's cache and W_k
# (shared memory, no copies) and runs the unchanged single-thread oracle on its own window.
_W = {}


def _oracle_worker_init(shm_names, shapes, meta):
    import numpy as np
    from multiprocessing import shared_memory
    import oracle
    oracle.lib()
    blocks = [shared_memory.SharedMemory(name=n) for n in shm_names]
    _W["blocks"] = blocks  # keep the mappings alive
    _W["cache"] = np.ndarray(shapes[0], dtype=np.uint16, buffer=blocks[0].buf)
    _W["w_k"] = np.ndarray(shapes[1], dtype=np.uint16, buffer=blocks[1].buf)
    _W["meta"] = meta


def _oracle_worker_run(window):
    """Runs the oracle on rows [start, start + rows); returns (rows written, seconds)."""
    import oracle
    start, rows, sub_bro, sub_co = window
    m = _W["meta"]
    view = oracle.PagedCacheView(_W["cache"], m["ls"], m["ps"], m["ss"], m["num_pages"],
                                 m["page_size"], m["page_table"], m["page_table"].shape[1])
    t0 = time.perf_counter()
    st, lat, kb, written = oracle.decompress_k(view, m["layer_idx"], sub_bro, sub_co, m["batch"],
                                               rows, m["R"], m["P"], _W["w_k"])
    return int(written.sum()), time.perf_counter() - t0


class OraclePool:
    """The CPU oracle on every host core: one spawned process per core, each running the
    unchanged single-thread oracle on a disjoint window of consecutive rows.  Rows are
    independent, so the windows together compute the same rows one oracle call would."""

    def __init__(self, d, workers=None):
        import multiprocessing as mp
        import numpy as np
        from multiprocessing import shared_memory
        self.d = d
        try:
            cores = len(os.sched_getaffinity(0))
        except AttributeError:
            cores = os.cpu_count() or 1
        self.workers = workers or cores
        self.blocks = []
        arrays = [np.ascontiguousarray(d.cache), np.ascontiguousarray(d.w_k)]
        for arr in arrays:
            blk = shared_memory.SharedMemory(create=True, size=max(arr.nbytes, 1))
            np.ndarray(arr.shape, dtype=arr.dtype, buffer=blk.buf)[...] = arr
            self.blocks.append(blk)
        ls, ps, ss = d.strides
        meta = {"ls": ls, "ps": ps, "ss": ss, "num_pages": d.num_pages, "page_size": d.page_size,
                "page_table": d.page_table, "layer_idx": d.layer_idx, "batch": d.batch,
                "R": d.kv_lora_rank, "P": d.rope_dim}
        ctx = mp.get_context("spawn")  # no fork of a process that holds a CUDA context
        self.pool = ctx.Pool(self.workers, initializer=_oracle_worker_init,
                             initargs=([b.name for b in self.blocks],
                                       [arrays[0].shape, arrays[1].shape], meta))

    def run(self, start, rows_per_worker):
        """One parallel pass: worker i takes rows [start + i * rows_per_worker, ...).
        Returns (rows written, wall seconds, summed worker seconds)."""
        windows = []
        for i in range(self.workers):
            s0 = start + i * rows_per_worker
            sub_bro, sub_co = _sub_problem(self.d, s0, rows_per_worker)
            windows.append((s0, rows_per_worker, sub_bro, sub_co))
        t0 = time.perf_counter()
        res = self.pool.map(_oracle_worker_run, windows, chunksize=1)
        wall = time.perf_counter() - t0
        return sum(r for r, _ in res), wall, sum(t for _, t in res)

    def close(self):
        self.pool.close()
        self.pool.join()
        for b in self.blocks:
            b.close()
            b.unlink()


def cpu_baseline_sample(d, sample_rows, rows_per_core):
    """The oracle, as it stands, on this host: one thread on the first `sample_rows` rows,
    and every core at once on `rows_per_core` consecutive rows each (gather + fp64 triple
    loop).  Reported as TFLOP/s; the all-cores figure is the line's value."""
    import oracle
    from util import cache_view

    n = min(sample_rows, d.buffer_length)
    t0 = time.perf_counter()
    st, lat, kb, written = oracle.decompress_k(cache_view(d), d.layer_idx, d.buffer_row_offsets,
                                               d.cache_offsets, d.batch, n, d.kv_lora_rank,
                                               d.rope_dim, d.w_k)
    t1 = time.perf_counter() - t0
    flop_row = 2 * d.kv_lora_rank * d.n_out
    single = {"value": flop_row * int(written.sum()) / t1 / 1e12, "unit": "TFLOP/s", "cores": 1,
              "sample": f"first {n} rows of {d.name}; {t1:.1f} s", "seconds": t1}
    pool = OraclePool(d)
    try:
        pool.run(0, 2)  # each worker imports the oracle and maps the shared cache
        rows, wall, busy = pool.run(0, rows_per_core)
    finally:
        pool.close()
    return {"value": flop_row * rows / wall / 1e12, "unit": "TFLOP/s", "cores": pool.workers,
            "kind": "oracle",
            "sample": f"{pool.workers} processes (one per host core), each the single-thread "
                      f"oracle on {rows_per_core} consecutive rows of {d.name} "
                      f"({rows} rows in all, gather + {d.n_out} fp64 dot products of "
                      f"{d.kv_lora_rank} per row); {wall:.1f} s wall, "
                      f"{busy:.1f} s of worker time",
            "seconds": wall, "single_thread": single}


# ----------------------------------------------------------------------------------------
# reference arm: the CPU oracle
# ----------------------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    import workloads
    sys.path.insert(0, os.path.join(ROOT, "tests"))

    d = workloads.WORKLOADS["deepseek_v3_bf16_decompress"]()
    per_core = args.ref_rows
    pool = OraclePool(d)
    span = per_core * pool.workers
    try:
        pool.run(0, 2)  # each worker imports the oracle and maps the shared cache

        # each step: a different window of rows, one slice per core, each a sub-problem of
        # the same workload
        def step(i):
            start = (i * span) % max(1, d.buffer_length - span)
            return pool.run(start, per_core)

        for i in range(args.warmup):
            step(i)
        done = 0
        wall = 0.0
        for i in range(args.steps):
            rows, w, _ = step(args.warmup + i)
            done += rows
            wall += w
    finally:
        pool.close()
    flop = 2 * done * d.kv_lora_rank * d.n_out
    value = flop / wall / 1e12
    sample = (f"{span} consecutive rows of {d.name} per step, {per_core} on each of "
              f"{pool.workers} processes (one per host core) running the single-thread oracle "
              f"(gather + {d.n_out} fp64 dot products of {d.kv_lora_rank} per row)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wall / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": d.name, "batch": d.batch, "buffer_length": d.buffer_length,
                       "kv_lora_rank": d.kv_lora_rank, "qk_rope_head_dim": d.rope_dim,
                       "n_out": d.n_out, "page_size": d.page_size},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": pool.workers,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=768,
                    help="rows of the workload the single-thread CPU oracle leg computes")
    ap.add_argument("--cpu-rows-per-core", type=int, default=192,
                    help="rows each host core computes in the all-cores CPU oracle leg")
    ap.add_argument("--ref-rows", type=int, default=4,
                    help="rows per host core per step of the reference (oracle) arm")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus > 1 and world == 1 and "RANK" not in os.environ:
        ap.error("--gpus > 1 must be launched with torch.distributed.run (one rank per GPU)")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
