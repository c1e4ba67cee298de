"""Benchmark of the fused Hadamard-rotated ternary GEMV on GB300.

Default workload: FFN gate/up decode projection, PQ2_0_G128 n=17408 k=5120,
M=1 bf16 activation, seed 1 (synthetic inputs with the pages' distributions).
One step = one call of ninfer_ternary_matmul (rotate + decode + GEMV) on one
activation row. Inputs are resident in HBM; L2 reuse is defeated by cycling a
pool of weight-payload copies whose total size is more than 3x the L2 cache.
Steps are captured in CUDA graphs and timed with CUDA events on the launching
stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--no-extra]
  python bench.py --workload gateup|ffn_gate_up|down|down_m8|head|head_m8|head_ptq1|head_ptq1_m8|
                             prefill|prefill_down|embed|embed_ptq1|tiny   (one workload alone)
  python bench.py --impl reference ...   (the fp64 CPU oracle on the host cores)

Without --workload, gate/up is the headline and the FFN down (PTQ1_0, M = 1
and M = 8) and the output head (both formats) are timed in the same run, each
in its own graphs over its own payload pool, under "workloads".
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "fused ternary GEMV weight GB/s & % of HBM roofline at 17408x5120; tokens/s"
FALLBACK_HBM_GBS = 6800.0


def algorithmic_bytes(w, M: int) -> dict:
    """Bytes the method must move per call: packed planes + activations + signs + fp32 output.
    The embedding moves the gathered rows' planes, the ids, the signs and the fp32 rows."""
    groups = -(-w.k // 128)
    per_group = 34 if w.fmt == "PQ2_0_G128" else 28
    if w.kind == "embed":
        cnt = synth.EMBED_COUNT
        weights = cnt * groups * per_group
        return {"weights": weights, "x": cnt * 4, "signs": w.k * 2, "y": cnt * w.k * 4,
                "total": weights + cnt * 4 + w.k * 2 + cnt * w.k * 4}
    weights = w.mats * w.n * groups * per_group
    xb = M * w.k * (4 if w.x_dtype == "f32" else 2)
    sb = w.mats * w.k * 2
    yb = M * w.n * 4
    return {"weights": weights, "x": xb, "signs": sb, "y": yb, "total": weights + xb + sb + yb}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(kernel_tag: str, workload: str, source_files):
    """Per-launch DRAM bytes from the committed ncu summary for this kernel and
    workload, or None when absent or when the kernel sources changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path, encoding="utf-8").read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt)
    if not m or not h or h.group(1) != sources_sha256(source_files):
        return None
    return float(m.group(1))


def sources_sha256(files) -> str:
    d = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(ROOT, f), "rb") as fh:
            d.update(fh.read())
    return d.hexdigest()


_COMMON = ["bit_gemv_gb300/csrc/gemv_common.cu", "bit_gemv_gb300/csrc/async.cuh",
           "bit_gemv_gb300/csrc/device.cuh", "bit_gemv_gb300/csrc/gemv.h"]
GEMV_SOURCES = ["bit_gemv_gb300/csrc/gemv_pq2_int.cu", "bit_gemv_gb300/csrc/act16.cuh",
                "bit_gemv_gb300/csrc/rot2.cuh"] + _COMMON
KERNEL_TAG = "gemv"


def dominant_kernel(w):
    """(profile tag, source files) of the kernel that dominates one step of workload w."""
    if w.kind == "embed":
        return "embed", ["bit_gemv_gb300/csrc/embed.cu"] + _COMMON
    if w.mats == 2 and w.fmt == "PQ2_0_G128" and w.M == 1:
        return KERNEL_TAG, GEMV_SOURCES + ["bit_gemv_gb300/csrc/ffn.cu"]
    if w.fmt == "PQ2_0_G128" and w.M == 1:
        return KERNEL_TAG, GEMV_SOURCES
    if w.fmt == "PQ2_0_G128" and w.M <= 8:
        return "gemv_mma", ["bit_gemv_gb300/csrc/gemv_pq2_mma.cu", "bit_gemv_gb300/csrc/act16.cuh"] + _COMMON
    if w.fmt == "PQ2_0_G128":
        return "gemm_tc", ["bit_gemv_gb300/csrc/gemm_tc.cu"] + _COMMON
    if w.M == 1:
        return "gemv_ptq1", ["bit_gemv_gb300/csrc/gemv_ptq1_int.cu", "bit_gemv_gb300/csrc/act16.cuh",
                             "bit_gemv_gb300/csrc/rot2.cuh"] + _COMMON
    if w.M <= 8:
        return "gemv_ptq1_mma", ["bit_gemv_gb300/csrc/gemv_ptq1_mma.cu", "bit_gemv_gb300/csrc/act16.cuh"] + _COMMON
    return "gemm_tc", ["bit_gemv_gb300/csrc/gemm_tc.cu", "bit_gemv_gb300/csrc/transcode.cu"] + _COMMON


def measured_tensor_peak():
    """Dense binary16 tensor peak (TFLOP/s): the measured bf16 burst figure
    (binary16 and bfloat16 run at the same nominal rate)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["bf16_tflops"]), "measured bf16_tflops (burst; f16 rate equal)"
    except Exception:
        return 1900.0, "fallback"


# ------------------------------------------------------------------ clocks ---
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_dir: str | None = None):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(out_dir or tempfile.gettempdir(), f"bench_clocks_rank{gpu_index}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- our arm ---
# Workloads timed in the same run as the default headline (gate/up), each with
# its own graph of back-to-back calls: the other 17408 x 5120 decode shape (FFN
# down, PTQ1_0, M = 1 and M = 8) and the output head in both formats.
EXTRA_WORKLOADS = ("down", "down_m8", "head", "head_ptq1")
EXTRA_STEPS = {"down": 20000, "down_m8": 20000, "head": 3000, "head_ptq1": 3000}

_CASES = {}


def _case(w):
    """Inputs of workload w; workloads drawn from the same preset shape and seed
    (the head in both formats) share one draw."""
    key = (w.n, w.k, w.M if w.kind != "embed" else 1, w.seed, w.mats, w.kind == "embed", w.x_dtype)
    if key not in _CASES:
        _CASES.clear()
        _CASES[key] = synth.make_case(w, with_ids=w.kind == "embed")
    return _CASES[key]


class _Setup:
    """Device buffers and the per-call step of one workload: a pool of payload
    copies larger than 3x L2 (cycled call by call), the activation, the signs,
    the output and the workspace, all resident in HBM."""

    def __init__(self, name, dev):
        import torch

        import bit_gemv_gb300 as nt

        self.nt = nt
        self.w = w = synth.WORKLOADS[name]
        c = _case(w)
        self.embed = w.kind == "embed"
        payload_host = nt.ninfer_ternary_pack(w.fmt, c.values, c.scales)
        up_host = nt.ninfer_ternary_pack(w.fmt, c.up[0], c.up[1]) if w.mats == 2 else None
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.pool = max(2, -(-3 * self.l2 // (w.mats * payload_host.size)))
        self.pool_bytes = self.pool * w.mats * payload_host.size
        self.payloads = [torch.from_numpy(payload_host).to(dev) for _ in range(self.pool)]
        del payload_host
        self.signs = torch.from_numpy(c.signs.view(np.int16)).to(dev)
        if w.mats == 2:
            self.payloads_up = [torch.from_numpy(up_host).to(dev) for _ in range(self.pool)]
            self.signs_up = torch.from_numpy(c.up[2].view(np.int16)).to(dev)
        M = w.M
        if w.x_dtype == "bf16":
            self.x_host = torch.from_numpy(c.x_raw[:M].view(np.int16)).view(torch.bfloat16)
        else:
            self.x_host = torch.from_numpy(c.x[:M])
        self.x = self.x_host.to(dev)
        self.y = torch.empty((synth.EMBED_COUNT, w.k) if self.embed else (M, w.n), dtype=torch.float32, device=dev)
        self.ids_host = torch.from_numpy(c.ids) if self.embed else None
        self.ids = self.ids_host.to(dev) if self.embed else None
        if w.mats == 2:
            ws_bytes = nt.ninfer_ternary_gate_up_workspace(w.fmt, w.n, w.k, M, True, True)
        else:
            ws_bytes = nt.ninfer_ternary_matmul_workspace(w.fmt, w.n, w.k, M, True)
        self.ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def step(self, i):
        w, nt = self.w, self.nt
        if self.embed:
            nt.ninfer_ternary_embed(w.fmt, self.payloads[i % self.pool], w.n, w.k, self.ids, self.signs, out=self.y)
        elif w.mats == 2:
            nt.ninfer_ternary_gate_up(w.fmt, self.payloads[i % self.pool], self.payloads_up[i % self.pool], w.n, w.k,
                                      self.x, self.signs, self.signs_up, y=self.y, workspace=self.ws)
        else:
            nt.ninfer_ternary_matmul(w.fmt, self.payloads[i % self.pool], w.n, w.k, self.x, self.signs, y=self.y,
                                     workspace=self.ws)


def _capture(stream, fn, count, offset=0):
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(count):
                fn(offset + i)
    return g


HOLD_CYCLES = 300_000      # about 0.15 ms at 2 GHz: longer than the submission of the graphs


def _timed_graphs(stream, graphs, warm_replays, world, dev):
    """Replay graphs (each a list replayed in order) after warm-up replays of the
    first; CUDA events on the launching stream, barrier + synchronize on both
    sides; the slowest rank's milliseconds."""
    import torch

    with torch.cuda.stream(stream):
        for _ in range(warm_replays):
            graphs[0].replay()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        # a short spin kernel holds the idle stream while the host records the start
        # event and submits the graphs, so that the timed region begins with the
        # first step on the device instead of waiting for the host's submission
        # (the blocking-kernel technique of NVIDIA's nvbench); it runs before the
        # start event and is not part of any step
        torch.cuda._sleep(HOLD_CYCLES)
        e0.record(stream)
        for gr in graphs:
            gr.replay()
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    if world > 1:
        ms = max_over_ranks(ms, dev)
    return ms


def _graph_set(stream, fn, steps, per_graph):
    full, rem = divmod(steps, per_graph)
    g_main = _capture(stream, fn, per_graph) if full else None
    g_rem = _capture(stream, fn, rem, per_graph * full) if rem else None
    return ([g_main] * full) + ([g_rem] if g_rem is not None else [])


def _roofline(w, M, s_step, traffic):
    nbytes = algorithmic_bytes(w, M)
    if M > 8:
        return tensor_roofline(M, w.n, w.k, s_step, traffic)
    achieved = nbytes["total"] / s_step / 1e9
    peak, peak_kind = measured_peaks()
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs (copy)",
            "frac_of_8000_nominal": round(achieved / 8000, 4)}


def _measure_extra(name, stream, dev, world, steps, warmup):
    """One more workload timed in the same run: its own graphs of back-to-back
    calls over its own payload pool."""
    su = _Setup(name, dev)
    w = su.w
    with torch_stream(stream):
        for i in range(max(warmup, 3)):
            su.step(i)
    stream.synchronize()
    graphs = _graph_set(stream, su.step, steps, min(steps, 1000))
    ms = _timed_graphs(stream, graphs, max(1, -(-warmup // min(steps, 1000))), world, dev)
    s_step = ms / steps / 1e3
    tag, srcs = dominant_kernel(w)
    res = {"format": w.fmt, "n": w.n, "k": w.k, "M": w.M, "steps": steps, "ms_per_step": round(ms / steps, 6),
           "value": round(job_value(algorithmic_bytes(w, w.M)["weights"], world, s_step), 2), "unit": "GB/s",
           "projection_tokens_per_s": round(world * w.M / s_step, 1),
           "roofline": _roofline(w, w.M, s_step, profile_traffic(tag, name, srcs)),
           "gpu_launches": steps * kernels_per_step(w),
           "l2": f"rotating pool of {su.pool} payload copies ({su.pool_bytes / 1e6:.0f} MB > 3x L2)"}
    del su, graphs
    import torch

    torch.cuda.empty_cache()
    return res


def torch_stream(stream):
    import torch

    return torch.cuda.stream(stream)


def run_ours(args, rank: int, world: int, local_rank: int):
    import torch

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    name = args.workload or "gateup"
    su = _Setup(name, dev)
    w = su.w
    n, k, M = w.n, w.k, w.M
    nbytes = algorithmic_bytes(w, M)
    stream = torch.cuda.Stream(dev)

    # e2e buffers: pinned host inputs (activations, or token ids) in, pinned host result out
    in_dev = su.ids if su.embed else su.x
    in_host = su.ids_host if su.embed else su.x_host
    x_pin = [in_host.clone().pin_memory() for _ in range(su.pool)]
    y_pin = [torch.empty(tuple(su.y.shape), dtype=torch.float32).pin_memory() for _ in range(su.pool)]

    def step_e2e(i):
        in_dev.copy_(x_pin[i % su.pool], non_blocking=True)
        su.step(i)
        y_pin[i % su.pool].copy_(su.y, non_blocking=True)

    per_graph = min(args.steps, 1000)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):     # eager warm-up (module load, first launches)
            su.step(i)
    stream.synchronize()
    g_main = _graph_set(stream, su.step, args.steps, per_graph)
    g_e2e = _graph_set(stream, step_e2e, args.steps, per_graph)
    warm_replays = max(1, -(-args.warmup // per_graph))

    clocks = ClockSampler(local_rank, args.clocks_dir)
    clocks.start()
    ms_total = _timed_graphs(stream, g_main, warm_replays, world, dev)
    clock_info = clocks.stop()
    ms_e2e = _timed_graphs(stream, g_e2e, warm_replays, world, dev)

    # eager calls (no graph): what a caller that launches each projection
    # itself sees, host-side argument checks and launch set-up included
    eager_calls = min(args.steps, 2000)
    with torch.cuda.stream(stream):
        for i in range(20):
            su.step(i)
    stream.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ea.record(stream)
        for i in range(eager_calls):
            su.step(i)
        eb.record(stream)
    eb.synchronize()
    eager_us = ea.elapsed_time(eb) / eager_calls * 1e3

    torch.cuda.synchronize()
    ms_step = ms_total / args.steps
    s_step = ms_step / 1e3
    value = job_value(nbytes["weights"], world, s_step)
    e2e_s = ms_e2e / args.steps / 1e3
    tag, srcs = dominant_kernel(w)
    traffic = profile_traffic(tag, name, srcs)
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": path_dtype(w),
        "data": "synthetic",
        "config": {"workload": name, "format": w.fmt, "n": n, "k": k, "M": M, "x_dtype": w.x_dtype,
                   "seed": w.seed, "rotate": True, "projections": w.mats,
                   **({"rows_gathered": synth.EMBED_COUNT} if su.embed else {}),
                   "l2": f"rotating pool of {su.pool} payload copies ({su.pool_bytes / 1e6:.0f} MB > 3x L2 "
                         f"{su.l2 / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}"},
        "projection_tokens_per_s": round(world * (synth.EMBED_COUNT if su.embed else M) / s_step, 1),
        "roofline": _roofline(w, M, s_step, traffic),
        "e2e": {"value": round(job_value(nbytes["weights"], world, e2e_s), 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(in_host.numel() * in_host.element_size()),
                "d2h_bytes_per_step": int(su.y.numel() * 4), "ms_per_step": round(ms_e2e / args.steps, 6)},
        "eager_us_per_call": round(eager_us, 3),
        "clocks": clock_info,
        "gpu_launches": args.steps * kernels_per_step(w),
    }
    del g_main, g_e2e, su
    torch.cuda.empty_cache()
    extras = EXTRA_WORKLOADS if args.workload is None and not args.no_extra else ()
    if extras:
        clocks2 = ClockSampler(local_rank, args.clocks_dir)
        clocks2.start()
        res["workloads"] = {}
        for nm in extras:
            res["workloads"][nm] = _measure_extra(nm, stream, dev, world, min(EXTRA_STEPS[nm], args.steps), args.warmup)
            res["gpu_launches"] += res["workloads"][nm]["gpu_launches"]
        res["workloads_clocks"] = clocks2.stop()
    return res


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time: every rank contributes its own and gets the
    maximum (a collective on the process group; then a barrier)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_value(weight_bytes_per_rank: int, world: int, s_step: float) -> float:
    """Whole-job weight GB/s: every rank streams its own replica's weights once
    per step, so the job moves world times the per-rank bytes in s_step."""
    return world * weight_bytes_per_rank / s_step / 1e9


def path_dtype(w) -> str:
    """Arithmetic type of the path that serves workload w."""
    if w.kind == "embed":
        return "f32"     # dequantised weights and the inverse transform in fp32
    if w.M == 1:
        return "int16*ternary->int32->f32"
    return "f16*f16->f32"


def tensor_roofline(M, n, k, s_step, traffic):
    """Prefill: the contraction after expansion, 2*M*n*k flops per call."""
    tflops = 2.0 * M * n * k / s_step / 1e12
    peak, kind = measured_tensor_peak()
    return {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(tflops / peak, 4), "traffic": traffic, "peak_source": kind}


def kernels_per_step(w) -> int:
    """Kernels one projection launches: the M = 1 decode kernels rotate x
    themselves (one kernel, whatever k); the PTQ1_0 M <= 8 kernel rotates x
    itself and, with more than one 1024-block, is followed by the block
    reduction; the PQ2_0 M <= 8, prefill and general paths run a prep or
    transform kernel and then the main one. The fused gate/up pair at PQ2_0,
    M = 1 is one kernel, and so is the embedding."""
    if w.kind == "embed":
        return 1
    if w.mats == 2 and w.fmt == "PQ2_0_G128" and w.M == 1:
        return 1
    if w.mats == 2:      # two projections, then the SwiGLU kernel
        import dataclasses
        return 2 * kernels_per_step(dataclasses.replace(w, mats=1)) + 1
    if w.M == 1:
        return 1
    if w.fmt == "PTQ1_0_G128" and w.M <= 8:
        return 2 if w.k > 1024 else 1
    if w.fmt == "PTQ1_0_G128":
        return 3     # planes rewritten as PQ2_0, rotation to binary16, tensor-core GEMM
    return 2


# ------------------------------------------------------------ CPU oracle ---
def cpu_oracle_sample(workload: str, rows: int, reps: int) -> dict:
    """Time the fp64 oracle on `rows` rows of the workload (single thread)."""
    import oracle

    w = synth.WORKLOADS[workload]
    if w.kind == "embed":
        # the same work per call: EMBED_COUNT rows gathered from a `rows`-row slice
        c = synth.make_case(w, n=rows, with_ids=True)
        payload = oracle.pack_planes(w.fmt, c.values, c.scales)
        D = synth.bf16_bits_to_f32(c.signs)
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle.embed_rows(w.fmt, payload, rows, w.k, c.ids, D)
        dt = (time.perf_counter() - t0) / reps
        return {"seconds_per_call": dt, "weight_bytes": algorithmic_bytes(w, 1)["weights"], "rows": rows}
    c = synth.make_case(w, n=rows)
    payload = oracle.pack_planes(w.fmt, c.values, c.scales)
    D = synth.bf16_bits_to_f32(c.signs)
    if w.mats == 2:
        payload_up = oracle.pack_planes(w.fmt, c.up[0], c.up[1])
        D_up = synth.bf16_bits_to_f32(c.up[2])
    t0 = time.perf_counter()
    for _ in range(reps):
        if w.mats == 2:
            oracle.gate_up_swiglu(w.fmt, payload, payload_up, rows, w.k, c.x, D, D_up)
        else:
            oracle.ternary_matmul(w.fmt, payload, rows, w.k, c.x, D)
    dt = (time.perf_counter() - t0) / reps
    groups = -(-w.k // 128)
    wbytes = w.mats * rows * groups * (34 if w.fmt == "PQ2_0_G128" else 28)
    return {"seconds_per_call": dt, "weight_bytes": wbytes, "rows": rows}


def run_cpu_child(workload: str, rows: int, reps: int, threads: int = 1) -> dict:
    env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads))
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-child", workload, str(rows), str(reps)],
                         capture_output=True, text=True, env=env, timeout=900)
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    return json.loads(out.stdout.strip().splitlines()[-1])


def cpu_baseline(workload: str) -> dict:
    res = _cpu_baseline_one(workload, 1)
    cores = os.cpu_count() or 1
    if cores > 1:
        # the same sample with the host's BLAS on every core (the dense transform
        # and contraction of the oracle are BLAS calls; its plane decode is not)
        allc = _cpu_baseline_one(workload, cores)
        res["all_cores"] = {"value": allc["value"], "unit": allc["unit"], "cores": cores,
                            "seconds_per_call": allc["seconds_per_call"]}
    return res


def _cpu_baseline_one(workload: str, threads: int) -> dict:
    w = synth.WORKLOADS[workload]
    rows = min(w.n, 17408)
    r = run_cpu_child(workload, rows, 2, threads)
    gbs = r["weight_bytes"] / r["seconds_per_call"] / 1e9
    if w.kind == "embed":
        return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                "sample": f"{synth.EMBED_COUNT} rows gathered from a {rows}-row slice of the {workload} matrix "
                          f"(the same work per call), 2 calls, fp64 numpy, {threads} thread(s)",
                "seconds_per_call": round(r["seconds_per_call"], 4)}
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {w.n} rows of the {workload} workload, 2 calls, fp64 numpy, {threads} thread(s)",
            "seconds_per_call": round(r["seconds_per_call"], 4),
            "tokens_per_s_full_matrix": round(w.M / (r["seconds_per_call"] * w.n / rows), 4)}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return None
    w = synth.WORKLOADS[args.workload]
    # size each step's row sample so that warm-up + timed steps take ~2 minutes
    cal = run_cpu_child(args.workload, min(w.n, 256), 1)
    per_row = cal["seconds_per_call"] / min(w.n, 256)
    rows = int(max(1, min(w.n, 120.0 / (args.steps + args.warmup) / per_row)))
    run_cpu_child(args.workload, rows, args.warmup)
    r = run_cpu_child(args.workload, rows, max(args.steps, 1))
    gbs = r["weight_bytes"] / r["seconds_per_call"] / 1e9
    sample = f"each step: {rows} of {w.n} rows of the {args.workload} workload, fp64 numpy oracle, 1 thread"
    return {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["seconds_per_call"] * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "format": w.fmt, "n": w.n, "k": w.k, "M": w.M, "x_dtype": w.x_dtype,
                   "seed": w.seed, "rotate": True, "projections": w.mats},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    if len(sys.argv) > 1 and sys.argv[1] == "--cpu-child":
        print(json.dumps(cpu_oracle_sample(sys.argv[2], int(sys.argv[3]), int(sys.argv[4]))))
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None, choices=sorted(synth.WORKLOADS),
                    help="time one workload alone (default: gate/up as the headline, plus the down and head "
                         "workloads in the same run)")
    ap.add_argument("--no-extra", action="store_true", help="time the headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-dir", default=None, help="where to keep the raw nvidia-smi samples (default: temp dir)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        args.workload = args.workload or "gateup"
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.workload or "gateup")
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
