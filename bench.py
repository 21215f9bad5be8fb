#!/usr/bin/env python
"""Benchmark of the block-scaled packed-precision hot path on GB300.

Headline workload (the largest single-GPU configuration): nvfp4 prefill GEMM
M = N = K = 8192, both operands e2m1 with ue4m3 scales per 16 and an fp32
tensor factor, quantized beforehand from bf16 N(0, 1) (A) and N(0, 0.02) (W);
one step = the tcgen05 block-scaled GEMM (fp32 accumulate, bf16 out).

  value       GEMM TFLOP/s of the step (2*M*N*K / step time), summed over ranks
              (each rank runs its own independent replica: weak scaling).
  roofline    the step's kernel, achieved vs the dense fp4 tensor peak (the
              measured bf16 peak in MEASURED_PEAKS.json times the nominal ratio).
  e2e         the same metric through the public API with host buffers: the
              step's quantized operands copied from pinned host memory, the bf16
              output copied back, inside the timed region.
  configs     every other configuration, each with its own time and roofline:
              the decode GEMV at M = 1, 8, 32 (HBM GB/s), the W6A8 GEMM (fp8/fp6
              tensor peak) with the small-M e2m3 quantizer, the one-row GEMV and
              the W6A6 step (batched quantize + GEMM); L2 flushed and warm.
  cpu_baseline  the CPU oracle on a bounded sample of the step, at 1 core and at
              every host core, extrapolated to the step.

--workload selects a single workload (its line alone).  L2 is flushed before
every timed step (a 256 MiB write, then a 256 MiB read of another buffer so no
dirty lines remain); the warm figures replay without the flush.  Each step is
captured once as a CUDA graph with event nodes at its two ends and replayed
(device time).  A second capture with an event node after every op gives the
per-op split and the dominant op's duration for the roofline.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = ("nvfp4_prefill_gemm_8192", "nvfp4_decode_gemv_Mx28672x8192", "w6a8_e4m3xe2m3_4096x14336x4096",
             "mxfp6_e3m2_w6a6_128x4096x4096", "nvfp4_gemv_1x256x256")
HEADLINE = WORKLOADS[0]
METRIC = "block-scaled GEMM TFLOP/s & decode GEMV HBM GB/s, as fraction of GB300 roofline"
L2_FLUSH_BYTES = 256 << 20
# A decode step runs the GEMV of several layers back to back; the decode
# workload's step is this many GEMVs, each over its own copy of the quantized
# weight at distinct addresses (every copy larger than L2), so each launch
# streams its weight from HBM and the per-launch figure is the step time over
# the launches.
DECODE_LAYERS = 4


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# Dense tensor-core peak of a block-scaled kind, from the measured bf16 peak and
# the nominal dense ratios (bf16 2.25, fp8/fp6 4.5, fp4 13.5 PFLOP/s).
def tensor_peak(kind, pk, sustained=False):
    base = pk["bf16_sus"] if sustained and pk.get("bf16_sus") else pk["bf16"]
    return base * {"fp4": 13.5 / 2.25, "fp8f6": 4.5 / 2.25}[kind]


def src_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_scaled_precision_packed_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel, workload, m=None):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the kernel sources as they are now (else None); m: the decode GEMV's rows."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(f"{kernel}@{workload}@M{m}") if m is not None else None
    e = e or d.get(f"{kernel}@{workload}")
    if not e or e.get("src_sha") != src_sha():
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"bsq_clocks_gpu{gpu_index}_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            self.proc.wait()
            self.f.close()
        self.rows = self._read()
        try:
            os.unlink(self.path)
        except OSError:
            pass

    def _read(self):
        rows = []
        try:
            lines = open(self.path).read().splitlines()
        except OSError:
            return rows
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        return rows

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = self.rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [r[0] for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": rows[0][1], "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------- workloads ----
class Workload:
    """Holds device inputs/outputs; step() runs the hot path once on `stream`;
    ops() lists (name, launch fn, algorithmic bytes, flops, bound, peak kind)."""

    def __init__(self, name, dev, gemv_m=32, cache=None):
        import torch
        from block_scaled_precision_packed_gb300 import bsq, synthetic as S
        self.name, self.dev, self.bsq, self.torch = name, dev, bsq, torch
        cfg = S.WORKLOADS[name]
        self.cfg = cfg
        t = lambda a: torch.from_numpy(a.view({2: np.int16, 4: np.int32, 1: np.uint8}[a.dtype.itemsize])).to(dev)
        if name == "mxfp6_e3m2_w6a6_128x4096x4096":
            M, N, K = cfg["M"], cfg["N"], cfg["K"]
            self.M, self.N, self.K = M, N, K
            a = S.normal_bf16((M, K), cfg["a_std"], cfg["seed"] + 1, cfg["outlier_frac"], cfg["outlier_mult"])
            w = S.normal_bf16((N, K), cfg["w_std"], cfg["seed"] + 2, cfg["outlier_frac"], cfg["outlier_mult"])
            self.host_in = {"a": a, "w": w}
            self.a, self.w = t(a).view(torch.bfloat16), t(w).view(torch.bfloat16)
            self.ca = torch.empty((M, 3 * K // 4), dtype=torch.uint8, device=dev)
            self.cw = torch.empty((N, 3 * K // 4), dtype=torch.uint8, device=dev)
            self.sa = torch.empty(bsq.scale_bytes(M, K // 32), dtype=torch.uint8, device=dev)
            self.sw = torch.empty(bsq.scale_bytes(N, K // 32), dtype=torch.uint8, device=dev)
            self.ga = torch.empty(1, dtype=torch.float32, device=dev)
            self.gw = torch.empty(1, dtype=torch.float32, device=dev)
            self.wsq = torch.empty(bsq.quantize_batch_workspace_bytes(), dtype=torch.uint8, device=dev)
            self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            self.flops = 2.0 * M * N * K
            qa_bytes = M * K * 2 + M * 3 * K // 4 + bsq.scale_bytes(M, K // 32)
            qw_bytes = N * K * 2 + N * 3 * K // 4 + bsq.scale_bytes(N, K // 32)
            g_bytes = M * 3 * K // 4 + N * 3 * K // 4 + bsq.scale_bytes(M, K // 32) + bsq.scale_bytes(N, K // 32) + M * N * 2
            # A and W quantized by one batched launch (each with its own amax / s_global)
            qitems = [(self.a, self.ca, self.sa, self.ga), (self.w, self.cw, self.sw, self.gw)]
            self._ops = [
                ("quantize_AW_e3m2", lambda s: bsq.quantize_mxfp6_batch_(qitems, 0, self.wsq, s),
                 qa_bytes + qw_bytes, 0.0, "hbm", None),
                ("gemm_e3m2xe3m2", lambda s: bsq.gemm_mxfp6_(self.ca, 0, self.sa, self.ga, self.cw, 0, self.sw, self.gw,
                                                             self.y, M, N, K, s),
                 g_bytes, self.flops, "hbm", "fp8f6"),
            ]
            self.units = ("TFLOP/s", self.flops / 1e12)
            self.launches_per_step = None
        elif name == "nvfp4_decode_gemv_Mx28672x8192":
            N, K = cfg["N"], cfg["K"]
            M = gemv_m
            self.M, self.N, self.K = M, N, K
            cache = {} if cache is None else cache
            if "decode_w" not in cache:     # one quantized weight, copied per layer, serves every M
                w = S.normal_bf16((N, K), cfg["w_std"], cfg["seed"] + 1)
                wd = t(w).view(torch.bfloat16)
                cw, sw, gw = bsq.quantize_nvfp4(wd)
                del wd, w
                cache["decode_w"] = [(cw, sw, gw)] + [(cw.clone(), sw.clone(), gw.clone())
                                                      for _ in range(DECODE_LAYERS - 1)]
            self.layers = cache["decode_w"]
            self.cw, self.sw, self.gw = self.layers[0]
            x = S.normal_bf16((M, K), cfg["x_std"], cfg["seed"] + 2 + M)
            self.host_in = {"x": x}
            self.x = t(x).view(torch.bfloat16)
            self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            self.ys = [self.y] + [torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                                  for _ in range(DECODE_LAYERS - 1)]
            self.flops = 2.0 * M * N * K * DECODE_LAYERS
            by = N * K // 2 + bsq.scale_bytes(N, K // 16) + M * K * 2 + M * N * 2

            def layer(l):
                cw, sw, gw = self.layers[l]
                return lambda s: bsq.gemv_nvfp4_(self.x, cw, sw, gw, self.ys[l], N, K, s)
            self._ops = [(f"gemv_nvfp4[layer {l}]", layer(l), by, self.flops / DECODE_LAYERS, "hbm", None)
                         for l in range(DECODE_LAYERS)]
            self.units = ("GB/s", by * DECODE_LAYERS / 1e9)
            self.same_kernel_ops = True
        elif name == "nvfp4_gemv_1x256x256":
            M, N, K = cfg["M"], cfg["N"], cfg["K"]
            self.M, self.N, self.K = M, N, K
            x = S.normal_bf16((M, K), cfg["x_std"], cfg["seed"])
            self.host_in = {"x": x}
            self.x = t(x).view(torch.bfloat16)
            self.cw = t(S.random_words((N, K // 8), cfg["seed"] + 1))
            self.sw = t(S.choice_bytes(bsq.scale_bytes(N, K // 16), cfg["seed"] + 2, S.UE4M3_POW2_M4_TO_P4))
            self.gw = torch.tensor([cfg["g_w"]], device=dev)
            self.y = torch.empty((M, N), dtype=torch.float32, device=dev)
            self.flops = 2.0 * M * N * K
            by = N * K // 2 + bsq.scale_bytes(N, K // 16) + M * K * 2 + M * N * 4
            self._ops = [("gemv_nvfp4", lambda s: bsq.gemv_nvfp4_(self.x, self.cw, self.sw, self.gw, self.y, N, K, s),
                          by, self.flops, "hbm", None)]
            self.units = ("GB/s", by / 1e9)
        elif name == "nvfp4_prefill_gemm_8192":
            M, N, K = cfg["M"], cfg["N"], cfg["K"]
            self.M, self.N, self.K = M, N, K
            a = S.normal_bf16((M, K), cfg["a_std"], cfg["seed"] + 1)
            w = S.normal_bf16((N, K), cfg["w_std"], cfg["seed"] + 2)
            self.ca, self.sa, self.ga = bsq.quantize_nvfp4(t(a).view(torch.bfloat16))
            self.cw, self.sw, self.gw = bsq.quantize_nvfp4(t(w).view(torch.bfloat16))
            # end to end: the quantized operands (codes, scales, global factors) come from the host
            self.host_in = operand_host_copies(self, ("ca", "sa", "ga", "cw", "sw", "gw"))
            self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            self.flops = 2.0 * M * N * K
            by = (M + N) * K // 2 + bsq.scale_bytes(M, K // 16) + bsq.scale_bytes(N, K // 16) + M * N * 2
            self._ops = [("gemm_nvfp4", lambda s: bsq.gemm_nvfp4_(self.ca, self.sa, self.ga, self.cw, self.sw, self.gw,
                                                                   self.y, M, N, K, s),
                          by, self.flops, "tensor", "fp4")]
            self.units = ("TFLOP/s", self.flops / 1e12)
        elif name == "w6a8_e4m3xe2m3_4096x14336x4096":
            M, N, K = cfg["M"], cfg["N"], cfg["K"]
            self.M, self.N, self.K = M, N, K
            a = S.normal_bf16((M, K), cfg["a_std"], cfg["seed"] + 1)
            w = S.normal_bf16((N, K), cfg["w_std"], cfg["seed"] + 2)
            self.ca, self.sa, self.ga = bsq.quantize_mxfp6(t(a).view(torch.bfloat16), "e4m3")
            self.cw, self.sw, self.gw = bsq.quantize_mxfp6(t(w).view(torch.bfloat16), "e2m3")
            self.host_in = operand_host_copies(self, ("ca", "sa", "ga", "cw", "sw", "gw"))
            self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            self.flops = 2.0 * M * N * K
            by = M * K + N * 3 * K // 4 + bsq.scale_bytes(M, K // 32) + bsq.scale_bytes(N, K // 32) + M * N * 2
            self._ops = [("gemm_e4m3xe2m3", lambda s: bsq.gemm_mxfp6_(self.ca, 2, self.sa, self.ga, self.cw, 1, self.sw,
                                                                       self.gw, self.y, M, N, K, s),
                          by, self.flops, "tensor", "fp8f6")]
            self.units = ("TFLOP/s", self.flops / 1e12)
        else:
            raise ValueError(name)

    def ops(self):
        return self._ops

    def step(self, stream):
        for _, fn, *_ in self._ops:
            fn(stream)


def operand_host_copies(wl, names):
    """Host copies of a product workload's device operands (raw bytes), for
    the end-to-end arm, which copies them in from pinned host memory every step."""
    return {n: getattr(wl, n).contiguous().view(-1).cpu().numpy().view(np.uint8) for n in names}


def max_over_ranks(ms, dist, device):
    """The slowest rank's time (every rank gets it): replicas report the
    whole job's throughput over the time of the last one to finish."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step, world, ms):
    """Whole-job throughput: every rank runs its own replica of the step."""
    return units_per_step * world / (ms / 1e3)


class Timer:
    """Device timing of a workload's step: the step captured as a CUDA graph
    (event nodes at its ends) and replayed, L2 flushed before each replay (cold)
    or not (warm); a second capture with an event node after every op gives the
    per-op split (its event nodes add a little time per op)."""

    def __init__(self, dev, stream, args, dist):
        import torch
        self.torch, self.dev, self.stream, self.args, self.dist = torch, dev, stream, args, dist
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        # after the write, a read of a second buffer of the same size leaves L2
        # holding clean lines, so the step does not pay for the flush's write-backs
        self.flush_b = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.flush_sink = torch.zeros((), dtype=torch.int64, device=dev)

    def capture(self, ops, per_op):
        torch, stream = self.torch, self.stream
        n = len(ops)
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n + 1)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            evs[0].record(stream)
            for j, (_, fn, *_r) in enumerate(ops):
                fn(stream)
                if per_op or j == n - 1:
                    evs[j + 1].record(stream)
        return graph, evs

    def replay(self, g, i, cold=True):
        torch, stream = self.torch, self.stream
        with torch.cuda.stream(stream):
            if cold:
                self.flush.fill_(i + 1000)
                torch.sum(self.flush_b, dim=0, dtype=torch.int64, out=self.flush_sink)
            g.replay()
        stream.synchronize()

    def run(self, wl, clock=None):
        """{cold_ms, warm_ms, op_ms [per op, cold], launches_per_step}; the
        cold timed region is the K steps between a barrier and a synchronize,
        its mean taken as the slowest rank's."""
        from block_scaled_precision_packed_gb300 import bsq
        torch, stream, args, dist = self.torch, self.stream, self.args, self.dist
        ops = wl.ops()
        n = len(ops)
        with torch.cuda.stream(stream):
            for _ in range(2):
                wl.step(stream)                     # loads kernels before capture
        torch.cuda.synchronize()
        bsq.reset_launch_counts()
        graph, evs = self.capture(ops, False)
        launches = sum(bsq.launch_count(k) for k in bsq.KERNEL_IDS)
        graph_ops, evs_ops = self.capture(ops, True)
        for i in range(args.warmup):
            self.replay(graph, i)
            self.replay(graph_ops, i)
        cold = np.zeros(args.steps)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        with clock if clock is not None else _NoClock():
            for i in range(args.steps):
                self.replay(graph, i)
                cold[i] = evs[0].elapsed_time(evs[n])
            torch.cuda.synchronize()
        if dist:
            dist.barrier()
        op_ms = np.zeros((args.steps, n))
        for i in range(args.steps):
            self.replay(graph_ops, i)
            for j in range(n):
                op_ms[i, j] = evs_ops[j].elapsed_time(evs_ops[j + 1])
        warm = np.zeros(args.steps)
        for i in range(args.warmup + args.steps):
            self.replay(graph, i, cold=False)
            if i >= args.warmup:
                warm[i - args.warmup] = evs[0].elapsed_time(evs[n])
        cold_ms = max_over_ranks(float(cold.mean()), dist, self.dev)
        warm_ms = max_over_ranks(float(warm.mean()), dist, self.dev)
        return {"cold_ms": cold_ms, "warm_ms": warm_ms, "op_ms": op_ms.mean(axis=0), "launches_per_step": launches}


class _NoClock:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def roofline(wl, op_ms, pk, workload, gemv_m=None, step_ms=None):
    """The dominant op's achieved rate against its peak: algorithmic bytes (HBM
    bound) or flops (tensor bound) per launch over its mean duration.  A step
    of launches of one kernel (the decode layers) takes the step time over its
    launches as that duration."""
    ops = wl.ops()
    d = int(np.argmax(op_ms))
    name, _, by, fl, bound, pkind = ops[d]
    dur_s = op_ms[d] / 1e3
    if getattr(wl, "same_kernel_ops", False) and step_ms is not None:
        name = name.split("[")[0]
        dur_s = step_ms / len(ops) / 1e3
    if bound == "hbm":
        achieved, peak, ru = by / dur_s / 1e9, pk["hbm"], "GB/s"
    else:
        achieved, peak, ru = fl / dur_s / 1e12, tensor_peak(pkind, pk), "TFLOP/s"
    return {"bound": bound, "kernel": name, "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": ru,
            "frac": round(achieved / peak, 4), "peak_source": pk["src"] + (" (burst)" if bound == "tensor" else ""),
            "algorithmic": by if bound == "hbm" else fl,
            "traffic": traffic_for(name, workload, gemv_m if workload == "nvfp4_decode_gemv_Mx28672x8192" else None),
            "ms": round(dur_s * 1e3, 5)}


def config_entry(wl, t, pk, workload, gemv_m=None):
    """One configuration's figures for the line: its step time (L2 flushed and
    warm), throughput in its unit, per-op split and roofline."""
    unit, per_step = wl.units
    extra = {}
    if getattr(wl, "same_kernel_ops", False):
        n = len(wl.ops())
        extra = {"launches_per_step": n, "us_per_launch": round(t["cold_ms"] * 1e3 / n, 2)}
    return {**extra, "us": round(t["cold_ms"] * 1e3, 2), "us_warm_l2": round(t["warm_ms"] * 1e3, 2),
            "value": round(per_step / (t["cold_ms"] / 1e3), 2), "unit": unit,
            "per_op_us": {wl.ops()[j][0]: round(float(t["op_ms"][j]) * 1e3, 2) for j in range(len(wl.ops()))},
            "roofline": roofline(wl, t["op_ms"], pk, workload, gemv_m, t["cold_ms"])}


def run_bsq(args, rank, world, dev_index):
    import torch
    from block_scaled_precision_packed_gb300 import bsq
    torch.cuda.set_device(dev_index)
    dev = torch.device("cuda", dev_index)
    bsq.load()
    pk = peaks()
    stream = torch.cuda.Stream(device=dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
    timer = Timer(dev, stream, args, dist)
    cache = {}
    wl = Workload(args.workload, dev, gemv_m=args.gemv_m, cache=cache)
    with ClockSampler(dev_index) as clk:
        t = timer.run(wl)
    unit, per_step = wl.units
    step_ms = t["cold_ms"]
    value = job_throughput(per_step, world, step_ms)
    roof = roofline(wl, t["op_ms"], pk, args.workload, args.gemv_m, t["cold_ms"])
    per_op = {wl.ops()[j][0]: round(float(t["op_ms"][j]) * 1e3, 2) for j in range(len(wl.ops()))}
    launches = t["launches_per_step"] * args.steps
    e2e = end_to_end(wl, timer, args, dist, dev, per_step, world)
    flush, flush_b, flush_sink = timer.flush, timer.flush_b, timer.flush_sink
    extras = {}
    if args.workload == "w6a8_e4m3xe2m3_4096x14336x4096":
        extras["quantizer_small_m_us"] = small_m_quantizer_us(wl, dev, stream, flush, flush_b, flush_sink, args)
    if args.workload == "mxfp6_e3m2_w6a6_128x4096x4096":
        extras.update(w6a6_next_rows(wl, dev, stream, timer, args, pk))
    configs = None
    if args.all_configs:
        del wl
        configs = {}
        for M in (1, 8, 32):
            w = Workload("nvfp4_decode_gemv_Mx28672x8192", dev, gemv_m=M, cache=cache)
            configs.setdefault("nvfp4_decode_gemv_Mx28672x8192", {})[f"M={M}"] = \
                config_entry(w, timer.run(w), pk, "nvfp4_decode_gemv_Mx28672x8192", M)
            del w
        cache.clear()
        w = Workload("w6a8_e4m3xe2m3_4096x14336x4096", dev)
        e = config_entry(w, timer.run(w), pk, "w6a8_e4m3xe2m3_4096x14336x4096")
        e["quantizer_small_m_us"] = small_m_quantizer_us(w, dev, stream, flush, flush_b, flush_sink, args)
        configs["w6a8_e4m3xe2m3_4096x14336x4096"] = e
        del w
        w = Workload("nvfp4_gemv_1x256x256", dev)
        configs["nvfp4_gemv_1x256x256"] = config_entry(w, timer.run(w), pk, "nvfp4_gemv_1x256x256")
        del w
        w = Workload("mxfp6_e3m2_w6a6_128x4096x4096", dev)
        e = config_entry(w, timer.run(w), pk, "mxfp6_e3m2_w6a6_128x4096x4096")
        e["next"] = w6a6_next_rows(w, dev, stream, timer, args, pk)
        configs["mxfp6_e3m2_w6a6_128x4096x4096"] = e
        del w
    return dict(value=value, unit=unit, step_ms=step_ms, warm_ms=t["warm_ms"], roofline=roof, per_op_us=per_op,
                e2e=e2e, launches=launches, clocks=clk.summary(), extras=extras, configs=configs)


def end_to_end(wl, timer, args, dist, dev, per_step, world):
    """The step through the public API with host buffers: every step copies
    its inputs in from pinned host memory and its output back (L2 flushed
    before each step as in the timed region)."""
    import torch
    if not wl.host_in:
        return None
    stream = timer.stream
    # flat 16-bit views of both sides (any operand dtype of even byte size)
    pinned = {k: torch.from_numpy(np.ascontiguousarray(v).reshape(-1).view(np.int16)).pin_memory()
              for k, v in wl.host_in.items()}
    dst = {k: getattr(wl, k).reshape(-1).view(torch.int16) for k in pinned}
    yh = torch.empty(wl.y.shape, dtype=wl.y.dtype).pin_memory()
    h2d = sum(v.numel() * 2 for v in pinned.values())
    d2h = wl.y.numel() * wl.y.element_size()
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            timer.flush.fill_(i)
            if i >= args.warmup:
                e_ev[i - args.warmup][0].record(stream)
            for k in pinned:
                dst[k].copy_(pinned[k], non_blocking=True)
            wl.step(stream)
            yh.copy_(wl.y, non_blocking=True)
            if i >= args.warmup:
                e_ev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in e_ev])), dist, dev)
    return {"value": round(job_throughput(per_step, world, e_ms), 3), "unit": wl.units[0],
            "ms_per_step": round(e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def w6a6_next_rows(wl, dev, stream, timer, args, pk):
    """The W6A6 layer's next rows of the path: the fused activation quantizer,
    the byte-container quantizer, the grouped (MoE) layer and the GEMM with the
    activation quantizer inside it."""
    f, fb, fs = timer.flush, timer.flush_b, timer.flush_sink
    return {"fused_activation_quantizer": fused_act_quantizer_us(wl, dev, stream, f, fb, fs, args),
            "byte_container_quantizer": byte_container_quantizer_us(wl, dev, stream, f, fb, fs, args),
            "grouped_moe": grouped_moe_us(wl, dev, stream, f, fb, fs, args, pk),
            "gemm_with_fused_activation_quantizer": fused_quant_a_gemm_us(wl, dev, stream, f, fb, fs, args)}


def graph_call_us(fn, stream, flush, flush_b, flush_sink, args):
    """Mean device time of one call of fn(stream), captured as a graph with
    event nodes at its ends and replayed with the L2 flushed before each run."""
    import torch
    with torch.cuda.stream(stream):
        fn(stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True, external=True)
    e1 = torch.cuda.Event(enable_timing=True, external=True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        e0.record(stream)
        fn(stream)
        e1.record(stream)
    ts = []
    for i in range(args.warmup + args.steps):
        with torch.cuda.stream(stream):
            flush.fill_(i + 3000)
            torch.sum(flush_b, dim=0, dtype=torch.int64, out=flush_sink)
            g.replay()
        stream.synchronize()
        if i >= args.warmup:
            ts.append(e0.elapsed_time(e1) * 1e3)
    return float(np.mean(ts))


def fused_act_quantizer_us(wl, dev, stream, flush, flush_b, flush_sink, args):
    """The W6A6 layer's activation side with the activation fused into the
    quantizer (bsq_quantize_mxfp6_act): ReLU^2 of [M, K] and SiLU(gate) * up of
    [M, 2K] -> e3m2 codes + UE8M0 scales, M = 128, K = 4096, inputs N(0, 1)."""
    import torch
    from block_scaled_precision_packed_gb300 import bsq, synthetic as S
    M, K = wl.M, wl.K
    out = {"M": M, "K": K, "format": "e3m2, UE8M0 per 32"}
    for name, act, kin in (("relu2", bsq.ACT_RELU2, K), ("silu_mul", bsq.ACT_SILU_MUL, 2 * K)):
        x = S.normal_bf16((M, kin), 1.0, wl.cfg["seed"] + 20 + act)
        xd = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
        codes = torch.empty((M, 3 * K // 4), dtype=torch.uint8, device=dev)
        scales = torch.empty(bsq.scale_bytes(M, K // 32), dtype=torch.uint8, device=dev)
        sg = torch.empty(1, dtype=torch.float32, device=dev)
        ws = torch.empty(max(16, bsq.quantize_workspace_bytes(M, K)), dtype=torch.uint8, device=dev)
        us = graph_call_us(lambda s: bsq.quantize_mxfp6_act_(xd, K, act, 0, codes, scales, sg, None, ws, s),
                           stream, flush, flush_b, flush_sink, args)
        by = M * kin * 2 + M * 3 * K // 4 + bsq.scale_bytes(M, K // 32)
        out[name] = {"us": round(us, 2), "algorithmic_bytes": by, "GB/s": round(by / (us * 1e-6) / 1e9, 1)}
    return out


def fused_quant_a_gemm_us(wl, dev, stream, flush, flush_b, flush_sink, args):
    """The W6A6 product with the activation quantizer fused into the GEMM
    (bsq_gemm_mxfp6_quant_a: x bf16 [128, 4096] quantized to e3m2 inside the
    GEMM against the e3m2 weight), beside the same product as two calls
    (bsq_quantize_mxfp6 of x, then bsq_gemm_mxfp6); W is quantized beforehand."""
    import torch
    from block_scaled_precision_packed_gb300 import bsq, synthetic as S
    M, N, K = wl.M, wl.N, wl.K
    c = wl.cfg
    x = S.normal_bf16((M, K), c["a_std"], c["seed"] + 30, outlier_frac=c["outlier_frac"], outlier_mult=c["outlier_mult"])
    w = S.normal_bf16((N, K), c["w_std"], c["seed"] + 31, outlier_frac=c["outlier_frac"], outlier_mult=c["outlier_mult"])
    xd = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    Wc, sW, gW = bsq.quantize_mxfp6(torch.from_numpy(w.view(np.int16)).to(dev).view(torch.bfloat16), "e3m2")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    sg = torch.empty(1, dtype=torch.float32, device=dev)
    wsq = torch.empty(bsq.gemm_quant_a_workspace_bytes(), dtype=torch.uint8, device=dev)
    codes = torch.empty((M, 3 * K // 4), dtype=torch.uint8, device=dev)
    scales = torch.empty(bsq.scale_bytes(M, K // 32), dtype=torch.uint8, device=dev)
    ws = torch.empty(max(16, bsq.quantize_workspace_bytes(M, K)), dtype=torch.uint8, device=dev)
    fused = graph_call_us(lambda s: bsq.gemm_mxfp6_quant_a_(xd, 0, Wc, 0, sW, gW, Y, sg, wsq, M, N, K, s),
                          stream, flush, flush_b, flush_sink, args)

    def two(s):
        bsq.quantize_mxfp6_(xd, 0, codes, scales, sg, ws, s)
        bsq.gemm_mxfp6_(codes, 0, scales, sg, Wc, 0, sW, gW, Y, M, N, K, s)
    two_us = graph_call_us(two, stream, flush, flush_b, flush_sink, args)
    return {"M": M, "N": N, "K": K, "format": "bf16 x -> e3m2 in the GEMM, e3m2 W", "fused_us": round(fused, 2),
            "quantize_then_gemm_us": round(two_us, 2),
            "TFLOP/s": round(2 * M * N * K / (fused * 1e-6) / 1e12, 1)}


def grouped_moe_us(wl, dev, stream, flush, flush_b, flush_sink, args, pk):
    """The W6A6 layer as 8 experts (grouped MoE layout): A [8, 512, 4096] with
    seeded row counts (mean ~256 routed rows per expert), W [8, 4096, 4096],
    both e3m2.  Times the grouped activation quantizer (per-expert global scales
    given) and the grouped tcgen05 GEMM over all experts; TFLOP/s counts only the
    routed rows."""
    import torch
    from block_scaled_precision_packed_gb300 import bsq, synthetic as S
    G, R, N, K = 8, 512, wl.N, wl.K
    rc = np.random.default_rng(wl.cfg["seed"] + 40).integers(64, 449, G).astype(np.int32)
    rct = torch.from_numpy(rc).to(dev)
    x = torch.from_numpy(S.normal_bf16((G * R, K), 1.0, wl.cfg["seed"] + 41).view(np.int16)).to(dev)
    x = x.view(torch.bfloat16).view(G, R, K)
    A = torch.empty((G, R, 3 * K // 4), dtype=torch.uint8, device=dev)
    sA = torch.empty((G, bsq.scale_bytes(R, K // 32)), dtype=torch.uint8, device=dev)
    gA = torch.empty(G, dtype=torch.float32, device=dev)
    gsa = torch.full((G,), 12544.0 / 4.5, dtype=torch.float32, device=dev)
    W = torch.empty((G, N, 3 * K // 4), dtype=torch.uint8, device=dev)
    sW = torch.empty((G, bsq.scale_bytes(N, K // 32)), dtype=torch.uint8, device=dev)
    gW = torch.empty(G, dtype=torch.float32, device=dev)
    for g in range(G):                                  # weights: quantized once, outside the timing
        wg = torch.from_numpy(S.normal_bf16((N, K), 0.02, wl.cfg["seed"] + 50 + g).view(np.int16)).to(dev)
        wg = wg.view(torch.bfloat16).view(1, N, K)
        gsw = torch.full((1,), 12544.0 / float(wg.float().abs().max()), dtype=torch.float32, device=dev)
        bsq.quantize_grouped_mxfp6_(wg, torch.tensor([N], dtype=torch.int32, device=dev), gsw, 0, W[g:g + 1],
                                    sW[g:g + 1], gW[g:g + 1])
        del wg
    Y = torch.empty((G, R, N), dtype=torch.bfloat16, device=dev)
    q_us = graph_call_us(lambda s: bsq.quantize_grouped_mxfp6_(x, rct, gsa, 0, A, sA, gA, s),
                         stream, flush, flush_b, flush_sink, args)
    g_us = graph_call_us(lambda s: bsq.gemm_grouped_mxfp6_(A, 0, sA, gA, W, 0, sW, gW, rct, Y, G, R, N, K, s),
                         stream, flush, flush_b, flush_sink, args)
    flops = 2.0 * float(rc.sum()) * N * K
    tf = flops / (g_us * 1e-6) / 1e12
    peak = tensor_peak("fp8f6", pk)
    return {"experts": G, "rows_per_expert": R, "routed_rows": [int(v) for v in rc], "N": N, "K": K,
            "format": "e3m2 x e3m2, UE8M0 per 32", "quantize_us": round(q_us, 2), "gemm_us": round(g_us, 2),
            "gemm_TFLOP/s": round(tf, 1), "gemm_frac_of_fp8f6_peak": round(tf / peak, 4)}


def byte_container_quantizer_us(wl, dev, stream, flush, flush_b, flush_sink, args):
    """The W6A6 weight quantized with fp6 byte-container output
    (bsq_quantize_mxfp6_containers): bf16 [N, K] -> e3m2 codes one per byte."""
    import torch
    from block_scaled_precision_packed_gb300 import bsq
    N, K = wl.N, wl.K
    codes = torch.empty((N, K), dtype=torch.uint8, device=dev)
    scales = torch.empty(bsq.scale_bytes(N, K // 32), dtype=torch.uint8, device=dev)
    sg = torch.empty(1, dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, bsq.quantize_workspace_bytes(N, K)), dtype=torch.uint8, device=dev)
    us = graph_call_us(lambda s: bsq.quantize_mxfp6_containers_(wl.w, 0, codes, scales, sg, ws, s),
                       stream, flush, flush_b, flush_sink, args)
    by = N * K * 2 + N * K + bsq.scale_bytes(N, K // 32)
    return {"N": N, "K": K, "format": "e3m2 byte containers, UE8M0 per 32", "us": round(us, 2),
            "algorithmic_bytes": by, "GB/s": round(by / (us * 1e-6) / 1e9, 1)}


def small_m_quantizer_us(wl, dev, stream, flush, flush_b, flush_sink, args):
    """The W6A8 layer's activation-side quantizer at decode sizes: bf16 [M, K]
    -> e2m3 codes + UE8M0 scales for M in {1, 4, 16}, K = 4096 (one launch each),
    timed like the step (a captured graph with event nodes at its ends, L2
    flushed before every replay); mean microseconds per call."""
    import torch
    from block_scaled_precision_packed_gb300 import bsq, synthetic as S
    K = wl.K
    out = {}
    for M in (1, 4, 16):
        x = S.normal_bf16((M, K), wl.cfg["a_std"], wl.cfg["seed"] + 10 + M)
        xd = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
        codes = torch.empty((M, 3 * K // 4), dtype=torch.uint8, device=dev)
        scales = torch.empty(bsq.scale_bytes(M, K // 32), dtype=torch.uint8, device=dev)
        sg = torch.empty(1, dtype=torch.float32, device=dev)
        ws = torch.empty(max(16, bsq.quantize_workspace_bytes(M, K)), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            bsq.quantize_mxfp6_(xd, 1, codes, scales, sg, ws, stream)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True, external=True)
        e1 = torch.cuda.Event(enable_timing=True, external=True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e0.record(stream)
            bsq.quantize_mxfp6_(xd, 1, codes, scales, sg, ws, stream)
            e1.record(stream)
        ts = []
        for i in range(args.warmup + args.steps):
            with torch.cuda.stream(stream):
                flush.fill_(i + 2000)
                torch.sum(flush_b, dim=0, dtype=torch.int64, out=flush_sink)
                g.replay()
            stream.synchronize()
            if i >= args.warmup:
                ts.append(e0.elapsed_time(e1) * 1e3)
        out[f"M={M}"] = round(float(np.mean(ts)), 2)
    out["K"] = K
    out["format"] = "bf16 -> e2m3, UE8M0 per 32"
    return out


# ----------------------------------------------------------- CPU oracle arm ---
def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


# Output rows x weight rows of the product the oracle computes per sample: a
# single-core sample (a few seconds of CPU work) and a 16x larger one for all
# host cores, taken on the workload's own quantized operands.
ORACLE_SAMPLE = {1: (16, 256), 0: (32, 2048)}


class OracleSample:
    """A bounded sample of one step of a workload for the CPU oracle: the
    operands are the oracle's own quantization of the workload's bf16 inputs
    (only the rows the sample needs; the tensor amax spans the whole tensor),
    the product is a block of output rows x weight rows, and the step's time is
    the sample's scaled by the step's outputs over the sample's."""

    def __init__(self, workload, threads, gemv_m=32):
        import oracle as O
        from block_scaled_precision_packed_gb300 import synthetic as S
        self.O, self.workload, self.threads = O, workload, threads
        cfg = S.WORKLOADS[workload]
        mr, nr = ORACLE_SAMPLE[1 if threads == 1 else 0]
        if workload == "nvfp4_gemv_1x256x256":
            M, N, K = cfg["M"], cfg["N"], cfg["K"]
            self.x = S.normal_bf16((M, K), cfg["x_std"], cfg["seed"])
            self.W = S.random_words((N, K // 8), cfg["seed"] + 1)
            self.sw = S.choice_bytes(O.scale_bytes(N, K // 16), cfg["seed"] + 2, S.UE4M3_POW2_M4_TO_P4)
            self.mr, self.nr, self.scale = M, N, 1.0
            self.desc = f"the whole product [{M},{N}], K = {K}"
            self.args = (M, N, K)
            return
        if workload == "nvfp4_decode_gemv_Mx28672x8192":
            M, N, K = gemv_m, cfg["N"], cfg["K"]
            w = S.normal_bf16((N, K), cfg["w_std"], cfg["seed"] + 1)
            rows = np.arange(nr, dtype=np.int64)
            self.W, sb, g = O.quantize_nvfp4_rows(w, rows)
            self.sw = _swizzle(O, sb)
            self.g = g
            self.x = S.normal_bf16((M, K), cfg["x_std"], cfg["seed"] + 2 + M)
            self.mr, self.nr, self.scale = M, nr, N / nr * DECODE_LAYERS
            self.desc = (f"GEMV outputs [{M},{nr}] of [{M},{N}] (weight rows quantized by the oracle), scaled by "
                         f"{N}/{nr} and by the step's {DECODE_LAYERS} layers")
            self.args = (M, nr, K)
            return
        M, N, K = cfg["M"], cfg["N"], cfg["K"]
        mr = min(mr, M)
        a = S.normal_bf16((M, K), cfg["a_std"], cfg["seed"] + 1, cfg.get("outlier_frac", 0.0),
                          cfg.get("outlier_mult", 20.0))
        w = S.normal_bf16((N, K), cfg["w_std"], cfg["seed"] + 2, cfg.get("outlier_frac", 0.0),
                          cfg.get("outlier_mult", 20.0))
        ra, rw = np.arange(mr, dtype=np.int64), np.arange(nr, dtype=np.int64)
        self.a, self.w, self.rw = a, w, rw
        if workload == "nvfp4_prefill_gemm_8192":
            self.A, sa, self.ga = O.quantize_nvfp4_rows(a, ra)
            self.W, sw, self.gw = O.quantize_nvfp4_rows(w, rw)
        else:
            fa, fw = (O.E3M2, O.E3M2) if workload.startswith("mxfp6") else (O.E4M3, O.E2M3)
            self.fa, self.fw = fa, fw
            self.A, sa, self.ga = O.quantize_mx_rows(a, fa, ra)
            self.W, sw, self.gw = O.quantize_mx_rows(w, fw, rw)
        self.sa, self.sw = _swizzle(O, sa), _swizzle(O, sw)
        self.mr, self.nr, self.scale = mr, nr, (M / mr) * (N / nr)
        self.desc = (f"GEMM outputs [{mr},{nr}] of [{M},{N}] on the oracle's quantization of the workload's "
                     f"operands, scaled by area" + (f"; plus quantize A whole and W rows 0..{nr - 1} (scaled by "
                                                    f"{N}/{nr})" if workload.startswith("mxfp6") else ""))
        self.args = (mr, nr, K)
        self.NW = N

    def step_seconds(self):
        """One sample's time scaled to the full step."""
        O, th = self.O, self.threads
        t0 = time.perf_counter()
        if self.workload == "nvfp4_gemv_1x256x256":
            O.gemv_nvfp4(self.x, self.W, self.sw, 0.5, *self.args, threads=th)
        elif self.workload == "nvfp4_decode_gemv_Mx28672x8192":
            O.gemv_nvfp4(self.x, self.W, self.sw, self.g, *self.args, threads=th)
        elif self.workload == "nvfp4_prefill_gemm_8192":
            O.gemm_nvfp4(self.A, self.sa, self.ga, self.W, self.sw, self.gw, *self.args, threads=th)
        else:
            O.gemm_mx(self.A, self.fa, self.sa, self.ga, self.W, self.fw, self.sw, self.gw, *self.args, threads=th)
        t = (time.perf_counter() - t0) * self.scale
        if self.workload.startswith("mxfp6"):          # the W6A6 step quantizes both operands too
            t0 = time.perf_counter()
            O.quantize_mx(self.a, self.fa)
            t1 = time.perf_counter()
            O.quantize_mx_rows(self.w, self.fw, self.rw)
            t += (t1 - t0) + (time.perf_counter() - t1) * self.NW / self.rw.size
        return t


def _swizzle(O, plain):
    rows, blocks = plain.shape
    buf = np.zeros(O.scale_bytes(rows, blocks), np.uint8)
    for r in range(rows):
        for b in range(blocks):
            buf[O.swz_offset(r, b, blocks)] = plain[r, b]
    return buf


def cpu_baseline(workload, gemv_m, unit):
    """The oracle as it stands on this host: one sample at 1 core, one (16x
    larger) at every core; value = the step's units per extrapolated second."""
    import oracle as O
    O.build()
    per_step = per_step_units(workload, gemv_m)
    out = {"kind": "oracle", "unit": unit}
    for threads, key in ((1, "one_core"), (0, "all_cores")):
        smp = OracleSample(workload, threads, gemv_m)
        t = smp.step_seconds()
        out[key] = {"value": per_step / t, "cores": 1 if threads == 1 else host_cores(),
                    "ms_per_step_extrapolated": round(t * 1e3, 1), "sample": smp.desc}
    # the headline figure: all host cores
    out.update(value=out["all_cores"]["value"], cores=out["all_cores"]["cores"], sample=out["all_cores"]["sample"],
               host_cpu_count=os.cpu_count())
    return out


def config_cpu_baselines(configs):
    """The oracle at 1 core and at every host core on each other configuration
    (the same bounded samples as the headline's cpu_baseline)."""
    import oracle as O
    O.build()
    for name, entry in configs.items():
        subs = [(k, int(k[2:])) for k in entry] if name == "nvfp4_decode_gemv_Mx28672x8192" else [(None, 32)]
        for key, m in subs:
            e = entry[key] if key else entry
            unit = e["unit"]
            per_step = per_step_units(name, m)
            out = {"kind": "oracle", "unit": unit}
            for threads, leg in ((1, "one_core"), (0, "all_cores")):
                smp = OracleSample(name, threads, m)
                t = smp.step_seconds()
                out[leg] = {"value": per_step / t, "cores": 1 if threads == 1 else host_cores(),
                            "ms_per_step_extrapolated": round(t * 1e3, 3), "sample": smp.desc}
            e["cpu_baseline"] = out


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="bsq", choices=["bsq", "reference"])
    ap.add_argument("--workload", default=None, choices=WORKLOADS,
                    help=f"one workload alone (default: {HEADLINE} with every other configuration in 'configs')")
    ap.add_argument("--gemv-m", type=int, default=32, choices=[1, 8, 32])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    args.all_configs = args.workload is None
    if args.workload is None:
        args.workload = HEADLINE

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl_cfg = workload_config(args.workload, args.gemv_m)
    unit = "GB/s" if "gemv" in args.workload else "TFLOP/s"

    if args.impl == "reference":
        # The CPU oracle as it stands, on this arm's workload, metric and sample
        # (every host core); rank 0 only.
        if rank != 0:
            return
        import oracle as O
        O.build()
        smp = OracleSample(args.workload, 0, args.gemv_m)
        times = []
        for i in range(args.warmup + args.steps):
            t = smp.step_seconds()
            if i >= args.warmup:
                times.append(t)
        step_s = float(np.mean(times))
        per_step = per_step_units(args.workload, args.gemv_m)
        v = per_step / step_s
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(args.workload),
                "data": "synthetic (seeded; shapes and distributions of the workload)", "config": wl_cfg,
                "cpu_baseline": {"kind": "oracle", "value": v, "unit": unit, "cores": host_cores(),
                                 "sample": smp.desc + f"; extrapolated per step, {args.steps} steps timed"},
                "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = run_bsq(args, rank, world, local)
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    cpu = None if args.no_cpu_baseline else cpu_baseline(args.workload, args.gemv_m, r["unit"])
    line = {"metric": METRIC, "value": round(r["value"], 3), "unit": r["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["step_ms"], 5),
            "ms_per_step_warm_l2": round(r["warm_ms"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(args.workload),
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": dict(wl_cfg, parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
            "roofline": r["roofline"], "per_op_us": r["per_op_us"], "e2e": r["e2e"],
            "gpu_launches": int(r["launches"]), "clocks": r["clocks"], "cpu_baseline": cpu}
    line.update(r["extras"])
    if r["configs"] is not None:
        if not args.no_cpu_baseline:
            config_cpu_baselines(r["configs"])
        line["configs"] = r["configs"]
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def workload_config(workload, gemv_m):
    c = {"workload": workload,
         "l2": "flushed before every timed step (256 MiB write, then a read pass); warm-L2 figures replay "
               "without the flush",
         "timing": "step captured as a CUDA graph (event nodes at its ends only) and replayed; per-op split from "
                   "a second capture with an event node after each op"}
    if workload == "nvfp4_decode_gemv_Mx28672x8192":
        c["M"] = gemv_m
        c["layers"] = DECODE_LAYERS
        c["step"] = (f"{DECODE_LAYERS} decode GEMVs back to back, each over its own copy of the quantized weight "
                     f"(distinct addresses, each larger than L2); L2 flushed before the step")
    return c


def per_step_units(workload, gemv_m):
    from block_scaled_precision_packed_gb300 import synthetic as S
    cfg = S.WORKLOADS[workload]
    if workload == "nvfp4_decode_gemv_Mx28672x8192":
        N, K, M = cfg["N"], cfg["K"], gemv_m
        sb = -(-N // 128) * 128 * (-(-(K // 16) // 4) * 4)
        return DECODE_LAYERS * (N * K // 2 + sb + M * K * 2 + M * N * 2) / 1e9
    if workload == "nvfp4_gemv_1x256x256":
        N, K, M = cfg["N"], cfg["K"], cfg["M"]
        return (N * K // 2 + N * K // 16 + M * K * 2 + M * N * 4) / 1e9
    return 2.0 * cfg["M"] * cfg["N"] * cfg["K"] / 1e12


def dtype_of(workload):
    return {"mxfp6_e3m2_w6a6_128x4096x4096": "e3m2 x e3m2 (UE8M0/32), fp32 accumulate, bf16 out",
            "nvfp4_decode_gemv_Mx28672x8192": "bf16 x nvfp4 (e2m1, ue4m3/16), fp32 accumulate, bf16 out",
            "nvfp4_gemv_1x256x256": "bf16 x nvfp4, fp32 accumulate, fp32 out",
            "nvfp4_prefill_gemm_8192": "nvfp4 x nvfp4, fp32 accumulate, bf16 out",
            "w6a8_e4m3xe2m3_4096x14336x4096": "e4m3 x e2m3 (UE8M0/32), fp32 accumulate, bf16 out"}[workload]


if __name__ == "__main__":
    main()
