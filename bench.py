#!/usr/bin/env python
"""Benchmark of the block-scaled packed-precision hot path on GB300.

Default workload (the one the headline metric is quoted on): MX-FP6 e3m2 W6A6,
A bf16 [128, 4096] and W bf16 [4096, 4096] ~ N(0, 0.02) with 1% outliers x20.
One step = quantize A and W (one batched launch; each tensor its own amax
global scale, exact ceil UE8M0, RNE encode, 4-in-3 packing) + the tcgen05
block-scaled GEMM (fp32 accumulate, bf16 out) -- every row of the hot path
this workload exercises.

  value       GEMM TFLOP/s of the whole step (2*M*N*K / step time), summed over
              ranks (each rank runs its own independent replica: weak scaling).
  roofline    the step's dominant op (largest device time), achieved vs the
              measured peak in MEASURED_PEAKS.json.
  e2e         the same metric through the public API with host buffers: the
              step's bf16 inputs copied from pinned host memory, the bf16 output
              copied back, inside the timed region.
  cpu_baseline  the CPU oracle on a bounded sample of the same step, extrapolated.

Other workloads (--workload) measure the decode GEMV, the nvfp4 prefill GEMM
and the W6A8 GEMM the same way.  L2 is flushed before every timed step (a
256 MiB write, then a 256 MiB read of another buffer so no dirty lines remain).
The step is captured once as a CUDA graph with event nodes at its two ends and
replayed (device time).  A second capture with an event node after every op,
replayed after the timed steps, gives the per-op split and the dominant op's
duration for the roofline.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = ("mxfp6_e3m2_w6a6_128x4096x4096", "nvfp4_decode_gemv_Mx28672x8192", "nvfp4_prefill_gemm_8192",
             "w6a8_e4m3xe2m3_4096x14336x4096", "nvfp4_gemv_1x256x256")
METRIC = "block-scaled GEMM TFLOP/s & decode GEMV HBM GB/s, as fraction of GB300 roofline"
L2_FLUSH_BYTES = 256 << 20


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
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_rank{gpu_index}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
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

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
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

    def __init__(self, name, dev, gemv_m=32):
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
            w = S.normal_bf16((N, K), cfg["w_std"], cfg["seed"] + 1)
            wd = t(w).view(torch.bfloat16)
            self.cw, self.sw, self.gw = bsq.quantize_nvfp4(wd)
            del wd
            x = S.normal_bf16((M, K), cfg["x_std"], cfg["seed"] + 2 + M)
            self.host_in = {"x": x}
            self.x = t(x).view(torch.bfloat16)
            self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            self.flops = 2.0 * M * N * K
            by = N * K // 2 + bsq.scale_bytes(N, K // 16) + M * K * 2 + M * N * 2
            self._ops = [("gemv_nvfp4", lambda s: bsq.gemv_nvfp4_(self.x, self.cw, self.sw, self.gw, self.y, N, K, s),
                          by, self.flops, "hbm", None)]
            self.units = ("GB/s", by / 1e9)
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


def run_bsq(args, rank, world, dev_index):
    import torch
    from block_scaled_precision_packed_gb300 import bsq
    torch.cuda.set_device(dev_index)
    dev = torch.device("cuda", dev_index)
    bsq.load()
    pk = peaks()
    wl = Workload(args.workload, dev, gemv_m=args.gemv_m)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    # after the write, a read of a second buffer of the same size leaves L2
    # holding clean lines, so the step does not pay for the flush's write-backs
    flush_b = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
    ops = wl.ops()

    # The step is captured once as a CUDA graph and replayed: the timed region
    # measures device time, not the host's launch rate.  The timed graph has
    # event nodes only at its two ends; a second capture with an event node
    # after every op, replayed for the same number of steps after the timed
    # region, gives the per-op split (its event nodes add a little time per op,
    # so the split slightly overstates each op).  The L2 flush runs outside the
    # graphs, before every step.
    n_ops = len(ops)
    with torch.cuda.stream(stream):
        for i in range(2):
            wl.step(stream)                     # loads kernels before capture
    torch.cuda.synchronize()

    def capture(per_op):
        # external events become event-record nodes inside the captured graph
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n_ops + 1)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            evs[0].record(stream)
            for j, (_, fn, *_r) in enumerate(ops):
                fn(stream)
                if per_op or j == n_ops - 1:
                    evs[j + 1].record(stream)
        return graph, evs

    bsq.reset_launch_counts()
    graph, evs = capture(False)
    launches_per_step = sum(bsq.launch_count(k) for k in bsq.KERNEL_IDS)
    graph_ops, evs_ops = capture(True)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            for g in (graph, graph_ops):
                flush.fill_(i)
                g.replay()
    torch.cuda.synchronize()

    def flushed_replay(g, i):
        with torch.cuda.stream(stream):
            flush.fill_(i + 1000)
            torch.sum(flush_b, dim=0, dtype=torch.int64, out=flush_sink)
            g.replay()
        stream.synchronize()

    # ---- timed region: K steps, L2 flushed before each ----
    step_ms_all = np.zeros(args.steps)
    op_ms = np.zeros((args.steps, n_ops))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev_index) as clk:
        for i in range(args.steps):
            flushed_replay(graph, i)
            step_ms_all[i] = evs[0].elapsed_time(evs[n_ops])
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        # per-op split (same flush, the instrumented capture)
        for i in range(args.steps):
            flushed_replay(graph_ops, i)
            for j in range(n_ops):
                op_ms[i, j] = evs_ops[j].elapsed_time(evs_ops[j + 1])
        torch.cuda.synchronize()
    launches = launches_per_step * args.steps
    if dist:
        dist.barrier()
    step_ms = max_over_ranks(float(step_ms_all.mean()), dist, dev)
    unit, per_step = wl.units
    value = job_throughput(per_step, world, step_ms)

    # dominant op and its roofline
    mean_op = op_ms.mean(axis=0)
    d = int(np.argmax(mean_op))
    name, _, by, fl, bound, pkind = ops[d]
    dur_s = mean_op[d] / 1e3
    if bound == "hbm":
        achieved, peak, ru = by / dur_s / 1e9, pk["hbm"], "GB/s"
    else:
        achieved, peak, ru = fl / dur_s / 1e12, tensor_peak(pkind, pk), "TFLOP/s"
    roof = {"bound": bound, "kernel": name, "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": ru,
            "frac": round(achieved / peak, 4), "peak_source": pk["src"] + (" (burst)" if bound == "tensor" else ""),
            "algorithmic": by if bound == "hbm" else fl,
            "traffic": traffic_for(name, args.workload,
                                   args.gemv_m if args.workload == "nvfp4_decode_gemv_Mx28672x8192" else None),
            "ms": round(float(mean_op[d]), 5)}
    per_op = {ops[j][0]: round(float(mean_op[j]) * 1e3, 2) for j in range(n_ops)}

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if wl.host_in:
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
                flush.fill_(i)
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
        e2e = {"value": round(job_throughput(per_step, world, e_ms), 3), "unit": unit, "ms_per_step": round(e_ms, 4),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    small_m = small_m_quantizer_us(wl, dev, stream, flush, flush_b, flush_sink, args) \
        if args.workload == "w6a8_e4m3xe2m3_4096x14336x4096" else None
    w6a6 = args.workload == "mxfp6_e3m2_w6a6_128x4096x4096"
    fused_act = fused_act_quantizer_us(wl, dev, stream, flush, flush_b, flush_sink, args) if w6a6 else None
    containers = byte_container_quantizer_us(wl, dev, stream, flush, flush_b, flush_sink, args) if w6a6 else None
    grouped = grouped_moe_us(wl, dev, stream, flush, flush_b, flush_sink, args, peaks()) if w6a6 else None
    quant_a = fused_quant_a_gemm_us(wl, dev, stream, flush, flush_b, flush_sink, args) if w6a6 else None
    return dict(value=value, unit=unit, step_ms=step_ms, roofline=roof, per_op_us=per_op, e2e=e2e,
                launches=launches, clocks=clk.summary(), wl=wl, small_m=small_m, fused_act=fused_act,
                containers=containers, grouped=grouped, quant_a=quant_a)


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
def oracle_sample(workload, rows_w):
    """Time the oracle on a bounded sample of one step; returns (seconds for a
    full step, extrapolated; description)."""
    import oracle as O
    from block_scaled_precision_packed_gb300 import synthetic as S
    cfg = S.WORKLOADS[workload]
    if workload == "mxfp6_e3m2_w6a6_128x4096x4096":
        M, N, K = cfg["M"], cfg["N"], cfg["K"]
        a = S.normal_bf16((M, K), cfg["a_std"], cfg["seed"] + 1, cfg["outlier_frac"], cfg["outlier_mult"])
        w = S.normal_bf16((N, K), cfg["w_std"], cfg["seed"] + 2, cfg["outlier_frac"], cfg["outlier_mult"])
        rows = np.arange(rows_w, dtype=np.int64)
        t0 = time.perf_counter()
        ca, sa, ga = O.quantize_mx(a, O.E3M2)
        t1 = time.perf_counter()
        cw, uw, gw = O.quantize_mx_rows(w, O.E3M2, rows)
        t2 = time.perf_counter()
        sw = np.zeros(O.scale_bytes(rows_w, K // 32), np.uint8)
        for r in range(rows_w):
            for b in range(K // 32):
                sw[O.swz_offset(r, b, K // 32)] = uw[r, b]
        t3 = time.perf_counter()
        O.gemm_mx(ca, O.E3M2, sa, ga, cw, O.E3M2, sw, gw, M, rows_w, K, threads=1)
        t4 = time.perf_counter()
        full = (t1 - t0) + (t2 - t1) * N / rows_w + (t4 - t3) * N / rows_w
        return full, f"quantize A [{M},{K}] whole, W rows 0..{rows_w - 1} of {N} (tensor amax over all of W), " \
                     f"GEMM outputs [{M},{rows_w}]; W quantize and GEMM scaled by {N}/{rows_w}"
    if workload in ("nvfp4_decode_gemv_Mx28672x8192", "nvfp4_gemv_1x256x256"):
        N, K = cfg["N"], cfg["K"]
        M = 32 if "Ms" in cfg else cfg["M"]
        rows_w = min(rows_w, N)
        x = S.normal_bf16((M, K), cfg["x_std"], cfg["seed"] + 2)
        W = S.random_words((rows_w, K // 8), cfg["seed"] + 1)
        sc = S.choice_bytes(O.scale_bytes(rows_w, K // 16), cfg["seed"] + 2, list(range(0x20, 0x60)))
        t0 = time.perf_counter()
        O.gemv_nvfp4(x, W, sc, 1.0, M, rows_w, K, threads=1)
        t1 = time.perf_counter()
        return (t1 - t0) * N / rows_w, f"GEMV outputs [{M},{rows_w}] of [{M},{N}], scaled by {N}/{rows_w}"
    # GEMM workloads: a block of output rows against a block of W rows
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    mr = 16
    if workload == "nvfp4_prefill_gemm_8192":
        A = S.random_words((mr, K // 8), 1)
        W = S.random_words((rows_w, K // 8), 2)
        sa = S.choice_bytes(O.scale_bytes(mr, K // 16), 3, list(range(0x20, 0x60)))
        sw = S.choice_bytes(O.scale_bytes(rows_w, K // 16), 4, list(range(0x20, 0x60)))
        t0 = time.perf_counter()
        O.gemm_nvfp4(A, sa, 1.0, W, sw, 1.0, mr, rows_w, K, threads=1)
    else:
        A = S.random_bytes(mr * K, 1).reshape(mr, K) & 0x7E
        W = S.random_bytes(rows_w * 3 * K // 4, 2).reshape(rows_w, 3 * K // 4)
        sa = S.choice_bytes(O.scale_bytes(mr, K // 32), 3, list(range(120, 134)))
        sw = S.choice_bytes(O.scale_bytes(rows_w, K // 32), 4, list(range(120, 134)))
        t0 = time.perf_counter()
        O.gemm_mx(A, O.E4M3, sa, 1.0, W, O.E2M3, sw, 1.0, mr, rows_w, K, threads=1)
    t1 = time.perf_counter()
    return (t1 - t0) * (M / mr) * (N / rows_w), f"GEMM outputs [{mr},{rows_w}] of [{M},{N}], scaled by area"


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="bsq", choices=["bsq", "reference"])
    ap.add_argument("--workload", default=WORKLOADS[0], choices=WORKLOADS)
    ap.add_argument("--gemv-m", type=int, default=32, choices=[1, 8, 32])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl_cfg = {"workload": args.workload}
    if args.workload == "nvfp4_decode_gemv_Mx28672x8192":
        wl_cfg["M"] = args.gemv_m

    if args.impl == "reference":
        # The CPU oracle as it stands, on this arm's workload and metric; rank 0 only.
        if rank != 0:
            return
        import oracle as O
        O.build()
        rows = 8
        unit = "GB/s" if "gemv" in args.workload else "TFLOP/s"
        times, desc = [], ""
        for i in range(args.warmup + args.steps):
            t, desc = oracle_sample(args.workload, rows)
            if i >= args.warmup:
                times.append(t)
        step_s = float(np.mean(times))
        per_step = per_step_units(args.workload, args.gemv_m)
        v = per_step / step_s
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(args.workload),
                "data": "synthetic", "config": wl_cfg,
                "cpu_baseline": {"kind": "oracle", "value": v, "unit": unit, "cores": 1, "sample": desc},
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
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as O
        O.build()
        t, desc = oracle_sample(args.workload, 256 if args.workload.startswith("mxfp6") else 16)
        per_step = per_step_units(args.workload, args.gemv_m)
        cpu = {"kind": "oracle", "value": per_step / t, "unit": r["unit"], "cores": 1, "sample": desc,
               "ms_per_step_extrapolated": round(t * 1e3, 1)}
    line = {"metric": METRIC, "value": round(r["value"], 3), "unit": r["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["step_ms"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(args.workload),
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": dict(wl_cfg, l2="flushed before every timed step (256 MiB write, then a read pass)",
                           timing="step captured as a CUDA graph (event nodes at its ends only) and replayed; "
                                  "per-op split from a second capture with an event node after each op",
                           parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
            "roofline": r["roofline"], "per_op_us": r["per_op_us"], "e2e": r["e2e"],
            "gpu_launches": int(r["launches"]), "clocks": r["clocks"], "cpu_baseline": cpu}
    if r["small_m"] is not None:
        line["quantizer_small_m_us"] = r["small_m"]
    if r["fused_act"] is not None:
        line["fused_activation_quantizer"] = r["fused_act"]
    if r["containers"] is not None:
        line["byte_container_quantizer"] = r["containers"]
    if r["grouped"] is not None:
        line["grouped_moe"] = r["grouped"]
    if r["quant_a"] is not None:
        line["gemm_with_fused_activation_quantizer"] = r["quant_a"]
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def per_step_units(workload, gemv_m):
    from block_scaled_precision_packed_gb300 import synthetic as S
    cfg = S.WORKLOADS[workload]
    if workload == "nvfp4_decode_gemv_Mx28672x8192":
        N, K, M = cfg["N"], cfg["K"], gemv_m
        sb = -(-N // 128) * 128 * (-(-(K // 16) // 4) * 4)
        return (N * K // 2 + sb + M * K * 2 + M * N * 2) / 1e9
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
