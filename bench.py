#!/usr/bin/env python
"""Benchmark of the GB300 Simple GLA mixer (one JSON line on rank 0).

Headline: chunked-forward tokens/s on the Laplace-layer workload (B=8, T=2048, H=16, d_k=96,
d_v=192, bf16 operands, fp32 state), inputs resident in HBM.  The same line carries the other
hot-path rows measured the same way: decode tokens/s at 1,280 sequences x 24 layers (64 steps),
the chunked backward, and the packed varlen forward; each with its roofline against the measured
GB300 peaks.  `e2e` repeats the headline through host buffers (copies inside the timed region),
`cpu_baseline` times the fp64 oracle on the host cores.  `--impl reference` times the oracle alone.

Multi-GPU: every rank runs the same workload on its own GPU (independent replicas, no
collective on the data path; scaling "weak"); values are summed over ranks, times are the max.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GLA chunked-fwd tokens/s (H16,dk96,dv192); decode tok/s at 1280 seqs"
DK, DV, H = 96, 192, 16

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) from the ncu captures summarised in
# profiles/, per unit of work; reported only while the kernel source is byte-identical to the one
# profiled (SHA-256 prefix), else null.
PROFILED_TRAFFIC = {
    # B=8 T=2048 H=16 forward: 245.515008 MB read + 81.780480 MB written, one launch
    "fwd": ("linear_attention_recurrence_simple_gb300/csrc/gla_chunk_tc.cu", "d75fb5f6c49d8cfb",
            327295488.0, "per launch of the B=8 T=2048 H=16 forward"),
    # 49,152-state pool: 3.662106 GB read + 3.583718 GB written; traffic scales with the pool
    "decode": ("linear_attention_recurrence_simple_gb300/csrc/gla_decode.cu", "a4a26403a2ad2cf8",
               7245823744.0 / 49152, "per state per step"),
    # the same pool in bf16: 1.849750 GB read + 1.771710 GB written
    "decode_bf16_state": ("linear_attention_recurrence_simple_gb300/csrc/gla_decode.cu", "a4a26403a2ad2cf8",
                          3621459200.0 / 49152, "per state per step"),
    # the fused norm-gate step on the fp32 pool: 3.680801 GB read + 3.583189 GB written
    "decode_norm_gate": ("linear_attention_recurrence_simple_gb300/csrc/gla_decode.cu", "a4a26403a2ad2cf8",
                         7263989504.0 / 49152, "per state per step"),
    # the same forward with the self-augmentation step: 244.934400 MB read + 82.883328 MB written
    "fwd_aug": ("linear_attention_recurrence_simple_gb300/csrc/gla_chunk_tc.cu", "d75fb5f6c49d8cfb",
                327817728.0, "per launch of the B=8 T=2048 H=16 augmented forward"),
    # head RMSNorm + gate, 16,384 x 16 rows: 201.355776 MB read + 70.854144 MB written (part of y
    # is still in L2 when the kernel ends), one launch
    "norm_gate": ("linear_attention_recurrence_simple_gb300/csrc/gla_norm.cu", "4987f08ea9f6d8e4",
                  272209920.0, "per launch of the 16,384 x 16 rows"),
    # the MXFP8 pool: 972.095744 MB read + 892.485120 MB written
    "decode_mxfp8_state": ("linear_attention_recurrence_simple_gb300/csrc/gla_mxfp8.cu", "158873036f51e740",
                           1864580864.0 / 49152, "per state per step"),
    # the all-fp32 mode's forward: 404.469504 MB read + 183.305728 MB written (part of o is still
    # in L2 when the kernel ends), one launch
    "fwd_fp32": ("linear_attention_recurrence_simple_gb300/csrc/gla_simt.cu", "f1b9f51523b1e5ae",
                 587775232.0, "per launch of the B=8 T=2048 H=16 fp32 forward"),
    # the all-fp32 mode's backward, its three launches per call: dq 509.635328 + 91.569152 MB,
    # dk 519.081984 + 97.524480 MB, dv 414.296064 + 177.118720 MB (read + written)
    "bwd_fp32": ("linear_attention_recurrence_simple_gb300/csrc/gla_simt.cu", "f1b9f51523b1e5ae",
                 1809225728.0, "per call (three launches) of the B=8 T=2048 H=16 fp32 backward"),
}


def profiled_traffic(row, units=1.0):
    import hashlib
    path, sha, per_unit, _ = PROFILED_TRAFFIC[row]
    try:
        with open(os.path.join(ROOT, path), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != sha:
                return None
    except OSError:
        return None
    return int(per_unit * units)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for_smi(torch):
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        first = vis.split(",")[0] if vis else str(torch.cuda.current_device())
        return first


# ------------------------------------------------------------------------------------------
# timing
# ------------------------------------------------------------------------------------------
class Dist:
    def __init__(self, torch):
        self.torch = torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.device = "cpu"

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist
            self.device = "cuda" if backend == "nccl" else "cpu"

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x):
        if not self.pg:
            return x
        t = self.torch.tensor([x], dtype=self.torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def timed(torch, dist, fn, steps, warmup):
    """W untimed calls, then exactly K calls between a barrier + synchronize on both sides, timed
    by one pair of CUDA events around the K calls (nothing else in the stream between them).
    A ~0.2 ms device-side sleep is queued just before the start event, so that the first timed
    call is already queued when the region opens (otherwise the host's time to issue that call
    counts as device time, about 36 us per region).
    Then K more calls, each bracketed by its own events, for the per-call (kernel) time.
    Returns (ms per step over the region, mean ms per call from per-call events)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    dist.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(400_000)  # cycles (~0.2 ms); outside the timed region
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    region = start.elapsed_time(end) / steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda._sleep(400_000)
    for i in range(steps):
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    per_call = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return region, per_call


# GB300 datasheet figures (nominal, per GPU): HBM3e bandwidth and dense bf16 tensor throughput.
# The roofline's `frac` is against the measured copy bandwidth / cuBLAS throughput of
# MEASURED_PEAKS.json; `frac_of_datasheet` is the same achieved figure against these.
DATASHEET = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}
# fp32 FMA on the CUDA cores: 152 SMs x 128 fp32 lanes x 2 flops x 2,070 MHz (the maximum SM clock)
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def roofline(bytes_, flops, secs, peaks, bound="hbm"):
    if bound == "hbm":
        ach = bytes_ / secs / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": None,
                "peak_source": peaks["source"] + " copy bandwidth",
                "frac_of_datasheet": round(ach / DATASHEET["hbm_gbs"], 4),
                "datasheet_peak": DATASHEET["hbm_gbs"],
                "algorithmic_bytes": int(bytes_), "flops": int(flops),
                "tensor_frac": round(flops / secs / 1e12 / peaks["bf16_tflops"], 4)}
    ach = flops / secs / 1e12
    if bound == "alu":
        return {"bound": "alu", "achieved": round(ach, 2), "peak": round(FP32_ALU_TFLOPS, 2), "unit": "TFLOP/s",
                "frac": round(ach / FP32_ALU_TFLOPS, 4), "traffic": None,
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2,070 MHz",
                "algorithmic_bytes": int(bytes_), "flops": int(flops),
                "hbm_frac": round(bytes_ / secs / 1e9 / peaks["hbm_gbs"], 4)}
    return {"bound": "tensor", "achieved": round(ach, 2), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4), "traffic": None,
            "frac_of_datasheet": round(ach / DATASHEET["bf16_tflops"], 4),
            "datasheet_peak": DATASHEET["bf16_tflops"]}


def bwd_bytes(tokens, n_seq):
    """q, k, v, dO read and dq, dk, dv written once each (bf16), plus dhT read and dh0 written."""
    return tokens * H * (4 * DK + 3 * DV) * 2 + 2 * n_seq * H * DK * DV * 4


def fwd_bytes(tokens, n_seq, with_h0):
    io = tokens * H * (2 * DK * 2 + 2 * DV * 2)
    return io + n_seq * H * DK * DV * 4 * (2 if with_h0 else 1)


def fwd_flops(tokens):
    return tokens * H * 2 * (128 * DK + 128 * DV + 2 * DK * DV)


# ------------------------------------------------------------------------------------------
# rows
# ------------------------------------------------------------------------------------------
def bench_fwd(torch, gla, wl, dist, args, peaks):
    w = wl.layer()
    g = w.device_inputs()
    o = torch.empty_like(g["v"])
    hT = torch.empty((w.n_seq, H, DK, DV), dtype=torch.float32, device="cuda")
    fn = lambda: gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], w.scale, o=o, hT=hT)
    region, per_call = timed(torch, dist, fn, args.steps, args.warmup)
    region = dist.max(region)
    per_call = dist.max(per_call)
    tokens = w.tokens
    res = {
        "workload": w.name, "tokens": tokens, "ms_per_step": region,
        "value": tokens * dist.world / (region / 1e3),
        "roofline": roofline(fwd_bytes(tokens, w.n_seq, False), fwd_flops(tokens), region / 1e3,
                             peaks),
        "kernel_ms": per_call, "launches_per_step": 1,
    }
    res["roofline"]["traffic"] = profiled_traffic("fwd")
    # e2e through the C ABI with host buffers (gla_chunk_fwd_host): every step copies q, k, v in
    # from pinned host memory and o, hT back out, inside the library, pipelined with the compute
    # over pieces of the batch (sub-batches of whole sequences, or with more pieces than
    # sequences, parts of each sequence cut at chunk boundaries and chained through the state);
    # the step's region covers all of it.
    hq, hk, hv = (x.cpu().pin_memory() for x in (g["q"], g["k"], g["v"]))
    ho, hh = torch.empty_like(o, device="cpu").pin_memory(), torch.empty_like(hT, device="cpu").pin_memory()
    B_, T_, H_ = g["q"].shape[:3]
    ws_host = torch.empty(gla.gla_chunk_fwd_host_workspace_bytes(B_, T_, H_, 0), dtype=torch.uint8, device="cuda")
    pieces = max(1, args.e2e_parts)

    def e2e():
        gla.gla_chunk_fwd_host(hq, hk, hv, g["log_lambda"], w.scale, o=ho, hT=hh, pieces=pieces, workspace=ws_host)
    e_region, _ = timed(torch, dist, e2e, args.steps, args.warmup)
    e_region = dist.max(e_region)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hh.numel() * hh.element_size()
    res["e2e"] = {"value": tokens * dist.world / (e_region / 1e3), "unit": "tokens/s",
                  "ms_per_step": e_region, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                  "call": "gla_chunk_fwd_host (pinned host q, k, v in; o, hT out)",
                  "pipeline": f"{pieces} pieces: host-to-device copies, forward and device-to-host copies "
                              f"overlapped on three streams inside the library"}
    # the pipelined results are the plain call's results
    ref_o, ref_h = o.clone(), hT.clone()
    gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], w.scale, o=ref_o, hT=ref_h)
    torch.cuda.synchronize()
    res["e2e"]["matches_device_call"] = bool(torch.equal(ho, ref_o.cpu()) and torch.equal(hh, ref_h.cpu()))
    del g, o, hT, hq, hk, hv, ho, hh, ws_host
    return res


def bench_fwd_fp32(torch, gla, wl, dist, args, peaks):
    """The all-fp32 mode's forward (fp32 q, k, v, o; the CUDA-core kernels that serve the 1e-4
    accuracy bar) on the forward workload's shapes.  Its bytes: fp32 q, k, v in and o out (twice
    the bf16 path's) plus hT."""
    w = wl.layer()
    g = w.device_inputs()
    q, k, v = (g[x].float() for x in ("q", "k", "v"))
    del g["q"], g["k"], g["v"]
    o = torch.empty_like(v)
    hT = torch.empty((w.n_seq, H, DK, DV), dtype=torch.float32, device="cuda")
    fn = lambda: gla.gla_chunk_fwd(q, k, v, g["log_lambda"], w.scale, o=o, hT=hT)
    region, per_call = timed(torch, dist, fn, max(3, args.steps // 4), args.warmup)
    region, per_call = dist.max(region), dist.max(per_call)
    tokens = w.tokens
    byts = tokens * H * (2 * DK * 4 + 2 * DV * 4) + w.n_seq * H * DK * DV * 4
    res = {"workload": w.name.replace("bf16", "fp32") + " (all-fp32 mode)", "tokens": tokens, "ms_per_step": region,
           "value": tokens * dist.world / (region / 1e3), "unit": "tokens/s",
           "roofline": roofline(byts, fwd_flops(tokens), region / 1e3, peaks, bound="alu"), "kernel_ms": per_call,
           "launches_per_step": 1}
    res["roofline"]["traffic"] = profiled_traffic("fwd_fp32")
    del g, q, k, v, o, hT
    return res


def bench_fwd_aug(torch, gla, wl, dist, args, peaks):
    """The forward with the self-augmentation step (gla_chunk_fwd_aug) on the same workload;
    aug_balance ~ N(0, 10^2) spreads the gate over the sigmoid (q, k ~ N(0, 1/96))."""
    import glasynth as gs
    w = wl.layer()
    g = w.device_inputs()
    aug = torch.from_numpy(gs.normal(11, 9, (H, DK), 10.0)).cuda()
    o = torch.empty_like(g["v"])
    hT = torch.empty((w.n_seq, H, DK, DV), dtype=torch.float32, device="cuda")
    fn = lambda: gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], w.scale, o=o, hT=hT,
                                   aug=aug)
    region, per_call = timed(torch, dist, fn, args.steps, args.warmup)
    region, per_call = dist.max(region), dist.max(per_call)
    tokens = w.tokens
    res = {"workload": w.name + " + self-augmentation", "tokens": tokens, "ms_per_step": region,
           "value": tokens * dist.world / (region / 1e3), "unit": "tokens/s",
           "roofline": roofline(fwd_bytes(tokens, w.n_seq, False) + H * DK * 4,
                                fwd_flops(tokens) + tokens * H * 2 * (DK + DV), region / 1e3, peaks),
           "kernel_ms": per_call, "launches_per_step": 1}
    res["roofline"]["traffic"] = profiled_traffic("fwd_aug")
    del g, o, hT, aug
    return res


def bench_norm_gate(torch, gla, wl, dist, args, peaks):
    """Per-tier Head RMSNorm + SiLU gate (gla_head_norm_gate) on the forward workload's output
    shape: o and g [8 x 2048, 16, 192] bf16 read once, y written once; four tiers of four heads."""
    import glasynth as gs
    w = wl.layer()
    rows = w.tokens
    o = torch.from_numpy(gs.normal(13, 1, (rows, H, DV))).cuda().to(torch.bfloat16)
    g = torch.from_numpy(gs.normal(13, 2, (rows, H, DV), 2.0)).cuda().to(torch.bfloat16)
    wt = (1.0 + torch.from_numpy(gs.normal(13, 3, (4, DV), 0.3))).cuda()
    tier = (torch.arange(H, dtype=torch.int32) // 4).cuda()
    y = torch.empty_like(o)
    fn = lambda: gla.gla_head_norm_gate(o, g, wt, tier, y=y)
    region, per_call = timed(torch, dist, fn, args.steps, args.warmup)
    region, per_call = dist.max(region), dist.max(per_call)
    byts = 3 * rows * H * DV * 2 + 4 * DV * 4 + H * 4
    res = {"workload": "head RMSNorm + SiLU gate, 16,384 rows x 16 heads x 192 bf16, 4 tiers",
           "tokens": rows, "ms_per_step": region, "value": rows * dist.world / (region / 1e3),
           "unit": "tokens/s", "roofline": roofline(byts, rows * H * DV * 8, region / 1e3, peaks),
           "kernel_ms": per_call, "launches_per_step": 1}
    res["roofline"]["traffic"] = profiled_traffic("norm_gate")
    del o, g, wt, tier, y
    return res


def bench_fwd_split(torch, gla, wl, dist, args, peaks):
    """One long sequence (131,072 tokens, H=16, bf16): the sequence-split forward
    (gla_chunk_fwd_split, segment length chosen by the library) against the plain packed forward,
    whose 48 units (16 heads x 3 d_v tiles) each run 1,024 chunks on one SM."""
    import glasynth as gs
    T = 131072
    q = torch.from_numpy(gs.normal(14, 1, (T, H, DK), DK ** -0.5)).cuda().to(torch.bfloat16)
    k = torch.from_numpy(gs.normal(14, 2, (T, H, DK), DK ** -0.5)).cuda().to(torch.bfloat16)
    v = torch.from_numpy(gs.normal(14, 3, (T, H, DV))).cuda().to(torch.bfloat16)
    ll = torch.from_numpy(gs.laplace_log_lambda(H)).cuda()
    o = torch.empty_like(v)
    hT = torch.empty((1, H, DK, DV), dtype=torch.float32, device="cuda")
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    ws_plain = torch.empty(gla.gla_workspace_bytes(1, H), dtype=torch.uint8, device="cuda")
    scale = DK ** -0.5
    plain = lambda: gla.gla_chunk_fwd(q, k, v, ll, scale, cu_seqlens=cu, o=o, hT=hT, workspace=ws_plain)
    p_region, _ = timed(torch, dist, plain, max(3, args.steps // 4), args.warmup)
    import numpy as np
    cu_h = np.array([0, T], np.int32)
    seg = gla.gla_split_choose_seg_chunks([T], H)
    ws = torch.empty(gla.load_library().gla_split_workspace_bytes(cu_h.ctypes.data_as(__import__("ctypes").c_void_p),
                                                                  1, H, 0), dtype=torch.uint8, device="cuda")
    split = lambda: gla.gla_chunk_fwd_split(q, k, v, ll, [T], seg_chunks=0, scale=scale, o=o, hT=hT,
                                            workspace=ws)
    region, per_call = timed(torch, dist, split, max(3, args.steps // 4), args.warmup)
    region, p_region = dist.max(region), dist.max(p_region)
    res = {"workload": f"one sequence of 131,072 tokens, H=16, bf16, {seg}-chunk segments (seg_chunks=0)",
           "tokens": T, "seg_chunks": seg,
           "ms_per_step": region, "value": T * dist.world / (region / 1e3), "unit": "tokens/s",
           "plain_forward_ms": p_region,
           "roofline": roofline(fwd_bytes(T, 1, False), fwd_flops(T), region / 1e3, peaks),
           "launches_per_step": 5}
    del q, k, v, o, hT, ws, ws_plain
    return res


def bench_varlen(torch, gla, wl, dist, args, peaks):
    w = wl.varlen()
    g = w.device_inputs()
    o = torch.empty_like(g["v"])
    hT = torch.empty((w.n_seq, H, DK, DV), dtype=torch.float32, device="cuda")
    ws = torch.empty(gla.gla_workspace_bytes(w.n_seq, H), dtype=torch.uint8, device="cuda")
    fn = lambda: gla.gla_chunk_fwd(g["q"], g["k"], g["v"], g["log_lambda"], w.scale, h0=g["h0"],
                                   cu_seqlens=g["cu_seqlens"], o=o, hT=hT, workspace=ws)
    region, per_call = timed(torch, dist, fn, args.steps, args.warmup)
    region, per_call = dist.max(region), dist.max(per_call)
    res = {"workload": w.name, "tokens": w.tokens, "ms_per_step": region,
           "value": w.tokens * dist.world / (region / 1e3), "unit": "tokens/s",
           "roofline": roofline(fwd_bytes(w.tokens, w.n_seq, True), fwd_flops(w.tokens),
                                region / 1e3, peaks),
           "launches_per_step": 2}
    del g, o, hT
    return res


def bench_bwd(torch, gla, wl, dist, args, peaks):
    w = wl.layer(with_grad=True)
    g = w.device_inputs()
    fn = lambda: gla.gla_chunk_bwd(g["q"], g["k"], g["v"], g["log_lambda"], g["dO"], w.scale,
                                   dhT=g["dhT"])
    region, per_call = timed(torch, dist, fn, args.steps, args.warmup)
    region, per_call = dist.max(region), dist.max(per_call)
    tokens = w.tokens
    byts = bwd_bytes(tokens, w.n_seq)
    flops = tokens * H * 2 * (128 * DV + 128 * DK + 2 * DK * DV      # dq scan
                              + 128 * DV + 128 * DK + 128 * DK + 128 * DV + 4 * DK * DV)  # dk, dv scan
    res = {"workload": w.name, "tokens": tokens, "ms_per_step": region,
           "value": tokens * dist.world / (region / 1e3), "unit": "tokens/s",
           "roofline": roofline(byts, flops, region / 1e3, peaks), "launches_per_step": 5}
    del g
    return res


def bench_bwd_fp32(torch, gla, wl, dist, args, peaks):
    """The all-fp32 mode's backward (the CUDA-core scans) on the backward workload's shapes, with
    fp32 q, k, v, dO and gradients."""
    w = wl.layer(with_grad=True)
    g = w.device_inputs()
    q, k, v, dO = (g[x].float() for x in ("q", "k", "v", "dO"))
    for x in ("q", "k", "v", "dO"):
        del g[x]
    fn = lambda: gla.gla_chunk_bwd(q, k, v, g["log_lambda"], dO, w.scale, dhT=g["dhT"])
    region, per_call = timed(torch, dist, fn, max(3, args.steps // 4), args.warmup)
    region, per_call = dist.max(region), dist.max(per_call)
    tokens = w.tokens
    byts = 2 * bwd_bytes(tokens, w.n_seq) - 2 * w.n_seq * H * DK * DV * 4  # fp32 rows, the states as before
    flops = tokens * H * 2 * (128 * DV + 128 * DK + 2 * DK * DV + 128 * DV + 128 * DK + 128 * DK + 128 * DV
                              + 4 * DK * DV)
    res = {"workload": w.name.replace("bf16", "fp32") + " (all-fp32 mode)", "tokens": tokens, "ms_per_step": region,
           "value": tokens * dist.world / (region / 1e3), "unit": "tokens/s",
           "roofline": roofline(byts, flops, region / 1e3, peaks, bound="alu"), "launches_per_step": 3}
    res["roofline"]["traffic"] = profiled_traffic("bwd_fp32")
    del g, q, k, v, dO
    return res


def bench_decode(torch, gla, wl, dist, args, peaks, aug=False, bf16_state=False, norm_gate=False):
    """``aug``: the step with the self-augmentation copy of v (gla_decode_step_aug), 16 steps;
    ``bf16_state``: the same pool stored in bf16 (gla_decode_step_bf16_state), 16 steps;
    ``norm_gate``: the step with the per-tier Head RMSNorm + SiLU gate fused into its epilogue
    (gla_decode_step_norm_gate: y instead of o, a gate stream g per step, four tiers of four
    heads), 16 steps."""
    import glasynth as gs
    w = wl.DecodeWorkload(seqs=args.decode_seqs, layers=args.decode_layers)
    state = w.device_state()
    if bf16_state:
        state = state.to(torch.bfloat16)
    ll = torch.from_numpy(w.log_lambda).cuda()
    a = torch.from_numpy(gs.normal(12, 9, (H, DK), 10.0)).cuda() if aug else None
    steps = [w.device_step(s) for s in range(min(w.steps, 4))]  # 4 distinct token sets, cycled
    o = torch.empty((w.N, H, DV), dtype=torch.bfloat16, device="cuda")
    it = [0]
    if norm_gate:
        from glasynth.device import normal as dnormal
        gs_ = [dnormal((w.N, H, DV), 12, 40 + i, 2.0) for i in range(len(steps))]
        wt = (1.0 + torch.from_numpy(gs.normal(12, 41, (4, DV), 0.3))).cuda()
        tier = (torch.arange(H, dtype=torch.int32) // 4).cuda()

    def fn():
        i = it[0] % len(steps)
        b = steps[i]
        it[0] += 1
        if norm_gate:
            gla.gla_decode_step_norm_gate(b["q"], b["k"], b["v"], ll, state, gs_[i], wt, tier, scale=w.scale,
                                          y=o)
        else:
            gla.gla_decode_step(b["q"], b["k"], b["v"], ll, state, w.scale, o=o, aug=a)
    n = 16 if (aug or bf16_state or norm_gate) else w.steps
    region, per_call = timed(torch, dist, fn, n, max(args.warmup, 3))
    region, per_call = dist.max(region), dist.max(per_call)
    state_bytes = 2 * w.N * H * DK * DV * (2 if bf16_state else 4)
    io_bytes = w.N * H * (2 * DK * 2 + 2 * DV * 2)
    res = {"workload": f"decode {w.seqs} seqs x {w.layers} layers H=16 "
                       + ("bf16" if bf16_state else "fp32") + " state bf16 io"
                       + (" + self-augmentation" if aug else "")
                       + (" + fused head RMSNorm/SiLU gate (y out)" if norm_gate else ""), "steps": n,
           "ms_per_step": region,
           "value": w.seqs * dist.world / (region / 1e3), "unit": "tokens/s",
           "token": "one new token per sequence through all 24 layers",
           "roofline": roofline(state_bytes, 2 * 2 * w.N * H * DK * DV, region / 1e3, peaks),
           "io_bytes_outside_roofline": io_bytes, "launches_per_step": 1}
    res["roofline"]["algorithmic_bytes_note"] = ("bf16" if bf16_state else "fp32") + " state read + write per step"
    if norm_gate:
        res["io_bytes_outside_roofline"] += w.N * H * DV * 2
    row = "decode_bf16_state" if bf16_state else "decode_norm_gate" if norm_gate else "decode"
    res["roofline"]["traffic"] = None if aug else profiled_traffic(row, w.N * H)
    del state, steps, o, a
    return res


def bench_decode_mxfp8(torch, gla, wl, dist, args, peaks):
    """The decode step on the same pool stored as MXFP8 (gla_decode_step_mxfp8_state: E4M3 codes
    plus one E8M0 scale per 32 values, 19,008 bytes per state against 73,728 in fp32), built on
    the device from the pool's fp32 states (2,048 pool rows at a time); 16 steps."""
    from glasynth import TID
    from glasynth.device import normal as dnormal
    w = wl.DecodeWorkload(seqs=args.decode_seqs, layers=args.decode_layers)
    codes = torch.empty((w.N, H, DK, DV), dtype=torch.uint8, device="cuda")
    scales = torch.empty((w.N, H, DK, DV // 32), dtype=torch.uint8, device="cuda")
    for r0 in range(0, w.N, 2048):
        r1 = min(w.N, r0 + 2048)
        x = dnormal((r1 - r0, H, DK, DV), w.seed, TID["state"], w.state_sigma, torch.float32,
                    start=r0 * H * DK * DV)
        gla.gla_state_to_mxfp8(x, codes[r0:r1], scales[r0:r1])
        del x
    ll = torch.from_numpy(w.log_lambda).cuda()
    steps = [w.device_step(s) for s in range(4)]
    o = torch.empty((w.N, H, DV), dtype=torch.bfloat16, device="cuda")
    it = [0]

    def fn():
        b = steps[it[0] % len(steps)]
        it[0] += 1
        gla.gla_decode_step_mxfp8_state(b["q"], b["k"], b["v"], ll, codes, scales, w.scale, o=o)
    n = 16
    region, per_call = timed(torch, dist, fn, n, max(args.warmup, 3))
    region, per_call = dist.max(region), dist.max(per_call)
    state_bytes = 2 * w.N * H * (DK * DV + DK * DV // 32)
    res = {"workload": f"decode {w.seqs} seqs x {w.layers} layers H=16 MXFP8 state bf16 io", "steps": n,
           "ms_per_step": region, "value": w.seqs * dist.world / (region / 1e3), "unit": "tokens/s",
           "token": "one new token per sequence through all 24 layers",
           "roofline": roofline(state_bytes, 2 * 2 * w.N * H * DK * DV, region / 1e3, peaks),
           "io_bytes_outside_roofline": w.N * H * (2 * DK * 2 + 2 * DV * 2), "launches_per_step": 1}
    res["roofline"]["algorithmic_bytes_note"] = "MXFP8 state (codes + scales) read + write per step"
    res["roofline"]["traffic"] = profiled_traffic("decode_mxfp8_state", w.N * H)
    del codes, scales, steps, o
    return res


def cpu_baseline_fwd(seconds_budget=10.0):
    """The oracle as it stands on the host cores: whole sequences of the B=8, T=2048, H=16
    workload (all 16 heads each), cycling over the 8 sequences until about `seconds_budget` of
    oracle time has been spent."""
    import numpy as np

    import oracle
    from glasynth import workloads as wl
    oracle.build()
    w = wl.layer()
    cores = oracle.hardware_threads()
    done_tokens, t_total, seqs = 0, 0.0, 0
    inputs = {}
    while t_total < seconds_budget and seqs < 512:
        n = seqs % w.n_seq
        if n not in inputs:
            units = [w.host_unit(n, h) for h in range(H)]
            inputs[n] = tuple(np.concatenate([u[x] for u in units], axis=1) for x in ("q", "k", "v"))
        q, k, v = inputs[n]
        t0 = time.perf_counter()
        oracle.fwd(q, k, v, w.log_lambda, w.scale, nthreads=0)
        t_total += time.perf_counter() - t0
        done_tokens += w.lengths[n]
        seqs += 1
    return {"value": done_tokens / t_total, "unit": "tokens/s", "cores": min(cores, H),
            "kind": "oracle",
            "sample": f"{seqs} sequence passes (T=2048, all 16 heads; cycling over the 8 sequences) "
                      f"of the B=8 T=2048 H=16 forward workload, fp64 per-token recurrence, "
                      f"{min(cores, H)} threads (one per head), {t_total:.1f} s of oracle time"}


def run_reference(args):
    """`--impl reference`: the fp64 oracle timed on the host cores, one sequence per step."""
    import numpy as np

    import oracle
    from glasynth import workloads as wl
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    oracle.build()
    w = wl.layer()
    units = [w.host_unit(0, h) for h in range(H)]
    q = np.concatenate([u["q"] for u in units], axis=1)
    k = np.concatenate([u["k"] for u in units], axis=1)
    v = np.concatenate([u["v"] for u in units], axis=1)
    step = lambda: oracle.fwd(q, k, v, w.log_lambda, w.scale, nthreads=0)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    cores = min(oracle.hardware_threads(), H)
    value = w.lengths[0] / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": 8, "T": 2048, "H": H, "dk": DK, "dv": DV,
                       "sample_per_step": "sequence 0 (2048 tokens, 16 heads)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "one T=2048 sequence (16 heads) of the B=8 workload per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def free_port():
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_ranks(args):
    """`--gpus N` without a launcher around it: run this script as N ranks, one per GPU, under
    torch.distributed.run on 127.0.0.1 (the same command line a scaling driver uses).  Returns
    the launcher's exit status, or None when this process is already a rank (or N = 1)."""
    world = os.environ.get("WORLD_SIZE")
    if world is not None:
        if int(world) != args.gpus:
            raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}: the launcher and "
                             f"the flag disagree on the number of ranks")
        return None
    if args.gpus <= 1:
        return None
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           f"--master-port={free_port()}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def run_launcher_check(args):
    """`--launcher-check`: exercises the rank launch, the barrier and the max-over-ranks timing on
    CPU ranks (gloo) with no GPU and no GLA work; prints a line that says so (no metric value).
    Used by the CPU tests of the multi-rank path."""
    import torch
    dist = Dist(torch)
    dist.init("gloo")
    dist.barrier()
    t0 = time.perf_counter()
    time.sleep(0.001 * (dist.rank + 1))
    dist.barrier()
    secs = dist.max(time.perf_counter() - t0)
    if dist.rank == 0:
        print(json.dumps({"launcher_check": True, "n_gpus": dist.world, "value": None,
                          "max_rank_seconds": secs}), flush=True)
    dist.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--rows", default="fwd,bwd,varlen,decode,fwd_aug,norm_gate,decode_aug,decode_bf16_state,"
                    "fwd_split,decode_norm_gate,decode_mxfp8_state,fwd_fp32,bwd_fp32")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-seqs", type=int, default=1280,
                    help="sequences in the decode pool (1280 = the measured workload)")
    ap.add_argument("--decode-layers", type=int, default=24)
    ap.add_argument("--e2e-parts", type=int, default=8,
                    help="pieces of the e2e pipeline (copies overlapped with compute); more pieces than "
                         "sequences cut each sequence at chunk boundaries")
    ap.add_argument("--launcher-check", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)
    rc = launch_ranks(args)
    if rc is not None:
        return rc
    if args.launcher_check:
        return run_launcher_check(args)

    import torch

    import linear_attention_recurrence_simple_gb300 as gla
    from glasynth import workloads as wl
    dist = Dist(torch)
    torch.cuda.set_device(dist.local)
    dist.init("nccl")
    gla.load_library()
    peaks = load_peaks()
    rows = args.rows.split(",")
    out = {}
    sampler = ClockSampler(gpu_id_for_smi(torch))
    with sampler:
        if "fwd" in rows:
            out["fwd"] = bench_fwd(torch, gla, wl, dist, args, peaks)
        if "varlen" in rows:
            out["varlen"] = bench_varlen(torch, gla, wl, dist, args, peaks)
        if "bwd" in rows:
            out["bwd"] = bench_bwd(torch, gla, wl, dist, args, peaks)
        if "decode" in rows:
            out["decode"] = bench_decode(torch, gla, wl, dist, args, peaks)
        if "fwd_aug" in rows:
            out["fwd_aug"] = bench_fwd_aug(torch, gla, wl, dist, args, peaks)
        if "fwd_fp32" in rows:
            out["fwd_fp32"] = bench_fwd_fp32(torch, gla, wl, dist, args, peaks)
        if "bwd_fp32" in rows:
            out["bwd_fp32"] = bench_bwd_fp32(torch, gla, wl, dist, args, peaks)
        if "fwd_split" in rows:
            out["fwd_split"] = bench_fwd_split(torch, gla, wl, dist, args, peaks)
        if "norm_gate" in rows:
            out["norm_gate"] = bench_norm_gate(torch, gla, wl, dist, args, peaks)
        if "decode_aug" in rows:
            out["decode_aug"] = bench_decode(torch, gla, wl, dist, args, peaks, aug=True)
        if "decode_bf16_state" in rows:
            out["decode_bf16_state"] = bench_decode(torch, gla, wl, dist, args, peaks, bf16_state=True)
        if "decode_norm_gate" in rows:
            out["decode_norm_gate"] = bench_decode(torch, gla, wl, dist, args, peaks, norm_gate=True)
        if "decode_mxfp8_state" in rows:
            out["decode_mxfp8_state"] = bench_decode_mxfp8(torch, gla, wl, dist, args, peaks)
    err = gla.gla_get_device_error()
    clocks = sampler.summary()
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_fwd()
    if dist.rank == 0:
        f = out.get("fwd", {})
        line = {
            "metric": METRIC, "value": f.get("value"), "unit": "tokens/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": f.get("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded SplitMix64 / Box-Muller normal inputs, no dataset",
            "config": {"workload": f.get("workload"), "B": 8, "T": 2048, "H": H, "dk": DK, "dv": DV,
                       "chunk": 128, "accumulate": "fp32 state and accumulation",
                       "l2": "no flush: inputs of each call (201 MB) exceed the 129 MB L2",
                       "parallelism": f"replicas x{dist.world} (no collective)"},
            "roofline": f.get("roofline"), "e2e": f.get("e2e"),
            "gpu_launches": args.steps * f.get("launches_per_step", 1),
            "clocks": clocks, "cpu_baseline": cpu, "device_error": err,
            "rows": {k: v for k, v in out.items() if k != "fwd"},
        }
        # one compact entry per row, last on the line (ms per step, tokens/s, bytes counted,
        # fraction of the measured peak and of the datasheet peak)
        line["rows_summary"] = {
            k: {"ms": round(v["ms_per_step"], 4), "tok_s": round(v["value"], 1),
                "bytes": v["roofline"].get("algorithmic_bytes"), "frac": v["roofline"]["frac"],
                "frac_ds": v["roofline"].get("frac_of_datasheet")}
            for k, v in out.items()}
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
