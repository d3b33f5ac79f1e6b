#!/usr/bin/env python
"""Benchmark of the AWQ hot path on B300.

Workload (default): LLaMA-7B-shaped decode at M = 1 over the four
projections (fused qkv 12288x4096, o 4096x4096, fused gate+up 22016x4096,
down 4096x11008), fp16 weights ~ N(0, 0.02^2), activations ~ N(0,1) with 1%
of input channels x20, quantised to INT4 g128 by the AWQ search on 512
calibration tokens.  One step = the whole hot path on every projection:
act_stats -> act_mean -> search_scale (20 alphas) -> pack_int4 ->
repack_int4 (contiguous decode tiles), then an L2 flush, then the M = 1
decode matmul (w4a16_gemm_repacked) on every projection.

Headline ``value``: W4A16 GEMV HBM GB/s at M = 1, i.e. the algorithmic bytes
of the four decode matmuls (packed weights + scales/zeros + x + y) over
their CUDA-event time inside the timed steps.  ``ms_per_step`` is the whole
step.  ``roofline`` is for the dominant kernel of the step (the fused search
GEMM), ``roofline_gemv`` for the headline kernel.

``--impl reference`` times the CPU oracle on a bounded sample of the same
workload (the oracle is the reference implementation of this method here).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthgen as sg  # noqa: E402

METRIC = "W4A16 GEMV HBM GB/s (M=1) & GEMM TFLOP/s (M≥256), % of B300 roofline"
T_CAL = 512
N_ALPHA = 20
FLUSH_BYTES = 512 << 20          # > 4x the 126 MB L2
WORKLOAD = ("LLaMA-7B-shaped decode GEMV, M=1, projections qkv 12288x4096, o 4096x4096, "
            "gate_up 22016x4096, down 4096x11008; W ~ N(0,0.02^2) fp16, X ~ N(0,1) with 1% "
            "channels x20; INT4 g128 via AWQ search (20 alphas) on 512 calibration tokens")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# DRAM traffic of the fused search kernel, dram__bytes_read.sum +
# dram__bytes_write.sum summed over the four search launches of one step of
# this workload in one ncu capture, valid only while the kernel's sources (comments aside) are the ones
# captured.
SEARCH_TRAFFIC = {"bytes_per_step": 105576192 + 2854912 + 38526976 + 0 + 185360640 + 505344 +
                                    103335680 + 136704,
                  "src_sha": "640cf6c14483b9d7"}
SEARCH_SOURCES = ("tc.cu", "common.cuh", "kernels.cuh")


def gemv_bytes(N, K, M=1):
    return N * K // 2 + 4 * N * (K // 128) + 2 * M * K + 2 * M * N


def search_flop(N, K, T=T_CAL, n_alpha=N_ALPHA):
    return 2.0 * T * N * K * n_alpha


def search_flop_t(N, K, T=128 * 512, n_alpha=N_ALPHA):
    return 2.0 * T * N * K * n_alpha


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def strip_comments(text):
    """C/C++/CUDA source without its comments, trailing blanks and empty
    lines: the part of a kernel's source that its counters depend on.
    String and character literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
        elif text.startswith("/*", i):
            end = text.find("*/", i + 2)
            i = n if end < 0 else end + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def src_sha(names):
    """Hash of the named kernel sources, comments and layout excluded."""
    import hashlib
    h = hashlib.sha256()
    for name in names:
        path = os.path.join(ROOT, "weight_only_bit_stats_b300", "csrc", name)
        h.update(strip_comments(open(path).read()).encode())
    return h.hexdigest()[:16]


# ------------------------------------------------------------ multi-rank --

def rank_layer(rank):
    """Weak scaling across GPUs: rank r quantises and runs decoder layer r of
    the workload (every layer's statistics, search, pack and matmuls are
    independent), so the data path has no collective."""
    return rank


def max_over_ranks(values, device):
    """Each timing's maximum over all ranks (one all-reduce of the timings,
    outside the timed region); the values themselves on a single rank."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_value(bytes_per_rank_step, steps, max_ms, world):
    """Whole-job GB/s: the bytes all ranks processed over the slowest rank's
    time."""
    return world * bytes_per_rank_step * steps / (max_ms * 1e-3) / 1e9


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            except ValueError:
                continue
            rows.append((ts, parts))
        os.unlink(self.f.name)
        sel = [p for ts, p in rows if self.t0 - 1 <= ts <= self.t1 + 1] or [p for _, p in rows]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(p[2]) for p in sel if p[2].replace(".", "").isdigit()]
        mx = [float(p[3]) for p in sel if p[3].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in sel:
            for n, v in zip(names, p[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sel)}


# ------------------------------------------------------------- GPU arm ----

def run_ours(args, rank, world):
    import torch
    import weight_only_bit_stats_b300 as wb

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    layer = rank_layer(rank)
    projs = []
    for j, (name, N, K) in enumerate(sg.LLAMA7B_DECODE_PROJ):
        W, Xc, Xm, _ = sg.layer_inputs(layer, j, N, K, T_CAL, M=1)
        projs.append(dict(name=name, N=N, K=K, W_h=W, Xc_h=Xc, x_h=Xm))
    for p in projs:
        N, K = p["N"], p["K"]
        p["W"] = torch.from_numpy(p["W_h"]).to(dev)
        p["Xc"] = torch.from_numpy(p["Xc_h"]).to(dev)
        p["x"] = torch.from_numpy(p["x_h"]).to(dev)
        p["abs"] = torch.empty(K, dtype=torch.int64, device=dev)
        p["mean"] = torch.empty(K, dtype=torch.float64, device=dev)
        p["s"] = torch.empty(K, dtype=torch.float32, device=dev)
        p["mse"] = torch.empty(N_ALPHA, dtype=torch.float64, device=dev)
        p["best"] = torch.empty(1, dtype=torch.int32, device=dev)
        p["ws"] = wb.search_workspace(N, K, T_CAL, N_ALPHA, dev)
        p["cand"] = torch.empty((N_ALPHA, K), dtype=torch.float32, device=dev)
        p["cws"] = torch.empty(max(16, wb.lib().awq_candidate_scales_workspace_size(K, N_ALPHA)),
                               dtype=torch.uint8, device=dev)
        p["qw"] = torch.empty((N, K // 8), dtype=torch.int32, device=dev)
        p["sc"] = torch.empty((N, K // 128), dtype=torch.float16, device=dev)
        p["ze"] = torch.empty((N, K // 128), dtype=torch.float16, device=dev)
        p["y"] = torch.empty((1, N), dtype=torch.float16, device=dev)
        p["tiles"] = torch.empty(wb.lib().awq_repack_int4_bytes(N, K), dtype=torch.uint8,
                                 device=dev)
    # Decode matmuls may fetch their packed weights before the previous kernel
    # in the stream completes: in this step the first decode launch follows
    # the L2 flush kernels and each other one follows a decode launch (in the
    # e2e step the first follows the pack of another projection), so no
    # matmul's weights are written by the kernel just before it.
    wb.set_weight_prefetch(True)
    flush_w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)  # noqa: F841
    fence = torch.empty(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    E = lambda: torch.cuda.Event(enable_timing=True)

    def step(ev=None, evc=None):
        for i, p in enumerate(projs):
            if ev: ev[i][0].record(stream)
            wb.act_stats(p["Xc"], out=p["abs"])
            if ev: ev[i][1].record(stream)
            wb.act_mean(p["abs"], T_CAL, out=p["mean"])
            if ev: ev[i][2].record(stream)
            # the search as its two steps: the candidate scales, then the
            # search kernel on them (together what awq_search_scale runs;
            # the events between them time the search kernel's call alone)
            wb.candidate_scales(p["mean"], out=p["cand"], workspace=p["cws"])
            if evc: evc[i].record(stream)
            wb.search_mse(p["W"], p["Xc"], p["cand"], workspace=p["ws"],
                          out=(p["s"], p["mse"], p["best"]))
            if ev: ev[i][3].record(stream)
            wb.pack_int4(p["W"], p["s"], out=(p["qw"], p["sc"], p["ze"]))
            wb.repack_int4(p["qw"], p["sc"], p["ze"], out=p["tiles"])
            if ev: ev[i][4].record(stream)
        # L2 flush: write a buffer larger than L2, then read another one so the
        # cache holds clean lines when the decode matmuls start
        flush_w.fill_(1.0)
        torch.sum(flush_r, dim=0, out=flush_out)
        if ev: ev[4][0].record(stream)
        # a one-element kernel after the opening event: decode launches may
        # start early beside the kernel before them (programmatic dependent
        # launch), and this keeps any of their work out of the flush, i.e.
        # inside the timed segment
        fence.zero_()
        for p in projs:
            wb.w4a16_gemm_repacked(p["x"], p["tiles"], p["N"], out=p["y"])
        if ev: ev[4][1].record(stream)

    for _ in range(args.warmup):
        step()
    wb.sync_status()
    torch.cuda.synchronize()

    sampler = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.3)
    evs = [[[E() for _ in range(5)] for _ in range(5)] for _ in range(args.steps)]
    evcs = [[E() for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = E(), E()
    if sampler: sampler.mark_start()
    t_start.record(stream)
    for k in range(args.steps):
        step(evs[k], evcs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    if sampler: sampler.mark_end()
    if world > 1:
        dist.barrier()
    wb.sync_status()
    total_ms = t_start.elapsed_time(t_end)
    st = {"stats": 0.0, "mean": 0.0, "candidates": 0.0, "search": 0.0, "pack": 0.0,
          "flush": 0.0, "gemv": 0.0}
    per_search = [0.0] * 4
    for k in range(args.steps):
        e = evs[k]
        for i in range(4):
            st["stats"] += e[i][0].elapsed_time(e[i][1])
            st["mean"] += e[i][1].elapsed_time(e[i][2])
            st["candidates"] += e[i][2].elapsed_time(evcs[k][i])
            d = evcs[k][i].elapsed_time(e[i][3])
            st["search"] += d
            per_search[i] += d
            st["pack"] += e[i][3].elapsed_time(e[i][4])
        st["flush"] += e[3][4].elapsed_time(e[4][0])
        st["gemv"] += e[4][0].elapsed_time(e[4][1])
    clocks = sampler.stop() if sampler else None

    # per-projection decode times, outside the timed steps: each launch alone
    # after an L2 flush (and the same one-element fence kernel)
    # (all repetitions are queued before any is read, so the host never
    # leaves the GPU idle inside a timed launch)
    def alone(launch):
        # the host queues every repetition while the GPU sleeps, so no launch
        # waits for the host inside its events
        torch.cuda.synchronize()
        torch.cuda._sleep(100_000_000)
        evs_alone = []
        for _ in range(20):
            flush_w.fill_(1.0)
            torch.sum(flush_r, dim=0, out=flush_out)
            a, b = E(), E()
            a.record(stream)
            fence.zero_()
            launch()
            b.record(stream)
            evs_alone.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs_alone)

    per_gemv = [alone(lambda p=p: wb.w4a16_gemm_repacked(p["x"], p["tiles"], p["N"], out=p["y"]))
                for p in projs]
    per_gemv_plain = [alone(lambda p=p: wb.w4a16_gemm(p["x"], p["qw"], p["sc"], p["ze"],
                                                      out=p["y"])) for p in projs]

    # the same four-launch decode segment on the plain packed layout
    # (w4a16_gemm), for comparison with the repacked tiles
    seg_plain = []
    torch.cuda.synchronize()
    torch.cuda._sleep(100_000_000)
    for _ in range(20):
        flush_w.fill_(1.0)
        torch.sum(flush_r, dim=0, out=flush_out)
        a, b = E(), E()
        a.record(stream)
        fence.zero_()
        for p in projs:
            wb.w4a16_gemm(p["x"], p["qw"], p["sc"], p["ze"], out=p["y"])
        b.record(stream)
        seg_plain.append((a, b))
    torch.cuda.synchronize()
    seg_plain_ms = statistics.median(a.elapsed_time(b) for a, b in seg_plain)

    # Size-matched read ceiling: a plain streaming read (torch.sum) of as many
    # bytes as each decode launch moves, timed the same way.  Single launches
    # of 9-48 MB cannot reach the copy-bandwidth peak; this is what a read of
    # that size alone achieves on this GPU.
    read_ms = []
    for p in projs:
        buf = torch.ones(gemv_bytes(p["N"], p["K"]) // 4, dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        torch.cuda._sleep(100_000_000)
        evs_read = []
        for _ in range(20):
            flush_w.fill_(1.0)
            torch.sum(flush_r, dim=0, out=flush_out)
            a, b = E(), E()
            a.record(stream)
            fence.zero_()
            torch.sum(buf, dim=0, out=flush_out)
            b.record(stream)
            evs_read.append((a, b))
        torch.cuda.synchronize()
        read_ms.append(statistics.median(a.elapsed_time(b) for a, b in evs_read))
        del buf

    # max over ranks of the timed region and the GEMV segment
    total_ms, gemv_ms = max_over_ranks([total_ms, st["gemv"]], dev)
    bytes_step = sum(gemv_bytes(p["N"], p["K"]) for p in projs)
    flop_step = sum(search_flop(p["N"], p["K"]) for p in projs)
    value = job_value(bytes_step, args.steps, gemv_ms, world)
    peaks, peak_src = load_peaks()
    # the burst peak for a timed region shorter than a second (the clocks
    # stay at their maximum), the sustained peak for a seconds-long one
    search_peak_key, search_peak_kind = (("bf16_tflops", "burst") if total_ms < 1000.0
                                         else ("bf16_tflops_sustained", "sustained"))
    search_peak = peaks[search_peak_key]
    search_tf = flop_step * args.steps / (st["search"] * 1e-3) / 1e12
    gemv_gbs = bytes_step * args.steps / (st["gemv"] * 1e-3) / 1e9
    traffic = None
    if SEARCH_TRAFFIC and SEARCH_TRAFFIC.get("src_sha") == src_sha(SEARCH_SOURCES):
        traffic = SEARCH_TRAFFIC["bytes_per_step"] / len(projs)      # per launch
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "calibration_tokens": T_CAL, "alphas": N_ALPHA,
                   "l2": "flushed every step before the decode matmuls (512 MiB write + 512 MiB "
                         "read); the step's fp16 weights (405 MB) also exceed L2",
                   "parallelism": f"replicas x{world} (one layer per GPU, no collective)",
                   "value_basis": "decode-matmul algorithmic bytes (packed weights, scales, "
                                  "zero-points, x, y) / CUDA-event time of the decode segment "
                                  "of each timed step (the four launches back to back, after "
                                  "the L2 flush), over the repacked decode tiles",
                   "decode_overlap": "programmatic dependent launch with early weight fetch "
                                     "(awq_set_weight_prefetch 1): consecutive decode launches "
                                     "overlap; no launch's weights are written by the kernel "
                                     "just before it"},
        "roofline": {"kernel": "tc_kernel<search> (fused fake-quant + tcgen05 GEMM + MSE)",
                     "bound": "tensor", "achieved": round(search_tf, 2),
                     "peak": search_peak, "unit": "TFLOP/s",
                     "frac": round(search_tf / search_peak, 4),
                     "peak_source": f"{peak_src} bf16 dense {search_peak_kind} (fp16 nominal = "
                                    f"bf16; timed region {total_ms / 1e3:.2f} s)",
                     "traffic": traffic,
                     "traffic_note": "DRAM bytes per search launch, mean of the step's four "
                                     "(ncu); the algorithmic bytes (W and Xcal read once, "
                                     "candidate scales) are within a few percent",
                     "timing": "CUDA events around each awq_search_mse call of the timed "
                               "steps: the search kernel with its 1/s pre-pass and final "
                               "reduction (the candidate scales are the separate "
                               "'candidates' stage)"},
        "roofline_gemv": {"kernel": "gemv_tiles_kernel<1,16> (4 launches per step)", "bound": "hbm",
                          "achieved": round(gemv_gbs, 1), "peak": peaks["hbm_gbs"],
                          "unit": "GB/s", "frac": round(gemv_gbs / peaks["hbm_gbs"], 4),
                          "peak_source": f"{peak_src} copy bandwidth",
                          "size_matched_read_gbs": round(bytes_step / (sum(read_ms) * 1e-3) / 1e9, 1),
                          "size_matched_read_note": "torch.sum over each launch's byte count, "
                                                    "one launch at a time after the L2 flush; "
                                                    "sum of bytes / sum of times",
                          "plain_layout_segment_gbs": round(bytes_step / (seg_plain_ms * 1e-3) / 1e9, 1),
                          "plain_layout_note": "the same four launches with w4a16_gemm on the "
                                               "plain packed layout, median of 20 segments"},
        "stages_ms_per_step": {k: round(v / args.steps, 4) for k, v in st.items()},
        "per_projection": {p["name"]: {"search_ms": round(per_search[i] / args.steps, 4),
                                       "gemv_us_alone": round(per_gemv[i] * 1e3, 2),
                                       "gemv_plain_us_alone": round(per_gemv_plain[i] * 1e3, 2),
                                       "gemv_gbs_alone": round(gemv_bytes(p["N"], p["K"]) /
                                                               (per_gemv[i] * 1e-3) / 1e9, 1),
                                       "read_us_alone": round(read_ms[i] * 1e3, 2)}
                           for i, p in enumerate(projs)},
        # per projection and step: stats, mean, two candidate-scale kernels, 1/s,
        # search, finalize, pack, repack, decode
        "gpu_launches": args.steps * 4 * 10,
        "clocks": clocks,
    }
    if not args.no_e2e:
        out["e2e"] = run_e2e(args, projs, dev, stream, world, fence)
    if not args.no_prefill:
        for p in projs:     # release the decode workload before the large prefill layers
            for k in ("W", "Xc", "ws", "x", "y"):
                p.pop(k, None)
        torch.cuda.empty_cache()

        def flush():
            flush_w.fill_(1.0)
            torch.sum(flush_r, dim=0, out=flush_out)
        out["gemm_m_ge_256"] = run_prefill(args, dev, stream, flush, peaks, peak_src)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args, budget_s=args.cpu_budget, projs=projs)
    return out


# ------------------------------------------------- full LLaMA-7B pass --

FULL_T = 128 * 512                 # calibration tokens per layer input
FULL_M = (1, 16, 64, 256)
FULL_WORKLOAD = ("full LLaMA-7B-shaped quantisation pass: per decoder layer, statistics of its "
                 "four inputs over 128 x 512 = 65536 calibration tokens, G/T = X^T X / T per "
                 "input, the 20-alpha search of each of the 7 linears (q, k, v, o 4096x4096; "
                 "gate, up 11008x4096; down 4096x11008) through G/T, INT4 g128 pack and decode "
                 "repack, then w4a16 matmuls at M in {1, 16, 64, 256}; W ~ N(0,0.02^2), X ~ "
                 "N(0,1) with 1% channels x20")


def gram_flop(N, K, n_alpha=N_ALPHA):
    return 2.0 * N * K * K * n_alpha


def run_full_pass(args, rank, world):
    """The full LLaMA-7B-shaped quantisation pass on a sample of decoder
    layers: one step is one layer's whole pass.  The layers' inputs (3 GB of calibration tokens
    per layer) are generated on the host and uploaded before the timed region;
    they exceed L2 many times over, so no flush is needed."""
    import torch
    import weight_only_bit_stats_b300 as wb
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    n_layers = max(1, args.steps)
    layer_ids = [(rank * n_layers + i) % 32 for i in range(n_layers)]
    t_gen = time.perf_counter()
    layers = []
    for li in layer_ids:
        L = {"id": li, "x": [], "lin": []}
        for idx, (name, K) in enumerate(sg.LLAMA7B_LAYER_INPUTS):
            L["x"].append(torch.from_numpy(sg.layer_activations(li, idx, FULL_T, K)).to(dev))
        for j, (name, N, K) in enumerate(sg.LLAMA7B_LAYER_LINEARS):
            W, _, Xm, _ = sg.layer_inputs(li, j, N, K, 0, M=max(FULL_M))
            L["lin"].append(dict(name=name, N=N, K=K, W=torch.from_numpy(W).to(dev),
                                 xm=torch.from_numpy(Xm).to(dev)))
        layers.append(L)
    t_gen = time.perf_counter() - t_gen
    # buffers shared by every layer
    ws_gram = {K: torch.empty(wb.lib().awq_gram_workspace_size(FULL_T, K), dtype=torch.uint8,
                              device=dev) for _, K in sg.LLAMA7B_LAYER_INPUTS}
    G = {idx: torch.empty((K, K), dtype=torch.float16, device=dev)
         for idx, (_, K) in enumerate(sg.LLAMA7B_LAYER_INPUTS)}
    abs_sum = {idx: torch.empty(K, dtype=torch.int64, device=dev)
               for idx, (_, K) in enumerate(sg.LLAMA7B_LAYER_INPUTS)}
    mean = {idx: torch.empty(K, dtype=torch.float64, device=dev)
            for idx, (_, K) in enumerate(sg.LLAMA7B_LAYER_INPUTS)}
    out = []
    for j, (name, N, K) in enumerate(sg.LLAMA7B_LAYER_LINEARS):
        out.append(dict(
            s=torch.empty(K, dtype=torch.float32, device=dev),
            mse=torch.empty(N_ALPHA, dtype=torch.float64, device=dev),
            best=torch.empty(1, dtype=torch.int32, device=dev),
            ws=torch.empty(max(16, wb.lib().awq_search_gram_workspace_size(N, K, N_ALPHA)),
                           dtype=torch.uint8, device=dev),
            qw=torch.empty((N, K // 8), dtype=torch.int32, device=dev),
            sc=torch.empty((N, K // 128), dtype=torch.float16, device=dev),
            ze=torch.empty((N, K // 128), dtype=torch.float16, device=dev),
            tiles=torch.empty(wb.lib().awq_repack_int4_bytes(N, K), dtype=torch.uint8, device=dev),
            y=torch.empty((max(FULL_M), N), dtype=torch.float16, device=dev),
            gws=torch.empty(max(16, max(wb.lib().w4a16_gemm_workspace_size(M, N, K)
                                        for M in FULL_M)), dtype=torch.uint8, device=dev)))
    stream = torch.cuda.current_stream()
    E = lambda: torch.cuda.Event(enable_timing=True)
    stages = ("stats", "gram", "search", "pack", "matmul_m1", "matmul_m16", "matmul_m64",
              "matmul_m256")

    def step(L, ev=None):
        rec = (lambda k: ev[k].record(stream)) if ev else (lambda k: None)
        rec(0)
        for idx, X in enumerate(L["x"]):
            wb.act_stats(X, out=abs_sum[idx])
            wb.act_mean(abs_sum[idx], FULL_T, out=mean[idx])
        rec(1)
        for idx, X in enumerate(L["x"]):
            wb.gram(X, out=G[idx], workspace=ws_gram[X.shape[1]])
        rec(2)
        for j, lin in enumerate(L["lin"]):
            idx = sg.LLAMA7B_LINEAR_INPUT[j]
            o = out[j]
            wb.search_scale_gram(lin["W"], G[idx], mean[idx], workspace=o["ws"],
                                 out=(o["s"], o["mse"], o["best"]))
        rec(3)
        for j, lin in enumerate(L["lin"]):
            o = out[j]
            wb.pack_int4(lin["W"], o["s"], out=(o["qw"], o["sc"], o["ze"]))
            wb.repack_int4(o["qw"], o["sc"], o["ze"], out=o["tiles"])
        rec(4)
        for k, M in enumerate(FULL_M):
            for j, lin in enumerate(L["lin"]):
                o = out[j]
                if M <= 16:
                    wb.w4a16_gemm_repacked(lin["xm"][:M], o["tiles"], lin["N"], out=o["y"][:M])
                else:
                    wb.w4a16_gemm(lin["xm"][:M], o["qw"], o["sc"], o["ze"], out=o["y"][:M])
            rec(5 + k)

    for _ in range(max(3, args.warmup)):
        step(layers[0])
    wb.sync_status()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.3)
    evs = [[E() for _ in range(len(stages) + 1)] for _ in layers]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = E(), E()
    if sampler: sampler.mark_start()
    t0.record(stream)
    for L, ev in zip(layers, evs):
        step(L, ev)
    t1.record(stream)
    torch.cuda.synchronize()
    if sampler: sampler.mark_end()
    if world > 1:
        dist.barrier()
    wb.sync_status()
    total_ms = max_over_ranks([t0.elapsed_time(t1)], dev)[0]
    st = {k: 0.0 for k in stages}
    for ev in evs:
        for k, name in enumerate(stages):
            st[name] += ev[k].elapsed_time(ev[k + 1])
    clocks = sampler.stop() if sampler else None
    nl = len(layers)
    lin = sg.LLAMA7B_LAYER_LINEARS
    inputs = sg.LLAMA7B_LAYER_INPUTS
    gram_form_flop = sum(2.0 * FULL_T * K * K for _, K in inputs)
    search_flop = sum(gram_flop(N, K) for _, N, K in lin)
    direct_flop = sum(search_flop_t(N, K) for _, N, K in lin)
    bytes_m = {M: sum(gemv_bytes(N, K, M) for _, N, K in lin) for M in FULL_M}
    flop_m = {M: sum(2.0 * M * N * K for _, N, K in lin) for M in FULL_M}
    mm = {}
    for k, M in enumerate(FULL_M):
        ms = st[stages[4 + k]] / nl
        mm[f"M={M}"] = {"ms": round(ms, 4), "gbs": round(bytes_m[M] / (ms * 1e-3) / 1e9, 1),
                        "tflops": round(flop_m[M] / (ms * 1e-3) / 1e12, 2)}
    value = job_value(bytes_m[1], nl, max_over_ranks([st["matmul_m1"]], dev)[0], world)
    peaks, peak_src = load_peaks()
    search_tf = search_flop * nl / (st["search"] * 1e-3) / 1e12
    peak_key, peak_kind = (("bf16_tflops", "burst") if total_ms < 1000.0
                           else ("bf16_tflops_sustained", "sustained"))
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": nl, "warmup": max(3, args.warmup), "ms_per_step": round(total_ms / nl, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": FULL_WORKLOAD + f"; sample of {nl} of the 32 decoder layers "
                                               f"(layers {layer_ids})",
                   "calibration_tokens": FULL_T, "alphas": N_ALPHA, "M": list(FULL_M),
                   "search_route": "Gram matrix (awq_gram + awq_search_scale_gram)",
                   "l2": "inputs exceed L2 (3 GB of calibration tokens per layer)",
                   "value_basis": "M = 1 matmul algorithmic bytes of the 7 linears / CUDA-event "
                                  "time of the M = 1 segment, per layer",
                   "parallelism": f"replicas x{world} (own layers per GPU, no collective)"},
        "seconds_per_layer": round(total_ms / nl / 1e3, 4),
        "projected_32_layers_s": round(32 * total_ms / nl / 1e3, 3),
        "stages_ms_per_layer": {k: round(v / nl, 4) for k, v in st.items()},
        "roofline": {"kernel": "tc_kernel<3> (Gram-route search: fake-quant producer + tcgen05 "
                               "E (G/T) + residual-column epilogue)",
                     "bound": "tensor", "achieved": round(search_tf, 2),
                     "peak": peaks[peak_key], "unit": "TFLOP/s",
                     "frac": round(search_tf / peaks[peak_key], 4),
                     "peak_source": f"{peak_src} bf16 dense {peak_kind} (fp16 nominal = bf16)",
                     "traffic": None,
                     "timing": "CUDA events around the 7 awq_search_scale_gram calls of a layer"},
        "search": {"gram_route_flop_per_layer": search_flop,
                   "gram_formation_flop_per_layer": gram_form_flop,
                   "direct_route_flop_per_layer": direct_flop,
                   "gram_formation_tflops": round(gram_form_flop * nl / (st["gram"] * 1e-3) / 1e12,
                                                  1),
                   "direct_equivalent_tflops": round(direct_flop * nl / ((st["search"] + st["gram"])
                                                                        * 1e-3) / 1e12, 1)},
        "matmul_per_layer": mm,
        "host_generation_s": round(t_gen, 1),
        "gpu_launches": nl * (4 * 2 + 4 * 2 + 7 * 4 + 7 * 2 + 7 * len(FULL_M)),
        "clocks": clocks,
    }
    return res


PREFILL_M = (256, 1024, 4096)
PREFILL_REPS = 10


def run_prefill(args, dev, stream, flush, peaks, peak_src):
    """The metric's GEMM half: w4a16_gemm TFLOP/s at M >= 256 on the
    LLaMA-70B-shaped prefill projections (gate+up 57344x8192, down
    8192x28672; W ~ N(0, 0.015^2) fp16 packed to INT4 g128 on the device,
    X ~ N(0,1) with 1% channels x20).  Each rep is timed alone with CUDA
    events after an L2 flush; the median rep is reported."""
    import torch
    import weight_only_bit_stats_b300 as wb
    E = lambda: torch.cuda.Event(enable_timing=True)
    res = {}
    best_frac = None
    total_flop = total_ms = 0.0
    for j, (name, N, K) in enumerate(sg.LLAMA70B_PREFILL_PROJ):
        W_h, _, X_h, _ = sg.layer_inputs(2, j, N, K, 0, M=max(PREFILL_M), sigma=0.015)
        W = torch.from_numpy(W_h).to(dev)
        del W_h
        qw, sc, ze = wb.pack_int4(W)
        del W
        X = torch.from_numpy(X_h).to(dev)
        Y = torch.empty((max(PREFILL_M), N), dtype=torch.float16, device=dev)
        for M in PREFILL_M:
            x, y = X[:M], Y[:M]
            for _ in range(3):
                wb.w4a16_gemm(x, qw, sc, ze, out=y)
            times = []
            for _ in range(PREFILL_REPS):
                flush()
                a, b = E(), E()
                a.record(stream)
                wb.w4a16_gemm(x, qw, sc, ze, out=y)
                b.record(stream)
                b.synchronize()
                times.append(a.elapsed_time(b))
            ms = statistics.median(times)
            flop = 2.0 * M * N * K
            tf = flop / (ms * 1e-3) / 1e12
            res.setdefault(f"M={M}", {})[name] = {"ms": round(ms, 4), "tflops": round(tf, 1)}
            total_flop += flop
            total_ms += ms
        del qw, sc, ze, X, Y
        torch.cuda.empty_cache()
    wb.sync_status()
    tf_all = total_flop / (total_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"kernel": "tc_kernel<gemm> (TMA + producer dequant + tcgen05/TMEM)",
            "workload": "LLaMA-70B-shaped prefill: gate_up 57344x8192, down 8192x28672, "
                        "M in {256, 1024, 4096}, INT4 g128, W ~ N(0,0.015^2)",
            "per_shape": res, "bound": "tensor", "achieved": round(tf_all, 1), "unit": "TFLOP/s",
            "peak": peak, "frac": round(tf_all / peak, 4),
            "peak_source": f"{peak_src} bf16 dense burst (each launch is timed alone; fp16 "
                           "nominal = bf16)",
            "timing": f"median of {PREFILL_REPS} reps per shape, L2 flushed before each rep; "
                      "achieved = total flop / total median time over the six shapes"}


def run_e2e(args, projs, dev, stream, world, fence):
    """Same step through the public API from pinned HOST buffers: every
    step copies its inputs host->device and its results device->host."""
    import torch
    import weight_only_bit_stats_b300 as wb
    h2d = d2h = 0
    for p in projs:
        p["W_pin"] = torch.from_numpy(p["W_h"]).pin_memory()
        p["Xc_pin"] = torch.from_numpy(p["Xc_h"]).pin_memory()
        p["x_pin"] = torch.from_numpy(p["x_h"]).pin_memory()
        p["out_pin"] = [torch.empty(t.shape, dtype=t.dtype).pin_memory()
                        for t in (p["qw"], p["sc"], p["ze"], p["s"], p["best"], p["y"])]
        h2d += p["W_pin"].nbytes + p["Xc_pin"].nbytes + p["x_pin"].nbytes
        d2h += sum(t.nbytes for t in p["out_pin"])

    # Two streams: host->device copies of projection j+1 overlap the compute
    # of projection j, and each projection's packed weights go back to the
    # host while later projections compute.  The next step's copies wait
    # until this step's compute has released the buffers.
    copy_stream = torch.cuda.Stream(device=dev)
    E = lambda: torch.cuda.Event()
    released = E()
    released.record(stream)

    def step():
        done_in, done_pack = [], []
        copy_stream.wait_event(released)
        for p in projs:
            with torch.cuda.stream(copy_stream):
                p["W"].copy_(p["W_pin"], non_blocking=True)
                p["Xc"].copy_(p["Xc_pin"], non_blocking=True)
                p["x"].copy_(p["x_pin"], non_blocking=True)
            e = E()
            e.record(copy_stream)
            done_in.append(e)
        for p, e in zip(projs, done_in):
            stream.wait_event(e)
            wb.act_stats(p["Xc"], out=p["abs"])
            wb.act_mean(p["abs"], T_CAL, out=p["mean"])
            wb.search_scale(p["W"], p["Xc"], p["mean"], workspace=p["ws"],
                            out=(p["s"], p["mse"], p["best"]))
            wb.pack_int4(p["W"], p["s"], out=(p["qw"], p["sc"], p["ze"]))
            wb.repack_int4(p["qw"], p["sc"], p["ze"], out=p["tiles"])
            e2 = E()
            e2.record(stream)
            done_pack.append(e2)
        for p, e2 in zip(projs, done_pack):
            copy_stream.wait_event(e2)
            with torch.cuda.stream(copy_stream):
                for dst, src in zip(p["out_pin"][:5], (p["qw"], p["sc"], p["ze"], p["s"], p["best"])):
                    dst.copy_(src, non_blocking=True)
        fence.zero_()
        for p in projs:
            wb.w4a16_gemm_repacked(p["x"], p["tiles"], p["N"], out=p["y"])
        released.record(stream)
        copy_stream.wait_event(released)
        with torch.cuda.stream(copy_stream):
            for p in projs:
                p["out_pin"][5].copy_(p["y"], non_blocking=True)
        done_out = E()
        done_out.record(copy_stream)
        stream.wait_event(done_out)

    for _ in range(max(1, min(args.warmup, 3))):
        step()
    torch.cuda.synchronize()
    n = max(1, min(args.steps, 10))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks([a.elapsed_time(b) / n], dev)[0]
    bytes_step = sum(gemv_bytes(p["N"], p["K"]) for p in projs)
    return {"value": round(job_value(bytes_step, 1, ms, world), 3), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "steps": n,
            "basis": "decode-matmul algorithmic bytes / whole-step time with host buffers "
                     "(fp16 weights and calibration tokens in, packed weights, s, alpha, y out; "
                     "copies overlap compute on a second stream)"}


# ------------------------------------------------------- oracle (CPU) arm --

def oracle_step(projs, rows_search):
    """One bounded sample of the step on the CPU oracle; returns timings."""
    import oracle as orc
    t = {"quant": 0.0, "gemv": 0.0}
    for p in projs:
        t0 = time.perf_counter()
        m = orc.act_mean(orc.act_stats(p["Xc_h"]), T_CAL)
        s, _, _ = orc.search_scale(p["W_h"][:rows_search], p["Xc_h"], m)
        q = orc.pack_int4(p["W_h"], s)
        t1 = time.perf_counter()
        orc.w4a16_gemm(p["x_h"], *q)
        t2 = time.perf_counter()
        t["quant"] += t1 - t0
        t["gemv"] += t2 - t1
    return t


def _oracle_projs():
    projs = []
    for j, (name, N, K) in enumerate(sg.LLAMA7B_DECODE_PROJ):
        W, Xc, Xm, _ = sg.layer_inputs(0, j, N, K, T_CAL, M=1)
        projs.append(dict(name=name, N=N, K=K, W_h=W, Xc_h=Xc, x_h=Xm))
    return projs


ROWS_SEARCH = 16
SAMPLE = ("per step, each of the four projections: statistics over all 512 calibration tokens, "
          f"the 20-alpha search on the first {ROWS_SEARCH} weight rows, INT4 pack of all rows, "
          "and the M=1 decode matmul over all rows (value = its GB/s)")


def cpu_baseline(args, budget_s=20.0, projs=None):
    import oracle as orc
    orc.build()
    projs = projs or _oracle_projs()
    bytes_step = sum(gemv_bytes(p["N"], p["K"]) for p in projs)
    oracle_step(projs, ROWS_SEARCH)            # warm-up (page-in, thread pools)
    t_gemv = t_quant = 0.0
    n = 0
    t_begin = time.perf_counter()
    while n < 1 or (time.perf_counter() - t_begin < budget_s and n < 50):
        t = oracle_step(projs, ROWS_SEARCH)
        t_gemv += t["gemv"]
        t_quant += t["quant"]
        n += 1
    return {"value": round(bytes_step * n / t_gemv / 1e9, 4), "unit": "GB/s",
            "cores": os.cpu_count(), "kind": "oracle", "sample": SAMPLE,
            "steps": n, "oracle_gemv_s_per_step": round(t_gemv / n, 4),
            "oracle_quant_s_per_step": round(t_quant / n, 4)}


def run_reference(args):
    import oracle as orc
    orc.build()
    projs = _oracle_projs()
    bytes_step = sum(gemv_bytes(p["N"], p["K"]) for p in projs)
    for _ in range(args.warmup):
        oracle_step(projs, ROWS_SEARCH)
    t_gemv = t_quant = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        t = oracle_step(projs, ROWS_SEARCH)
        t_gemv += t["gemv"]
        t_quant += t["quant"]
    wall = time.perf_counter() - t0
    value = bytes_step * args.steps / t_gemv / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": 1, "calibration_tokens": T_CAL,
                       "alphas": N_ALPHA},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": SAMPLE},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "oracle_quant_s_per_step": round(t_quant / args.steps, 4)}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 50; with --workload llama7b_full: decoder "
                         "layers, default 2)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="do not report the separate M >= 256 GEMM measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--workload", choices=["llama7b_decode", "llama7b_full"],
                    default="llama7b_decode",
                    help="llama7b_full: the full LLaMA-7B quantisation pass, one step per "
                         "decoder layer (steps = layers sampled)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 2 if args.workload == "llama7b_full" else 50
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    out = run_full_pass(args, rank, world) if args.workload == "llama7b_full" else \
        run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
