#!/usr/bin/env python3
"""Benchmark of the block-scaled FP4 routed-MoE layer on GB300.

Default workload: DeepSeek-V4-Flash decode, T=64 tokens, H=4096, I=2048,
E=256, top-k 6, swiglu_limit 10. Weights are NVFP4, quantised from seeded
synthetic N(0, 0.02) values. Activations are seeded, with 1% outliers x20.
A step is one pass of the whole layer: route, quantise+scatter,
W1+SwiGLU+requant, W2, combine, issued by one moe_forward call. The
per-stage split comes from a second pass that makes the four stage calls
separately, with CUDA events between them. Workloads with a shared expert
(dsv4_flash_decode_shared_T64) also run its three block-FP8 kernels on a side
stream beside the routed path (as moe_forward_shared does), and the combine
adds its output.

Prints ONE JSON line (rank 0). value = tokens/s over all ranks, with inputs
resident in HBM; e2e = the same metric through moe_forward with pinned host
buffers, with the host<->device copies inside the timed region. The
roofline section is for the dominant kernel (the W1 grouped GEMM), timed with
CUDA events inside the timed region on the stream it runs on.

--impl reference times the CPU oracle on a bounded token sample of the same
workload. It is the reference arm. The pages ship no runnable
implementation of this layer.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthgen as sg  # noqa: E402

METRIC = "MoE layer tokens/s (DSV4 shape) + achieved HBM GB/s / FP4 tensor-pipe % on 1 GB300"
FALLBACK_HBM_GBS = 6800.0


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one W1 GEMM launch per workload, from a
# one-pass ncu capture summarised under profiles/. A figure holds only for the GEMM sources it was taken
# with, so it is reported while their hash matches and as null otherwise.
W1_TRAFFIC = {
    # workload name: (bytes per launch, sha256 of the GEMM sources)
    "dsv4_flash_decode_T64": (1948672512 + 7872768, "75391954e7b25c7165249bf2d4b6525bdb0df307ccb299a98605588f4e41fb4c"),
}
GEMM_SOURCES = ("block_scaled_fp4_top_gb300/csrc/gemm.cu", "block_scaled_fp4_top_gb300/csrc/gemm_wide.cu",
                "block_scaled_fp4_top_gb300/csrc/gemm_sched.cuh", "block_scaled_fp4_top_gb300/csrc/common.cuh")


def gemm_sources_sha() -> str:
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def w1_traffic(workload: str):
    t = W1_TRAFFIC.get(workload)
    return float(t[0]) if t is not None and t[1] == gemm_sources_sha() else None


def max_over_ranks(v: float, world: int, device) -> float:
    """The largest v over all ranks: the job takes as long as its slowest replica."""
    if world <= 1:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, steps: int, ms_max: float) -> float:
    """Whole-job throughput of `world` replicas that each ran `steps` steps of `tokens_per_rank` tokens."""
    return tokens_per_rank * world * steps / (ms_max * 1e-3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.idx = gpu_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        if self.proc is None:
            return None
        rows = [r.split(",") for r in getattr(self, "out", "").strip().splitlines() if r.strip()]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def setup_layer(wl, max_tokens):
    import torch
    from block_scaled_fp4_top_gb300 import _lib, api
    from synthgen import gpu as sgpu
    if wl.w_format == _lib.W_MXFP4:
        return setup_mx_layer(wl, max_tokens)
    if wl.w_format == 2:   # the TP3 shard's MXFP4 weights on the NVFP4 path
        return setup_mx_nvfp4_layer(wl, max_tokens)
    cfg = api.config(wl.H, wl.I, wl.E, wl.k, max_tokens, wl.swiglu_limit, shared_inter=wl.shared_I,
                     ep_first=wl.ep_first, ep_count=wl.ep_count)
    layer = api.MoELayer(cfg)
    n_local = wl.ep_count or wl.E   # expert parallelism: local expert l is global expert ep_first + l
    for e0 in range(0, n_local, 16):
        n = min(16, n_local - e0)
        layer.quantize_weights(1, e0, sgpu.expert_w1(wl, wl.ep_first + e0, n))
        layer.quantize_weights(2, e0, sgpu.expert_w2(wl, wl.ep_first + e0, n))
    if wl.shared_I:
        layer.quantize_shared_weights(1, sgpu.shared_w1(wl))
        layer.quantize_shared_weights(2, sgpu.shared_w2(wl))
    bias = sg.router_bias_f32(wl)
    layer.set_router(sgpu.router(wl), None if bias is None else torch.from_numpy(bias).cuda())
    layer.calibrate(sgpu.activations(wl, sg.WARMUP_SEED))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # drop the fp32 weight staging buffers
    return cfg, layer


def setup_mx_nvfp4_layer(wl, max_tokens):
    """Rank 0 of the TP3 MXFP4 shard (as setup_mx_layer builds it), its weights converted to the NVFP4 operand
    form on the GPU (fp4moe_mxfp4_as_nvfp4), then calibrated like the NVFP4 layer."""
    import dataclasses
    import torch
    from block_scaled_fp4_top_gb300 import api
    from synthgen import gpu as sgpu
    _, mx = setup_mx_layer(dataclasses.replace(wl, w_format=1), max_tokens)
    cfg = api.config(wl.H, wl.I, wl.E, wl.k, max_tokens, wl.swiglu_limit, inter_logical=wl.I_logical)
    layer = api.MoELayer(cfg)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    layer.load_mxfp4_weights(1, 0, mx.weights.w1_fp4, mx.weights.w1_sf, err)
    layer.load_mxfp4_weights(2, 0, mx.weights.w2_fp4, mx.weights.w2_sf, err)
    torch.cuda.synchronize()
    if int(err[0].item()) != 0:
        raise RuntimeError(f"fp4moe_mxfp4_as_nvfp4: error word {int(err[0].item()):#x}")
    del mx
    layer.set_router(sgpu.router(wl), None)
    layer.calibrate(sgpu.activations(wl, sg.WARMUP_SEED))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return cfg, layer


def setup_mx_layer(wl, max_tokens, rank=0, tp=3):
    """Rank `rank` of a TP `tp` MXFP4 shard: the full-width synthetic experts (intermediate 2048) cut in logical
    units, zero past the logical width, quantised by the library."""
    import dataclasses
    import torch
    from block_scaled_fp4_top_gb300 import _lib, api
    from synthgen import gpu as sgpu
    I_full = 2048
    Il, Ik = wl.I_logical, wl.I
    full = dataclasses.replace(wl, I=I_full, I_logical=I_full)
    cfg = api.config(wl.H, Ik, wl.E, wl.k, max_tokens, wl.swiglu_limit, inter_logical=Il, w_format=_lib.W_MXFP4)
    layer = api.MoELayer(cfg)
    a = rank * Il
    n = max(0, min(Il, I_full - a))
    for e0 in range(0, wl.E, 8):
        c = min(8, wl.E - e0)
        w1f = sgpu.expert_w1(full, e0, c)
        w1 = torch.zeros(c, 2 * Ik, wl.H, dtype=torch.float32, device="cuda")
        w1[:, :n] = w1f[:, a:a + n]
        w1[:, Ik:Ik + n] = w1f[:, I_full + a:I_full + a + n]
        del w1f
        layer.quantize_weights(1, e0, w1)
        w2f = sgpu.expert_w2(full, e0, c)
        w2 = torch.zeros(c, wl.H, Ik, dtype=torch.float32, device="cuda")
        w2[:, :, :n] = w2f[:, :, a:a + n]
        del w2f
        layer.quantize_weights(2, e0, w2)
    layer.set_router(sgpu.router(wl), None)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return cfg, layer


def build_step(wl, cfg, layer, x, y, dev, n_stage_steps):
    """The layer's hot path as the four C-ABI calls (route, quantise-scatter, W1, W2 + combine) on
    preallocated buffers. step(e, es) records CUDA events e[0..4] between the calls (and es[0..1] around the
    shared expert on its side stream) when given them."""
    import torch
    from block_scaled_fp4_top_gb300 import api
    W = layer.weights
    T, H, k, E = wl.T, wl.H, wl.k, wl.E
    E_loc = wl.ep_count or E   # counts, offsets and padded offsets are per local expert
    mx = wl.w_format == 1
    i32 = dict(dtype=torch.int32, device=dev)
    cap = api.capacity_rows(cfg, T)
    bufs = dict(logits=torch.empty(T, E, dtype=torch.float32, device=dev), ids=torch.empty(T * k, **i32),
                w=torch.empty(T * k, dtype=torch.float32, device=dev), counts=torch.empty(E_loc, **i32),
                offsets=torch.empty(E_loc, **i32), poff=torch.empty(E_loc, **i32), slot=torch.empty(T * k, **i32),
                por=torch.empty(cap, **i32),
                # slot activations: NVFP4 codes + scales, or bf16 rows for MXFP4 layers
                a1=torch.empty(cap * H * 2 if mx else cap * H // 2, dtype=torch.uint8, device=dev),
                a1sf=torch.empty(16 if mx else cap * H // 16, dtype=torch.uint8, device=dev),
                a2=torch.empty(cap * wl.I * 2 if mx else cap * wl.I // 2, dtype=torch.uint8, device=dev),
                a2sf=torch.empty(16 if mx else cap * wl.I // 16, dtype=torch.uint8, device=dev))
    se = wl.shared_I > 0
    ep = wl.ep_count > 0
    if se:   # the shared expert's fp32 output rows
        bufs["o_shared"] = torch.empty(T, H, dtype=torch.float32, device=dev)
    if se or ep:   # the routed W2 rows, combined in a separate pass (with the slot mask under EP)
        bufs["o_pairs"] = torch.empty(T * k, H, dtype=torch.bfloat16, device=dev)   # bf16 pair rows
    b = bufs
    stream = torch.cuda.current_stream()
    n_stage = 5
    se_ev = None
    if se:   # the shared expert runs beside the routed path, as moe_forward_shared runs it
        side = torch.cuda.Stream()
        fork_ev, join_ev = torch.cuda.Event(), torch.cuda.Event()
        se_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_stage_steps)]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_stage + 1)] for _ in range(n_stage_steps)]

    def step(e=None, es=None):
        if se:
            fork_ev.record(stream)
            side.wait_event(fork_ev)
            if es is not None:
                es[0].record(side)
            api.moe_shared_expert(cfg, T, x, layer.shared, b["o_shared"], layer.ws, stream=side)
            if es is not None:
                es[1].record(side)
            join_ev.record(side)
        if e is not None:
            e[0].record(stream)
        api.moe_route(cfg, T, x, layer.router_w, layer.router_bias, b["logits"], b["ids"], b["w"], b["counts"],
                      b["offsets"], b["poff"], b["slot"], b["por"], layer.ws)
        if e is not None:
            e[1].record(stream)
        api.moe_quantize_scatter(cfg, T, x, layer.gs1, b["slot"], b["a1"], b["a1sf"], layer.ws)
        if e is not None:
            e[2].record(stream)
        api.moe_grouped_gemm_w1_swiglu(cfg, T, b["a1"], b["a1sf"], b["poff"], b["por"], W.w1_fp4, W.w1_sf,
                                       layer.alpha1, layer.gs2, b["a2"], b["a2sf"], layer.ws)
        if e is not None:
            e[3].record(stream)
        if se or ep:
            api.moe_grouped_gemm_w2(cfg, T, b["a2"], b["a2sf"], b["poff"], b["por"], W.w2_fp4, W.w2_sf,
                                    layer.alpha2, b["o_pairs"], layer.ws)
            if se:
                stream.wait_event(join_ev)
            api.moe_combine_shared(cfg, T, b["o_pairs"], b["w"], b["slot"] if ep else None,
                                   b["o_shared"] if se else None, y)
            if e is not None:
                e[4].record(stream)
            return
        api.moe_grouped_gemm_w2_combine(cfg, T, b["a2"], b["a2sf"], b["poff"], b["por"], W.w2_fp4, W.w2_sf,
                                        layer.alpha2, b["w"], y, layer.ws)
        if e is not None:
            e[4].record(stream)

    return step, bufs, ev, se_ev


def e2e_pipeline(layer, x, y, stream):
    """The end-to-end loop as a caller would pipeline it: every step copies its input from pinned host memory,
    runs moe_forward and copies its output back to pinned host memory. The copies run on a second stream
    with two device buffers each way, so step i's output copy and step i + 1's input copy overlap the
    compute of the steps around them; events keep every buffer's reuse ordered. run(n) runs n steps and
    returns CUDA events recorded before the first input copy and after the last output copy; last(n) is the
    host copy of the output of the last of those n steps."""
    import torch
    copy = torch.cuda.Stream()
    x_host = torch.empty_like(x, device="cpu").pin_memory()
    x_host.copy_(x.cpu())
    y_host = [torch.empty_like(y, device="cpu").pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    y_dev = [torch.empty_like(y) for _ in range(2)]
    ev = lambda: torch.cuda.Event()
    x_ready, done, y_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def run(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        copy.wait_stream(stream)
        e0.record(copy)
        with torch.cuda.stream(copy):
            x_dev[0].copy_(x_host, non_blocking=True)
        x_ready[0].record(copy)
        for i in range(n):
            b = i & 1
            stream.wait_event(x_ready[b])            # this step's input is on the device
            stream.wait_event(y_free[b])             # its output buffer was copied out two steps ago
            layer.forward(x_dev[b], y_dev[b])
            done[b].record(stream)
            with torch.cuda.stream(copy):
                if i + 1 < n:                        # the next input, once step i - 1 no longer reads its buffer
                    copy.wait_event(done[1 - b])
                    x_dev[1 - b].copy_(x_host, non_blocking=True)
                    x_ready[1 - b].record(copy)
                copy.wait_event(done[b])             # this step's output, once it is written
                y_host[b].copy_(y_dev[b], non_blocking=True)
                y_free[b].record(copy)
        e1.record(copy)
        return e0, e1
    run.last = lambda n: y_host[(n - 1) & 1]
    return run


def run_ours(args, wl, rank, world):
    import torch
    from block_scaled_fp4_top_gb300 import api
    from synthgen import gpu as sgpu
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg, layer = setup_layer(wl, wl.T)
    T, H, k, E = wl.T, wl.H, wl.k, wl.E
    E_loc = wl.ep_count or E   # counts, offsets and padded offsets are per local expert
    mx = wl.w_format == 1
    se = wl.shared_I > 0
    ep = wl.ep_count > 0
    x = sgpu.activations(wl, sg.EVAL_SEED + rank)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    n_stage_steps = min(args.steps, 200)
    step, b, ev, se_ev = build_step(wl, cfg, layer, x, y, dev, n_stage_steps)

    for _ in range(args.warmup):
        step()
        layer.forward(x, y)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # the timed region: moe_forward (one C-ABI call per step, the layer as a caller runs it) back to back,
    # events only at its two ends, so each kernel's prologue still overlaps its predecessor's tail
    # (programmatic dependent launch)
    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)  # let the sampler start before the timed region
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            layer.forward(x, y)
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    err = layer.read_error()
    if err != 0:
        raise RuntimeError(f"device error word {err:#x}")
    # the stage split, from a second pass with events between the calls: an event between two launches ends
    # the overlap, so these durations are serialised ones and their sum exceeds the step time above
    for i in range(n_stage_steps):
        step(ev[i], se_ev[i] if se else None)
    torch.cuda.synchronize()
    stage_names = ["route", "quantize_scatter", "w1_swiglu_requant", "w2_combine"]
    stage_ms = {n: float(np.mean([e[j].elapsed_time(e[j + 1]) for e in ev])) for j, n in enumerate(stage_names)}
    if se:   # on the side stream, beside the routed stages
        stage_ms["shared_expert"] = float(np.mean([e[0].elapsed_time(e[1]) for e in se_ev]))

    counts = b["counts"].cpu().numpy()
    n_active = int((counts > 0).sum())
    R = int(b["poff"][-1].item())
    I = wl.I
    sfdiv = 32 if mx else 16  # elements per block scale
    w1_bytes = n_active * (2 * I * H // 2 + 2 * I * H // sfdiv)
    w2_bytes = n_active * (H * I // 2 + H * I // sfdiv)
    if mx:   # A1 real rows read, A2 real rows written: bf16 rows
        act1 = T * k * H * 2 + T * k * I * 2
    else:
        act1 = T * k * (H // 2 + H // 16) + T * k * (I // 2 + I // 16)
    layer_bytes = w1_bytes + w2_bytes + E * H * 2 + 2 * T * H * 2
    if se:
        Is = wl.shared_I
        # codes and block scales of both matrices; x read, its FP8 codes written and read, h codes written and
        # read, fp32 output rows written and read back by the combine
        se_bytes = 3 * Is * H + 3 * (Is // 128) * (H // 128) * 4 + T * H * 2 + 2 * T * H + 2 * T * Is + 2 * T * H * 4
        layer_bytes += se_bytes
    peak, peak_kind = peaks()
    w1_ms = stage_ms["w1_swiglu_requant"]
    achieved = (w1_bytes + act1) / (w1_ms * 1e-3) / 1e9
    step_ms = ms / args.steps

    # ---------------- e2e: moe_forward with pinned host buffers, copies inside the timed region
    e2e_run = e2e_pipeline(layer, x, y, stream)
    e2e_run(args.warmup)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = e2e_run(args.steps)
    torch.cuda.synchronize()
    # the pipelined steps give the output of the eager steps above, bit for bit
    assert torch.equal(e2e_run.last(args.steps), y.cpu()), "e2e output differs from the timed steps' output"
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    assert layer.read_error() == 0

    # ---------------- the per-batch activation scale (fp4moe_batch_gs1), timed alone: one launch per call
    bgs = None
    if not mx:
        gs1_keep, a1_keep = layer.gs1.clone(), layer.alpha1.clone()
        for _ in range(3):
            layer.batch_gs1(x)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        reps = 50
        g0.record(stream)
        for _ in range(reps):
            layer.batch_gs1(x)
        g1.record(stream)
        torch.cuda.synchronize()
        layer.gs1.copy_(gs1_keep)
        layer.alpha1.copy_(a1_keep)
        bgs_us = g0.elapsed_time(g1) * 1e3 / reps
        bgs_bytes = T * H * 2 + E_loc * 8   # x read once; the weight scales read and alpha written
        bgs = {"us": bgs_us, "algorithmic_bytes": bgs_bytes, "achieved_gbs": bgs_bytes / (bgs_us * 1e-6) / 1e9,
               "launches": 1}
    assert layer.read_error() == 0

    out = {
        "metric": METRIC, "value": job_tokens_per_s(T, world, args.steps, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": ("mxfp4 weights x bf16 activations (exact bf16 expansion, fp32 accumulate)" if mx
                                                         else "mxfp4 weights (e8m0 scales as exact e4m3 powers of two) x nvfp4 activations, fp32 accumulate"
                                                         if wl.w_format == 2
                                                         else "nvfp4 (e2m1 x e2m1, e4m3 block scales, fp32 accumulate)"),
        "data": "synthetic (seeded SplitMix64 / Irwin-Hall normal; NVFP4 weights quantised from N(0,0.02))",
        "config": {"workload": wl.name, "T": T, "H": H, "I": I, "E": E, "top_k": k, "swiglu_limit": wl.swiglu_limit,
                   "parallelism": f"replicas x{world}", "l2": "inputs larger than L2: ~2.8 GB of expert weights "
                   "streamed per step (L2 129 MB)"},
        "us_per_layer": step_ms * 1e3,
        "layer_hbm_gbs": layer_bytes / (step_ms * 1e-3) / 1e9,
        "layer_algorithmic_bytes": layer_bytes, "n_active_experts": n_active, "padded_rows": R,
        "stages_us": {n: v * 1e3 for n, v in stage_ms.items()},
        "stages_note": f"serialised: a second pass of {n_stage_steps} steps with CUDA events between the calls, "
                       "which stop each kernel's prologue from overlapping its predecessor; the step time above has "
                       "no events inside",
        "roofline": {"kernel": "mx_gemm_kernel<W1 SwiGLU bf16>" if mx else "grouped_gemm_wide_kernel<W1 SwiGLU requant>",
                     "bound": "hbm", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_kind": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": w1_bytes + act1, "traffic": w1_traffic(wl.name)},
        # route: router_mma + router_refine + layout_small (T*k <= 4096) or + hist, scan, slots;
        # then quantise-scatter, W1, W2, combine
        "gpu_launches": ((3 if T * k <= 4096 else 5) + 4 + (3 if se else 0)) * args.steps,
        "e2e": {"value": job_tokens_per_s(T, world, args.steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2},
        "clocks": clk.summary(),
        "batch_gs1": bgs,
    }
    if ep:
        out["config"]["expert_parallel"] = {"ep_first": wl.ep_first, "ep_count": wl.ep_count,
                                            "note": "one rank's share: routing over all experts, GEMMs over the local ones"}
    if se:
        se_ms = stage_ms["shared_expert"]
        se_gbs = se_bytes / (se_ms * 1e-3) / 1e9
        out["shared_expert"] = {"kernels": "se_quant_x, se_gemm<W1 SwiGLU requant>, se_gemm<W2>",
                                "stream": "a side stream beside route + routed experts, joined before the combine",
                                "shared_inter": Is, "us": se_ms * 1e3, "algorithmic_bytes": se_bytes,
                                "achieved_gbs": se_gbs, "frac_hbm": se_gbs / peak,
                                "tflops": 2 * T * 3 * Is * H / (se_ms * 1e-3) / 1e12}
    return out


def fp4_dense_peak(dev):
    """The dense NVFP4 tensor-core rate of this GPU, measured: fp4moe_tensor_peak_probe at N = 128 and 256
    (one CTA per SM issuing back-to-back M = 128, K = 64 block-scaled MMAs on shared-memory operands), timed with
    CUDA events on its stream after two warm-up launches."""
    import torch
    from block_scaled_fp4_top_gb300 import api
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    err = torch.zeros(4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    by_n, us = {}, {}
    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)
        for n, iters in ((128, 40000), (256, 20000)):
            for _ in range(2):
                api.fp4moe_tensor_peak_probe(n, iters, err)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 5
            e0.record(stream)
            for _ in range(reps):
                api.fp4moe_tensor_peak_probe(n, iters, err)
            e1.record(stream)
            torch.cuda.synchronize()
            sec = e0.elapsed_time(e1) * 1e-3 / reps
            by_n[str(n)] = nsm * iters * 4 * 2 * 128 * n * 64 / sec / 1e12
            us[str(n)] = sec * 1e6
    if int(err[0].item()) != 0:
        raise RuntimeError("tensor peak probe: a bounded wait ran out")
    return {"tflops": max(by_n.values()), "tflops_by_n": by_n, "us_per_launch_by_n": us, "sms": nsm,
            "kernel": "tensor_peak_kernel: tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X, "
                      "M=128, K=64, operands in shared memory", "clocks": clk.summary()}


def run_prefill(args, dev, fp4_peak_tflops):
    """The Zipf-routed prefill workload (T = 8192, DSV4 shapes), timed like the decode step (moe_forward back to
    back, then the four stage calls with events between them for the split), with the layer's HBM fraction and
    the GEMMs' tensor-pipe share of the measured FP4 peak."""
    import torch
    from synthgen import gpu as sgpu
    wl = sg.DSV4_PREFILL_ZIPF
    cfg, layer = setup_layer(wl, wl.T)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    x = sgpu.activations(wl, sg.EVAL_SEED)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    steps, n_stage_steps = args.prefill_steps, min(args.prefill_steps, 50)
    step, b, ev, _ = build_step(wl, cfg, layer, x, y, dev, n_stage_steps)
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        step()
        layer.forward(x, y)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            layer.forward(x, y)
        t1.record(stream)
        torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    for i in range(n_stage_steps):
        step(ev[i])
    torch.cuda.synchronize()
    err = layer.read_error()
    if err != 0:
        raise RuntimeError(f"prefill: device error word {err:#x}")
    names = ["route", "quantize_scatter", "w1_swiglu_requant", "w2_combine"]
    st = {n: float(np.mean([e[j].elapsed_time(e[j + 1]) for e in ev])) for j, n in enumerate(names)}
    counts = b["counts"].cpu().numpy()
    n_active = int((counts > 0).sum())
    w1_bytes = n_active * (2 * I * H // 2 + 2 * I * H // 16)
    w2_bytes = n_active * (H * I // 2 + H * I // 16)
    a1 = T * k * (H // 2 + H // 16)    # A1 rows: written by the scatter, read by W1
    a2 = T * k * (I // 2 + I // 16)    # A2 rows: written by W1, read by W2
    layer_bytes = w1_bytes + w2_bytes + E * H * 2 + 2 * T * H * 2 + 2 * (a1 + a2)
    flops_w1, flops_w2 = 2 * T * k * 2 * I * H, 2 * T * k * I * H
    hbm, hbm_kind = peaks()
    us = ms * 1e3
    w1_s, w2_s = st["w1_swiglu_requant"] * 1e-3, st["w2_combine"] * 1e-3
    return {
        "workload": wl.name, "T": T, "us_per_layer": us, "tokens_per_s": T / (ms * 1e-3), "steps": steps,
        "n_active_experts": n_active, "padded_rows": int(b["poff"][-1].item()), "max_tokens_per_expert":
            int(counts.max()), "zero_token_experts": int((counts == 0).sum()),
        "layer_algorithmic_bytes": layer_bytes,
        "layer_hbm_gbs": layer_bytes / (ms * 1e-3) / 1e9, "layer_hbm_frac": layer_bytes / (ms * 1e-3) / 1e9 / hbm,
        "hbm_peak_gbs": hbm, "hbm_peak_kind": hbm_kind,
        "flops": flops_w1 + flops_w2,
        "tensor_pipe_frac_layer": (flops_w1 + flops_w2) / (ms * 1e-3) / 1e12 / fp4_peak_tflops,
        "fp4_peak_tflops": fp4_peak_tflops,
        "stages_us": {n: v * 1e3 for n, v in st.items()},
        "stages_note": f"serialised: {n_stage_steps} steps with CUDA events between the calls",
        "w1": {"us": w1_s * 1e6, "algorithmic_bytes": w1_bytes + a1 + a2, "hbm_frac": (w1_bytes + a1 + a2) / w1_s / 1e9 / hbm,
               "tflops": flops_w1 / w1_s / 1e12, "tensor_pipe_frac": flops_w1 / w1_s / 1e12 / fp4_peak_tflops},
        "w2_combine": {"us": w2_s * 1e6, "algorithmic_bytes": w2_bytes + a2 + T * H * 2,
                       "hbm_frac": (w2_bytes + a2 + T * H * 2) / w2_s / 1e9 / hbm,
                       "tflops": flops_w2 / w2_s / 1e12, "tensor_pipe_frac": flops_w2 / w2_s / 1e12 / fp4_peak_tflops},
        "clocks": clk.summary(),
        "l2": "inputs larger than L2: ~3.4 GB of expert weights streamed per step (L2 129 MB)",
    }


def run_route_only(args, wl, dev):
    """moe_route alone on the workload's batch (x, router and bias from the seeded generator; no expert weights
    are made): --warmup untimed calls, then --steps calls back to back between two CUDA events. A small case for
    profiler captures of the routing kernels, not the bench line."""
    import torch
    from synthgen import gpu as sgpu
    from block_scaled_fp4_top_gb300 import api
    T = wl.T
    cfg = api.config(wl.H, wl.I, wl.E, wl.k, T, wl.swiglu_limit)
    i32 = dict(dtype=torch.int32, device=dev)
    bufs = [torch.empty(T, wl.E, dtype=torch.float32, device=dev), torch.empty(T * wl.k, **i32),
            torch.empty(T * wl.k, dtype=torch.float32, device=dev), torch.empty(wl.E, **i32),
            torch.empty(wl.E, **i32), torch.empty(wl.E, **i32), torch.empty(T * wl.k, **i32),
            torch.empty(api.capacity_rows(cfg, T), **i32)]
    ws = torch.zeros(api.workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    x = sgpu.activations(wl, sg.EVAL_SEED)
    wr = sgpu.router(wl)
    bias = sg.router_bias_f32(wl)
    bias_t = None if bias is None else torch.from_numpy(bias).to(dev)
    for _ in range(args.warmup):
        api.moe_route(cfg, T, x, wr, bias_t, *bufs, ws)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        api.moe_route(cfg, T, x, wr, bias_t, *bufs, ws)
    t1.record()
    torch.cuda.synchronize()
    err = api.fp4moe_read_error(ws)
    if err != 0:
        raise RuntimeError(f"route: device error word {err:#x}")
    return {"route_only": wl.name, "T": T, "E": wl.E, "steps": args.steps, "warmup": args.warmup,
            "us_per_call": t0.elapsed_time(t1) * 1e3 / args.steps}


def run_side_workload(args, wl, dev):
    """A second workload measured in the same run, the way the decode line is (run_ours), cut to its figures."""
    import copy
    sub = copy.copy(args)
    sub.steps, sub.warmup = args.side_steps, max(3, min(args.warmup, 10))
    r = run_ours(sub, wl, 0, 1)
    keep = ("us_per_layer", "value", "layer_hbm_gbs", "layer_algorithmic_bytes", "n_active_experts", "stages_us",
            "dtype", "clocks")
    out = {"workload": wl.name, "T": wl.T, "steps": sub.steps, **{k: r[k] for k in keep}}
    out["tokens_per_s"] = out.pop("value")
    out["w1"] = {k: r["roofline"][k] for k in ("kernel", "achieved", "peak", "frac", "algorithmic_bytes_per_launch")}
    out["e2e_tokens_per_s"] = r["e2e"]["value"]
    return out


def run_graph_sweep(args, dev):
    """Config-5 style batch sweep: the decode-shape layer captured in one CUDA graph per T over fixed-capacity
    buffers; each replay is timed alone (CUDA events around the replay) after a write of 256 MB that flushes
    L2, so even the smallest batches stream their experts' weights from HBM."""
    import torch
    from synthgen import gpu as sgpu
    wl = sg.DSV4_DECODE
    Ts = (1, 8, 64, 512, 4096)
    cfg, layer = setup_layer(wl, max(Ts))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    hbm, _ = peaks()
    res = []
    for T in Ts:
        x = sgpu.activations(wl, sg.EVAL_SEED, T=T)
        y = torch.empty(T, wl.H, dtype=torch.bfloat16, device=dev)
        ids = torch.empty(T * wl.k, dtype=torch.int32, device=dev)
        layer.forward(x, y, ids)   # eager first: load-time set-up of the launch path happens outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer.forward(x, y, ids)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        n_active = int(np.unique(ids.cpu().numpy()).size)
        tot = 0.0
        for _ in range(args.side_steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1)
        us = tot * 1e3 / args.side_steps
        nbytes = n_active * (2 * wl.I * wl.H * 9 // 16 + wl.H * wl.I * 9 // 16) + wl.E * wl.H * 2 + 2 * T * wl.H * 2
        res.append({"T": T, "us_per_replay": us, "tokens_per_s": T / (us * 1e-6), "n_active_experts": n_active,
                    "algorithmic_bytes": nbytes, "hbm_frac": nbytes / (us * 1e-6) / 1e9 / hbm})
        del g
    if layer.read_error() != 0:
        raise RuntimeError("graph sweep: device error word set")
    return {"workload": "dsv4_flash_decode graph replay per T", "replays_per_T": args.side_steps,
            "l2": "256 MB written before every replay (L2 flushed); events around the replay only", "by_T": res}


class OracleSample:
    """The oracle, as it stands, on the first n_tokens of the evaluation batch.

    The expert weights those tokens route to are quantised once, here: that is load time, outside every
    timed region. run(rows) then times the oracle's layer on those token rows (routing, experts, combine).
    """

    def __init__(self, wl, n_tokens: int):
        import dataclasses
        from oracle import moe, mxfp4
        self.wl, self.n = wl, n_tokens
        self.x = sg.activations_bf16(wl, sg.EVAL_SEED, T=n_tokens)
        self.wr = sg.router_bf16(wl)
        self.bias = sg.router_bias_f32(wl)
        ids, _ = moe.topk_softmax(moe.router_logits(self.x, self.wr, self.bias), wl.k)
        self.cache = {}
        self.mx = wl.w_format == 1
        self.full = dataclasses.replace(wl, I=2048, I_logical=2048)
        self.plan = mxfp4.tp_plan(2048, 3, 32, 128)
        for e in np.unique(ids):
            if not wl.ep_count or wl.ep_first <= e < wl.ep_first + wl.ep_count:
                self.expert(int(e))
        self.shared = None
        if wl.shared_I:
            from oracle import fp8block
            self.shared = fp8block.quantize_shared(sg.shared_w1_f32(wl), sg.shared_w2_f32(wl))
        # the timing needs plausible global scales, not calibrated ones: take gs1 from the sample's amax
        self.gs1 = np.float32(2688.0) / np.float32(np.abs(sg.bf16_bits_to_f32(self.x)).max())
        self.gs2 = np.float32(2688.0 / 100.0)

    def expert(self, e: int):
        from oracle import moe, mxfp4
        if e not in self.cache:
            wl = self.wl
            if self.mx:   # rank 0 of the TP3 shard, as the GPU arm runs it
                self.cache[e] = mxfp4.mx_expert_shard(sg.expert_w1_f32(self.full, e), sg.expert_w2_f32(self.full, e),
                                                      self.plan, 0)
            elif wl.w_format == 2:   # the same shard in the NVFP4 operand form
                sh = mxfp4.mx_expert_shard(sg.expert_w1_f32(self.full, e), sg.expert_w2_f32(self.full, e), self.plan, 0)
                q1, s1, g1 = mxfp4.mx_as_nvfp4(sh.w1_q, sh.w1_s)
                q2, s2, g2 = mxfp4.mx_as_nvfp4(sh.w2_q, sh.w2_s)
                self.cache[e] = moe.QuantExpert(q1, s1, g1, q2, s2, g2)
            else:
                self.cache[e] = moe.quantize_expert(sg.expert_w1_f32(wl, e), sg.expert_w2_f32(wl, e))
        return self.cache[e]

    def run(self, rows) -> float:
        from oracle import fp8block, moe, mxfp4
        wl, x = self.wl, self.x[rows]
        t0 = time.perf_counter()
        l = moe.router_logits(x, self.wr, self.bias)
        ids, w = moe.topk_softmax(l, wl.k)
        if self.mx:
            mxfp4.mx_moe_tokens(x, ids, w, self.expert, wl.swiglu_limit)
        else:
            o_se = None if self.shared is None else fp8block.shared_out(x, self.shared, wl.swiglu_limit)
            if wl.ep_count:   # one rank's share: local ids, pairs held elsewhere masked
                from oracle import layout
                moe.moe_tokens(x, layout.local_ids(ids, wl.ep_first, wl.ep_count), w,
                               lambda le: self.expert(wl.ep_first + le), self.gs1, self.gs2, wl.swiglu_limit,
                               shared=o_se)
            else:
                moe.moe_tokens(x, ids, w, self.expert, self.gs1, self.gs2, wl.swiglu_limit, shared=o_se)
        return time.perf_counter() - t0


def oracle_sample_time(wl, n_tokens: int, repeats: int = 1):
    """The oracle on the first n_tokens of the evaluation batch, repeats times.

    Returns a dict: tokens/s and seconds of the layer (routing, experts, combine); weight_decode_s, the time
    to dequantise the weights of the experts those tokens route to into fp64 tables (the oracle does this
    inside its layer, once per expert per call, so it is part of the seconds, reported apart); prep_s, the
    load-time quantisation of those experts (untimed)."""
    from oracle import mxfp4, nvfp4
    t0 = time.perf_counter()
    sample = OracleSample(wl, n_tokens)
    prep = time.perf_counter() - t0
    dt = sum(sample.run(slice(0, n_tokens)) for _ in range(repeats))
    t0 = time.perf_counter()
    for qe in sample.cache.values():
        if sample.mx:
            mxfp4.mx_dequantize(qe.w1_q, qe.w1_s), mxfp4.mx_dequantize(qe.w2_q, qe.w2_s)
        else:
            nvfp4.dequantize(qe.w1_q, qe.w1_sf, qe.w1_gs), nvfp4.dequantize(qe.w2_q, qe.w2_sf, qe.w2_gs)
    decode = (time.perf_counter() - t0) * repeats
    return {"value": n_tokens * repeats / dt, "seconds": dt, "weight_decode_s": decode, "prep_s": prep,
            "experts": len(sample.cache)}


def oracle_single_thread(wl_name: str, n_tokens: int):
    """oracle_sample_time in a child process whose BLAS and OpenMP pools hold one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1", NUMEXPR_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-only", "--workload", wl_name,
                        "--oracle-tokens", str(n_tokens)], capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout).strip().splitlines()[-1:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_info():
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    model = ""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    return cores, model


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=sg.DSV4_DECODE.name, choices=sorted(sg.WORKLOADS))
    ap.add_argument("--oracle-tokens", type=int, default=2)
    ap.add_argument("--reference-budget", type=float, default=60.0,
                    help="--impl reference: stop timing oracle steps once they took this many seconds")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the FP4 peak probe and the Zipf prefill measurement that follow the decode run")
    ap.add_argument("--prefill-steps", type=int, default=50)
    ap.add_argument("--side-steps", type=int, default=30,
                    help="steps of the TP3 MXFP4 workloads and replays per T of the graph sweep in the default run")
    ap.add_argument("--oracle-only", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--route-only", action="store_true",
                    help="time moe_route alone on the workload (a small case for profiler captures)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override E (smaller case for profiler captures; the default is the workload's E)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = sg.WORKLOADS[args.workload]
    if args.experts:
        import dataclasses
        wl = dataclasses.replace(wl, E=args.experts, name=f"{wl.name}_E{args.experts}")
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.oracle_only:   # the single-thread leg of the CPU baseline, run as a child process
        print(json.dumps(oracle_sample_time(wl, args.oracle_tokens)))
        return

    if args.impl == "reference":
        if rank != 0:
            return
        cores, model = cpu_info()
        # Each step is the oracle on one token of a fixed pool (the batch's first --oracle-tokens tokens, their
        # experts prepared once, untimed). The oracle takes seconds per token, so the run stops once the timed
        # steps pass --reference-budget seconds, or after --steps, whichever comes first, and reports how many
        # steps it timed; warm-up is at most one step (the oracle has nothing to warm up).
        sample = OracleSample(wl, args.oracle_tokens)
        n_warm = min(args.warmup, 1)
        for i in range(n_warm):
            sample.run([i % sample.n])
        per_step = []
        while len(per_step) < max(args.steps, 1) and sum(per_step) < args.reference_budget:
            per_step.append(sample.run([len(per_step) % sample.n]))
        steps = len(per_step)
        val = steps / sum(per_step)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": 1,
            "steps": steps, "steps_requested": args.steps, "warmup": n_warm, "warmup_requested": args.warmup,
            "reference_budget_s": args.reference_budget, "ms_per_step": 1e3 * sum(per_step) / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
                                            "top_k": wl.k},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"one token per step, cycling over the first {args.oracle_tokens} tokens of "
                                       f"the {wl.name} batch; {steps} steps timed ({model})"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    from block_scaled_fp4_top_gb300 import build as libbuild  # noqa: F401  (the library must exist)
    from block_scaled_fp4_top_gb300 import _lib
    _lib.load()
    if args.route_only:
        if rank == 0:
            print(json.dumps(run_route_only(args, wl, torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))))))
        return
    out = run_ours(args, wl, rank, world)
    if rank == 0 and not args.no_prefill and wl.name == sg.DSV4_DECODE.name and world == 1:
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
        peak = fp4_dense_peak(dev)
        out["fp4_dense_peak"] = peak
        torch.cuda.empty_cache()
        out["prefill"] = run_prefill(args, dev, peak["tflops"])
        torch.cuda.empty_cache()
        # config 4 (the TP3 MXFP4 shard): the bf16-activation path and the NVFP4-operand variant
        out["tp3_mxfp4"] = [run_side_workload(args, w, dev) for w in (sg.TP3_MXFP4, sg.TP3_MXFP4_NVACT)]
        torch.cuda.empty_cache()
        out["graph_sweep"] = run_graph_sweep(args, dev)
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        cores, model = cpu_info()
        allc = oracle_sample_time(wl, args.oracle_tokens)
        one = oracle_single_thread(wl.name, args.oracle_tokens)
        out["cpu_baseline"] = {
            "value": allc["value"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {args.oracle_tokens} tokens of the {wl.name} batch ({allc['experts']} experts), "
                      f"{allc['seconds']:.1f} s on all {cores} cores (numpy BLAS default threads)",
            "cpu_model": model,
            "all_cores": {"value": allc["value"], "seconds": allc["seconds"], "threads": cores,
                          "weight_decode_s": allc["weight_decode_s"]},
            "single_thread": {k: one.get(k) for k in ("value", "seconds", "weight_decode_s", "error") if k in one},
            "weight_prep_s": allc["prep_s"],
            "note": "weight_decode_s: dequantising the sample's experts to fp64 tables, a part of the seconds that "
                    "the oracle repeats on every call; weight_prep_s: their quantisation at load time, untimed"}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
