#!/usr/bin/env python
"""Benchmark of the GB300 MoE layer (forward of a Kimi-class layer with skewed routing by default).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl mok|reference]

One step = one pass of the whole layer forward over one batch of T tokens: router GEMM + top-k,
pull-schedule counting sort, pull gather, gate/up GEMM + SwiGLU, down GEMM + router weight,
fixed-order combine (training workloads add the backward).  Inputs are synthetic, seeded, and
resident in HBM before the timed region; the gigabytes of expert weights read every step exceed
the 129 MB L2, so no explicit flush is needed.  Prints ONE JSON line on rank 0.

--impl reference times the float64 CPU oracle (as it stands) on the host cores on a bounded
sample of the same workload, one sampled token per step.

Multi-GPU (torchrun, N > 1): every rank runs an independent replica of the workload on its own
GPU (the layer has no exchange step on one node here); barrier + max-over-ranks timing only.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(PEAKS_FALLBACK)
    d["source"] = "fallback"
    return d


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def dist_init(world):
    if world > 1:
        import torch.distributed as dist

        if not dist.is_initialized():
            dist.init_process_group("gloo")


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def dist_max(value, world):
    """Max of a float over ranks (timing plumbing only, CPU tensors over gloo)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, tokens_per_rank, steps, ms_max):
    """Tokens per second of the whole job: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (ms_max / 1e3)


# ------------------------------------------------------------------ clocks during the timed region
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ algorithmic work model
def work_model(shape, counts):
    """Algorithmic FLOPs and HBM bytes per step for the whole layer and per kernel.
    counts: tokens per routed expert (for the active-expert weight bytes)."""
    T, d, E, k, F, Fs, ns = shape.T, shape.d, shape.E, shape.k, shape.F, shape.F_shared, shape.n_shared
    R = T * k
    Rs = R + T * ns
    Hs = R * F + T * ns * Fs          # elements of one [rows, F] activation, routed + shared
    e_act = sum(1 for c in counts if c > 0)
    wb = 2  # bf16
    train = shape.backward
    m = {}
    m["route"] = {"flops": 2.0 * T * d * E, "bytes": wb * (T * d + d * E) + 8.0 * T * k}
    # x is read once (repeated rows of a token hit L2), every destination row written once
    m["gather"] = {"flops": 0.0, "bytes": wb * (T * d + R * d) + 4.0 * R}
    # gate/up: the active weight sets, x once (the re-reads of a token's gathered rows are the
    # kernel's own materialisation, not algorithmic), h written (and G, U saved for training)
    m["gemm_fwd_gate_up"] = {
        "flops": 2.0 * (R * 2 * F * d + T * ns * 2 * Fs * d),
        "bytes": wb * (e_act * 2.0 * d * F + ns * 2.0 * d * Fs + T * d + Hs * (3 if train else 1))}
    m["gemm_fwd_down"] = {
        "flops": 2.0 * (R * F * d + T * ns * Fs * d),
        "bytes": wb * (e_act * 1.0 * F * d + ns * 1.0 * Fs * d + Hs + Rs * d)}
    m["combine"] = {"flops": 0.0, "bytes": wb * (Rs * d + T * d) + 8.0 * R}
    layer_flops = T * (2.0 * d * E + (k * 6.0 * d * F) + ns * 6.0 * d * Fs)
    if shape.dtype == "mxfp8":
        wq = 1.0 + 1.0 / 32  # E4M3 byte + one UE8M0 byte per 32
        m["mx_quantize"] = {"flops": 0.0, "bytes": T * d * (wb + wq)}
        m["gather_bytes"] = {"flops": 0.0, "bytes": wq * (T * d + R * d) + 4.0 * R}
        m["gemm_fwd_gate_up_mx"] = {  # (training: G and U saved in fp32)
            "flops": m["gemm_fwd_gate_up"]["flops"], "dtype": "fp8",
            "bytes": wq * (e_act * 2.0 * d * F + ns * 2.0 * d * Fs + T * d + Hs)
            + (8.0 * Hs if train else 0.0)}
        m["gemm_fwd_down_mx"] = {
            "flops": m["gemm_fwd_down"]["flops"], "dtype": "fp8",
            "bytes": wq * (e_act * 1.0 * F * d + ns * 1.0 * Fs * d + Hs) + wb * Rs * d}
    if shape.dtype == "nvfp4":
        wq = 0.5 + 1.0 / 16  # an E2M1 nibble + one E4M3 byte per 16 (the per-matrix scales: noise)
        m["nv_quantize_x"] = {"flops": 0.0, "bytes": T * d * (wb + 2.0)}  # bf16 in, f16 values out
        m["gemm_fwd_gate_up_nv"] = {  # f16 products at the bf16 rate; x values once, h written
            "flops": m["gemm_fwd_gate_up"]["flops"], "dtype": "f16",
            "bytes": wq * (e_act * 2.0 * d * F + ns * 2.0 * d * Fs) + 2.0 * (T * d + Hs)}
        m["gemm_fwd_down_nv"] = {
            "flops": m["gemm_fwd_down"]["flops"], "dtype": "f16",
            "bytes": wq * (e_act * 1.0 * F * d + ns * 1.0 * Fs * d) + 2.0 * Hs + wb * Rs * d}
    if train:
        m["gather_dy"] = {"flops": 0.0, "bytes": wb * (T * d + R * d) + 4.0 * R}
        m["gemm_bwd_da"] = {  # a = dY Wd^T; reads G, U; writes dG, dU, w*h
            "flops": 2.0 * (R * F * d + T * ns * Fs * d),
            "bytes": wb * (e_act * 1.0 * F * d + ns * 1.0 * Fs * d + Rs * d + 5.0 * Hs) + 4.0 * R * 16}
        m["router_bwd"] = {"flops": 0.0, "bytes": 4.0 * T * E + wb * T * E + 4.0 * R * 16}
        m["gemm_bwd_dx"] = {  # dX = dG Wg^T + dU Wu^T (+ dl Wr^T)
            "flops": 2.0 * (R * 2 * F * d + T * ns * 2 * Fs * d + T * E * d),
            "bytes": wb * (e_act * 2.0 * d * F + ns * 2.0 * d * Fs + 2.0 * Hs + Rs * d + T * E)}
        m["gemm_bwd_dw"] = {  # dWg, dWu, dWd (written for every expert) and x^T dl
            "flops": 2.0 * (3.0 * (R * F * d + T * ns * Fs * d) + T * d * E),
            "bytes": wb * (3.0 * (E * d * F + ns * d * Fs) + 2.0 * Rs * d + 3.0 * Hs + d * E)}
        if shape.dtype == "mxfp8":
            wq = 1.0 + 1.0 / 32
            ops_t = 2.0 * Rs * d + 3.0 * Hs  # token-axis operands: x, dY, dG, dU, w*h
            m["gemm_bwd_da_mx"] = {  # reads dY codes, W_down codes, fp32 G, U; writes the codes of
                # dG, dU along F and of dG, dU, w*h along tokens
                "flops": m["gemm_bwd_da"]["flops"], "dtype": "fp8",
                "bytes": wq * (e_act * 1.0 * F * d + ns * 1.0 * Fs * d + Rs * d + 5.0 * Hs)
                + 4.0 * 2.0 * Hs + 4.0 * R * (F // 128)}
            m["gemm_bwd_dx_mx"] = {
                "flops": 2.0 * (R * 2 * F * d + T * ns * 2 * Fs * d), "dtype": "fp8",
                "bytes": wq * (e_act * 2.0 * d * F + ns * 2.0 * d * Fs + 2.0 * Hs) + wb * Rs * d}
            m["gemm_bwd_dx"] = {"flops": 2.0 * T * E * d, "bytes": wb * (T * E + d * E + T * d)}
            m["gemm_bwd_dw_mx"] = {
                "flops": 2.0 * 3.0 * (R * F * d + T * ns * Fs * d), "dtype": "fp8",
                "bytes": wb * 3.0 * (E * d * F + ns * d * Fs) + wq * ops_t}
            m["gemm_bwd_dw"] = {"flops": 2.0 * T * d * E, "bytes": wb * (T * d + T * E + d * E)}
            # per launch (one per group: x and dY)
            m["mx_quantize_tokens"] = {"flops": 0.0,
                                       "bytes": (wb + wq) * 2.0 * Rs * d / (1.0 + ns)}
        layer_flops = 3.0 * layer_flops
    return m, layer_flops, e_act


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum, a one-pass ncu metric
# captured on the full-size workload) for (workload, kernel), valid only while the kernel source
# is the one that was captured (sha1 prefix of the file); None otherwise.
_GEMM_SRC = "mixture_experts_layer_14_gb300/csrc/moe_gemm.cu"
PROFILED_TRAFFIC = {
    # ncu captures of the Kimi-class forward at full size (4th step of a 3-warm-up bench run)
    ("kimi_skew_bf16_fwd", "gemm_fwd_gate_up"): ("296ca27805b4", 23.383e9 + 0.606e9, _GEMM_SRC),
    ("kimi_skew_bf16_fwd", "gemm_fwd_down"): ("296ca27805b4", 5.944e9 + 2.100e9, _GEMM_SRC),
    # the same one-pass capture on the other forward workloads at full size
    ("dsv3_bf16_fwd", "gemm_fwd_gate_up"): ("296ca27805b4", 15.922e9 + 0.152e9, _GEMM_SRC),
    ("dsv3_bf16_fwd", "gemm_fwd_down"): ("296ca27805b4", 7.715e9 + 0.520e9, _GEMM_SRC),
    ("dsv3_decode_t64", "gemm_fwd_gate_up"): ("296ca27805b4", 13.329e9 + 0.006e9, _GEMM_SRC),
    ("dsv3_decode_t64", "gemm_fwd_down"): ("296ca27805b4", 6.645e9 + 0.008e9, _GEMM_SRC),
    ("dsv3_mxfp8_fwd", "gemm_fwd_gate_up_mx"): ("296ca27805b4", 8.524e9 + 0.158e9, _GEMM_SRC),
    ("dsv3_mxfp8_fwd", "gemm_fwd_down_mx"): ("296ca27805b4", 4.048e9 + 1.036e9, _GEMM_SRC),
    ("dsv3_nvfp4_fwd", "gemm_fwd_gate_up_nv"): ("296ca27805b4", 5.503e9 + 0.150e9, _GEMM_SRC),
    ("dsv3_nvfp4_fwd", "gemm_fwd_down_nv"): ("296ca27805b4", 2.592e9 + 0.511e9, _GEMM_SRC),
    ("dsv3_nvfp4_decode_t64", "gemm_fwd_gate_up_nv"): ("296ca27805b4", 3.585e9 + 0.005e9, _GEMM_SRC),
    ("dsv3_nvfp4_decode_t64", "gemm_fwd_down_nv"): ("296ca27805b4", 1.786e9 + 0.008e9, _GEMM_SRC),
    # the training steps (4th step of a 3-warm-up run), forward and backward expert GEMMs
    ("dsv3_bf16_train", "gemm_fwd_gate_up"): ("296ca27805b4", 16.875e9 + 0.900e9, _GEMM_SRC),
    ("dsv3_bf16_train", "gemm_fwd_down"): ("296ca27805b4", 7.851e9 + 1.043e9, _GEMM_SRC),
    ("dsv3_bf16_train", "gemm_bwd_da"): ("296ca27805b4", 9.480e9 + 0.889e9, _GEMM_SRC),
    ("dsv3_bf16_train", "gemm_bwd_dx"): ("296ca27805b4", 16.556e9 + 1.049e9, _GEMM_SRC),
    ("dsv3_bf16_train", "gemm_bwd_dw"): ("296ca27805b4", 5.576e9 + 22.587e9, _GEMM_SRC),
    ("dsv3_mxfp8_train", "gemm_fwd_gate_up_mx"): ("296ca27805b4", 8.775e9 + 1.350e9, _GEMM_SRC),
    ("dsv3_mxfp8_train", "gemm_fwd_down_mx"): ("296ca27805b4", 4.048e9 + 1.036e9, _GEMM_SRC),
    ("dsv3_mxfp8_train", "gemm_bwd_da_mx"): ("296ca27805b4", 5.750e9 + 0.864e9, _GEMM_SRC),
    ("dsv3_mxfp8_train", "gemm_bwd_dx_mx"): ("296ca27805b4", 8.116e9 + 1.043e9, _GEMM_SRC),
    ("dsv3_mxfp8_train", "gemm_bwd_dw_mx"): ("296ca27805b4", 2.325e9 + 22.578e9, _GEMM_SRC),
}


def profiled_traffic(workload, name):
    import hashlib

    key = (workload, name)
    if key not in PROFILED_TRAFFIC:
        return None
    sha, nbytes, src = PROFILED_TRAFFIC[key]
    with open(os.path.join(ROOT, src), "rb") as f:
        if hashlib.sha1(f.read()).hexdigest()[:12] != sha:
            return None  # the kernel changed since the counters were taken
    return nbytes


# What each forward kernel's algorithmic bytes count (a kernel's own re-reads of rows it
# materialised, e.g. gathered token rows read once per N tile, are not counted).
BYTE_BASIS = {
    "gemm_fwd_gate_up": "active gate+up weight sets + x once (T d) + h written (+ G, U saved)",
    "gemm_fwd_gate_up_mx": "active gate+up E4M3 weights and scales + x codes once + h codes written",
    "gemm_fwd_gate_up_nv": "active gate+up E2M1 weights and E4M3 scales + x values (f16) once + h values (f16) written",
    "gemm_fwd_down_nv": "active down E2M1 weights and E4M3 scales + h values (f16) read + router-weighted rows Y_s written",
    "gemm_fwd_down": "active down weight sets + h read + router-weighted rows Y_s written",
    "gemm_fwd_down_mx": "active down E4M3 weights and scales + h codes read + Y_s written",
    "combine": "(k + 1) rows read + one row written per token",
    "gather": "x read once + every destination row written",
    "route": "x read once + W_router + top-k written",
}


SUSTAINED_AFTER_MS = 2000.0  # timed regions this long run under the power cap: sustained peak


def roofline_of(name, model, ms_per_launch, peaks, sustained=False):
    w = model[name]
    # the measured bf16 peak (burst for a short timed region, the seconds-long sustained figure
    # for a long one); an FP8 contraction takes it times the nominal fp8/bf16 ratio (2), an f16
    # one (the NVFP4 GEMMs' decoded operands) the bf16 figure itself
    base = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) if sustained else peaks["bf16_tflops"]
    tpeak = base * (2.0 if w.get("dtype") == "fp8" else 1.0)
    t_flop = w["flops"] / (tpeak * 1e12) if w["flops"] else 0.0
    t_byte = w["bytes"] / (peaks["hbm_gbs"] * 1e9)
    secs = ms_per_launch / 1e3
    if t_flop > t_byte:
        achieved = w["flops"] / secs / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": tpeak,
                "unit": "TFLOP/s", "frac": achieved / tpeak, "algorithmic_per_launch": w["flops"],
                "peak_dtype": w.get("dtype", "bf16"),
                "peak_kind": "sustained (power-capped loop)" if sustained else "burst"}
    achieved = w["bytes"] / secs / 1e9
    out = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": achieved / peaks["hbm_gbs"], "algorithmic_per_launch": w["bytes"]}
    if name in BYTE_BASIS:
        out["bytes_basis"] = BYTE_BASIS[name]
    return out


# ------------------------------------------------------------------ CPU oracle baseline
def oracle_sample_inputs(L, shape, tokens):
    """Host float64 copies of what the oracle needs for `tokens` (untimed set-up)."""
    import numpy as np
    import torch

    import oracle

    f64 = lambda t: t.detach().to("cpu").to(torch.float64).numpy()  # noqa: E731
    x = f64(L["x"][tokens])
    Wr = f64(L["W_router"])
    b = None if L["bias"] is None else f64(L["bias"])
    _, _, idx, _ = oracle.route(x, Wr, b, shape.k)
    experts = sorted(set(int(e) for e in np.asarray(idx).ravel()))
    Wg = {e: f64(L["W_gate"][e]) for e in experts}
    Wu = {e: f64(L["W_up"][e]) for e in experts}
    Wd = {e: f64(L["W_down"][e]) for e in experts}
    shared = (f64(L["Ws_gate"]), f64(L["Ws_up"]), f64(L["Ws_down"])) if shape.n_shared else None
    return dict(x=x, Wr=Wr, b=b, Wg=Wg, Wu=Wu, Wd=Wd, shared=shared)


def oracle_step(O, shape, rows):
    """One timed oracle step on sampled token rows: router, pull schedule, experts, combine."""
    import oracle

    x = O["x"][rows]
    l64, _, idx, w = oracle.route(x, O["Wr"], O["b"], shape.k)
    oracle.dispatch(idx, shape.E)
    return oracle.moe_forward(x, O["Wg"], O["Wu"], O["Wd"], O["shared"], idx, w)


def oracle_cores():
    try:
        import threadpoolctl

        info = threadpoolctl.threadpool_info()
        blas = [i.get("num_threads") for i in info if i.get("user_api") == "blas"]
        if blas:
            return int(max(blas))
    except ImportError:
        pass
    return os.cpu_count()


def cpu_baseline(L, shape, pool_tokens=2, budget_s=12.0, max_steps=64):
    tokens = list(range(pool_tokens))
    O = oracle_sample_inputs(L, shape, tokens)
    oracle_step(O, shape, [0])  # warm-up
    t_total, n = 0.0, 0
    while t_total < budget_s and n < max_steps:
        t0 = time.perf_counter()
        oracle_step(O, shape, [n % pool_tokens])
        t_total += time.perf_counter() - t0
        n += 1
    return {"value": n / t_total, "unit": "tokens/s", "cores": oracle_cores(), "kind": "oracle",
            "sample": (f"{n} steps of 1 token each, cycling over tokens 0..{pool_tokens - 1} of the "
                       f"{shape.name} batch (T={shape.T}); per step: float64 router over all "
                       f"{shape.E} experts, pull schedule, {shape.k} routed SwiGLU experts + the "
                       f"shared expert, combine; weights converted to float64 once, untimed")}


# ------------------------------------------------------------------ the GB300 arm
TIMING_EVERY = 4  # per-launch event timing on every 4th timed step
# NVFP4: calibrated amax of h for these synthetic inputs (SiLU(g) u with g, u about N(0, 1));
# the rare larger values saturate, as the recipe has it
NV_AMAX_H = 8.0


def measure(args, shape, steps, warmup, dev, world, peaks, L=None):
    """Times `steps` whole-layer steps of `shape` (forward, plus backward for training
    workloads).  Returns the measurement and the layer inputs."""
    import torch

    import mixture_experts_layer_14_gb300 as mok
    from mixture_experts_layer_14_gb300.synthetic import make_layer

    if L is None:
        L = make_layer(shape, dev, with_dy=shape.backward)
    mx = shape.dtype == "mxfp8"
    nv = shape.dtype == "nvfp4"
    D = mok.dims(shape.T, shape.d, shape.E, shape.k, shape.F, shape.F_shared, shape.n_shared,
                 mok.MOK_MXFP8 if mx else mok.MOK_NVFP4 if nv else mok.MOK_BF16)
    if mx or nv:  # weights are quantised once, outside the timed region
        L["prepared"] = mok.prepare_weights(D, L)
        if shape.backward:
            L["prepared_bwd"] = mok.prepare_weights_bwd(D, L)
    if nv:  # calibration: x's amax from the batch, h's the value calibrated for these inputs
        mok.nvfp4_set_activation_amax(D, L["prepared"], float(L["x"].abs().max()), NV_AMAX_H)
    layer = mok.MoELayer(D, L, dev)
    x = L["x"]
    torch.cuda.synchronize()

    def step():
        layer.forward(x, training=shape.backward)
        n = layer.last_launches  # router, dispatch and expert-forward kernels
        if shape.backward:
            layer.backward(x, L["dY"])
            n += layer.last_launches
        return n

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    counts = layer.routing["counts"].cpu().tolist()

    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index or 0)
    dist_barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    # per-launch CUDA events on every TIMING_EVERY-th timed step (they cost about 1% of a step)
    ev0.record(stream)
    launches = 0
    sampled = 0
    for i in range(steps):
        on = i % TIMING_EVERY == 0
        mok.timing_enable(on)
        sampled += on
        launches += step()
    ev1.record(stream)
    torch.cuda.synchronize()
    mok.timing_enable(False)
    clocks = sampler.stop()
    dist_barrier(world)
    ms = ev0.elapsed_time(ev1)
    kern = mok.timing_collect()
    for ws in (layer.ws, layer._ws_bwd):
        if ws is not None and mok.read_status(ws) != 0:
            raise RuntimeError(f"device status {mok.read_status(ws)} after the timed region")
    ms_max = dist_max(ms, world)

    model, layer_flops, e_act = work_model(shape, counts)
    sustained = ms >= SUSTAINED_AFTER_MS
    kernels = {}
    for name, (n, tms) in sorted(kern.items(), key=lambda kv: -kv[1][1]):
        entry = {"launches": n, "ms_total": round(tms, 4), "ms_per_launch": round(tms / max(n, 1), 5),
                 "share": round((tms / max(sampled, 1)) / max(ms / steps, 1e-9), 4)}
        if name in model:
            r = roofline_of(name, model, tms / max(n, 1), peaks, sustained)
            r["traffic"] = profiled_traffic(shape.name, name)
            entry["roofline"] = {k2: (round(v, 4) if isinstance(v, float) else v) for k2, v in r.items()}
        kernels[name] = entry
    dominant = max((n for n in kern if n in model), key=lambda n: kern[n][1])
    dn, dms = kern[dominant]
    roof = roofline_of(dominant, model, dms / dn, peaks, sustained)
    roof.update({"kernel": dominant, "traffic": profiled_traffic(shape.name, dominant),
                 "peak_source": "measured (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
                 else "fallback"})
    tflops = layer_flops * steps / (ms / 1e3) / 1e12
    tpeak = peaks["bf16_tflops"] * (2.0 if mx else 1.0)
    out = {
        "value": round(whole_job_value(world, shape.T, steps, ms_max), 1),
        "ms_per_step": round(ms_max / steps, 4),
        "tflops": round(tflops, 2),
        "tflops_frac_of_bf16_peak": round(tflops / peaks["bf16_tflops"], 4),
        "tflops_frac_of_dtype_peak": round(tflops / tpeak, 4),
        "dtype": "mxfp8 (e4m3 + ue8m0/32)" if mx else
                 "nvfp4 (e2m1 + e4m3/16 + fp32 per tensor; f16 tensor-core products)" if nv else "bf16",
        "roofline": {k2: (round(v, 4) if isinstance(v, float) else v) for k2, v in roof.items()},
        "kernels": kernels, "kernel_timing": f"CUDA events on {sampled} of the {steps} timed steps",
        "gpu_launches": launches, "clocks": clocks,
        "active_experts": e_act, "max_expert_rows": max(counts), "empty_experts": counts.count(0),
        "weight_gb_per_step": round(weight_bytes_per_step(shape, counts) / 1e9, 3),
    }
    if mx:  # context: the library's dense fp8 GEMM rate on this GPU (the roofline keeps 2 x bf16)
        f8 = fp8_cublas_tflops(dev)
        out["fp8_cublas_tflops_measured"] = f8
        out["tflops_frac_of_measured_fp8_gemm"] = round(tflops / f8, 4) if f8 else None
    del layer
    return out, L


def fp8_cublas_tflops(dev):
    """Dense e4m3 x e4m3 -> bf16 GEMM throughput of the library routine (torch._scaled_mm at
    8192^3, best of 10 CUDA-event-timed calls), reported beside the MXFP8 workload for context;
    None where the routine is unavailable."""
    import torch

    try:
        n = 8192
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        best = None
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return round(2.0 * n ** 3 / (best / 1e3) / 1e12, 1)
    except Exception as exc:
        print(f"fp8 GEMM rate unavailable: {exc!r}"[:300], file=sys.stderr)
        return None


def weight_bytes_per_step(shape, counts):
    """Bytes of expert weights one forward streams: every active routed expert and the shared."""
    b = {"mxfp8": 1.0 + 1.0 / 32, "nvfp4": 0.5 + 1.0 / 16}.get(shape.dtype, 2.0)
    e_act = sum(1 for c in counts if c > 0)
    return b * 3.0 * shape.d * (e_act * shape.F + shape.n_shared * shape.F_shared)


def config_of(shape, world):
    """The workload definition (identical in both arms); routing statistics are reported apart."""
    return {"workload": shape.name, "T": shape.T, "d": shape.d, "E": shape.E, "k": shape.k,
            "F": shape.F, "F_shared": shape.F_shared, "n_shared": shape.n_shared,
            "router_bias": shape.bias, "pass": "fwd+bwd" if shape.backward else "fwd",
            "expert_gemms": shape.dtype,
            "global_batch_tokens": world * shape.T, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2: every step streams the active experts' weights "
                  "(gigabytes) through the 129 MB L2, no flush needed"}


def metric_of(shape):
    return "MoE-layer fwd+bwd tokens/s" if shape.backward else "MoE-layer forward tokens/s"


def run_mok(args, shape, rank, world, local_rank):
    import torch

    import mixture_experts_layer_14_gb300 as mok
    from mixture_experts_layer_14_gb300.synthetic import WORKLOADS

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks = load_peaks()
    mok.set_forward_schedule(mok.SCHEDULE_FUSED if args.schedule == "fused" else mok.SCHEDULE_TWO_LAUNCHES)
    res, L = measure(args, shape, args.steps, args.warmup, dev, world, peaks)
    D = mok.dims(shape.T, shape.d, shape.E, shape.k, shape.F, shape.F_shared, shape.n_shared)
    e2e = None
    if not args.no_e2e and not shape.backward:
        e2e = run_e2e(args, mok, D, L, shape, dev, world)
    graph = None
    if not shape.backward and shape.dtype == "bf16":
        graph = run_graph(args, mok, D, L, shape, dev, world)
    line = {
        "metric": metric_of(shape),
        "value": res["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/sqrt(fan_in)) bf16 weights, random init)",
        "config": config_of(shape, world),
        "routing": {k2: res[k2] for k2 in ("active_experts", "max_expert_rows", "empty_experts",
                                           "weight_gb_per_step")},
        "tflops": res["tflops"], "tflops_frac_of_bf16_peak": res["tflops_frac_of_bf16_peak"],
        "roofline": res["roofline"], "kernels": res["kernels"], "kernel_timing": res["kernel_timing"],
        "gpu_launches": res["gpu_launches"], "forward_schedule": args.schedule,
        "clocks": res["clocks"], "e2e": e2e, "cuda_graph": graph,
    }
    for key in ("fp8_cublas_tflops_measured", "tflops_frac_of_measured_fp8_gemm"):
        if key in res:
            line[key] = res[key]
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(L, shape, budget_s=args.cpu_seconds)
    del L
    torch.cuda.empty_cache()
    if not args.no_extra:
        extra = {}
        for name in args.extra.split(","):
            if not name or name == shape.name:
                continue
            try:
                r, Lx = measure(args, WORKLOADS[name], min(args.steps, args.extra_steps), 3, dev, world, peaks)
                del Lx
                torch.cuda.empty_cache()
                r["metric"] = metric_of(WORKLOADS[name])
                r["kernels"] = {k2: v for k2, v in list(r["kernels"].items())[:6]}
                extra[name] = r
            except Exception as exc:  # report, do not hide the headline
                extra[name] = {"error": repr(exc)[:300]}
        line["workloads"] = extra
    return line


def run_graph(args, mok, D, L, shape, dev, world):
    """The same device-resident step replayed from a CUDA graph (route, pull schedule and expert
    forward captured once): the launch-overhead-free time of the layer."""
    import torch

    layer = mok.MoELayer(D, L, dev)
    x = L["x"]
    for _ in range(max(args.warmup, 1)):
        layer.forward(x)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer.forward(x)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x)
    for _ in range(max(args.warmup, 1)):
        graph.replay()
    torch.cuda.synchronize()
    dist_barrier(world)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = dist_max(e0.elapsed_time(e1), world)
    if mok.read_status(layer.ws) != 0:
        raise RuntimeError("device status after the graph replays")
    del graph, layer
    return {"value": round(world * shape.T * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
            "ms_per_step": round(ms / args.steps, 4)}


def run_e2e(args, mok, D, L, shape, dev, world):
    """Same metric through the host-buffer C-ABI call: H2D copy of x from pinned memory, the
    layer, D2H copy of y, every step."""
    import torch

    ws = torch.zeros(mok.workspace_size(D) + mok.host_extra_size(D), dtype=torch.uint8, device=dev)
    xh = L["x"].cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    for _ in range(max(args.warmup, 1)):
        mok.layer_forward_host(D, L, xh, yh, ws)
    torch.cuda.synchronize()
    dist_barrier(world)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        mok.layer_forward_host(D, L, xh, yh, ws)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = dist_max(e0.elapsed_time(e1), world)
    nbytes = shape.T * shape.d * 2
    return {"value": round(world * shape.T * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
            "ms_per_step": round(ms / args.steps, 4)}


# ------------------------------------------------------------------ the reference arm (oracle)
def run_reference(args, shape, rank, world, local_rank):
    import torch

    from mixture_experts_layer_14_gb300.synthetic import make_layer

    dev = torch.device("cuda", local_rank) if torch.cuda.is_available() else torch.device("cpu")
    if dev.type == "cuda":
        torch.cuda.set_device(local_rank)
    L = make_layer(shape, dev)
    pool = 2
    O = oracle_sample_inputs(L, shape, list(range(pool)))
    del L
    for i in range(args.warmup):
        oracle_step(O, shape, [i % pool])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_step(O, shape, [i % pool])
    secs = time.perf_counter() - t0
    value = args.steps / secs
    sample = (f"1 token per step cycling over tokens 0..{pool - 1} of the {shape.name} batch "
              f"(T={shape.T}): float64 router, pull schedule, {shape.k} routed experts + shared, "
              f"combine; weights converted to float64 once, untimed")
    return {
        "metric": metric_of(shape), "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(shape, world),
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": oracle_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    from mixture_experts_layer_14_gb300.synthetic import WORKLOADS

    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mok", "reference"], default="mok")
    ap.add_argument("--workload", default="kimi_skew_bf16_fwd", choices=sorted(WORKLOADS))
    ap.add_argument("--schedule", choices=["two_launches", "fused"], default="two_launches",
                    help="schedule of the bf16 forward's expert GEMMs (mok_set_forward_schedule)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--extra", default="dsv3_bf16_fwd,dsv3_bf16_train,dsv3_mxfp8_fwd,"
                    "dsv3_mxfp8_train,dsv3_decode_t64,dsv3_nvfp4_fwd,dsv3_nvfp4_decode_t64")
    ap.add_argument("--extra-steps", type=int, default=30)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_env()
    shape = WORKLOADS[args.workload]
    if args.impl == "reference":
        if rank != 0:
            return 0
        line = run_reference(args, shape, rank, world, local_rank)
    else:
        dist_init(world)
        line = run_mok(args, shape, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
