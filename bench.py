"""Benchmark of the sparse MoE feed-forward block on GB300.

Default workload (N=1): prefill of T=4096 tokens through one MoE layer
(d=2048, 256 experts top-8 + 1 shared, F=512, bf16 weights and activations,
fp32 accumulation), plus the batch-1 decode path over a stack of 40 distinct
layers with a fresh token per step.  `value` is prefill tokens/s; the decode
figures (microseconds per layer) are reported under "decode", and those of the
same stack with 4-bit group-affine expert weights under "decode_q4"; batches of
2..64 tokens through one layer under "small_batch"; the Gated DeltaNet scan of
one layer over a 2K-token prompt under "gdn".  `--no-side` leaves out every
object but the 4K prefill (for profiling); `--workload prefill_q4` prints the
4-bit prefill alone.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload prefill4k|skew16k|long128k|decode|decode_q4|small_batch|gdn2k|prefill_q4|tiny]
                    [--no-decode] [--no-side] [--no-cpu]

Timing: W untimed warm-up steps, then K timed steps, each bracketed by CUDA
events on the launching stream; a 256 MiB buffer is written between timed
steps to flush L2 (outside the events).  The per-kernel split (and the
roofline's kernel duration) comes from a second pass of K steps with events
around every kernel.  End to end ("e2e"): K steps through the host-buffer call
issued back to back, each copying its batch in from pinned host memory and its
result out, with one event pair around all of them.  Multi-GPU (torchrun): every rank runs
its own replica (tokens are independent; no collective on the data path),
value = all ranks' tokens / the slowest rank's time ("scaling": "weak").
The reference arm (--impl reference) times the CPU oracle on the host cores on
a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import sparse_mixture_experts_gemm_gb300 as moe  # noqa: E402
from sparse_mixture_experts_gemm_gb300 import synth  # noqa: E402

METRIC = "MoE block tokens/s (4K prefill) & decode µs/layer (batch 1); % of roofline"
D, F, E, K = 2048, 512, 256, 8

WORKLOADS = {
    "prefill4k": dict(T=4096, chunk=4096, seed=2, zipf=False, d=D, F=F, E=E, k=K, dtype="bf16"),
    "skew16k": dict(T=16384, chunk=16384, seed=3, zipf=True, d=D, F=F, E=E, k=K, dtype="bf16"),
    "long128k": dict(T=131072, chunk=8192, seed=4, zipf=False, d=D, F=F, E=E, k=K, dtype="bf16"),
    "tiny": dict(T=32, chunk=32, seed=0, zipf=False, d=512, F=128, E=256, k=8, dtype="f32"),
}


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm=j["hbm_gbs"], bf16=j["bf16_tflops"], bf16_sus=j["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ------------------------------------------------------------------ helpers
class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self) -> dict:
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


def make_layer(cfg: dict, dev, seed: int):
    w = synth.layer_weights(seed, cfg["d"], cfg["F"], cfg["E"], 1, cfg["dtype"], dev)
    bias = synth.zipf_bias(seed, cfg["E"], 1.2).to(dev) if cfg.get("zipf") else None
    layer = moe.MoELayer(w, cfg["k"], max_tokens=cfg["chunk"], bias=bias)
    return layer, w, bias


# DRAM bytes of one batch-1 layer (kernels A + B + C, reads; nothing is
# written back during them), from one ncu capture of the same kernel build.
DECODE_TRAFFIC_LAYER = 7_378_688 + 33_601_536 + 18_958_848
# The same for the 4-bit layer.
DECODE_Q4_TRAFFIC_LAYER = 1_082_368 + 10_668_032 + 5_349_632
# DRAM bytes (read + write) of one gate/up GEMM launch at T = 4096, from one
# ncu capture of the same kernel build.
GEMM1_TRAFFIC_4K = 1_095_424_512 + 7_973_888


def algorithmic_prefill(cfg: dict, counts: np.ndarray, T: int) -> dict:
    """Algorithmic work of one prefill pass: FLOPs and the minimum HBM bytes
    (weights of every expert with at least one row + shared + router, x read
    once, out written once)."""
    d, Fd, k = cfg["d"], cfg["F"], cfg["k"]
    es = 2 if cfg["dtype"] == "bf16" else 4
    active = int((counts > 0).sum())
    A = T * k
    flops = 2 * T * d * cfg["E"] + 6 * (A + T) * d * Fd
    w_bytes = (active + 1) * 3 * Fd * d * es + cfg["E"] * d * es
    bytes_ = w_bytes + 2 * T * d * es
    # gate/up GEMM alone: its weights, the tokens (each row is fetched once
    # from memory; its k + 1 uses gather it again from L2), the h it writes
    g1_bytes = (active + 1) * 2 * Fd * d * es + T * d * es + (A + T) * Fd * es
    g1_flops = 4 * (A + T) * d * Fd
    return dict(flops=flops, bytes=bytes_, active=active, g1_bytes=g1_bytes, g1_flops=g1_flops)


def flush_l2(buf):
    buf.fill_(1)


def workload_config(cfg: dict, wl_name: str, world: int) -> dict:
    """The line's `config` object: the same for both arms of one workload."""
    T = cfg["T"]
    return {
        "workload": f"{wl_name}: T={T} tokens through one MoE layer, d={cfg['d']}, "
                    f"{cfg['E']} experts top-{cfg['k']} + 1 shared, F={cfg['F']}"
                    + (", Zipf(1.2) router bias" if cfg["zipf"] else "")
                    + (f", chunks of {cfg['chunk']}" if cfg["chunk"] < T else ""),
        "tokens_per_step": T, "chunk": cfg["chunk"], "d_model": cfg["d"],
        "n_experts": cfg["E"], "top_k": cfg["k"], "d_ff": cfg["F"], "n_shared": 1,
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        "l2": "flushed between timed steps (256 MiB write outside the events)",
    }


# ------------------------------------------------------------------ our arm
def timed_steps(layer, x, out, steps, flush_buf, st, profile=False):
    """Per-step milliseconds of `steps` forwards, L2 flushed before each
    (outside the events).  profile: also time every kernel with the library's
    events on the launching stream and return {kind: (ms, launches)} as well.
    Those events make the front end drain before each next launch, so a
    profiled step runs longer than a plain one; the plain times are the step
    times, the profiled ones give the per-kernel split."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    if profile:
        moe.moe_profile(layer.handle, True)
    for i in range(steps):
        flush_l2(flush_buf)
        evs[i][0].record(st)
        layer.forward(x, out)
        evs[i][1].record(st)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    if not profile:
        return times
    prof = moe.moe_profile_read(layer.handle)
    moe.moe_profile(layer.handle, False)
    return times, prof


def bench_prefill(cfg, dev, steps, warmup, flush_buf):
    layer, w, bias = make_layer(cfg, dev, cfg["seed"])
    T = cfg["T"]
    x = synth.tokens(cfg["seed"] + 1000, T, cfg["d"], cfg["dtype"], dev)
    out = torch.empty_like(x)
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        layer.forward(x, out)
    torch.cuda.synchronize()
    rc, det = layer.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} ({det}) after warm-up")
    chunk_counts = []
    for c0 in range(0, T, cfg["chunk"]):
        _, _, cnt = layer.route(x[c0:c0 + cfg["chunk"]])
        chunk_counts.append(cnt.cpu().numpy())
    torch.cuda.synchronize()

    with Clocks(dev.index or 0) as clk:
        times = timed_steps(layer, x, out, steps, flush_buf, st)
    times_prof, prof = timed_steps(layer, x, out, steps, flush_buf, st, profile=True)
    rc, det = layer.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} ({det}) in timed region")

    # end to end through the host-buffer call (moe_forward_host): every step
    # copies its batch in from pinned host memory and its result back out, and
    # the handle overlaps one batch's copies with its neighbours' forwards.
    # Two batches (the tokens and a permutation of them) alternate.
    xh = [x.cpu().pin_memory(), x.roll(1, 0).cpu().pin_memory()]
    oh = [torch.empty_like(xh[0]).pin_memory() for _ in range(2)]
    for i in range(max(3, warmup)):
        layer.forward_host(xh[i % 2], oh[i % 2])
    layer.host_join()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for i in range(steps):
        layer.forward_host(xh[i % 2], oh[i % 2])
    layer.host_join()
    b.record(st)
    torch.cuda.synchronize()
    e2e_times = [a.elapsed_time(b) / steps] * steps
    rc, det = layer.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} ({det}) in the end-to-end steps")

    # the copies alone, for comparison with the step time
    c_ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    xd_ = torch.empty_like(x)
    for _ in range(2):
        c_ev[0].record(st)
        xd_.copy_(xh[0], non_blocking=True)
        c_ev[1].record(st)
        oh[0].copy_(xd_, non_blocking=True)
        c_ev[2].record(st)
        torch.cuda.synchronize()
    copy_ms = {"h2d": c_ev[0].elapsed_time(c_ev[1]), "d2h": c_ev[1].elapsed_time(c_ev[2])}

    # the same one step at a time: copy in, forward, copy out, L2 flushed between
    xd = torch.empty_like(x)
    od = torch.empty_like(x)
    for _ in range(max(1, warmup)):
        xd.copy_(xh[0], non_blocking=True)
        layer.forward(xd, od)
        oh[0].copy_(od, non_blocking=True)
    torch.cuda.synchronize()
    ser_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
    for i in range(steps):
        flush_l2(flush_buf)
        ser_ev[i][0].record(st)
        xd.copy_(xh[0], non_blocking=True)
        layer.forward(xd, od)
        oh[0].copy_(od, non_blocking=True)
        ser_ev[i][1].record(st)
    torch.cuda.synchronize()
    serial_times = [a_.elapsed_time(b_) for a_, b_ in ser_ev]
    res = dict(times=times, times_prof=times_prof, prof=prof, clocks=clk.summary(),
               e2e_times=e2e_times,
               serial_times=serial_times, copy_ms=copy_ms,
               counts=chunk_counts, h2d=xh[0].numel() * xh[0].element_size(),
               d2h=oh[0].numel() * oh[0].element_size(), layer=layer, w=w, bias=bias, x=x)
    return res


def gemm_kernels(chunk: int) -> dict:
    """The grouped-GEMM kernels that bf16 chunks of `chunk` tokens run on under
    the library's default options (two-CTA MMA for the gate/up GEMM from 8,192
    tokens and for the down GEMM from 16,384; cluster pairs of one-CTA MMAs
    for the down GEMM from 8,192; one CTA per tile below)."""
    gu = ("gemm2sm_kernel<EPI_SWIGLU> (two-CTA MMA, 256 x 256 tiles)" if chunk >= 8192
          else "gemm_kernel<bf16, EPI_SWIGLU, 256> (one CTA per 128 x 256 tile)")
    if chunk >= 16384:
        dn = "gemm2sm_kernel<EPI_STORE> (two-CTA MMA, 256 x 256 tiles)"
    elif chunk >= 8192:
        dn = "gemm_kernel<bf16, EPI_STORE, 256, pair> (cluster pairs sharing weight tiles)"
    else:
        dn = "gemm_kernel<bf16, EPI_STORE, 256> (one CTA per 128 x 256 tile)"
    return {"gate_up": gu, "down": dn}


def bench_prefill_side(name, dev, steps, warmup, flush_buf, pk) -> dict:
    """Another prefill configuration through the same kernels as the main
    line (skewed 16K, 128K in 8K chunks): step time, whole-step roofline and
    the per-kernel split from a second, event-profiled pass."""
    cfg = WORKLOADS[name]
    layer, w, bias = make_layer(cfg, dev, cfg["seed"])
    T = cfg["T"]
    x = synth.tokens(cfg["seed"] + 1000, T, cfg["d"], cfg["dtype"], dev)
    out = torch.empty_like(x)
    st = torch.cuda.current_stream()
    try:
        for _ in range(warmup):
            layer.forward(x, out)
        torch.cuda.synchronize()
        counts = [layer.route(x[c0:c0 + cfg["chunk"]])[2].cpu().numpy()
                  for c0 in range(0, T, cfg["chunk"])]
        with Clocks(dev.index or 0) as clk:
            times = timed_steps(layer, x, out, steps, flush_buf, st)
        times_prof, prof = timed_steps(layer, x, out, steps, flush_buf, st, profile=True)
        rc, det = layer.status()
        if rc != 0:
            raise RuntimeError(f"{name} device status {rc} ({det})")
    finally:
        layer.close()
    ms = statistics.mean(times)
    work = [algorithmic_prefill(cfg, c, min(cfg["chunk"], T - i * cfg["chunk"]))
            for i, c in enumerate(counts)]
    flops = sum(w_["flops"] for w_ in work)
    byts = sum(w_["bytes"] for w_ in work)
    t_tensor, t_hbm = flops / (pk["bf16"] * 1e12), byts / (pk["hbm"] * 1e9)
    per_step = {k_: v[0] / max(steps, 1) for k_, v in prof.items() if v[1] > 0}
    g1_ms = prof["gemm_gate_up"][0] / max(prof["gemm_gate_up"][1], 1)
    g2_ms = prof["gemm_down"][0] / max(prof["gemm_down"][1], 1)
    g1_flops = sum(w_["g1_flops"] for w_ in work) / len(work)
    g2_flops = g1_flops / 2  # the down projection: half the gate/up multiply-adds
    return {
        "workload": workload_config(cfg, name, 1)["workload"],
        "tokens_per_s": T / (ms * 1e-3), "ms_per_step": ms,
        "ms_per_step_with_kernel_events": statistics.mean(times_prof),
        "flops_per_step": flops, "algorithmic_bytes_per_step": byts,
        "gemm_kernels": gemm_kernels(cfg["chunk"]),
        "experts_with_rows_per_chunk": [int((c > 0).sum()) for c in counts],
        "largest_group_rows": int(max(c.max() for c in counts)),
        "block_roofline": {"bound": "tensor" if t_tensor >= t_hbm else "hbm",
                           "t_roof_ms": max(t_tensor, t_hbm) * 1e3,
                           "frac": max(t_tensor, t_hbm) * 1e3 / ms,
                           "tensor_frac_of_measured_burst": t_tensor * 1e3 / ms,
                           "tensor_frac_of_measured_sustained":
                               flops / (ms * 1e-3) / (pk["bf16_sus"] * 1e12),
                           "hbm_frac_of_measured": t_hbm * 1e3 / ms},
        "gemm_tensor_frac_of_measured_burst": {
            "gate_up": g1_flops / (g1_ms * 1e-3) / (pk["bf16"] * 1e12),
            "down": g2_flops / (g2_ms * 1e-3) / (pk["bf16"] * 1e12)},
        "kernels_ms_per_step": per_step,
        "kernel_times_from": "event pair around every kernel on the launching stream "
                             "(second pass of the same steps)",
        "gpu_launches": sum(v[1] for v in prof.values()),
        "clocks": clk.summary(),
    }


def bench_prefill_q4(cfg, dev, steps, warmup, flush_buf, pk) -> dict:
    """The same prefill with 4-bit group-affine expert weights (seeded random
    codes, scales and biases; bf16 router and tokens): the grouped GEMMs
    dequantise each weight block on the chip."""
    d, F, E, k, T = cfg["d"], cfg["F"], cfg["E"], cfg["k"], cfg["T"]
    w = synth.q4_layer_weights(cfg["seed"] + 7, d, F, E, 1, dev)
    layer = moe.Q4Layer(w, k, max_tokens=cfg["chunk"])
    x = synth.tokens(cfg["seed"] + 1000, T, d, "bf16", dev)
    out = torch.empty_like(x)
    st = torch.cuda.current_stream()
    try:
        for _ in range(warmup):
            layer.forward(x, out)
        torch.cuda.synchronize()
        _, _, cnt = layer.route(x[:cfg["chunk"]])
        counts = cnt.cpu().numpy()
        with Clocks(dev.index or 0) as clk:
            times = timed_steps(layer, x, out, steps, flush_buf, st)
        times_prof, prof = timed_steps(layer, x, out, steps, flush_buf, st, profile=True)
        rc, det = layer.status()
        if rc != 0:
            raise RuntimeError(f"4-bit prefill device status {rc} ({det})")
        small = bench_small_batch(layer, cfg, dev, flush_buf, pk, q4=True)
    finally:
        layer.close()
    ms = statistics.mean(times)
    active = int((counts > 0).sum())
    A = T * k
    flops = 2 * T * d * E + 6 * (A + T) * d * F
    q4b = 0.5 + 4 / 64  # bytes per weight: codes, bf16 scale and bias per 64
    byts = (active + 1) * 3 * F * d * q4b + E * d * 2 + 2 * T * d * 2
    per = {kk: v[0] / max(v[1], 1) for kk, v in prof.items() if v[1] > 0}
    g1_ms = per.get("gemm_gate_up", 0.0)
    g1_flops = 4 * (A + T) * d * F
    return {
        "tokens_per_s": T / (ms * 1e-3), "ms_per_step": ms,
        "ms_per_step_with_kernel_events": statistics.mean(times_prof),
        "workload": f"prefill T={T} (d={d}, {E} experts top-{k} + 1 shared, F={F}), 4-bit "
                    "group-affine expert weights (64 per group, bf16 scale and bias), bf16 "
                    "router and tokens, L2 flushed between steps",
        "flops_per_step": flops, "algorithmic_bytes_per_step": byts,
        "roofline": {"bound": "tensor", "achieved": g1_flops / (g1_ms * 1e-3) / 1e12,
                     "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": g1_flops / (g1_ms * 1e-3) / 1e12 / pk["bf16"], "traffic": None,
                     "kernel": "gemm_gate_up (4-bit weights)",
                     "peak_source": f"{pk['src']} bf16_tflops"} if g1_ms > 0 else None,
        "whole_step_floors_us": {"tensor": flops / (pk["bf16"] * 1e12) * 1e6,
                                 "hbm": byts / (pk["hbm"] * 1e9) * 1e6},
        "kernels_ms_per_step": per, "clocks": clk.summary(),
        "gpu_launches": sum(v[1] for v in prof.values()) // max(steps, 1) * steps,
        "small_batch": small,
    }


def slowest_rank_ms(total_ms: float, steps: int, world: int, device=None) -> float:
    """Mean step time of the slowest rank: each rank passes the sum of its
    timed steps, the MAX over ranks (all_reduce on the default process group)
    is divided by the step count.  One rank: its own mean."""
    if world <= 1:
        return total_ms / steps
    import torch.distributed as dist
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item() / steps


def whole_job_rate(units_per_rank: float, ms_per_step: float, world: int) -> float:
    """Units all ranks process per second, timed by the slowest rank."""
    return world * units_per_rank / (ms_per_step / 1e3)


def bench_small_batch(layer, cfg, dev, flush_buf, pk, iters=50, q4=False) -> dict:
    """Batches of 2..64 tokens through the same layer (the verification shape
    of speculative decoding): one routing launch, then the grouped GEMV on all
    SMs (at most 16 tokens with bf16 weights, 32 with 4-bit ones) or the
    grouped GEMMs, the combine; eager calls as
    a user makes them, L2 flushed before each.  q4: the layer has 4-bit expert
    weights (0.5625 bytes a weight)."""
    d, F, E, k = cfg["d"], cfg["F"], cfg["E"], cfg["k"]
    st = torch.cuda.current_stream()
    out = {}
    for T in (2, 4, 8, 16, 32, 64):
        x = synth.tokens(cfg["seed"] + 5000 + T, T, d, "bf16", dev)
        for _ in range(5):
            layer.forward(x)
        _, _, cnt = layer.route(x)
        active = int((cnt > 0).sum().item())
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(iters)]
        for a, b in evs:
            flush_l2(flush_buf)
            a.record(st)
            layer.forward(x)
            b.record(st)
        torch.cuda.synchronize()
        rc, det = layer.status()
        if rc != 0:
            raise RuntimeError(f"small-batch device status {rc} ({det})")
        us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)
        byts = (active + 1) * 3 * F * d * (0.5 + 4 / 64 if q4 else 2) + E * d * 2
        out[str(T)] = {"us_per_layer_median": us, "experts_touched": active,
                       "algorithmic_bytes": byts,
                       "hbm_frac_of_measured": byts / (us * 1e-6) / (pk["hbm"] * 1e9)}
    return {"workload": "T = 2, 4, 8, 16, 32, 64 tokens through one layer (d=2048, 256 experts top-8 + "
                        "1 shared, F=512, " + ("4-bit group-affine expert weights, bf16 router "
                                               "and tokens" if q4 else "bf16") +
                        "), eager calls, L2 flushed before each, median of "
                        f"{iters}", "by_T": out, "gpu_launches_per_layer": 4}


GDN = {"T": 2048, "Hk": 16, "Hv": 32, "dk": 128, "dv": 128, "seed": 31}
# DRAM bytes (read + write) of one scan launch on that workload, from an ncu
# capture; None: the kernel this workload runs (two column groups per CTA) has
# not been captured since it changed
GDN_TRAFFIC_2K = None


def bench_gdn(dev, flush_buf, pk, iters=20, cpu_tokens=64) -> dict:
    """Gated DeltaNet scan of one layer over a 2,048-token prompt (16 key heads,
    32 value heads, d_k = d_v = 128, fp32 state in registers), L2 flushed
    before each call; the oracle timed beside it on a bounded sample."""
    c = GDN
    inp = synth.gdn_inputs(c["seed"], c["T"], c["Hk"], c["Hv"], c["dk"], c["dv"], dev, state=True)
    st = torch.cuda.current_stream()
    o = torch.empty((c["T"], c["Hv"], c["dv"]), dtype=torch.bfloat16, device=dev)
    s_out = torch.empty_like(inp["state"])
    args = (inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], inp["state"])
    for _ in range(3):
        moe.gdn_scan(*args, out=o, state_out=s_out)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    with Clocks(dev.index or 0) as clk:
        for a, b in evs:
            flush_l2(flush_buf)
            a.record(st)
            moe.gdn_scan(*args, out=o, state_out=s_out)
            b.record(st)
        torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)
    cols = c["Hv"] * c["dv"]
    fma = c["T"] * cols * 3 * c["dk"]  # recall, read-out and update per state entry and token
    byts = (2 * c["T"] * c["Hk"] * c["dk"] * 2 + 2 * c["T"] * cols * 2 + 2 * c["T"] * c["Hv"] * 4
            + 2 * cols * c["dk"] * 4)
    peak = 152 * 128 * 2 * 2.07e9 / 1e12  # fp32 lanes x 2 flops x maximum SM clock
    res = {
        "workload": f"Gated DeltaNet scan, one layer: T={c['T']} tokens, {c['Hk']} key heads, "
                    f"{c['Hv']} value heads, d_k=d_v={c['dk']}, bf16 q/k/v, fp32 gate, "
                    "strength and state, L2 flushed before each call",
        "us_per_layer_median": us, "tokens_per_s": c["T"] / (us * 1e-6),
        "us_per_token": us / c["T"],
        "roofline": {"bound": "alu", "achieved": 2 * fma / (us * 1e-6) / 1e12, "peak": peak,
                     "unit": "TFLOP/s", "frac": 2 * fma / (us * 1e-6) / 1e12 / peak,
                     "traffic": GDN_TRAFFIC_2K, "algorithmic_bytes": byts,
                     "hbm_frac_of_measured": byts / (us * 1e-6) / (pk["hbm"] * 1e9),
                     "peak_source": "152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz (nominal)"},
        "clocks": clk.summary(), "gpu_launches": iters,
    }
    if cpu_tokens:
        import oracle
        cpu = {k: (None if v is None else v[:cpu_tokens].cpu()) for k, v in inp.items()
               if k != "state"}
        bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
        t0 = time.perf_counter()
        oracle.gdn_scan(bits(cpu["q"]), bits(cpu["k"]), bits(cpu["v"]), cpu["alpha"].numpy(),
                        cpu["beta"].numpy(), inp["state"].cpu().numpy())
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": cpu_tokens / dt, "unit": "tokens/s", "cores": 1,
                               "kind": "oracle",
                               "sample": f"first {cpu_tokens} of the {c['T']} tokens, all heads, "
                                         f"{dt:.2f} s, numpy float64"}
    return res


def bench_decode(dev, steps, warmup, n_layers=40, q4=False):
    cfg = WORKLOADS["prefill4k"]
    layers = []
    for l in range(n_layers):
        if q4:
            w = synth.q4_layer_weights(1000 + l, cfg["d"], cfg["F"], cfg["E"], 1, dev)
            layer = moe.Q4Layer(w, cfg["k"])
            layer.keep = w
        else:
            layer, w, _ = make_layer(dict(cfg, chunk=1), dev, 1000 + l)
        layers.append(layer)
    d = cfg["d"]
    xs = synth.tokens(1, steps + warmup, d, "bf16", dev)
    x_in = torch.empty((1, d), dtype=torch.bfloat16, device=dev)
    outs = [torch.empty((1, d), dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    st = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(st):
        x_in.copy_(xs[0:1])
        for l, layer in enumerate(layers):  # eager pass (also loads everything)
            layer.forward(x_in, outs[l], stream=st)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for l, layer in enumerate(layers):
                layer.forward(x_in, outs[l], stream=st)
        for i in range(warmup):
            x_in.copy_(xs[i:i + 1])
            g.replay()
        st.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        with Clocks(dev.index or 0) as clk:
            for i in range(steps):
                x_in.copy_(xs[warmup + i:warmup + i + 1])
                evs[i][0].record(st)
                g.replay()
                evs[i][1].record(st)
            st.synchronize()
        # per-kernel split on one eager step with events between the kernels
        for layer in layers:
            moe.moe_profile(layer.handle, True)
        for l, layer in enumerate(layers):
            layer.forward(x_in, outs[l], stream=st)
        st.synchronize()
        split = {}
        for layer in layers:
            for kname, (ms, n) in moe.moe_profile_read(layer.handle).items():
                a = split.setdefault(kname, [0.0, 0])
                a[0] += ms
                a[1] += n
            moe.moe_profile(layer.handle, False)
    for layer in layers:
        rc, det = layer.status(st)
        if rc != 0:
            raise RuntimeError(f"decode device status {rc} ({det})")
    times = [a.elapsed_time(b) for a, b in evs]
    for layer in layers:
        layer.close()
    del g
    return dict(times=times, clocks=clk.summary(), split=split, n_layers=n_layers, q4=q4)


# ------------------------------------------------------------------ oracle arm
def oracle_prefill_rate(cfg, w, x, bias, n_tokens, nthreads, min_seconds=0.0, max_passes=1):
    """Oracle tokens/s on the first n_tokens of the batch (host cores): passes
    over the sample repeat until min_seconds have passed (at most max_passes).
    Returns (tokens/s, seconds, passes)."""
    import oracle
    oracle.build()

    def npv(t):
        t = t.detach().contiguous().cpu()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 \
            else t.numpy()

    wr, wg, wu, wd = npv(w["Wr"]), npv(w["Wg"]), npv(w["Wu"]), npv(w["Wd"])
    sg, su, sd = npv(w["Sg"]), npv(w["Su"]), npv(w["Sd"])
    xs = npv(x[:n_tokens])
    b = None if bias is None else bias.detach().cpu().numpy()
    t0 = time.perf_counter()
    passes = 0
    while True:
        oracle.forward(xs, wr, list(wg), list(wu), list(wd), cfg["k"], sg=sg, su=su, sd=sd, bias=b,
                       nthreads=nthreads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= max_passes:
            break
    return n_tokens * passes / dt, dt, passes


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill4k",
                    choices=["prefill4k", "skew16k", "long128k", "tiny", "decode", "decode_q4",
                             "small_batch", "gdn2k", "prefill_q4"])
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--decode-layers", type=int, default=40,
                    help="distinct layers in the decode stack (40 in the benchmark; fewer for profiling)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="only the 4K prefill: no 16K/128K, 4-bit, small-batch or scan objects")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--oracle-seconds", type=float, default=10.0,
                    help="minimum host seconds of the oracle baseline (whole passes)")
    ap.add_argument("--oracle-tokens", type=int, default=1 << 30,
                    help="tokens of the batch the CPU baseline runs on (about 10-30 s)")
    ap.add_argument("--reference-tokens", type=int, default=256,
                    help="tokens per step of the reference (oracle) arm")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")

    wl_name = ("prefill4k" if args.workload.startswith("decode")
               or args.workload in ("small_batch", "gdn2k", "prefill_q4") else args.workload)
    cfg = WORKLOADS[wl_name]
    pk = peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, cfg, wl_name)
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    moe.build()
    flush_buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()

    if args.workload.startswith("decode"):
        dec = bench_decode(dev, args.decode_steps, max(args.warmup, 50), args.decode_layers,
                           q4=args.workload == "decode_q4")
        emit_decode_line(args, dec, pk, world)
        return

    if args.workload == "gdn2k":
        g = bench_gdn(dev, flush_buf, pk, iters=args.steps, cpu_tokens=0 if args.no_cpu else 64)
        print(json.dumps({
            "metric": "Gated DeltaNet scan time per layer, 2K-token prompt",
            "value": g["us_per_layer_median"], "unit": "us/layer", "n_gpus": world,
            "steps": args.steps, "warmup": 3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)",
            "config": {"workload": g["workload"]}, "roofline": g["roofline"],
            "clocks": g["clocks"], "gpu_launches": g["gpu_launches"], "gdn": g}))
        return

    if args.workload == "prefill_q4":
        q = bench_prefill_q4(cfg, dev, args.steps, args.warmup, flush_buf, pk)
        print(json.dumps({
            "metric": "prefill tokens/s, 4-bit expert weights", "value": q["tokens_per_s"],
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": q["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
            "config": {"workload": q["workload"]}, "roofline": q["roofline"],
            "clocks": q["clocks"], "gpu_launches": q["gpu_launches"], "prefill_q4": q}))
        return

    if args.workload == "small_batch":
        layer, _, _ = make_layer(cfg, dev, cfg["seed"])
        try:
            sb = bench_small_batch(layer, cfg, dev, flush_buf, pk, iters=args.steps)
        finally:
            layer.close()
        t16 = sb["by_T"]["16"]
        print(json.dumps({
            "metric": "small-batch layer time at T=16", "value": t16["us_per_layer_median"],
            "unit": "us/layer", "n_gpus": world, "steps": args.steps, "warmup": 5,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded)", "config": {"workload": sb["workload"]},
            "small_batch": sb}))
        return

    res = bench_prefill(cfg, dev, args.steps, args.warmup, flush_buf)
    T = cfg["T"]
    ms = statistics.mean(res["times"])
    ms_max = slowest_rank_ms(sum(res["times"]), len(res["times"]), world, dev)
    value = whole_job_rate(T, ms_max, world)
    e2e_ms = slowest_rank_ms(sum(res["e2e_times"]), len(res["e2e_times"]), world, dev)
    serial_ms = slowest_rank_ms(sum(res["serial_times"]), len(res["serial_times"]), world, dev)

    counts = np.sum(res["counts"], axis=0) if len(res["counts"]) == 1 else None
    work = [algorithmic_prefill(cfg, c, min(cfg["chunk"], T - i * cfg["chunk"]))
            for i, c in enumerate(res["counts"])]
    flops = sum(w_["flops"] for w_ in work)
    bytes_ = sum(w_["bytes"] for w_ in work)
    g1_ms, g1_n = res["prof"]["gemm_gate_up"]
    g1_avg = g1_ms / max(g1_n, 1)
    g1_bytes = sum(w_["g1_bytes"] for w_ in work) / len(work)
    g1_flops = sum(w_["g1_flops"] for w_ in work) / len(work)
    achieved = g1_bytes / (g1_avg / 1e3) / 1e9
    t_roof = max(flops / (pk["bf16"] * 1e12), bytes_ / (pk["hbm"] * 1e9))
    launches_per_step = 4 * len(work)  # router, gate/up, down, combine per chunk
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if cfg["dtype"] == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights)",
        "config": workload_config(cfg, wl_name, world),
        "roofline": {
            "kernel": "grouped gate/up GEMM + SiLU: " + gemm_kernels(cfg["chunk"])["gate_up"],
            "bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
            "frac": achieved / pk["hbm"],
            "traffic": GEMM1_TRAFFIC_4K if wl_name == "prefill4k" and GEMM1_TRAFFIC_4K else None,
            "peak_source": f"{pk['src']} hbm_gbs",
            "algorithmic_bytes_per_launch": g1_bytes, "avg_launch_ms": g1_avg,
            "tensor_frac_of_measured_burst": g1_flops / (g1_avg / 1e3) / (pk["bf16"] * 1e12),
        },
        "block_roofline": {
            "flops_per_step": flops, "bytes_per_step": bytes_,
            "t_roof_ms": t_roof * 1e3, "frac": t_roof * 1e3 / ms,
            "bound": "hbm" if bytes_ / (pk["hbm"] * 1e9) >= flops / (pk["bf16"] * 1e12) else "tensor",
            "tensor_frac_of_measured_burst": flops / (ms / 1e3) / (pk["bf16"] * 1e12),
            "hbm_frac_of_measured": bytes_ / (ms / 1e3) / (pk["hbm"] * 1e9),
        },
        "kernels_ms_per_step": {k_: v[0] / max(args.steps, 1) for k_, v in res["prof"].items()
                                if v[1] > 0},
        "kernel_times_from": "a second pass of the same steps with an event pair around every "
                             "kernel on the launching stream (the events cost the step "
                             "launch overlap: see ms_per_step_with_kernel_events)",
        "ms_per_step_with_kernel_events": slowest_rank_ms(sum(res["times_prof"]),
                                                          len(res["times_prof"]), world, dev),
        "e2e": {"value": whole_job_rate(T, e2e_ms, world), "unit": "tokens/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "ms_per_step": e2e_ms, "copies_alone_ms": res["copy_ms"],
                "how": "moe_forward_host on pinned host buffers, steps issued back to back, "
                       "one moe_host_join, events around all steps; each batch's copies "
                       "overlap the neighbouring batches' forwards; no L2 flush (each "
                       f"step reads {bytes_ / 1e9:.3f} GB; L2 holds 0.13 GB)",
                "serial": {"value": whole_job_rate(T, serial_ms, world), "ms_per_step": serial_ms,
                           "how": "copy in, moe_forward, copy out per step, L2 flushed "
                                  "between steps outside the events"}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": res["clocks"],
    }
    if not args.no_decode and wl_name == "prefill4k":
        dec = bench_decode(dev, args.decode_steps, max(args.warmup, 50), args.decode_layers)
        line["decode"] = decode_summary(dec, pk)
        dec = bench_decode(dev, args.decode_steps, max(args.warmup, 50), args.decode_layers,
                           q4=True)
        line["decode_q4"] = decode_summary(dec, pk)
        # decode launches are counted in their own objects
    if wl_name == "prefill4k" and not args.no_side:
        for side in ("skew16k", "long128k"):
            line[side] = bench_prefill_side(side, dev, args.steps, args.warmup, flush_buf, pk)
        line["prefill_q4"] = bench_prefill_q4(cfg, dev, args.steps, args.warmup, flush_buf, pk)
        line["small_batch"] = bench_small_batch(res["layer"], cfg, dev, flush_buf, pk)
        line["gdn"] = bench_gdn(dev, flush_buf, pk, cpu_tokens=64 if rank == 0 else 0)
    if rank == 0 and not args.no_cpu:
        nthr = host_threads()
        n_tok = min(args.oracle_tokens, T)
        rate, dt, passes = oracle_prefill_rate(cfg, res["w"], res["x"], res["bias"], n_tok, nthr,
                                               min_seconds=args.oracle_seconds, max_passes=8)
        what = (f"the whole {T}-token batch" if n_tok == T
                else f"first {n_tok} of the {T} tokens of the same batch")
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": nthr, "kind": "oracle",
                                "sample": f"{what}, {passes} pass(es) in {dt:.1f} s, "
                                          f"{cpu_model()}"}
    res["layer"].close()
    line["summary"] = summary_of(line)  # last key: the record keeps the line's tail
    if rank == 0:
        print(json.dumps(line))


def summary_of(line: dict) -> dict:
    """The headline figures of every object of the line, in a few hundred
    bytes: prefill 4K, decode, the other prefill configurations, 4-bit
    weights, small batches and the scan."""
    r3 = lambda v: None if v is None else round(v, 3)  # noqa: E731
    main = line["config"]["workload"].split(":")[0]
    out = {main: {"Mtok_s": r3(line["value"] / 1e6), "ms": r3(line["ms_per_step"]),
                         "block_frac": r3(line["block_roofline"]["frac"]),
                         "gate_up_hbm_frac": r3(line["roofline"]["frac"]),
                         "e2e_Mtok_s": r3(line["e2e"]["value"] / 1e6)}}
    for key in ("decode", "decode_q4"):
        if key in line:
            dsum = line[key]
            out[key] = {"us_per_layer": r3(dsum["us_per_layer_median"]),
                        "hbm_frac": r3(dsum["roofline"]["frac"])}
    for key in ("skew16k", "long128k"):
        if key in line:
            o = line[key]
            out[key] = {"Mtok_s": r3(o["tokens_per_s"] / 1e6), "ms": r3(o["ms_per_step"]),
                        "block_frac": r3(o["block_roofline"]["frac"]),
                        "bound": o["block_roofline"]["bound"],
                        "gate_up_tensor_frac": r3(o["gemm_tensor_frac_of_measured_burst"]["gate_up"])}
    if "prefill_q4" in line:
        out["prefill_q4"] = {"ms": r3(line["prefill_q4"]["ms_per_step"])}
    for key in ("small_batch",):
        if key in line:
            out[key] = {T: {"us": r3(v["us_per_layer_median"]), "hbm_frac": r3(v["hbm_frac_of_measured"])}
                        for T, v in line[key]["by_T"].items()}
    if "gdn" in line:
        out["gdn_us"] = r3(line["gdn"]["us_per_layer_median"])
    return out


def decode_summary(dec, pk) -> dict:
    per_layer_us = [t * 1e3 / dec["n_layers"] for t in dec["times"]]
    med = statistics.median(per_layer_us)
    p90 = float(np.percentile(per_layer_us, 90))
    q4 = dec.get("q4", False)
    # router rows (bf16) + the k + 1 experts' three matrices: 2 bytes a weight,
    # or 4-bit codes plus a bf16 scale and bias per 64 weights (0.5625 bytes)
    byts = E * D * 2 + (K + 1) * 3 * F * D * (0.5 + 4 / 64 if q4 else 2)
    achieved = byts / (med * 1e-6) / 1e9
    split = {k_: v[0] * 1e3 / max(v[1], 1) for k_, v in dec["split"].items() if v[1] > 0}
    return {
        "us_per_layer_median": med, "us_per_layer_p90": p90,
        "tokens_per_s": 1e6 / (med * dec["n_layers"]),
        "layers": dec["n_layers"], "steps": len(dec["times"]),
        "workload": f"batch-1 decode: one fresh token per step through {dec['n_layers']} "
                    "distinct layers (d=2048, 256 experts top-8 + 1 shared, F=512, "
                    + ("4-bit group-affine expert weights, bf16 router and tokens"
                       if q4 else "bf16") + "), CUDA graph per step",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                     "frac": achieved / pk["hbm"],
                     "traffic": DECODE_Q4_TRAFFIC_LAYER if q4 else DECODE_TRAFFIC_LAYER,
                     "algorithmic_bytes_per_layer": byts,
                     "peak_source": f"{pk['src']} hbm_gbs"},
        "eager_us_per_launch": split,
        "gpu_launches": 3 * dec["n_layers"] * len(dec["times"]),
        "clocks": dec["clocks"],
    }


def emit_decode_line(args, dec, pk, world):
    s = decode_summary(dec, pk)
    line = {
        "metric": METRIC, "value": s["us_per_layer_median"], "unit": "us/layer",
        "n_gpus": world, "steps": len(dec["times"]), "warmup": max(args.warmup, 50),
        "ms_per_step": statistics.mean(dec["times"]), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded)", "config": {"workload": s["workload"]},
        "roofline": s["roofline"], "gpu_launches": s["gpu_launches"], "clocks": s["clocks"],
        "decode": s,
    }
    print(json.dumps(line))


def run_reference(args, cfg, wl_name):
    """The CPU oracle on the host cores, same metric and config as our arm.
    Each step is a bounded sample of the workload (the first
    --reference-tokens tokens of the same batch, through the same layer):
    `ms_per_step` is the time of that sample, `value` the tokens it processed
    per second; --warmup untimed steps come first."""
    import oracle
    oracle.build()
    T = cfg["T"]
    w = synth.layer_weights(cfg["seed"], cfg["d"], cfg["F"], cfg["E"], 1, cfg["dtype"], "cpu")
    x = synth.tokens(cfg["seed"] + 1000, T, cfg["d"], cfg["dtype"], "cpu")
    bias = synth.zipf_bias(cfg["seed"], cfg["E"], 1.2) if cfg["zipf"] else None
    nthr = host_threads()
    n_tok = min(args.reference_tokens, T)
    for _ in range(args.warmup):
        oracle_prefill_rate(cfg, w, x, bias, n_tok, nthr)
    dts = []
    for _ in range(args.steps):
        _, dt, _ = oracle_prefill_rate(cfg, w, x, bias, n_tok, nthr)
        dts.append(dt)
    ms = statistics.mean(dts) * 1e3
    rate = n_tok / (ms / 1e3)
    sample = (f"first {n_tok} of the {T} tokens of the same batch per step "
              f"({ms / 1e3:.2f} s per step), {nthr} threads, {cpu_model()}")
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights)",
        "config": workload_config(cfg, wl_name, 1),
        "tokens_timed_per_step": n_tok,
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": nthr, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
