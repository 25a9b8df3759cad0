#!/usr/bin/env python3
"""Throughput of one TSP transformer layer forward (bf16) on GB300.

One step = one tsp_layer_fwd call on the whole workload: zigzag permute, the
QKV projection over all weight shards with the fused K/V gather, the
zigzag-balanced causal flash attention, the output projection accumulated over
shards (+ residual), the gate/up projection with the fused SiLU*up epilogue,
the down projection accumulated over the MLP ring's shards (+ residual) and
the unpermute.  Default workload: D = 8 virtual ranks, batch 2, seq 16384,
hidden 4096, 32 heads x 128, SwiGLU ffn 14336 (the 7B dense decoder shape).

Prints one JSON line.  `value` is layer-forward TFLOP/s with inputs resident
in device memory; `e2e` repeats the measurement through the public API with
the input copied from pinned host memory and the output copied back inside
the timed region.  After the timed region the line also times, at the same
size, the zigzag permute, the K/V all-gather and the unpermute called on their
own (HBM-bound; `layout_kernels`, `roofline_hbm`).  `--impl reference` times
the fp64 CPU oracle instead (on a bounded prefix of the same workload,
single-threaded).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from folded_tensor_sequence_gb300.configs import BY_NAME, LAYER_7B_S16K  # noqa: E402
from folded_tensor_sequence_gb300.replicas import max_over_ranks, rank_env, whole_job_rate  # noqa: E402

METRIC = "TSP layer fwd TFLOP/s & tokens/s (bf16) at 1 GB300; % of dense bf16 tensor peak"
# (for the training workload the same metric counts the step's model flops, 3x the forward)
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch
# of a step's kernel, keyed by (step, workload), with the kernel source file
# and the first 16 hex digits of its sha256 when the counters were taken
# (one-pass capture of the full-size launch, see profiles/).  A workload
# without its own capture, or a source changed since, reports null.
NCU_TRAFFIC = {
    ("gate/up projection", "bf16_D8_b2_s16384_h4096"):
        (2174.07e6 + 926.63e6, "folded_tensor_sequence_gb300/csrc/gemm_tc.cu", "16a0278f61e1aa96"),
    # the same launch (M, N, K and kernel) as the multi-head workload's gate/up projection
    ("gate/up projection", "bf16_gqa8_D8_b2_s16384_h4096"):
        (2174.07e6 + 926.63e6, "folded_tensor_sequence_gb300/csrc/gemm_tc.cu", "16a0278f61e1aa96"),
    ("attention", "bf16_D8_b2_s16384_h4096"):
        (833.823e6 + 250.399e6, "folded_tensor_sequence_gb300/csrc/attn_fwd_tc.cu", "6c52c6aefe671f3b"),
    ("attention", "bf16_D8_b1_s65536_h4096"):
        (2278.46e6 + 567.390e6, "folded_tensor_sequence_gb300/csrc/attn_fwd_tc.cu", "6c52c6aefe671f3b"),
    ("attention bwd fused", "bf16_fwdbwd_D8_b2_s16384_h4096"):
        (1643.48e6 + 1040.48e6, "folded_tensor_sequence_gb300/csrc/attn_bwd_tc.cu", "908c433fee92d1ce"),
    ("attention bwd fused", "bf16_fwdbwd_D8_b1_s8192_h4096"):
        (406.761e6 + 222.230e6, "folded_tensor_sequence_gb300/csrc/attn_bwd_tc.cu", "908c433fee92d1ce"),
    ("attention bwd fused", "bf16_fwdbwd_gqa8_D8_b1_s8192_h4096"):
        (651.287e6 + 289.550e6, "folded_tensor_sequence_gb300/csrc/attn_bwd_tc.cu", "908c433fee92d1ce"),
    ("kv gather (standalone)", "bf16_D8_b2_s16384_h4096"):
        (536.906e6 + 485.511e6, "folded_tensor_sequence_gb300/csrc/layout.cu", "b3e6ab7624313095"),
    ("zigzag permute (standalone)", "bf16_D8_b2_s16384_h4096"):
        (268.450e6 + 216.774e6, "folded_tensor_sequence_gb300/csrc/layout.cu", "b3e6ab7624313095"),
    ("decode attention", "bf16_decode_D8_b1_ctx131072_h4096"):
        (2.15e9 + 0.00292e9, "folded_tensor_sequence_gb300/csrc/decode.cu", "3bfb1d17f6da32df"),
    ("decode attention", "bf16_decode_gqa8_D8_b4_ctx131072_h4096"):
        (2.15e9 + 0.00627e9, "folded_tensor_sequence_gb300/csrc/decode.cu", "3bfb1d17f6da32df"),
}


def ncu_traffic(step: str, workload: str):
    ent = NCU_TRAFFIC.get((step, workload))
    if not ent:
        return None
    import hashlib

    with open(os.path.join(ROOT, ent[1]), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return ent[0] if sha == ent[2] else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def host_cpu() -> dict:
    """The host the CPU baseline ran on: logical CPUs and the CPU model name."""
    import platform

    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.processor() or "unknown",
            "machine": platform.machine()}


# Dense bf16 tcgen05 rate per SM: one 128 x 256 x 16 MMA (2^20 flops) every 128
# SM cycles, timed on the GPU with clock64 around back-to-back MMAs on all SMs.
BF16_FLOPS_PER_SM_CYCLE = 8192


def nominal_bf16_tflops(num_sms: int, sm_mhz) -> float | None:
    """Dense bf16 tensor peak at a given SM clock (the clock-derived issue rate)."""
    if not sm_mhz:
        return None
    return BF16_FLOPS_PER_SM_CYCLE * num_sms * sm_mhz * 1e6 / 1e12


def step_work(cfg, cfg_det=False):
    """Algorithmic work per launch of each step: (flops, bytes, kernels launched);
    cfg_det: the backward runs the split (deterministic) attention kernels."""
    B, S, h, F, H, dh = cfg.batch, cfg.seq, cfg.hidden, cfg.ffn, cfg.heads, cfg.head_dim
    T = B * S
    e = 2 if cfg.dtype == "bf16" else 4
    hk = cfg.kv_hidden       # K/V width (h unless grouped-query attention)
    W3 = h + 2 * hk          # packed Q|K|V width
    attn = 4 * B * H * dh * S * (S + 1) // 2
    w = {
        "zigzag permute": (0, 2 * T * h * e, 1),
        "QKV projection": (2 * T * h * W3, (T * h + W3 * h + T * W3) * e, 1),
        "attention": (attn, (2 * T * h + 2 * T * hk) * e, 1),
        "output projection": (2 * T * h * h, (3 * T * h + h * h) * e, 1),
        "gate/up projection": (2 * T * h * 2 * F, (T * h + 2 * F * h + T * F) * e, 1),
        "down projection": (2 * T * F * h, (T * F + F * h + 2 * T * h) * e, 1),
        "zigzag unpermute": (0, 2 * T * h * e, 1),
    }
    if cfg.decode:
        # one token per sequence: every projection streams its weight, attention streams the cache
        return {
            "decode QKV projection": (0, (h * W3 + B * h + B * W3) * e, 1),
            "decode attention": (0, (2 * B * S * hk + 2 * B * h) * e, 2),
            "decode output projection": (0, (h * h + 3 * B * h) * e, 1),
            "decode gate/up projection": (0, (2 * F * h + B * h + B * F) * e, 1),
            "decode down projection": (0, (h * F + B * F + 2 * B * h) * e, 1),
        }
    if cfg.backward:
        w.update({
            "permute dy": (0, 2 * T * h * e, 1),
            "dM = dY Wd^T": (2 * T * h * F, (T * h + F * h + 4 * T * F) * e, 1),
            "dW_down": (2 * h * F * T, (T * h + T * F + h * F) * e, 1),
            "dH": (2 * T * 2 * F * h, (2 * T * F + 2 * F * h + 2 * T * h) * e, 1),
            "dW_gate_up": (2 * 2 * F * h * T, (2 * T * F + T * h + 2 * F * h) * e, 1),
            "dO": (2 * T * h * h, (2 * T * h + h * h) * e, 1),
            "dW_O": (2 * h * h * T, (2 * T * h + h * h) * e, 1),
            "transpose V^T": (0, 2 * T * hk * e, 1),
            "attention bwd": (2 * attn, (4 * T * h + 4 * T * hk) * e, 3),
            # rowsum(dO * O); zeroes the fp32 dQ accumulator when the fused kernel follows
            "attention bwd dsum": (0, 2 * T * h * e + (0 if cfg_det else 4 * T * h), 1),
            # model flops of the backward attention: 2 x the forward's (dP, dV, dK, dQ; the S
            # recompute is not counted).  Fused: one kernel, dQ added into the fp32 accumulator.
            "attention bwd fused": (2 * attn, (2 * T * h + 4 * T * hk) * e + 4 * T * h, 1),
            # split (deterministic): dK/dV computes dP, dV and dK; dQ computes dQ.  The S
            # recompute (both kernels) and the dQ kernel's second dP are not counted.
            "attention bwd dK/dV": (3 * attn // 2, (2 * T * h + 4 * T * hk) * e, 1),
            "attention bwd dQ": (attn // 2, (2 * T * h + 2 * T * hk) * e + 4 * T * h, 1),
            "assemble dQKV": (0, (T * W3 + 2 * T * hk) * e + 4 * T * h, 1),
            "dx": (2 * T * W3 * h, (T * W3 + W3 * h + 2 * T * h) * e, 1),
            "dW_QKV": (2 * W3 * h * T, (T * W3 + T * h + W3 * h) * e, 1),
            "unpermute dx": (0, 2 * T * h * e, 1),
        })
    return w


# The layout calls timed on their own after the layer (kernel table names get " (standalone)").
LAYOUT_STEPS = ("zigzag permute", "kv gather", "zigzag unpermute")


def time_layout(cfg, plan, x, steps: int, warmup: int, hbm_peak: float, dev):
    """The zigzag permute, the K/V all-gather and the unpermute called on their
    own through the C ABI at the workload's full size (inputs larger than L2),
    each timed with CUDA events on the launching stream.  Returns
    {name: {ms, gbs, frac, bytes}} with the algorithmic bytes of one launch."""
    import torch

    from folded_tensor_sequence_gb300 import tsp

    B, S, hk, dh = cfg.batch, cfg.seq, cfg.kv_hidden, cfg.head_dim
    e = x.element_size()
    T = B * S
    xz, xu = torch.empty_like(x), torch.empty_like(x)
    gen = torch.Generator(device=dev).manual_seed(1)
    kz = torch.randn(T, hk, generator=gen, device=dev).to(x.dtype)
    vz = torch.randn(T, hk, generator=gen, device=dev).to(x.dtype)
    k = torch.empty(B, cfg.kv_h, S, dh, dtype=x.dtype, device=dev)
    v = torch.empty_like(k)
    stream = torch.cuda.current_stream(dev)

    def once():
        tsp.tsp_zigzag_permute(plan, B, x, xz, stream)
        tsp.tsp_kv_gather(plan, B, kz, vz, k, v, stream)
        tsp.tsp_zigzag_unpermute(plan, B, xz, xu, stream)

    for _ in range(warmup):
        once()
    torch.cuda.synchronize(dev)
    tsp.tsp_profile_enable(True)
    for _ in range(steps):
        once()
    rows = tsp.tsp_profile_report()
    tsp.tsp_profile_enable(False)
    tsp.tsp_sync_check(stream)
    if not torch.equal(xu, x):
        raise RuntimeError("permute then unpermute did not give the input back")
    nbytes = {"zigzag permute": 2 * T * cfg.hidden * e, "zigzag unpermute": 2 * T * cfg.hidden * e,
              "kv gather": 4 * T * hk * e}
    out = {}
    for name, tot, cnt in rows:
        avg = tot / cnt
        gbs = nbytes[name] / (avg / 1e3) / 1e9
        out[name] = {"ms": round(avg, 4), "gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
                     "bytes": nbytes[name], "launches": cnt}
    del xz, xu, kz, vz, k, v
    return out


def time_rank_compute(cfg, plan, packed, x, steps: int, warmup: int, dev, layer_ms: float):
    """One rank's compute in a D-GPU TSP layer (tsp_rank_* calls), shards
    already in local memory: for every attention shard the projection of the
    rank's tokens, attention over the gathered K/V and the output projection,
    then the D steps of the MLP ring.  Timed with CUDA events for rank 0 and
    rank D-1 (the zigzag split gives every rank the same causal work).  The
    exchanges between GPUs are not part of it."""
    import torch

    from folded_tensor_sequence_gb300 import tsp, tsp_rank

    D, B = cfg.D, cfg.batch
    stream = torch.cuda.current_stream(dev)
    attn = [torch.empty(tsp.tsp_rank_shard_bytes(plan, tsp.TSP_SHARD_ATTENTION), dtype=torch.uint8, device=dev)
            for _ in range(D)]
    mlp = [torch.empty(tsp.tsp_rank_shard_bytes(plan, tsp.TSP_SHARD_MLP), dtype=torch.uint8, device=dev)
           for _ in range(D)]
    for s_ in range(D):
        tsp.tsp_rank_extract_shard(plan, packed, s_, tsp.TSP_SHARD_ATTENTION, attn[s_], stream)
        tsp.tsp_rank_extract_shard(plan, packed, s_, tsp.TSP_SHARD_MLP, mlp[s_], stream)
    xz = torch.empty_like(x)
    tsp.tsp_zigzag_permute(plan, B, x, xz, stream)
    xr = xz.view(D, -1, cfg.hidden)
    out = {}
    for r in sorted({0, D - 1}):
        layer = tsp_rank.RankLayer(plan, r, B, dev, stream)
        gen = torch.Generator(device=dev).manual_seed(2)
        layer.kv_all.copy_(torch.randn(layer.kv_all.shape, generator=gen, device=dev).to(layer.kv_all.dtype))

        def rank_step():
            for s_ in range(D):
                layer.project(xr[r], attn[s_])
                layer.attend(attn[s_], xr[r] if s_ == 0 else layer.h)
            for t in range(D):
                layer.mlp(mlp[(r - t) % D], layer.h if t == 0 else layer.y)

        for _ in range(warmup):
            rank_step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(steps):
            rank_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        tsp.tsp_profile_enable(True)
        rank_step()
        parts = {n: round(t, 4) for n, t, _ in tsp.tsp_profile_report()}
        tsp.tsp_profile_enable(False)
        out[f"rank {r}"] = {"ms": round(ms, 4), "tflops": round(cfg.fwd_flops() / D / ms / 1e9, 1),
                            "steps_ms": parts}
        del layer
    tsp.tsp_sync_check(stream)
    return {"per_rank": out, "ideal_ms": round(layer_ms / D, 4),
            "note": ("compute of one rank of a D-GPU TSP layer on this GPU (its 1/D of the tokens against every "
                     "weight shard, shards already local); ideal_ms = the one-GPU layer's time / D; the "
                     "broadcasts, the K/V all-gather and the ring hops between GPUs are not included")}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.out = None

    def __enter__(self):
        self.out = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", self.gpu], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.15)
        if self.proc:
            self.proc.terminate()
            self.proc.wait()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.seek(0)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.out.read().splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def sample_flops(cfg, prefix: int) -> int:
    """Algorithmic flops of the oracle's sample: the causal prefix of `prefix`
    positions of one sequence, or for a decode workload one decode step of one
    sequence (`prefix` unused)."""
    h, F, H, dh, hk = cfg.hidden, cfg.ffn, cfg.heads, cfg.head_dim, cfg.kv_hidden
    if cfg.decode:
        return cfg.with_(batch=1).decode_flops()
    return prefix * 2 * (h * (h + 2 * hk) + h * h + 3 * h * F) + 4 * H * dh * prefix * (prefix + 1) // 2


def run_oracle_sample(cfg, prefix: int, repeats: int, timeout: float = 1800.0):
    """Times the fp64 oracle, single-threaded, `repeats` times on the first `prefix` positions of batch 0.

    Causality makes the layer's outputs at those positions depend only on that
    prefix, so the sample is an exact slice of the workload.  Runs in a fresh
    interpreter with BLAS pinned to one thread; inputs are drawn once, outside
    the timed calls.  Returns (list of seconds, error text).
    """
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np, torch
from folded_tensor_sequence_gb300 import synth
from folded_tensor_sequence_gb300.configs import BY_NAME
from oracle import tsp_oracle as O
cfg = BY_NAME[{cfg.name!r}]
h, F, P, hk = cfg.hidden, cfg.ffn, {prefix}, cfg.kv_hidden
shapes = {{"Wq": (h, h), "Wk": (h, hk), "Wv": (h, hk), "Wo": (h, h), "Wg": (h, F), "Wu": (h, F), "Wd": (F, h)}}
w = {{k: synth.tensor_torch(k, s, (F if k == "Wd" else h) ** -0.5, cfg.dtype, 0, "cpu").double().numpy()
      for k, s in shapes.items()}}
secs = []
if cfg.decode:
    # one decode step of sequence 0 at position seq-1 against a seeded N(0,1) cache
    gen = torch.Generator().manual_seed(0)
    kc = torch.randn(1, cfg.seq, hk, generator=gen).to(torch.bfloat16).float().numpy()
    vc = torch.randn(1, cfg.seq, hk, generator=gen).to(torch.bfloat16).float().numpy()
    x = synth.tensor_torch("x", (1, h), 1.0, cfg.dtype, 0, "cpu").double().numpy()
    for _ in range({repeats}):
        t0 = time.perf_counter()
        y, _, _ = O.decode_step(x, w, cfg.heads, kc, vc, cfg.seq - 1)
        secs.append(time.perf_counter() - t0)
        assert np.isfinite(y).all()
else:
    x = synth.tensor_torch("x", (1, P, h), 1.0, cfg.dtype, 0, "cpu").double().numpy()
    for _ in range({repeats}):
        t0 = time.perf_counter()
        out = O.layer_fwd(x, w, cfg.heads)
        secs.append(time.perf_counter() - t0)
        assert np.isfinite(out["Y"]).all()
print(json.dumps({{"seconds": secs}}))
"""
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=timeout)
    except subprocess.TimeoutExpired:
        return None, "timed out"
    if r.returncode != 0:
        return None, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])["seconds"], None


def cpu_baseline(cfg, prefix: int):
    secs, err = run_oracle_sample(cfg, prefix, 1)
    if secs is None:
        return None, err
    fl = sample_flops(cfg, prefix)
    return {"value": round(fl / secs[0] / 1e12, 6), "unit": UNIT, "cores": 1, "kind": "oracle", "host": host_cpu(),
            "sample": (f"fp64 numpy oracle, 1 thread, one decode step of sequence 0 at position {cfg.seq - 1} "
                       if cfg.decode else f"fp64 numpy oracle, 1 thread, positions 0..{prefix - 1} of batch 0 ")
                      + f"({fl / 1e9:.1f} GFLOP algorithmic, {secs[0]:.1f} s)",
            "tokens_per_s": round((1 if cfg.decode else prefix) / secs[0], 2)}, None


def dist_env():
    e = rank_env()
    return e.world_size, e.rank, e.local_rank


def run_reference(args, cfg):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    prefix = args.ref_prefix
    secs, err = run_oracle_sample(cfg, prefix, args.warmup + args.steps)
    if secs is None:
        print(json.dumps({"impl": "reference", "unavailable": f"oracle run failed: {err.strip()[-200:]}"}))
        return 0
    timed = secs[args.warmup:]
    fl = sample_flops(cfg, prefix)
    total = sum(timed)
    value = fl * len(timed) / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(timed),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "D": cfg.D, "batch": cfg.batch, "seq": cfg.seq, "hidden": cfg.hidden,
                   "heads": cfg.heads, "head_dim": cfg.head_dim, "ffn": cfg.ffn,
                   "sample": (f"each step: one decode step of sequence 0 at position {cfg.seq - 1}" if cfg.decode
                              else f"each step: positions 0..{prefix - 1} of batch 0 (causal prefix, exact slice)")},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "host": host_cpu(),
                         "sample": (f"fp64 numpy oracle, 1 thread, one decode step of sequence 0 per step"
                                    if cfg.decode else
                                    f"fp64 numpy oracle, 1 thread, causal prefix of {prefix} tokens per step")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tsp", choices=["tsp", "reference"])
    ap.add_argument("--config", default=LAYER_7B_S16K.name, choices=sorted(BY_NAME))
    ap.add_argument("--cpu-prefix", type=int, default=512, help="tokens of the oracle's CPU baseline sample")
    ap.add_argument("--ref-prefix", type=int, default=64, help="tokens per step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rank-compute", action="store_true", help="skip timing one rank of a D-GPU TSP layer")
    ap.add_argument("--deterministic", action="store_true",
                    help="backward: split bitwise-reproducible kernels instead of the fused one")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    cfg = BY_NAME[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)

    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)

    # The CPU baseline runs first, in its own interpreter, before this process
    # does any heavy GPU work (rank 0 at N = 1 only).
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu, err = cpu_baseline(cfg, args.cpu_prefix)
        if cpu is None:
            cpu = {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "host": host_cpu(),
                   "sample": f"failed: {err[-300:]}"}

    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import synth, tsp

    B, S, h, F, hk = cfg.batch, cfg.seq, cfg.hidden, cfg.ffn, cfg.kv_hidden
    plan = tsp.plan_for(cfg)
    tsp.tsp_plan_set_deterministic(plan, 1 if args.deterministic else 0)
    shapes = {"Wq": (h, h), "Wk": (h, hk), "Wv": (h, hk), "Wo": (h, h), "Wg": (h, F), "Wu": (h, F), "Wd": (F, h)}
    canon = {k: synth.tensor_torch(k, s, (F if k == "Wd" else h) ** -0.5, cfg.dtype, 0, dev) for k, s in shapes.items()}
    packed = tsp.empty_packed(plan, dev)
    tsp.tsp_pack_weights(plan, canon, packed)
    del canon
    stream = torch.cuda.current_stream(dev)
    if cfg.decode:
        # one decode step per sequence at the last position of a full cache (seeded N(0,1) contents)
        gen = torch.Generator(device=dev).manual_seed(0)
        kc = torch.randn(B, cfg.kv_h, S, cfg.head_dim, generator=gen, device=dev).to(torch.bfloat16)
        vc = torch.randn(B, cfg.kv_h, S, cfg.head_dim, generator=gen, device=dev).to(torch.bfloat16)
        x = synth.tensor_torch("x", (B, h), 1.0, cfg.dtype, 0, dev)
        y = torch.empty_like(x)
        dwork = tsp.workspace(plan, B, tsp.TSP_OP_DECODE, dev)

        def step_io(ins, out):
            tsp.tsp_decode_step(plan, B, S - 1, ins[0], packed, kc, vc, out, dwork, stream)
    else:
        x = synth.tensor_torch("x", (B, S, h), 1.0, cfg.dtype, 0, dev)
        y = torch.empty_like(x)
        work = tsp.workspace(plan, B, tsp.TSP_OP_LAYER_FWD, dev)
    if cfg.decode:
        pass
    elif cfg.backward:
        # training step (no optimizer): forward keeping activations, then the full backward
        dy = synth.tensor_torch("dY", (B, S, h), 1.0, cfg.dtype, 0, dev)
        dx = torch.empty_like(x)
        grads = tsp.empty_packed(plan, dev)
        saved = torch.empty(tsp.tsp_saved_bytes(plan, B), dtype=torch.uint8, device=dev)
        bwork = tsp.workspace(plan, B, tsp.TSP_OP_LAYER_BWD, dev)

        def step_io(ins, out):
            tsp.tsp_layer_fwd(plan, B, ins[0], packed, y, saved, work, stream)
            tsp.tsp_layer_bwd(plan, B, ins[0], packed, saved, ins[1], out, grads, bwork, stream)
    else:
        def step_io(ins, out):
            tsp.tsp_layer_fwd(plan, B, ins[0], packed, out, None, work, stream)

    ins = [x, dy] if cfg.backward and not cfg.decode else [x]  # per-step inputs
    out = dx if cfg.backward and not cfg.decode else y          # per-step result

    def step():
        step_io(ins, out)

    for _ in range(args.warmup):
        step()
    tsp.tsp_sync_check(stream)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    # ---- device-resident timing ------------------------------------------
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    vis = [t.strip() for t in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if t.strip()]
    gpu_id = vis[dev.index] if dev.index < len(vis) else str(dev.index)
    with ClockSampler(gpu_id) as clk:
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        barrier()
    ms = ev0.elapsed_time(ev1)
    tsp.tsp_sync_check(stream)
    ms = max_over_ranks(ms, dev)
    clocks = clk.summary()
    # training step: model flops = 3x forward; decode: the step's projections and attention
    flops = cfg.decode_flops() if cfg.decode else cfg.fwd_flops() * (3 if cfg.backward else 1)
    tokens_per_step = B if cfg.decode else B * S
    ms_step = ms / args.steps
    value = whole_job_rate(ws, flops, args.steps, ms) / 1e12
    tokens_s = whole_job_rate(ws, tokens_per_step, args.steps, ms)

    # ---- spread of single steps (same stream, separate pass): min / median ---
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for ea, eb in evs:
        ea.record(stream)
        step()
        eb.record(stream)
    torch.cuda.synchronize(dev)
    per = sorted(ea.elapsed_time(eb) for ea, eb in evs)
    spread = {"min": round(per[0], 4), "median": round(statistics.median(per), 4), "max": round(per[-1], 4),
              "n": len(per), "note": "rank 0, one event pair per step, after the timed region"}

    # ---- per-kernel timing (same stream, separate pass) ---------------------
    tsp.tsp_profile_enable(True)
    for _ in range(args.steps):
        step()
    rows = tsp.tsp_profile_report()
    tsp.tsp_profile_enable(False)
    wk = step_work(cfg, args.deterministic)
    kernels = {}
    launches_per_step = 0
    for name, tot, cnt in rows:
        fl, by, nk = wk.get(name, (0, 0, 1))
        launches_per_step += nk * cnt / args.steps
        avg = tot / cnt
        kernels[name] = {"ms": round(avg, 4), "tflops": round(fl / avg / 1e9, 1) if fl else None,
                         "gbs": round(by / avg / 1e6, 1)}
    dom = max(rows, key=lambda r: r[1])
    peaks, peak_src = load_peaks()
    dname, dtot, dcnt = dom
    dfl, dby, _ = wk.get(dname, (0, 0, 1))
    davg_s = dtot / dcnt / 1e3
    traffic = ncu_traffic(dname, cfg.name)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nominal = nominal_bf16_tflops(num_sms, clocks.get("sm_mhz"))
    if dfl:
        # The timed region lasts well under a second, far from the seconds-long
        # power-capped loop behind the sustained figure: the burst peak applies.
        peak = peaks["bf16_tflops"]
        ach = dfl / davg_s / 1e12
        roof = {"bound": "tensor", "kernel": dname, "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "traffic": traffic,
                "peak_source": (f"{peak_src} bf16 burst (cuBLAS 8192^3, best of 10); the timed region is "
                                f"{args.steps} steps of {ms_step:.1f} ms, not a seconds-long sustained loop"),
                "algorithmic": f"{dfl / 1e12:.3f} TFLOP per launch",
                "frac_nominal": round(ach / nominal, 4) if nominal else None,
                "nominal_peak": round(nominal, 1) if nominal else None,
                "nominal_source": (f"{BF16_FLOPS_PER_SM_CYCLE} flop/cycle/SM x {num_sms} SMs x median SM clock "
                                   f"{clocks.get('sm_mhz')} MHz")}
    else:
        peak = peaks["hbm_gbs"]
        ach = dby / davg_s / 1e9
        roof = {"bound": "hbm", "kernel": dname, "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "traffic": traffic, "peak_source": f"{peak_src} HBM copy"}

    # ---- the layout kernels on their own (HBM-bound; full workload size) -----
    layout, roof_hbm = None, None
    if not cfg.decode:
        layout = time_layout(cfg, plan, x, args.steps, args.warmup, peaks["hbm_gbs"], dev)
        for name, ent in layout.items():
            kernels[name + " (standalone)"] = {"ms": ent["ms"], "tflops": None, "gbs": ent["gbs"]}
        hname = max(layout, key=lambda n: layout[n]["ms"])
        hent = layout[hname]
        roof_hbm = {"bound": "hbm", "kernel": hname, "achieved": hent["gbs"], "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": hent["frac"],
                    "traffic": ncu_traffic(hname + " (standalone)", cfg.name),
                    "peak_source": f"{peak_src} HBM copy (torch copy_ of 2 GiB)",
                    "algorithmic": f"{hent['bytes'] / 1e9:.3f} GB per launch (read + write)"}

    # ---- one rank of a D-GPU TSP layer (compute only) ------------------------
    rank_compute = None
    if not cfg.decode and not cfg.backward and cfg.D > 1 and not args.no_rank_compute:
        try:
            rank_compute = time_rank_compute(cfg, plan, packed, x, args.steps, args.warmup, dev, ms_step)
        except Exception as e:  # noqa: BLE001 -- e.g. a shape the per-rank calls do not take
            rank_compute = {"unavailable": str(e)[:300]}

    # ---- end to end through the API with host buffers -----------------------
    # Every step's inputs come from pinned host memory and its result goes back
    # to it.  As a caller overlapping I/O with the layer would, one copy stream
    # brings step i+1's inputs in and another takes step i's result out while
    # step i computes (the host link is full duplex; device inputs and outputs
    # are double-buffered, events order the reuse of each buffer).  Timed from
    # the first input copy to the last result copy.
    ins_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ins]
    for th, t in zip(ins_host, ins):
        th.copy_(t)
    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    dins = [ins, [torch.empty_like(t) for t in ins]]
    douts = [out, torch.empty_like(out)]
    cs_in, cs_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    d2h = [torch.cuda.Event() for _ in range(2)]
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cs_in)
    with torch.cuda.stream(cs_in):
        for t, th in zip(dins[0], ins_host):
            t.copy_(th, non_blocking=True)
        h2d[0].record(cs_in)
    for i in range(args.steps):
        k = i % 2
        stream.wait_event(h2d[k])
        if i >= 2:
            stream.wait_event(d2h[k])  # douts[k] has been read back
        step_io(dins[k], douts[k])
        done[k].record(stream)
        if i + 1 < args.steps:
            nk = (i + 1) % 2
            with torch.cuda.stream(cs_in):
                if i >= 1:
                    cs_in.wait_event(done[nk])  # dins[nk] no longer read by step i-1
                for t, th in zip(dins[nk], ins_host):
                    t.copy_(th, non_blocking=True)
                h2d[nk].record(cs_in)
        with torch.cuda.stream(cs_out):
            cs_out.wait_event(done[k])
            out_host.copy_(douts[k], non_blocking=True)
            d2h[k].record(cs_out)
    e1.record(cs_out)
    barrier()
    ems = max_over_ranks(e0.elapsed_time(e1), dev)
    tsp.tsp_sync_check(stream)
    e2e = {"value": round(whole_job_rate(ws, flops, args.steps, ems) / 1e12, 2), "unit": UNIT,
           "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in ins),
           "d2h_bytes_per_step": out.numel() * out.element_size(),
           "tokens_per_s": round(whole_job_rate(ws, tokens_per_step, args.steps, ems), 1)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "step_ms": spread,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (splitmix64 + Box-Muller, seed 0)",
            "tokens_per_s": round(tokens_s, 1),
            "pct_of_peak": {"burst": round(value / ws / peaks["bf16_tflops"], 4),
                            "sustained": round(value / ws / peaks["bf16_tflops_sustained"], 4),
                            "source": f"{peak_src} (cuBLAS-attained bf16 throughput)",
                            "nominal_at_median_clock": round(value / ws / nominal, 4) if nominal else None,
                            "nominal_2250": round(value / ws / 2250.0, 4)},
            "config": {"workload": cfg.name, "D": cfg.D, "batch": B, "seq": S, "hidden": h, "heads": cfg.heads,
                       "kv_heads": cfg.kv_h, "head_dim": cfg.head_dim, "ffn": F,
                       "step": ("decode: one token per sequence at position seq-1 of a full K/V cache"
                                if cfg.decode else ("layer forward + backward" if cfg.backward else "layer forward")),
                       **({"attention_backward": "split, bitwise reproducible" if args.deterministic
                           else "fused (dQ by fp32 L2 reductions)"} if cfg.backward and not cfg.decode else {}),
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single",
                       "l2": "inputs larger than L2 (%s %d MB, packed weights %d MB)" % (
                           "K/V cache" if cfg.decode else "x",
                           (2 * kc.numel() * kc.element_size() if cfg.decode else x.numel() * x.element_size()) >> 20,
                           sum(t.numel() * t.element_size() for t in (packed.qkv, packed.o, packed.gate_up,
                                                                        packed.down)) >> 20)},
            "roofline": roof,
            "roofline_hbm": roof_hbm,
            "layout_kernels": layout,
            "tsp_rank_compute": rank_compute,
            "kernels": kernels,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": int(round(launches_per_step)) * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
