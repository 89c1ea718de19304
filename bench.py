#!/usr/bin/env python
"""Throughput of the fine-grained MoE layer forward (Kimi-K2 shape) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

One step is one moe_layer_forward over one batch of T synthetic tokens: the
fused router, the dispatch, the grouped SwiGLU experts with the shared
expert, and the weighted combine -- every row of the hot path.  Inputs are
resident in HBM when the timed region starts; the expert weights (34 GB for
the K2 layer) exceed the 129 MB L2, so every step streams them from HBM.

With N > 1 (torchrun, one rank per GPU) every rank runs an independent
replica of the layer on its own batch (the layer has no exchange step on one
GPU; weak scaling); the time is the maximum over ranks.

``--impl reference`` times the CPU oracle instead, on bounded samples of the
same workload, on the host cores of rank 0.

Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
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

METRIC = "MoE layer tokens/s (K2 shape) + % of HBM / bf16 tensor roofline; router tokens/s"
UNIT = "tokens/s"
WORKLOADS = {
    "k2_prefill": "K2 MoE layer prefill with group-limited routing: T=8192 tokens, d_model=7168, "
                  "384 routed + 1 shared SwiGLU expert (intermediate 2048), top-8, n_group=8, "
                  "topk_group=4, scale 2.827, bf16 experts with fp32 accumulation, fp32 router, "
                  "x from a 32-cluster Gaussian mixture, bias U(-0.1,0.1)",
    "k2_decode": "K2 MoE layer decode: T=128 tokens, d_model=7168, 384 routed + 1 shared SwiGLU "
                 "expert (intermediate 2048), top-8, scale 2.827, bf16 experts, fp32 router, "
                 "x from a 32-cluster Gaussian mixture",
    "k3_latent": "K3-shaped latent MoE layer: T=4096, d_model=7168, latent 3584, 896 routed SwiGLU "
                 "experts (intermediate 3072), top-16, 2 shared experts at 7168 (intermediate "
                 "3072), scale 2.827, bf16 experts, fp32 router",
}
WORKLOADS["tiny"] = ("Tiny MoE layer, all fp32: T=64 tokens, d_model=256, 16 routed + 1 shared "
                     "SwiGLU expert (intermediate 64), top-4, n_group 1, scale 2.827 "
                     "(launch-bound; reported for its time per step)")
WORKLOADS["k2_router"] = ("K2 router alone: T=4096 tokens, x bf16 N(0,1), fp32 W_r [384 x 7168] "
                          "kaiming-uniform, bias U(-0.05,0.05), sigmoid + bias top-8 of 384, "
                          "n_group 1, weights renormalised x 2.827")
_FP8_NOTE = (" -- expert weights FP8 E4M3 with one fp32 scale per 128 x 128 block (dequantised "
             "to bf16 in shared memory; bf16 activations, fp32 accumulation)")
for _n in ("k2_decode", "k2_prefill", "k3_latent"):
    WORKLOADS[_n + "_fp8"] = WORKLOADS[_n].replace(", bf16 experts", "") + _FP8_NOTE
PROFILE_DIR = os.path.join(ROOT, "profiles")
# the roofline's live gate/up duration: events around that launch in every
# GU_EVERY-th timed step
GU_EVERY = 4


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="k2_prefill", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--cpu-sample-tokens", type=int, default=0,
                    help="tokens of the CPU oracle sample (default 1024, about 10 s on 16 "
                         "cores; 48 with FP8 weights, whose per-expert dequantisation "
                         "dominates the oracle's time)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="skip the companion workloads measured after the headline one")
    ap.add_argument("--extra-steps", type=int, default=30,
                    help="timed steps of each companion workload")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# Replica plumbing for N > 1.  The layer has no exchange step, so ranks meet
# only at the barriers around the timed region and in the max-over-ranks
# reduction of its duration; the helpers take the backend and the device of
# the reduction buffer so that the same code runs over gloo on CPU.

def init_ranks(torch, world, backend="nccl", device=None):
    if world > 1:
        import torch.distributed as dist
        kw = {"device_id": device} if backend == "nccl" and device is not None else {}
        dist.init_process_group(backend, **kw)


def barrier(torch, world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(torch, ms, world, device):
    """The slowest rank's duration: the job is done when its last rank is."""
    if world == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_rank, steps, ms_total):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (ms_total / 1e3)


def replica_seed(seed, rank):
    """Each replica draws its own batch; the weights keep the common seed."""
    return seed + 7919 * rank


def finish_ranks(torch, world):
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ------------------------------------------------------------------ clocks
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling every 100 ms while the timed region runs."""

    def __init__(self, device_id: str):
        fields = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw",
                  "clocks_event_reasons.active"] + ["clocks_event_reasons." + r for r in REASONS]
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.cmd = ["nvidia-smi", "--query-gpu=" + ",".join(fields), "--format=csv,noheader,nounits",
                    "-lms", "100", "-i", device_id, "-f", self.path]
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 5 + len(REASONS):
                        continue
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[5:]))
                    except ValueError:
                        continue
            os.unlink(self.path)
        except OSError:
            return None
        inside = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({REASONS[i] for r in inside for i, v in enumerate(r[4][:len(REASONS)])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


def device_id(torch, local_rank):
    try:
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(local_rank)


# --------------------------------------------------------- work accounting
def per_step_work(shape, counts):
    """Algorithmic bytes and flops of one layer step and of its kernels.

    Bytes count only what the method must touch: the weights of the experts
    actually selected (unique, from the per-expert counts), the shared
    experts, the router weight and bias, x once and y once.  H / Y round
    trips and gathered copies are implementation costs and are left out."""
    T, d, E, K = shape.T, shape.d_model, shape.E_routed, shape.K
    F, S, Fs, L = shape.d_ff, shape.E_shared, shape.d_ff_shared, shape.d_latent
    de = L if L else d
    U = int((counts > 0).sum())
    b16 = 4 if getattr(shape, "dtype", "bf16") == "f32" else 2  # activations and bf16 weights
    # expert weight bytes per element: bf16, or an FP8 code plus its share of
    # the block's fp32 scale
    bw = 1 + 4 / (128 * 128) if getattr(shape, "weights", "bf16") == "fp8" else b16
    w_gu = 2 * F * de * bw
    w_dn = de * F * bw
    ws_gu = 2 * Fs * d * bw
    ws_dn = d * Fs * bw
    xbytes = T * d * b16
    router_bytes = E * d * 4 + E * 4 + xbytes + T * K * 8
    # x is read once; with the latent form the routed experts read x_lat instead
    gate_up_bytes = U * w_gu + S * ws_gu + T * de * b16 + (T * d * b16 if (S and L) else 0)
    down_bytes = U * w_dn + S * ws_dn
    layer_bytes = U * (w_gu + w_dn) + S * (ws_gu + ws_dn) + E * d * 4 + E * 4 + 2 * xbytes
    if L:
        layer_bytes += 2 * L * d * b16
    flops_router = 2 * T * d * E
    flops_gate_up = 2 * T * K * de * 2 * F + 2 * T * S * d * 2 * Fs
    flops_down = 2 * T * K * F * de + 2 * T * S * Fs * d
    flops_proj = 2 * 2 * T * d * L if L else 0
    return {"U": U, "gate_up_bytes": int(gate_up_bytes), "down_bytes": int(down_bytes),
            "router_bytes": router_bytes, "layer_bytes": int(layer_bytes),
            "flops_router": flops_router, "flops_gate_up": flops_gate_up, "flops_down": flops_down,
            "flops_layer": flops_router + flops_gate_up + flops_down + flops_proj}


def kernel_source_hash():
    """Hash of the GEMM kernel's sources with comments and blank space
    removed, so that edits to comments keep a profile valid."""
    h = hashlib.sha256()
    for name in ("gemm_tc.cu", "common.cuh", "internal.h"):
        with open(os.path.join(ROOT, "fine_grained_sparse_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(config):
    """DRAM bytes per gate/up launch from the committed ncu summary, if it was
    taken on the current kernel source."""
    path = os.path.join(PROFILE_DIR, f"tc_gemm_gate_up_{config}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_b or not m_h or m_h.group(1) != kernel_source_hash():
        return None
    return float(m_b.group(1))


# ------------------------------------------------------------ CPU oracle leg
def is_fp8(shape):
    return getattr(shape, "weights", "bf16") == "fp8"


def expert_f64(shape, rec):
    """(W_gate, W_up, W_down) in fp64 from an expert's host tensors: (gate_up,
    down) bf16, or FP8 (gate_up codes, scales, down codes, scales), which the
    oracle dequantises."""
    import oracle
    if is_fp8(shape):
        gu = oracle.dequant_fp8_blocks(rec[0].numpy(), rec[1].numpy())
        dn = oracle.dequant_fp8_blocks(rec[2].numpy(), rec[3].numpy())
    else:
        gu, dn = (t.to(__import__("torch").float64).numpy() for t in rec)
    F = gu.shape[0] // 2
    return gu[:F], gu[F:], dn


def expert_record(shape, g, bank, e):
    """One expert's weights of a generated layer, copied to the host."""
    if is_fp8(shape):
        return tuple(g[f"{bank}_{m}_{k}"][e].cpu() for m in ("gate_up", "down") for k in "qs")
    return g[f"{bank}_gate_up"][e].cpu(), g[f"{bank}_down"][e].cpu()


def oracle_sample(shape, x_rows, W_r, bias, routed, shared, lat):
    """Run the oracle on the given token rows; returns (seconds, result).
    routed(e) / shared(s) give an expert's host tensors (see expert_f64); the
    conversion to fp64 (and the FP8 dequantisation) is part of the timed
    oracle work."""
    import torch
    import oracle
    f64 = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    t0 = time.perf_counter()
    res = oracle.moe_layer(
        f64(x_rows), f64(W_r), bias.numpy(),
        routed=lambda e: expert_f64(shape, routed(e)),
        shared=(lambda s: expert_f64(shape, shared(s))) if shape.E_shared else None,
        n_shared=shape.E_shared, K=shape.K, n_group=shape.n_group, topk_group=shape.topk_group,
        scale=shape.routed_scaling_factor, norm_topk_prob=shape.norm_topk_prob,
        W_lat_down64=f64(lat[0]) if lat else None, W_lat_up64=f64(lat[1]) if lat else None)
    return time.perf_counter() - t0, res


def cpu_baseline_from_device(shape, g, idx, n_tokens):
    """Oracle on n_tokens of the benchmarked batch (host cores).  The weights
    the sample selects are staged to host memory before the clock starts."""
    import numpy as np
    import torch
    T = shape.T
    rows = np.unique(np.linspace(0, T - 1, n_tokens).astype(int))
    experts = sorted(set(int(e) for e in idx[rows].reshape(-1)))
    host = {e: expert_record(shape, g, "W", e) for e in experts}

    def routed(e):
        if e not in host:  # the oracle chose an expert the device did not
            host[e] = expert_record(shape, g, "W", e)
        return host[e]

    sh = [expert_record(shape, g, "Ws", s) for s in range(shape.E_shared)]
    lat = (g["W_lat_down"].cpu(), g["W_lat_up"].cpu()) if shape.d_latent else None
    x_rows = g["x"][torch.as_tensor(rows, device=g["x"].device)].cpu()
    secs, _ = oracle_sample(shape, x_rows, g["W_r"].cpu(), g["bias"].cpu(), routed,
                            lambda s: sh[s], lat)
    cores = len(os.sched_getaffinity(0))
    return {"value": len(rows) / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} of the {T} tokens of the benchmarked batch, full layer "
                      f"(router over all {shape.E_routed} experts, {shape.K} routed + "
                      f"{shape.E_shared} shared SwiGLU experts each, fp64); {secs:.1f} s"}


# ------------------------------------------------------------------ own arm
def time_router(fgs, torch, cfg, T, gp, ws, nws, stream, reps=20):
    """Mean device time of moe_router on the benchmarked batch."""
    idx = torch.empty((T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.K), dtype=torch.float32, device="cuda")
    run = lambda: fgs.moe_router(cfg, T, gp["x"], gp["W_r"], gp["bias"], idx, w, ws, nws,  # noqa: E731
                                 stream=stream)
    for _ in range(3):
        run()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        run()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / reps


def run_router_only(args, fgs, torch, synth, shape, world, rank, local, steps, warmup,
                    full=True):
    """One step = one moe_router call (x, W_r and the bias resident).  The
    inputs (70 MB) fit in L2, so a 256 MB buffer is written between steps,
    outside the timed intervals, and the step time is the sum of the
    per-step event intervals."""
    import numpy as np
    T, K = shape.T, shape.K
    seed = synth.SEEDS[shape.name]
    g = synth.generate(shape, device="cuda", seed=seed)
    if rank:
        g["x"] = synth.activations(shape, "cuda", seed=replica_seed(seed, rank))
    # the fp32 router weight split once into its three bf16 terms (a load step)
    cfg = fgs.config(shape, router_weight=fgs.MOE_ROUTER_WEIGHT_SPLIT)
    W_s = fgs.split_router_weight(cfg, g["W_r"])
    nws = fgs.moe_workspace_size(cfg, T)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        fgs.moe_router(cfg, T, g["x"], W_s, g["bias"], idx, w, ws, nws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.zero_()
            step()
    stream.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    sampler = ClockSampler(device_id(torch, local)) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(torch, world)
    torch.cuda.synchronize()
    t0 = time.time()
    launches0 = fgs.moe_launch_count()
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush.zero_()  # L2 flush between steps, outside [a, b]
            a.record(stream)
            step()
            b.record(stream)
    launches = fgs.moe_launch_count() - launches0
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(torch, world)
    clocks = sampler.stop(t0, t1) if sampler else None
    ms_total = max_over_ranks(torch, sum(a.elapsed_time(b) for a, b in evs), world, "cuda")
    status = fgs.moe_get_device_status(ws, stream)
    if status:
        raise RuntimeError("device status after the timed steps: " + fgs.moe_status_string(status))
    ms_step = ms_total / steps
    peaks = load_peaks()
    d, E = shape.d_model, shape.E_routed
    flops_fp32 = 2 * T * d * E            # the method's fp32 GEMM
    flops_bf16 = 3 * flops_fp32           # executed: x times the three bf16 pieces of W_r
    tflops = flops_bf16 / (ms_step / 1e3) / 1e12
    bytes_alg = T * d * 2 + E * d * 4 + E * 4 + T * K * 8
    line = {
        "metric": METRIC, "value": round(job_tokens_per_s(world, T, steps, ms_total), 1),
        "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16x3 (fp32-exact products)",
        "data": "synthetic (seeded; x N(0,1) bf16, W_r kaiming-uniform fp32, bias U(-0.05,0.05))",
        "config": {"workload": WORKLOADS[shape.name], "name": shape.name, "tokens_per_step": T,
                   "l2": "inputs (70 MB) fit in L2: a 256 MB buffer is written between steps, "
                         "outside the timed intervals",
                   "router_weight": "fp32 W_r split once before timing into three bf16 terms "
                                    "(moe_split_router_weight)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        # the dominant kernel is the split-bf16 logits GEMM; the interval is
        # the whole moe_router call (logits GEMM and selection)
        "roofline": {"bound": "tensor", "kernel": "moe_router (tensor-core logits "
                     "GEMM + selection)", "achieved": round(tflops, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(tflops / peaks["bf16_tflops"], 4), "traffic": None,
                     "peak_source": peaks["source"] + " (bf16 burst)",
                     "algorithmic_flops_per_launch": flops_bf16,
                     "fp32_equivalent_tflops": round(flops_fp32 / (ms_step / 1e3) / 1e12, 2),
                     "algorithmic_bytes_per_launch": bytes_alg,
                     "hbm_frac": round(bytes_alg / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"], 4)},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if not full:
        return line
    # end to end: pinned host x in, routing (indices and weights) out
    x_host = g["x"].cpu().pin_memory()
    xd = torch.empty_like(g["x"])
    idx_h = torch.empty((T, K), dtype=torch.int32).pin_memory()
    w_h = torch.empty((T, K), dtype=torch.float32).pin_memory()
    e_steps = max(3, min(steps, 50))
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        es.record(stream)
        for _ in range(e_steps):
            xd.copy_(x_host, non_blocking=True)
            fgs.moe_router(cfg, T, xd, W_s, g["bias"], idx, w, ws, nws, stream=stream)
            idx_h.copy_(idx, non_blocking=True)
            w_h.copy_(w, non_blocking=True)
        ee.record(stream)
    ee.synchronize()
    e_ms = max_over_ranks(torch, es.elapsed_time(ee), world, "cuda")
    line["e2e"] = {"value": round(job_tokens_per_s(world, T, e_steps, e_ms), 1), "unit": UNIT,
                   "h2d_bytes_per_step": T * d * 2, "d2h_bytes_per_step": T * K * 8,
                   "steps": e_steps, "api": "moe_router (pinned host x in, idx and w out)"}
    if full and rank == 0 and not args.no_cpu_baseline:
        import oracle
        n = args.cpu_sample_tokens or T  # the oracle router takes seconds for the batch
        rows = torch.as_tensor(np.unique(np.linspace(0, T - 1, n).astype(int)), device="cuda")
        x64 = g["x"][rows].to(torch.float64).cpu().numpy()
        W64 = g["W_r"].to(torch.float64).cpu().numpy()
        b32 = g["bias"].cpu().numpy()
        t_0 = time.perf_counter()
        oracle.router_from_x(x64, W64, b32, K, shape.n_group, shape.topk_group)
        secs = time.perf_counter() - t_0
        line["cpu_baseline"] = {"value": len(rows) / secs, "unit": UNIT,
                                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": f"{len(rows)} of the {T} tokens, fp64 router "
                                          f"(logits, sigmoid, selection, weights); {secs:.2f} s"}
    return line


def run_layer(args, fgs, torch, synth, name, steps, warmup, world, rank, local, full=True):
    """One workload: its JSON fields (full: with the end-to-end and CPU legs)."""
    import numpy as np

    shape = synth.shape(name)
    if shape.router_only:
        return run_router_only(args, fgs, torch, synth, shape, world, rank, local, steps, warmup,
                               full)
    T = shape.T
    seed = synth.SEEDS[shape.name]
    g = synth.generate(shape, device="cuda", seed=seed)
    if rank:  # replicas: every rank its own batch, same weights
        g["x"] = synth.activations(shape, "cuda", seed=replica_seed(seed, rank))
    # bf16 banks packed, FP8 banks (config(shape) picks MOE_WEIGHTS_PACKED_FP8),
    # fp32 layers in the natural layout (their experts run on CUDA cores)
    fp32 = shape.dtype == "f32"
    cfg = (fgs.config(shape) if (is_fp8(shape) or fp32) else
           fgs.config(shape, weight_layout=fgs.MOE_WEIGHTS_PACKED))
    # one-time load step: weights rearranged into the order the tensor cores
    # stream (the natural copies stay for the CPU oracle leg)
    gp = (g if fp32 else fgs.pack_layer_weights_fp8(g) if is_fp8(shape) else
          fgs.pack_layer_weights(g))
    if not fp32:
        # the fp32 router weight split once into its three bf16 terms (the
        # form its tensor-core GEMM reads), also a load step
        cfg.router_weight = fgs.MOE_ROUTER_WEIGHT_SPLIT
        gp = dict(gp)
        gp["W_r"] = fgs.split_router_weight(cfg, g["W_r"])
    torch.cuda.synchronize()
    nws = fgs.moe_workspace_size(cfg, T)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    y = torch.empty((T, shape.d_model), dtype=g["x"].dtype, device="cuda")
    idx = torch.empty((T, shape.K), dtype=torch.int32, device="cuda")
    counts = torch.empty(shape.E_routed, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    nev = fgs.MOE_STAGE_COUNT + 1

    def step(events=None):
        fgs.moe_layer_forward(cfg, T, gp["x"], gp["W_r"], gp["bias"], gp["W_gate_up"],
                              gp["W_down"], gp.get("Ws_gate_up"), gp.get("Ws_down"),
                              gp.get("W_lat_down"), gp.get("W_lat_up"), y, idx, None, counts, ws,
                              nws, stage_events=events, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    stream.synchronize()
    status = fgs.moe_get_device_status(ws, stream)
    if status:
        raise RuntimeError("device status after warm-up: " + fgs.moe_status_string(status))

    # inside the timed region only the gate/up launch is bracketed by events,
    # in every GU_EVERY-th step (each recorded event keeps the kernels on its
    # two sides from overlapping, about 0.03 ms a step at K2 prefill); the
    # other stage times come from an instrumented pass after it
    gu_events = [[None, None, torch.cuda.Event(enable_timing=True),
                  torch.cuda.Event(enable_timing=True), None, None]
                 if i % GU_EVERY == 0 else None for i in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device_id(torch, local)) if rank == 0 else None
    if sampler:
        sampler.start()
    # a layer whose weights fit in L2 (the tiny configuration) gets an L2
    # flush between steps, outside per-step intervals; the K2/K3 weights
    # (tens of GB) stream from HBM whatever the order
    small = fp32 or sum(t.numel() * t.element_size() for k, t in g.items() if k != "x") < (256 << 20)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if small else None
    step_iv = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)] if small else None
    barrier(torch, world)
    torch.cuda.synchronize()
    t0 = time.time()
    launches0 = fgs.moe_launch_count()
    start.record(stream)
    with torch.cuda.stream(stream):
        for i in range(steps):
            if small:
                flush.zero_()
                step_iv[i][0].record(stream)
            step(gu_events[i])
            if small:
                step_iv[i][1].record(stream)
    end.record(stream)
    launches = fgs.moe_launch_count() - launches0
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(torch, world)
    clocks = sampler.stop(t0, t1) if sampler else None
    ms_local = (sum(a.elapsed_time(b) for a, b in step_iv) if small
                else start.elapsed_time(end))
    ms_total = max_over_ranks(torch, ms_local, world, "cuda")
    status = fgs.moe_get_device_status(ws, stream)
    if status:
        raise RuntimeError("device status after the timed steps: " + fgs.moe_status_string(status))
    router_ms = time_router(fgs, torch, cfg, T, gp, ws, nws, stream)
    gu_live_ms = statistics.mean(ev[2].elapsed_time(ev[3]) for ev in gu_events if ev)
    # stage breakdown: a few steps with every stage boundary recorded
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)]
                   for _ in range(min(steps, 10))]
    with torch.cuda.stream(stream):
        for evs in step_events:
            step(evs)
    stream.synchronize()
    stage_ms = [statistics.mean(ev[j].elapsed_time(ev[j + 1]) for ev in step_events)
                for j in range(nev - 1)]
    ms_step = ms_total / steps
    value = job_tokens_per_s(world, T, steps, ms_total)
    counts_h = counts.cpu().numpy()
    work = per_step_work(shape, counts_h)
    peaks = load_peaks()
    gu_ms = gu_live_ms  # the gate/up launch inside the timed region
    achieved = work["gate_up_bytes"] / (gu_ms / 1e3) / 1e9
    traffic = profiled_traffic(name)
    kernel = ("simt_gemm_kernel (expert gate/up + SwiGLU on CUDA cores, fp32; launch-bound at "
              "this size)" if fp32 else
              "tc_gemm_kernel (expert gate/up + SwiGLU, routed + shared)")
    roofline = {"bound": "hbm", "kernel": kernel,
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "peak_source": peaks["source"],
                "duration_samples": (f"events around the launch in {sum(1 for e in gu_events if e)}"
                                     f" of the {steps} timed steps (every {GU_EVERY}th)"),
                "algorithmic_bytes_per_launch": work["gate_up_bytes"],
                "tensor_frac_of_sustained": round(work["flops_gate_up"] / (gu_ms / 1e3) / 1e12
                                                  / peaks["bf16_tflops_sustained"], 4)}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if fp32 else "bf16",
        "data": ("synthetic (seeded; FP8 E4M3 expert weights, codes N(0,112^2) rounded by "
                 "torch's float8 cast, 128x128 block scales U(0.5,1.5)*0.02/112"
                 if is_fp8(shape) else
                 "synthetic (seeded; fp32 expert weights N(0,0.02)" if fp32 else
                 "synthetic (seeded; bf16 expert weights N(0,0.02)")
                + ", fp32 router weight kaiming-uniform, bias uniform; shapes of the pages' "
                  "K2/K3 layers)",
        "config": {"workload": WORKLOADS[name], "name": name, "tokens_per_step": T,
                   "weights": ("FP8 E4M3 + fp32 128x128 block scales, packed once before "
                               "timing (moe_pack_weights_fp8)" if is_fp8(shape) else
                               "fp32, natural layout" if fp32 else
                               "bf16, packed once before timing (moe_pack_weights)"),
                   "router_weight": ("fp32, natural" if fp32 else
                                     "fp32 W_r split once before timing into three bf16 terms "
                                     "(moe_split_router_weight)"),
                   "l2": ("inputs fit in L2: a 256 MB buffer is written between steps, outside "
                          "the timed per-step intervals" if small else
                          "inputs larger than L2: the selected experts' weights (tens of GB) "
                          "stream from HBM every step"),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline,
        "layer": {"hbm_frac": round(work["layer_bytes"] / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                  "tensor_frac_of_sustained": round(work["flops_layer"] / (ms_step / 1e3) / 1e12
                                                    / peaks["bf16_tflops_sustained"], 4),
                  "algorithmic_bytes": work["layer_bytes"], "flops": work["flops_layer"],
                  "unique_experts": work["U"]},
        # moe_router alone, timed apart from the layer steps
        "router": {"tokens_per_s": round(T / (router_ms / 1e3), 1), "ms": round(router_ms, 4),
                   "fp32_tflops": round(work["flops_router"] / (router_ms / 1e3) / 1e12, 2)},
        "stages_ms": {n: round(v, 4) for n, v in zip(fgs.STAGE_NAMES, stage_ms)},
        "stages_source": f"{len(step_events)} steps after the timed region with every stage "
                         "boundary recorded (the timed steps record only the gate/up launch)",
        "gpu_launches": launches,
        "clocks": clocks,
    }

    if not full:
        return line
    # end to end through the C ABI with host buffers (copies inside the region)
    x_host = g["x"].cpu().pin_memory()
    y_host = torch.empty((T, shape.d_model), dtype=g["x"].dtype).pin_memory()

    def step_host(fn):
        fn(cfg, T, x_host, gp["W_r"], gp["bias"], gp["W_gate_up"], gp["W_down"],
           gp.get("Ws_gate_up"), gp.get("Ws_down"), gp.get("W_lat_down"), gp.get("W_lat_up"),
           y_host, ws, nws, stream=stream)

    def time_host(fn, flush):
        for _ in range(2):
            step_host(fn)
        if flush:
            fgs.moe_layer_forward_host_flush(ws, stream=stream)
        stream.synchronize()
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        es.record(stream)
        for _ in range(e_steps):
            step_host(fn)
        # every step's y is on the host before the closing event
        if flush:
            fgs.moe_layer_forward_host_flush(ws, stream=stream)
        ee.record(stream)
        ee.synchronize()
        return max_over_ranks(torch, es.elapsed_time(ee), world, "cuda")

    e_steps = max(3, min(steps, 50))
    nbytes = T * shape.d_model * g["x"].element_size()
    # batches streamed through the pipelined call: each y leaves the device
    # while the next batch computes.  Each figure is the median of three runs
    # of e_steps steps (the host link is shared with the rest of the machine)
    e_ms = statistics.median(time_host(fgs.moe_layer_forward_host_pipelined, True)
                             for _ in range(3))
    line["e2e"] = {"value": round(job_tokens_per_s(world, T, e_steps, e_ms), 1), "unit": UNIT,
                   "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "steps": e_steps,
                   "runs": "median of 3 runs",
                   "api": "moe_layer_forward_host_pipelined (pinned host x and y; y of a batch "
                          "copied out during the next batch's forward; flushed before the "
                          "closing event)"}
    # the synchronous call: y valid as soon as the stream has passed the call
    s_ms = statistics.median(time_host(fgs.moe_layer_forward_host, False) for _ in range(3))
    line["e2e_sync"] = {"value": round(job_tokens_per_s(world, T, e_steps, s_ms), 1),
                        "unit": UNIT, "steps": e_steps, "runs": "median of 3 runs",
                        "api": "moe_layer_forward_host (pinned host x and y)"}

    fgs.moe_layer_forward_host_release(ws)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_from_device(shape, g, idx.cpu().numpy(),
                                                        args.cpu_sample_tokens or
                                                        (48 if is_fp8(shape) else 1024))
    return line




# Companion workloads measured in the same run as the headline one (each a
# short timed run of its own, with its own clocks): the other configurations
# of the benchmark set.
EXTRA = ["k2_decode", "k3_latent", "k2_router", "tiny"]
EXTRA_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "dtype", "roofline", "layer",
              "router", "stages_ms", "gpu_launches", "clocks", "config")


def run_own(args):
    import torch
    import synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_ranks(torch, world, "nccl", torch.device("cuda", local))
    try:
        import fine_grained_sparse_gb300 as fgs
    except ImportError:
        import __graft_entry__
        __graft_entry__.build()
        import fine_grained_sparse_gb300 as fgs

    line = run_layer(args, fgs, torch, synth, args.config, args.steps, args.warmup, world, rank,
                     local, full=True)
    torch.cuda.empty_cache()  # the workload's tensors died with its call
    if not args.no_extra_configs and args.config == "k2_prefill":
        extras = {}
        for name in EXTRA:
            sub = run_layer(args, fgs, torch, synth, name, args.extra_steps, 3, world, rank, local,
                            full=False)
            torch.cuda.empty_cache()
            extras[name] = {k: sub[k] for k in EXTRA_KEYS if k in sub}
        line["configs"] = extras
    if rank == 0:
        print(json.dumps(line), flush=True)
    finish_ranks(torch, world)


# ------------------------------------------------------------ reference arm
def run_reference_router(args, shape, x, W_r, bias, world):
    """The oracle router on 64 tokens of the batch per step."""
    import numpy as np
    import torch
    import oracle
    tokens_per_step = 64
    W64 = W_r.to(torch.float64).numpy()
    b32 = bias.numpy()
    times = []
    for i in range(args.warmup + args.steps):
        start = (i * tokens_per_step) % shape.T
        x64 = x[start:start + tokens_per_step].to(torch.float64).numpy()
        t0 = time.perf_counter()
        oracle.router_from_x(x64, W64, b32, shape.K, shape.n_group, shape.topk_group)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    secs = sum(times)
    value = tokens_per_step * len(times) / secs
    cores = len(os.sched_getaffinity(0))
    sample = (f"{tokens_per_step} consecutive tokens of the {shape.T}-token batch per step, fp64 "
              f"router (logits, sigmoid, selection, weights)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOADS[args.config], "name": args.config},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The CPU oracle on the same workload, one bounded sample per step."""
    import numpy as np
    import torch
    import oracle
    import synth

    world, rank, _ = dist_env()
    if rank != 0:
        return
    shape = synth.shape(args.config)
    seed = synth.SEEDS[shape.name]
    x = synth.activations(shape, "cpu", seed)
    W_r, bias = synth.router_params(shape, "cpu", seed)
    if shape.router_only:
        return run_reference_router(args, shape, x, W_r, bias, world)
    lat = synth.latent_projections(shape, "cpu", seed) if shape.d_latent else None
    draw_routed = synth.routed_expert_fp8 if is_fp8(shape) else synth.routed_expert
    draw_shared = synth.shared_expert_fp8 if is_fp8(shape) else synth.shared_expert
    sh = [draw_shared(shape, s, "cpu", seed) for s in range(shape.E_shared)]
    cache = {}

    def routed(e):
        if e not in cache:
            cache[e] = draw_routed(shape, e, "cpu", seed)
        return cache[e]

    # a pool of tokens whose experts are drawn once (drawing weights is not the
    # oracle's work); each step runs the oracle on the next token of the pool
    tokens_per_step = 1
    total = args.warmup + args.steps
    pool = np.random.default_rng(0).choice(shape.T, size=min(8, total), replace=False)
    pre = oracle.router_from_x(x[torch.as_tensor(pool)].to(torch.float64).numpy(),
                               W_r.to(torch.float64).numpy(), bias.numpy(), shape.K,
                               shape.n_group, shape.topk_group)
    for e in sorted(set(int(v) for v in pre["idx"].reshape(-1))):
        routed(e)
    times = []
    for i in range(total):
        rows = pool[i % len(pool): i % len(pool) + tokens_per_step]
        secs, _ = oracle_sample(shape, x[torch.as_tensor(rows)], W_r, bias, routed,
                                lambda s: sh[s], lat)
        if i >= args.warmup:
            times.append(secs)
    secs = sum(times)
    value = tokens_per_step * len(times) / secs
    cores = len(os.sched_getaffinity(0))
    sample = (f"{tokens_per_step} token per step, cycling over {len(pool)} tokens drawn from the "
              f"{shape.T}-token batch, full layer "
              f"(router over all {shape.E_routed} experts, {shape.K} routed + {shape.E_shared} "
              f"shared SwiGLU experts, fp64 oracle)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOADS[args.config], "name": args.config},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_own(args)


if __name__ == "__main__":
    main()
