#!/usr/bin/env python
"""Benchmark of the Kimi K3 latent routed-MoE layer forward on GB300.

One step = one forward of the whole layer (router, top-k, permutation, expert
GEMMs, combine + RMSNorm, up-projection, shared experts when configured) over
one batch of synthetic tokens, inputs resident in HBM, L2 flushed (512 MB
write) between steps outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]

Headline workload: the K3 decode batch of 16 tokens (config 1).  Without
--config the same run then measures the other K3 workloads (decode T=256,
prefill T=8192, prefill T=32768 with the Zipf selection bias and shared
experts, and that prefill with a moderate rank-based bias) with the same
steps, and reports each under detail.configs; --config C measures C alone.
Under torchrun every rank runs an independent replica on its own GPU (the
layer is token-parallel; no collective on the data path); the time is the max
over ranks and the value counts the tokens of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; decode expert-weight GB/s vs HBM peak; prefill TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) per touched expert per launch of the decode GEMVs, from
# ncu captures of 128-expert cases at the K3 shapes, scaled by the touched experts:
# the fused gate/up + down launch at T=16 (8-token tiles), the separate 16-token-tile
# launches at T=37 (4.6 rows per expert, as at T=256 with 896 experts).  They hold for
# the kernel sources (the .cu and the headers it includes) whose concatenation has the
# sha256 prefix given; any other source reports traffic null until it is captured again.
_CS = "latent_moe_layer_gb300/csrc/"
NCU_TRAFFIC = {"sources": [_CS + f for f in ("gemv_expert.cu", "gemv_expert.h", "wait.cuh", "ptx.cuh",
                                             "k3moe_internal.h")],
               "sha256_16": "6fe8398cb6a18084",
               "per_expert": {("gate_up+expert_down", "gemv"): 18.37e6, ("gate_up", "gemv"): 12.24e6,
                              ("expert_down", "gemv"): 5.883e6}}
EXTRA_WORKLOADS = [2, 3, 4, "moderate", "3a8"]


def sources_sha16(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic_per_expert():
    try:
        sha = sources_sha16(NCU_TRAFFIC["sources"])
    except OSError:
        return {}
    return NCU_TRAFFIC["per_expert"] if sha == NCU_TRAFFIC["sha256_16"] else {}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_name(cfg):
    s = (f"{cfg.name}: T={cfg.T} tokens, hidden {cfg.H}, latent {cfg.L}, {cfg.E} experts top-{cfg.K}, "
         f"expert inter {cfg.I}, MXFP4 experts, router {cfg.router_dtype}")
    if cfg.S:
        s += f", shared GLU {cfg.H}->{cfg.S}->{cfg.H} MXFP4"
    if cfg.select_bias:
        s += ", Zipf(1.1) selection bias"
    if getattr(cfg, "act", "silu") != "silu":
        s += f", {cfg.act} GLU"
    if getattr(cfg, "a8", False):
        s += ", MXFP8 activations into the routed experts"
    return s


# ------------------------------------------------------------------ accounting
def stage_work(cfg, touched, path_tensor):
    """Algorithmic bytes and flops per forward, per stage."""
    T, H, L, E, K, I, S = cfg.T, cfg.H, cfg.L, cfg.E, cfg.K, cfg.I, cfg.S
    R = T * K
    rb = 2 if cfg.router_dtype == "bf16" else 4
    act_b = 2 if path_tensor else 4
    mx = lambda rows, cols: rows * cols // 2 + rows * cols // 32
    w = {}
    w["router"] = (E * H * rb + T * H * 2 + T * E * 4, 2 * T * E * H)
    w["down_proj"] = (L * H * 2 + T * H * 2 + T * L * 2, 2 * T * L * H)
    w["topk"] = (T * E * 4 + R * 8, 0)
    w["permute"] = (R * 16, 0)
    w["gate_up"] = (touched * 2 * mx(I, L) + R * L * 2 + R * I * act_b, 4 * R * I * L)
    w["expert_down"] = (touched * mx(L, I) + R * I * act_b + R * L * act_b, 2 * R * L * I)
    w["combine_norm"] = (R * L * act_b + T * L * 2, 0)
    w["up_proj"] = (H * L * 2 + T * L * 2 + T * H * 4, 2 * T * H * L)
    if path_tensor:
        w["shared"] = ((2 * mx(S, H) + T * H * 2 + T * S * 2) if S else 0, 4 * T * S * H)
        w["shared_down"] = ((mx(H, S) + T * S * 2 + T * H * 8) if S else 0, 2 * T * H * S)
    else:
        w["shared"] = ((2 * mx(S, H) + mx(H, S) + T * H * 2 + T * H * 4) if S else 0, 6 * T * S * H)
    w["finish"] = (T * H * 6, 0)
    w["prep"] = (R * L * 4, 0)
    return w


def dominant_stage(stage_ms, work):
    """The stage with the largest time, its (bytes, flops) and whether it is the fused
    decode GEMV launch: that one is timed as the gate/up stage (no expert_down time) and
    does both projections' work."""
    fused = stage_ms.get("gate_up", 0) > 0 and stage_ms.get("expert_down", 0) == 0
    if fused:
        work = dict(work)
        work["gate_up"] = tuple(u + v for u, v in zip(work["gate_up"], work["expert_down"]))
    dom = max(stage_ms, key=lambda s: stage_ms[s])
    return dom, work[dom], fused


def load_summary(load, cfg, path_tensor):
    """Rows per expert (histogram over experts) and the tile padding of the expert GEMMs."""
    import numpy as np
    R = int(load.sum())
    srt = np.sort(load)[::-1]
    edges = [0, 1, 16, 64, 256, 1024, 4096, 1 << 30]
    hist = {f"{lo}-{hi - 1}" if hi < (1 << 30) else f">={lo}": int(((load >= lo) & (load < hi)).sum())
            for lo, hi in zip(edges[:-1], edges[1:])}
    # the expert GEMMs compute ceil(rows / 16) x 16 token columns per tile
    tile = 256 if path_tensor and R > cfg.E * 24 else 16
    computed = sum(int(-(-min(tile, c - t0) // 16) * 16) for c in load for t0 in range(0, int(c), tile))
    return {"rows": R, "max": int(srt[0]), "top16_share": round(float(srt[:16].sum()) / max(1, R), 4),
            "experts_by_rows": hist, "padding_fraction": round(1 - R / max(1, computed), 4)}


def expert_bytes(cfg):
    mx = lambda rows, cols: rows * cols // 2 + rows * cols // 32
    return 2 * mx(cfg.I, cfg.L) + mx(cfg.L, cfg.I)


# ------------------------------------------------------------------ clocks
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ oracle (CPU) timing
def oracle_sample_time(cfg, n_tokens, seed=0, min_seconds=0.0, dense=None):
    """Time the fp64 oracle on a fixed token sample, repeated until at least
    min_seconds have elapsed; returns (seconds, tokens processed, threads)."""
    import numpy as np
    from latent_moe_layer_gb300 import synth
    from oracle import oracle
    rng = np.random.default_rng(1234 + seed)
    rows = np.sort(rng.choice(cfg.T, min(n_tokens, cfg.T), replace=False))
    x = synth.gen_x(cfg, rows)
    dense = dense if dense is not None else synth.gen_dense(cfg)
    idx, _, _, _ = oracle.route(cfg, dense, x)
    experts = {int(e): synth.gen_expert(cfg, int(e)) for e in np.unique(idx)}
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.forward(cfg, dense, experts, x)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return dt, reps * len(rows), oracle.max_threads()


def cpu_sample_size(cfg):
    """Tokens of the oracle's timed sample: the whole batch up to 16 tokens, else 4-8."""
    return cfg.T if cfg.T <= 16 else (8 if cfg.T <= 256 else 4)


# ------------------------------------------------------------------ distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def reduce_max(v, world, device="cuda"):
    """Max of a per-rank scalar over all ranks (the job's wall time is the slowest replica)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_step, steps, max_total_ms, world):
    """Tokens/s of the whole job: every replica processes its own batch each step."""
    return world * tokens_per_step * steps / (max_total_ms / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ our arm
def workload_cfg(key, args=None):
    """The LayerConfig of a workload key (a config number or "moderate"), with
    the profiling overrides of args applied when given."""
    from latent_moe_layer_gb300 import synth
    if key == "3a8":            # the T=8192 prefill with MXFP8 activations (block-scaled expert GEMMs)
        cfg = synth.CONFIGS[3].with_a8(True)
        cfg = synth.LayerConfig(**{**cfg.__dict__, "name": cfg.name + "_a8"})
    else:
        cfg = synth.MODERATE_SKEW if key == "moderate" else synth.CONFIGS[key]
    if args is None:
        return cfg
    if args.experts:
        # reduced expert count: for profiler captures that must stay a few GB on the device
        cfg = synth.LayerConfig(**{**cfg.__dict__, "E": args.experts, "name": cfg.name + f"_E{args.experts}"})
    if args.tokens:
        cfg = synth.LayerConfig(**{**cfg.__dict__, "T": args.tokens, "name": cfg.name + f"_T{args.tokens}"})
    if args.act != "silu":
        cfg = synth.LayerConfig(**{**cfg.__dict__, "act": args.act, "name": cfg.name + f"_{args.act}"})
    if args.a8:
        cfg = synth.LayerConfig(**{**cfg.__dict__, "a8": True, "name": cfg.name + "_a8"})
    return cfg


class WeightCache:
    """One set of device weights at a time, keyed by everything but the
    selection bias (the moderate-skew workload reuses config 4's weights with
    its own bias)."""

    def __init__(self):
        self.key, self.dw = None, None

    def get(self, cfg):
        import copy
        import torch
        from latent_moe_layer_gb300 import k3moe, synth
        key = (cfg.wseed, cfg.H, cfg.L, cfg.E, cfg.I, cfg.S, cfg.exp_lo, cfg.exp_hi, cfg.router_dtype,
               cfg.select_bias)
        if key != self.key:
            self.key, self.dw = None, None
            torch.cuda.empty_cache()
            self.dw = k3moe.DeviceWeights(cfg)
            self.key = key
        dw = self.dw
        if cfg.select_bias and dw.cfg.bias != cfg.bias:
            dw = copy.copy(self.dw)
            dw.cfg = cfg
            dw.dense = copy.copy(self.dw.dense)
            dw.dense.select_bias = synth.gen_bias(cfg)
            dw.bias = torch.from_numpy(dw.dense.select_bias).cuda()
        return dw


def measure(cfg, dw, args, ctx, cpu_seconds, extras=True):
    """Time one workload: W warm-up and K timed steps (L2 flushed before each),
    then a profiled pass for stage times, the host-buffer e2e, the oracle on a
    token sample and the training-time extras.  Returns the JSON line's fields."""
    import numpy as np
    import torch
    from latent_moe_layer_gb300 import k3moe, synth
    world, rank, local, pk, pk_src, flush = (ctx[k] for k in ("world", "rank", "local", "pk", "pk_src",
                                                              "flush"))
    layer = k3moe.Layer(cfg, path=args.path)
    layer.load(dw)
    path_tensor = layer.path_for(cfg.T) == k3moe.PATH_TENSOR
    x = synth.gen_x(cfg)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    out = torch.empty_like(xd)
    idx = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device="cuda")
    wts = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device="cuda")
    ws = layer.workspace(cfg.T)

    def step():
        layer.forward(xd, out=out, idx_out=idx, w_out=wts, workspace=ws)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if layer.status() != 0:
        raise RuntimeError("device status after warm-up: %d" % layer.status())
    idx_np = idx.cpu().numpy()
    touched = int(np.unique(idx_np).size)
    load = np.bincount(idx_np.reshape(-1), minlength=cfg.E)

    # the timed steps run without per-stage events (they would sit between kernels
    # that otherwise launch back to back); a separate profiled pass gives the
    # stage times and the launch count
    layer.profile(False)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = Clocks(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = sum(a.elapsed_time(b) for a, b in ev)
    layer.profile(True)
    layer.profile_read()
    for i in range(min(args.steps, 20)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    nfw, stage_ms, stage_launch = layer.profile_read()
    layer.profile(False)
    st = layer.status()
    if st != 0:
        raise RuntimeError(f"device status {st}")
    total_ms = reduce_max(total_ms, world)
    ms_step = total_ms / args.steps
    value = whole_job_value(cfg.T, args.steps, total_ms, world)

    # roofline of the dominant stage
    work = stage_work(cfg, touched, path_tensor)
    dom, (b, f), fused = dominant_stage(stage_ms, work)
    per_launch_ms = stage_ms[dom] / max(1, nfw)
    decode = cfg.T <= 256
    if decode or f == 0:
        ach = b / (per_launch_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / pk["hbm_gbs"], 4), "traffic": None}
    elif getattr(cfg, "a8", False) and dom in ("gate_up", "expert_down") and ctx.get("mma_peaks"):
        # block-scaled kind::mxf8f6f4 expert GEMMs: the tensor cores' own rate for that kind
        ach = f / (per_launch_ms / 1e3) / 1e12
        peak = ctx["mma_peaks"]["mxf8f6f4_e2m1_e4m3_n224_tflops"]
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "traffic": None,
                "peak_kind": "tcgen05 kind::mxf8f6f4 E2M1 x E4M3, N 224, own microbenchmark (burst)"}
    else:
        ach = f / (per_launch_ms / 1e3) / 1e12
        peak = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "traffic": None, "peak_kind": "bf16 dense, sustained"}
    key = ("gate_up+expert_down" if fused and dom == "gate_up" else dom,
           "gemv" if (path_tensor and cfg.T * cfg.K <= cfg.E * 24) else "other")
    traffic = ncu_traffic_per_expert()
    if key in traffic:
        roof["traffic"] = round(traffic[key] * touched)
        roof["traffic_source"] = "ncu dram bytes per touched expert x touched experts"
    roof.update({"kernel_stage": dom + ("+expert_down (one launch)" if fused and dom == "gate_up" else ""),
                 "per_launch_ms": round(per_launch_ms, 4),
                 "algorithmic_bytes": b, "algorithmic_flops": f,
                 "peak_source": "own microbenchmark" if "own" in roof.get("peak_kind", "") else pk_src})

    # end to end through the host-buffer C-ABI call
    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(x.view(np.int16)).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        for _ in range(2):
            layer.forward_host(xh, oh, workspace=ws)
        ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        barrier(world)
        for i in range(args.steps):
            flush.zero_()
            ee[i][0].record()
            layer.forward_host(xh, oh, workspace=ws)
            ee[i][1].record()
        torch.cuda.synchronize()
        barrier(world)
        e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in ee), world)
        e2e = {"value": round(whole_job_value(cfg.T, args.steps, e_ms, world), 2), "unit": "tokens/s",
               "h2d_bytes_per_step": cfg.T * cfg.H * 2, "d2h_bytes_per_step": cfg.T * cfg.H * 2,
               "ms_per_step": round(e_ms / args.steps, 4)}

    # CPU baseline: the oracle on a bounded token sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = cpu_sample_size(cfg)
        dt, nt, thr = oracle_sample_time(cfg, n, min_seconds=cpu_seconds, dense=dw.dense)
        cpu = {"value": round(nt / dt, 4), "unit": "tokens/s", "cores": thr, "kind": "oracle",
               "sample": f"{n} tokens of {cfg.name} (fp64 oracle, all layer steps), repeated to "
                         f"{nt} tokens in {dt:.2f} s"}

    qb_line = qb_timing(layer, cfg, flush, pk) if (extras and cfg.select_bias) else None
    ep_line = ep_timing(layer, cfg, flush) if (extras and cfg.T >= 4096 and not args.no_ep) else None

    exp_ms = stage_ms["gate_up"] + stage_ms["expert_down"]
    detail = {
        "stage_ms_per_step": {k: round(v / max(1, nfw), 4) for k, v in stage_ms.items() if v > 0},
        "touched_experts": touched,
        "expert_load": load_summary(load, cfg, path_tensor),
        "expert_weight_gbs": round(touched * expert_bytes(cfg) / (exp_ms / max(1, nfw) / 1e3) / 1e9, 1)
        if exp_ms > 0 else None,
        "layer_tflops": round(sum(v[1] for v in work.values()) / (ms_step / 1e3) / 1e12, 3),
        "path": "tensor" if path_tensor else "generic",
    }
    if qb_line:
        detail["qb_bias_update"] = qb_line
    if ep_line:
        detail["expert_parallel_plan"] = ep_line
    res = {"value": round(value, 2), "unit": "tokens/s", "ms_per_step": round(ms_step, 4),
           "dtype": "f16" if path_tensor else "f32",
           "config": {"workload": workload_name(cfg), "tokens_per_step": cfg.T,
                      "l2": "flushed between steps (512 MB write, outside the timed events)",
                      "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                      "weights": "MXFP4 experts (E2M1 + E8M0/32), BF16 dense, seeded synthetic"},
           "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
           "gpu_launches": int(round(sum(stage_launch.values()) / max(1, nfw) * args.steps)), "clocks": clk,
           "detail": detail}
    del layer, ws
    return res


def qb_timing(layer, cfg, flush, pk):
    """Quantile-Balancing bias update (the training-time estimator of the
    selection bias), on seeded N(0, 1.5^2) router logits of this workload's shape."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(7)
    lg = torch.randn((cfg.T, cfg.E), generator=g, device="cuda") * 1.5
    b0 = torch.zeros(cfg.E, dtype=torch.float32, device="cuda")
    for _ in range(3):
        layer.qb_bias(lg, b0)
    # the logits (T E 4 bytes) may fit in L2: flush it before each timed call
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    torch.cuda.synchronize()
    for q0, q1 in ev:
        flush.zero_()
        q0.record()
        layer.qb_bias(lg, b0)
        q1.record()
    torch.cuda.synchronize()
    qms = sum(q0.elapsed_time(q1) for q0, q1 in ev) / len(ev)
    qbytes = 2 * cfg.T * cfg.E * 4                 # the logits are read twice
    return {"ms": round(qms, 4), "algorithmic_bytes": qbytes,
            "achieved_gbs": round(qbytes / (qms / 1e3) / 1e9, 1),
            "frac": round(qbytes / (qms / 1e3) / 1e9 / pk["hbm_gbs"], 4), "nbins": 1000}


def ep_timing(layer, cfg, flush):
    """Balanced expert-parallel plan and dispatch (the MoonEP step around the
    experts): R ranks each routing this workload's T tokens (top-K of seeded
    N(0, 1) logits); one source rank's dispatch timed."""
    import torch
    ep_line = {}
    g = torch.Generator(device="cuda").manual_seed(9)
    for R in (8, 64):
        if cfg.E % R:
            continue
        cnt = torch.empty((R, cfg.E), dtype=torch.int32, device="cuda")
        idx0 = None
        for q in range(R):
            lg = torch.randn((cfg.T, cfg.E), generator=g, device="cuda")
            top = torch.topk(lg, cfg.K, dim=1).indices.to(torch.int32).contiguous()
            cnt[q] = torch.bincount(top.flatten(), minlength=cfg.E).to(torch.int32)
            if q == 0:
                idx0 = top
        # each call captured once in a CUDA graph with preallocated outputs, so
        # the events see device time rather than the binding's host overhead
        plan = layer.ep_plan(cnt, cfg.T)
        dout = (torch.empty_like(idx0), torch.empty_like(idx0))
        dws = torch.empty(layer.ep_dispatch_workspace_bytes(cfg.T), dtype=torch.uint8, device="cuda")
        for _ in range(3):
            layer.ep_plan(cnt, cfg.T, out=plan)
            layer.ep_dispatch(idx0, 0, cnt, plan, out=dout, workspace=dws)
        torch.cuda.synchronize()
        g_plan, g_disp = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_plan):
            layer.ep_plan(cnt, cfg.T, out=plan)
        with torch.cuda.graph(g_disp):
            layer.ep_dispatch(idx0, 0, cnt, plan, out=dout, workspace=dws)
        n_rep = 20
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_rep)]
        torch.cuda.synchronize()
        for q0, q1 in ev:
            q0.record()
            g_plan.replay()
            q1.record()
        torch.cuda.synchronize()
        plan_ms = sum(q0.elapsed_time(q1) for q0, q1 in ev) / n_rep
        for q0, q1 in ev:
            flush.zero_()
            q0.record()
            g_disp.replay()
            q1.record()
        torch.cuda.synchronize()
        disp_ms = sum(q0.elapsed_time(q1) for q0, q1 in ev) / n_rep
        if layer.status() != 0:
            raise RuntimeError("expert-parallel plan or dispatch reported a device error")
        info = plan["info"].tolist()
        pairs = cfg.T * cfg.K
        dbytes = 12 * pairs                         # idx read, destination rank and row written
        ep_line[f"ranks_{R}"] = {
            "tokens_per_rank": cfg.T, "plan_us": round(plan_ms * 1e3, 1), "dispatch_us": round(disp_ms * 1e3, 1),
            "segments": info[0], "max_redundant_experts": info[1], "redundant_slots_per_rank": cfg.E // R,
            "dispatch_algorithmic_bytes": dbytes,
            "dispatch_gbs": round(dbytes / (disp_ms / 1e3) / 1e9, 1), "dispatch_launches": 4,
            "timing": "CUDA-graph replay of one call, events around the replay"}
    return ep_line


def run_ours(args):
    import torch
    import __graft_entry__ as ge

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    ge.build()
    pk, pk_src = peaks()
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    ctx = dict(world=world, rank=rank, local=local, pk=pk, pk_src=pk_src, flush=flush)
    if args.config is None or getattr(args, "a8", False) or args.config == "3a8":
        ctx["mma_peaks"] = measure_mma_peaks()
    cache = WeightCache()
    head_key = args.config if args.config is not None else 1
    cfg = workload_cfg(head_key, args)
    head = measure(cfg, cache.get(cfg), args, ctx, cpu_seconds=10.0)
    line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
            "data": "synthetic", "config": head["config"], "roofline": head["roofline"],
            "cpu_baseline": head["cpu_baseline"], "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"], "detail": head["detail"]}
    if args.config is None and not args.no_extra:
        # the other K3 workloads, same steps and warm-up, each with its own
        # timed region, clocks, roofline and oracle sample
        configs = {}
        for key in EXTRA_WORKLOADS:
            c = workload_cfg(key)
            r = measure(c, cache.get(c), args, ctx, cpu_seconds=4.0)
            configs[c.name] = {"workload": r["config"]["workload"], "tokens_per_step": c.T,
                               "ms_per_step": r["ms_per_step"], "value": r["value"], "unit": r["unit"],
                               "dtype": r["dtype"], "roofline": r["roofline"], "clocks": r["clocks"],
                               "cpu_baseline": r["cpu_baseline"], "e2e": r["e2e"],
                               "gpu_launches": r["gpu_launches"], **r["detail"]}
        line["detail"]["configs"] = configs
    if ctx.get("mma_peaks"):
        line["detail"]["mma_peaks"] = ctx["mma_peaks"]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm (the oracle)
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from latent_moe_layer_gb300 import synth
    from oracle import oracle
    import numpy as np
    oracle.build()
    cfg = workload_cfg(args.config if args.config is not None else 1)
    n = 2 if cfg.T <= 256 else 1
    rng = np.random.default_rng(99)
    dense = synth.gen_dense(cfg)
    samples = []
    for s in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(cfg.T, n, replace=False))
        x = synth.gen_x(cfg, rows)
        idx, _, _, _ = oracle.route(cfg, dense, x)
        experts = {int(e): synth.gen_expert(cfg, int(e)) for e in np.unique(idx)}
        t0 = time.perf_counter()
        oracle.forward(cfg, dense, experts, x)
        samples.append(time.perf_counter() - t0)
    timed = samples[args.warmup:]
    tot = sum(timed)
    val = n * args.steps / tot
    thr = oracle.max_threads()
    cpu = {"value": round(val, 4), "unit": "tokens/s", "cores": thr, "kind": "oracle",
           "sample": f"{n} random tokens of {cfg.name} per step (fp64 oracle, all layer steps)"}
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(cfg), "tokens_per_step": n},
            "cpu_baseline": cpu,
            "e2e": {"value": round(val, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def library_peaks(steps=50):
    """Context numbers for the roofline discussion (not used by the layer): dense
    GEMM throughput of the vendor library on this GPU at 8192^3 -- BF16
    (torch.matmul), FP8 E4M3 with per-tensor scales and, where this PyTorch build
    exposes it, MXFP8 (E4M3 with E8M0 scales per 32 values) through
    torch._scaled_mm.  Prints one JSON line."""
    import torch
    n = 8192
    out = {"shape": [n, n, n]}

    def timed(fn):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return round(2.0 * n ** 3 / (e0.elapsed_time(e1) / steps * 1e-3) / 1e12, 1)

    a = torch.randn(n, n, device="cuda", dtype=torch.bfloat16)
    b = torch.randn(n, n, device="cuda", dtype=torch.bfloat16)
    out["bf16_tflops"] = timed(lambda: a @ b)
    a8 = a.to(torch.float8_e4m3fn)
    b8 = b.to(torch.float8_e4m3fn).t().contiguous().t()      # column-major second operand
    one = torch.ones((), device="cuda", dtype=torch.float32)
    try:
        out["fp8_tensorwise_tflops"] = timed(lambda: torch._scaled_mm(a8, b8, one, one, out_dtype=torch.bfloat16))
    except Exception as ex:                                     # noqa: BLE001
        out["fp8_tensorwise_tflops"] = None
        out["fp8_tensorwise_error"] = str(ex).splitlines()[0][:200]
    try:
        e8 = getattr(torch, "float8_e8m0fnu")
        sa = torch.full((n, n // 32), 127, device="cuda", dtype=torch.uint8).view(e8)
        sb = torch.full((n, n // 32), 127, device="cuda", dtype=torch.uint8).view(e8)
        out["mxfp8_tflops"] = timed(lambda: torch._scaled_mm(a8, b8, sa, sb, out_dtype=torch.bfloat16))
    except Exception as ex:                                     # noqa: BLE001
        out["mxfp8_tflops"] = None
        out["mxfp8_error"] = str(ex).splitlines()[0][:200]
    out["device"] = torch.cuda.get_device_name(0)
    print(json.dumps(out))


def measure_mma_peaks(iters=4096):
    """TFLOP/s of back-to-back tcgen05.mma per kind (k3moe_mma_peak), one CTA per SM."""
    from latent_moe_layer_gb300 import k3moe
    out = {"method": "tcgen05.mma back to back, M 128, operands in shared memory, one CTA per SM, "
                     f"{iters} x 128 K per CTA, CUDA events"}
    for kind, ns in [("f16", (256, 224)), ("mxf8f6f4_e4m3", (256, 224)), ("mxf8f6f4_e2m1_e4m3", (256, 224, 192))]:
        for n in ns:
            k3moe.mma_peak(kind, n, iters // 8)        # warm the clocks
            out[f"{kind}_n{n}_tflops"] = round(k3moe.mma_peak(kind, n, iters), 1)
    return out


def mma_peaks(iters=4096):
    """The tensor cores' own rate for each MMA kind the expert GEMMs use: back-to-back
    tcgen05.mma on shared-memory operands, one CTA per SM (k3moe_mma_peak).  Prints
    one JSON line of TFLOP/s; the block-scaled A8 roofline divides by the E2M1 x E4M3
    figure at N = 224, the tile width of the block-scaled expert GEMMs."""
    import torch
    import __graft_entry__ as ge
    ge.build()
    out = measure_mma_peaks(iters)
    out["device"] = torch.cuda.get_device_name(0)
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=None,
                    help="measure one workload alone: 0-4, 'moderate' or '3a8' (default: config 1, then the others)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 generic, 2 tensor")
    ap.add_argument("--experts", type=int, default=0, help="override the expert count (profiling aid)")
    ap.add_argument("--tokens", type=int, default=0, help="override the token count (profiling aid)")
    ap.add_argument("--act", default="silu", choices=["silu", "situ"],
                    help="GLU activation (the workload's is SiLU; SiTU is the option the layer also supports)")
    ap.add_argument("--a8", action="store_true", help="MXFP8 activations into the routed experts (the A8 option)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ep", action="store_true", help="skip the expert-parallel plan timing (prefill configs)")
    ap.add_argument("--no-extra", action="store_true", help="measure the headline workload only")
    ap.add_argument("--mma-peaks", action="store_true",
                    help="print the tensor cores' own MMA rates (tcgen05 microbenchmark) and exit")
    ap.add_argument("--library-peaks", action="store_true",
                    help="print the vendor library's dense BF16 / FP8 / MXFP8 GEMM rates and exit")
    args = ap.parse_args()
    if args.config is not None and args.config not in ("moderate", "3a8"):
        args.config = int(args.config)
    if args.library_peaks:
        library_peaks()
        return
    if args.mma_peaks:
        mma_peaks()
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
