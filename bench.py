#!/usr/bin/env python3
"""Decode throughput of the routed sparse-MoE stack on GB300.

One step = one batch of B tokens through every MoE layer of the workload
(router -> top-k -> slot lookup -> int4 dequant gate/up + SwiGLU -> down +
weighted combine + sigmoid-gated shared expert -> renormalisation), through
the C ABI (moe_forward_decode_stack) with inputs resident in HBM.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores on the same workload instead (each step: one token through one
layer, which is 1/n_layers of a token of the metric's unit).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import dataclasses
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-stack decode tok/s; expert-weight HBM GB/s as fraction of GB300 peak"
FALLBACK_HBM_GBS = 6800.0
# DRAM bytes (read + write) of one decode-stack launch per layer: an ncu capture
# of the 35B-shaped int4 stack at batch 1 (4 layers, 68.025344 + 0.380160 MB),
# scaled by the layer count; valid for that workload and the current kernel
STACK_35B_DRAM_BYTES_PER_LAYER = 68.405504e6 / 4
FALLBACK_BF16_TFLOPS = 1700.0
PREFILL_METRIC = "MoE prefill tok/s; grouped-GEMM bf16 TFLOP/s as fraction of GB300 dense peak"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (default: 2048 decode, 1024 stress, 50 prefill)")
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="35b", choices=["tiny", "35b", "80b", "80b-prefill", "stress"])
    ap.add_argument("--tokens", type=int, default=0, help="prefill tokens per step (default: the workload's)")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--bits", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling cases)")
    ap.add_argument("--cpu-samples", type=int, default=64, help="(token, layer) samples of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-subrecords", action="store_true",
                    help="default run: skip the 80B decode (B = 1, 8, 64) and 80B prefill sub-records")
    ap.add_argument("--slots", type=int, default=0, help="stress: slots per layer (default: the workload's 128)")
    ap.add_argument("--policy", default="lfu", choices=list(POLICIES), help="stress: eviction policy")
    ap.add_argument("--aging", type=int, default=64, help="stress: calls between halvings of the aged LFU")
    ap.add_argument("--store-file", default="",
                    help="stress: read misses from this expert container (written first unless it matches)")
    ap.add_argument("--store-direct", action="store_true", help="stress: O_DIRECT reads of the container")
    ap.add_argument("--pool-sweep", action="store_true",
                    help="stress: one JSON line per (slots, policy) point on one loaded store instead of the bench line")
    ap.add_argument("--sweep-slots", default="16,32,64,128,256")
    ap.add_argument("--sweep-policies", default="lfu,lru,persist,aged")
    return ap.parse_args()


# eviction policies by name (MOE_EVICT_* values of the C ABI)
POLICIES = {"lfu": 0, "lru": 1, "persist": 2, "aged": 3}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 TFLOP/s, burst figure: the grouped GEMMs run a few hundred
    microseconds inside a step of about a millisecond, not a seconds-long loop."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured (burst)"
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured (sustained)"
    return FALLBACK_BF16_TFLOPS, "fallback"


def workload_desc(w, B, bits):
    return (f"{w.name} decode stack: {w.n_layers} MoE layers, hidden {w.hidden}, {w.n_experts} experts top-{w.top_k}, "
            f"expert inter {w.inter}, shared inter {w.shared_inter}, int{bits} group-64 affine, batch {B}"
            + (", Zipf(1.1) router bias" if w.zipf_s else "") + ", renormalised per layer, all experts resident")


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                try:
                    rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
                except ValueError:
                    pass
        os.unlink(self.path)
        if not rows:
            return None
        sm = [r[0] for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[2]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and --impl reference)
# --------------------------------------------------------------------------
def oracle_samples(w, bits, n_samples, threads):
    """(token, layer) samples with their routed experts drawn beforehand (untimed):
    token = a renormalised N(0,1) vector, the distribution of a layer input."""
    import oracle
    samples = []
    for i in range(n_samples):
        layer = i % w.n_layers
        x = oracle.renorm(synth.tokens(w.seed, 900000 + i, 1, w.hidden)[0])
        wr, wsg, beta = synth.layer_inputs(w, layer)
        lay = oracle.Layer(w.hidden, w.n_experts, w.top_k, w.inter, w.shared_inter, wr, wsg, {}, router_bias=beta,
                           shared=synth.expert(w.seed, layer, synth.SHARED, w.hidden, w.shared_inter, bits, w.sigma))
        _, idx, _, _ = lay.route(x)
        samples.append((layer, x, lay, [int(e) for e in idx]))
    with cf.ThreadPoolExecutor(threads) as ex:
        for (layer, x, lay, idx) in samples:
            ex_arrays = dict(zip(idx, ex.map(lambda e: synth.expert(w.seed, layer, e, w.hidden, w.inter, bits,
                                                                    w.sigma), idx)))
            lay.set_experts(ex_arrays)
    return samples


def time_oracle(samples, n_steps, threads):
    """Run n_steps (token, layer) oracle evaluations over `threads` host threads."""
    def run(i):
        _, x, lay, _ = samples[i % len(samples)]
        lay.token(x)
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(run, range(n_steps)))
    return time.perf_counter() - t0


def cpu_baseline(w, bits, n_samples):
    threads = os.cpu_count() or 1
    samples = oracle_samples(w, bits, min(n_samples, 32), threads)
    secs = time_oracle(samples, n_samples, threads)
    return {"value": (n_samples / w.n_layers) / secs, "unit": "tok/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_samples} (token, layer) evaluations of the fp64 scalar oracle (one token through one "
                      f"of the {w.n_layers} layers each, inputs renormalised N(0,1)), split over {threads} host "
                      f"threads; {secs:.1f} s wall"}


def max_over_ranks(ms: float, pg) -> float:
    """The slowest replica's time in ms (gloo all-reduce MAX, then a barrier);
    the identity on a single process."""
    if not pg:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    pg.barrier()
    return float(t.item())


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = synth.CONFIGS[args.config]
    bits = args.bits or w.bits
    threads = os.cpu_count() or 1
    samples = oracle_samples(w, bits, 32, threads)
    time_oracle(samples, max(args.warmup, 1), threads)
    secs = time_oracle(samples, args.steps, threads)
    value = (args.steps / w.n_layers) / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w, 1, bits), "step": "one token through one layer (1/n_layers token)"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} (token, layer) oracle evaluations over {threads} host threads"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# our path
# --------------------------------------------------------------------------
def decode_record(moe, ctx, w, bits, B, steps, warmup, local, pg, world, e2e_steps=0):
    """Time `steps` decode-stack steps of B tokens (inputs resident in HBM,
    CUDA events on the launching stream) on a loaded context; returns the
    measurement fields of a line: value, ms_per_step, roofline, clocks, launches."""
    import torch

    L, H, k = w.n_layers, w.hidden, w.top_k
    n_ring = 256
    X = torch.from_numpy(np.stack([synth.tokens(w.seed, s, B, H) for s in range(n_ring)])).cuda()
    y = torch.empty((B, H), device="cuda")
    st = torch.cuda.current_stream()
    # expert bytes actually read per step: (distinct routed experts + shared) x blob bytes, per layer
    blob = moe.moe_blob_bytes(H, w.inter, bits)
    sblob = moe.moe_blob_bytes(H, w.shared_inter, bits) if w.shared_inter else 0
    it = torch.empty((L, B, k), dtype=torch.int32, device="cuda")
    uniq = []
    for s in range(min(n_ring, 32)):
        moe.moe_forward_decode_stack(ctx, 0, L, X[s], B, y, 1e-6, None, it, None, st)
        idx = it.cpu().numpy()
        uniq.append(sum(len(np.unique(idx[l])) for l in range(L)))
    expert_bytes = float(np.mean(uniq)) * blob + L * sblob
    router_bytes = L * w.n_experts * H * 2
    for s in range(warmup):
        moe.moe_forward_decode_stack(ctx, 0, L, X[s % n_ring], B, y, 1e-6, None, None, None, st)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    l0 = moe.moe_launch_count(ctx)
    clk = ClockSampler(local)
    clk.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for s in range(steps):
        moe.moe_forward_decode_stack(ctx, 0, L, X[s % n_ring], B, y, 1e-6, None, None, None, st)
    e1.record(st)
    torch.cuda.synchronize()
    clocks = clk.stop()
    launches = moe.moe_launch_count(ctx) - l0
    ms = max_over_ranks(e0.elapsed_time(e1), pg)
    secs = ms / 1e3
    gbs = expert_bytes * steps / secs / 1e9
    peak, peak_kind = peaks()
    traffic = (STACK_35B_DRAM_BYTES_PER_LAYER * L
               if (w.name, B, bits, w.hidden, w.n_experts) == ("35b", 1, 4, 2048, 256) else None)
    rec = {
        "value": steps * B * world / secs, "unit": "tok/s", "ms_per_step": ms / steps, "steps": steps,
        "warmup": warmup, "batch": B,
        "expert_gbs": gbs, "hbm_frac": gbs / peak,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_kind": peak_kind, "traffic": traffic,
                     "traffic_unit": "DRAM bytes per launch (ncu, 4-layer capture scaled by layers)",
                     "kernel": ("decode stack (one persistent forward_decode_stack launch per step)" if launches == steps
                                else "decode stack (per-layer kernels, one forward_decode_stack call per step)"),
                     "bytes_per_launch": expert_bytes, "router_bytes_per_launch": router_bytes},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    if e2e_steps:
        # end to end through the public API with host buffers: pinned H2D of the
        # step's tokens, the stack, D2H of the step's output, every step
        xh = torch.from_numpy(np.stack([synth.tokens(w.seed, s, B, H) for s in range(n_ring)])).pin_memory()
        yh = torch.empty((B, H)).pin_memory()
        xd = torch.empty((B, H), device="cuda")
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for s in range(e2e_steps):
            xd.copy_(xh[s % n_ring], non_blocking=True)
            moe.moe_forward_decode_stack(ctx, 0, L, xd, B, y, 1e-6, None, None, None, st)
            yh.copy_(y, non_blocking=True)
            st.synchronize()
        e2e_s = time.perf_counter() - t0
        rec["e2e"] = {"value": e2e_steps * B * world / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": B * H * 4,
                      "d2h_bytes_per_step": B * H * 4, "steps": e2e_steps}
    return rec


def subrecords(args, moe, workload, local, pg, world):
    """The other single-GPU workloads as sub-records of the default line: the
    80B decode stack at 1, 8 and 64 tokens, then the 80B prefill layer."""
    out = []
    w = synth.CONFIGS["80b"]
    ctx = workload.create_loaded(w, w.bits, max_batch=max(w.batches))
    try:
        for B in w.batches:
            rec = decode_record(moe, ctx, w, w.bits, B, args.steps, max(args.warmup, 3), local, pg, world)
            rec = {"metric": METRIC, "workload": workload_desc(w, B, w.bits), **rec}
            out.append(rec)
    finally:
        moe.moe_destroy(ctx)
    wp = synth.CONFIGS["80b-prefill"]
    ctx = workload.create_loaded(wp, wp.bits, max_tokens=wp.prefill_tokens)
    try:
        rec = prefill_record(moe, ctx, wp, wp.bits, wp.prefill_tokens, args.steps, max(args.warmup, 3), local, pg,
                             world)
        out.append({"metric": PREFILL_METRIC, "workload": prefill_desc(wp, wp.prefill_tokens, wp.bits), **rec})
    finally:
        moe.moe_destroy(ctx)
    return out


def run_ours(args):
    import torch

    import int4_expert_streaming_gb300 as moe
    from int4_expert_streaming_gb300 import workload

    rank, world, local = dist_env()
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")  # replicas: host-side barrier and max only
        pg = dist
    torch.cuda.set_device(local)
    w = synth.CONFIGS[args.config]
    if args.layers:
        w = dataclasses.replace(w, n_layers=args.layers)
    bits = args.bits or w.bits
    B = args.batch
    L = w.n_layers
    moe.build()
    ctx = workload.create_loaded(w, bits, max_batch=B)
    try:
        rec = decode_record(moe, ctx, w, bits, B, args.steps, args.warmup, local, pg, world,
                            e2e_steps=0 if args.no_e2e else min(args.steps, 512))
    finally:
        moe.moe_destroy(ctx)
    line = {
        "metric": METRIC, "value": rec["value"], "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(w, B, bits), "batch": B, "layers": L, "bits": bits,
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "l2": f"inputs larger than L2: {rec['roofline']['bytes_per_launch'] / 1e6:.1f} MB of expert "
                         "weights per step"},
        "expert_gbs": rec["expert_gbs"], "hbm_frac": rec["hbm_frac"],
        "roofline": rec["roofline"],
        "gpu_launches": rec["gpu_launches"],
        "clocks": rec["clocks"],
        "e2e": rec.get("e2e"),
    }
    default_run = (args.config == "35b" and not args.layers and not args.bits and B == 1)
    if default_run and not args.no_subrecords:
        line["configs"] = subrecords(args, moe, workload, local, pg, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, bits, args.cpu_samples)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


# --------------------------------------------------------------------------
# prefill (one 80B-shaped layer, T tokens per step)
# --------------------------------------------------------------------------
def prefill_desc(w, T, bits):
    return (f"{w.name}: one MoE layer, hidden {w.hidden}, {w.n_experts} experts top-{w.top_k}, expert inter "
            f"{w.inter}, shared inter {w.shared_inter}, int{bits} group-64 affine, {T} tokens per step, "
            "Zipf(1.1) router bias, tokens sorted per expert into tcgen05 grouped GEMMs, all experts resident")


def prefill_cpu_baseline(w, bits, n_tokens):
    """The oracle's prefill definition on n_tokens of the workload (one layer), all host cores."""
    import oracle
    threads = os.cpu_count() or 1
    x = synth.tokens(w.seed, 900001, n_tokens, w.hidden)
    wr, wsg, beta = synth.layer_inputs(w, 0)
    router = oracle.Layer(w.hidden, w.n_experts, w.top_k, w.inter, w.shared_inter, wr, wsg, {}, router_bias=beta)
    need = sorted({int(e) for t in range(n_tokens) for e in router.route(x[t])[1]})
    with cf.ThreadPoolExecutor(threads) as ex:
        experts = dict(zip(need, ex.map(lambda e: synth.expert(w.seed, 0, e, w.hidden, w.inter, bits, w.sigma), need)))
    lay = oracle.Layer(w.hidden, w.n_experts, w.top_k, w.inter, w.shared_inter, wr, wsg, experts, router_bias=beta,
                       shared=synth.expert(w.seed, 0, synth.SHARED, w.hidden, w.shared_inter, bits, w.sigma))
    t0 = time.perf_counter()
    lay.tokens(x, prefill=True, threads=threads)
    secs = time.perf_counter() - t0
    return {"value": n_tokens / secs, "unit": "tok/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_tokens} tokens of the prefill layer through the fp64 scalar oracle (prefill definition: "
                      f"bf16 weights and x), split over {threads} host threads; {secs:.1f} s wall"}


def prefill_record(moe, ctx, w, bits, T, steps, warmup, local, pg, world, e2e_steps=0):
    """Time `steps` prefill calls of T tokens on a loaded context (CUDA events),
    with per-kernel device times; returns the measurement fields of a line."""
    import torch

    H, k = w.hidden, w.top_k
    n_ring = 5  # 5 x T x H fp32 inputs: larger than L2 at the workload's T
    X = torch.from_numpy(np.stack([synth.tokens(w.seed, s, T, H) for s in range(n_ring)])).cuda()
    y = torch.empty((T, H), device="cuda")
    st = torch.cuda.current_stream()
    flop = 2.0 * T * k * 3 * H * w.inter + 2.0 * T * 3 * H * w.shared_inter
    for s in range(warmup):
        moe.moe_forward_prefill(ctx, 0, X[s % n_ring], T, y, None, None, st)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    moe.moe_prefill_profile(ctx, True)
    l0 = moe.moe_launch_count(ctx)
    clk = ClockSampler(local)
    clk.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for s in range(steps):
        moe.moe_forward_prefill(ctx, 0, X[s % n_ring], T, y, None, None, st)
    e1.record(st)
    torch.cuda.synchronize()
    clocks = clk.stop()
    launches = moe.moe_launch_count(ctx) - l0
    kms, calls = moe.moe_prefill_kernel_ms(ctx)
    moe.moe_prefill_profile(ctx, False)
    ms = max_over_ranks(e0.elapsed_time(e1), pg)
    secs = ms / 1e3
    per_kernel = {n: v / calls for n, v in kms.items()}
    gemm_ms = per_kernel["gateup_gemm"] + per_kernel["down_gemm"]
    peak, peak_kind = tensor_peak()
    achieved = flop / (gemm_ms / 1e3) / 1e12
    rec = {
        "value": steps * T * world / secs, "unit": "tok/s", "ms_per_step": ms / steps, "steps": steps,
        "warmup": warmup, "tokens": T,
        "layer_tflops": flop / secs * steps / 1e12,
        "kernel_ms": per_kernel,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_kind": peak_kind, "traffic": None,
                     "kernel": "grouped GEMMs (gate/up + down), algorithmic FLOPs 2*T*k*3*H*I + 2*T*3*H*I_s",
                     "flops_per_launch": flop, "ms_per_launch": gemm_ms},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    if e2e_steps:
        xh = torch.from_numpy(np.stack([synth.tokens(w.seed, s, T, H) for s in range(2)])).pin_memory()
        yh = torch.empty((T, H)).pin_memory()
        xd = torch.empty((T, H), device="cuda")
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for s in range(e2e_steps):
            xd.copy_(xh[s % 2], non_blocking=True)
            moe.moe_forward_prefill(ctx, 0, xd, T, y, None, None, st)
            yh.copy_(y, non_blocking=True)
            st.synchronize()
        e2e_s = time.perf_counter() - t0
        rec["e2e"] = {"value": e2e_steps * T * world / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": T * H * 4,
                      "d2h_bytes_per_step": T * H * 4, "steps": e2e_steps}
    return rec


def run_prefill(args):
    import torch

    import int4_expert_streaming_gb300 as moe
    from int4_expert_streaming_gb300 import workload

    rank, world, local = dist_env()
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    torch.cuda.set_device(local)
    w = synth.CONFIGS[args.config]
    bits = args.bits or w.bits
    T = args.tokens or w.prefill_tokens
    moe.build()
    ctx = workload.create_loaded(w, bits, max_tokens=T)
    try:
        rec = prefill_record(moe, ctx, w, bits, T, args.steps, args.warmup, local, pg, world,
                             e2e_steps=0 if args.no_e2e else min(args.steps, 32))
        line = {
            "metric": PREFILL_METRIC, "value": rec["value"], "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": prefill_desc(w, T, bits), "tokens": T, "bits": bits,
                       "parallelism": "replicas" if world > 1 else "single-gpu",
                       "l2": "inputs larger than L2: 5 rotating token batches of "
                             f"{T * w.hidden * 4 / 1e6:.1f} MB plus the touched experts' weights"},
            "layer_tflops": rec["layer_tflops"],
            "kernel_ms": rec["kernel_ms"],
            "roofline": rec["roofline"],
            "gpu_launches": rec["gpu_launches"],
            "clocks": rec["clocks"],
            "e2e": rec.get("e2e"),
        }
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = prefill_cpu_baseline(w, bits, 16)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        moe.moe_destroy(ctx)
        if pg:
            pg.destroy_process_group()


# --------------------------------------------------------------------------
# streaming stress (pool of 128 of 512 slots per layer, store in pinned host memory)
# --------------------------------------------------------------------------
def host_link_probe_gbs(nbytes: int = 1 << 30) -> float:
    """Pinned host -> device copy bandwidth (one cudaMemcpyAsync per copy)."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        d.copy_(h, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    gbs = 5 * nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9
    del h, d
    return gbs


def run_stress(args):
    import torch

    import int4_expert_streaming_gb300 as moe
    from int4_expert_streaming_gb300 import workload

    rank, world, local = dist_env()
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    torch.cuda.set_device(local)
    w = synth.CONFIGS["stress"]
    if args.layers:
        w = dataclasses.replace(w, n_layers=args.layers)
    bits = args.bits or w.bits
    L, H, k = w.n_layers, w.hidden, w.top_k
    moe.build()
    link_peak = host_link_probe_gbs()
    if args.pool_sweep:
        if world > 1:
            raise SystemExit("--pool-sweep runs on one GPU")
        return run_pool_sweep(args, w, bits, link_peak)
    slots = args.slots or w.pool_slots
    store_kw = {}
    if args.store_file:
        ensure_store(w, bits, args.store_file)
        store_kw = dict(store_path=args.store_file, store_flags=moe.MOE_STORE_DIRECT if args.store_direct else 0)
    ctx = workload.create_loaded(w, bits, max_batch=1, pool_slots=slots, policy=POLICIES[args.policy],
                                 aging_period=args.aging, **store_kw)
    try:
        drift = workload.Drift(w)
        n_ring = 256
        X = torch.from_numpy(np.stack([synth.tokens(w.seed, s, 1, H) for s in range(n_ring)])).cuda()
        y = torch.empty((1, H), device="cuda")
        st = torch.cuda.current_stream()
        stride = moe.moe_blob_stride(H, w.inter, bits)
        sblob = moe.moe_blob_bytes(H, w.shared_inter, bits) if w.shared_inter else 0
        step = 0
        at64 = None

        def one_step(bias=None):
            nonlocal step, at64
            if bias is not None:
                moe.moe_set_router_bias_all(ctx, bias, st)
            elif step > 0:
                drift.advance(ctx, st)
            moe.moe_forward_decode_stack(ctx, 0, L, X[step % n_ring], 1, y, 1e-6, None, None, None, st)
            step += 1
            if step == 64:
                at64 = moe.moe_pool_stats(ctx)

        for _ in range(args.warmup):
            one_step()
        # the drifted router biases of the timed steps, computed ahead like the token batches
        sched = drift.schedule(args.steps)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        s0 = moe.moe_pool_stats(ctx)
        l0 = moe.moe_launch_count(ctx)
        clk = ClockSampler(local)
        clk.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(st)
        for i in range(args.steps):
            one_step(sched[i])
        e1.record(st)
        torch.cuda.synchronize()
        clocks = clk.stop()
        launches = moe.moe_launch_count(ctx) - l0
        ms = e0.elapsed_time(e1)
        s1 = moe.moe_pool_stats(ctx)
        ms = max_over_ranks(ms, pg)
        secs = ms / 1e3
        value = args.steps * world / secs

        def rate(a, b):
            h, m = b["hits"] - (a["hits"] if a else 0), b["misses"] - (a["misses"] if a else 0)
            return h / max(1, h + m)

        h2d = s1["h2d_bytes"] - s0["h2d_bytes"]
        h2d_ms = s1["h2d_ms"] - s0["h2d_ms"]
        expert_bytes = L * (k * stride + sblob)  # batch 1: k distinct routed experts + the shared one per layer
        peak, peak_kind = peaks()
        gbs = expert_bytes * args.steps / secs / 1e9
        e2e = None
        if not args.no_e2e:
            xh = torch.from_numpy(np.stack([synth.tokens(w.seed, s, 1, H) for s in range(n_ring)])).pin_memory()
            yh = torch.empty((1, H)).pin_memory()
            xd = torch.empty((1, H), device="cuda")
            n_e2e = min(args.steps, 64)
            sched_e2e = drift.schedule(n_e2e)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i in range(n_e2e):
                xd.copy_(xh[(step + i) % n_ring], non_blocking=True)
                moe.moe_set_router_bias_all(ctx, sched_e2e[i], st)
                moe.moe_forward_decode_stack(ctx, 0, L, xd, 1, y, 1e-6, None, None, None, st)
                yh.copy_(y, non_blocking=True)
                st.synchronize()
            step += n_e2e
            e2e_s = time.perf_counter() - t0
            e2e = {"value": n_e2e * world / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": H * 4,
                   "d2h_bytes_per_step": H * 4, "steps": n_e2e}
        line = {
            "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": (f"stress: {L}-layer 80B-shaped decode stack, int{bits} group-64, batch 1, "
                                    f"{slots} of {w.n_experts} slots per layer in HBM ({args.policy} eviction), "
                                    + (f"routed blobs in the expert container {args.store_file} (one "
                                       f"{'O_DIRECT ' if args.store_direct else ''}pread per miss into pinned "
                                       "staging), " if args.store_file else "full store in pinned host memory, ")
                                    + f"Zipf(1.1) routing with {w.drift_swaps} adjacent-rank swaps per "
                                    "layer per step (biases of the timed steps computed before timing and sent with "
                                    "one moe_set_router_bias_all per step), one persistent launch per step: a missed "
                                    "expert's rows are read by the kernel from host memory and written into its new "
                                    "slot, pool starts cold"),
                       "batch": 1, "layers": L, "bits": bits, "pool_slots": slots, "policy": args.policy,
                       "parallelism": "replicas" if world > 1 else "single-gpu",
                       "l2": "inputs larger than L2: each step reads its experts from the HBM pool or the host"},
            "pool": {"hit_rate_all": rate(None, s1), "hit_rate_after_step64": rate(at64, s1) if at64 else None,
                     "hit_rate_timed": rate(s0, s1), "misses_timed": s1["misses"] - s0["misses"],
                     "h2d_bytes_timed": h2d, "h2d_bytes_per_step": h2d / args.steps,
                     "h2d_copy_engine_ms_timed": h2d_ms,  # 0 when the kernel reads the misses itself
                     "host_link_gbs_wall": h2d / secs / 1e9, "host_link_probe_gbs": link_peak},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "peak_kind": peak_kind, "traffic": None,
                         "kernel": "streaming decode stack (one persistent launch per step; the host runs the "
                                   "pool on each published routing)",
                         "bytes_per_launch": expert_bytes},
            "gpu_launches": int(launches),
            "clocks": clocks,
            "e2e": e2e,
        }
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, bits, args.cpu_samples)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        moe.moe_destroy(ctx)
        if pg:
            pg.destroy_process_group()


def ensure_store(w, bits, path):
    """Write the workload's expert container at `path` unless one with its shape is there."""
    import int4_expert_streaming_gb300 as moe
    from int4_expert_streaming_gb300 import workload
    want = dict(n_layers=w.n_layers, n_experts=w.n_experts, hidden=w.hidden, inter=w.inter, bits=bits,
                stride=moe.moe_blob_stride(w.hidden, w.inter, bits))
    try:
        if moe.moe_store_info(path) == want:
            return
    except moe.MoeError:
        pass
    workload.write_store(w, path, bits=bits)


def run_pool_sweep(args, w, bits, link_peak):
    """Hit rate and throughput of the streaming stack against pool size and
    eviction policy.  One context reserves the largest size; before each point
    moe_pool_reset empties every layer's pool and switches size and policy, and
    the same token batches and the same drifting router biases replay from
    step 0.  Each point runs `warmup` untimed steps from the cold pool, then
    `steps` timed steps, and prints one JSON line."""
    import torch

    import int4_expert_streaming_gb300 as moe
    from int4_expert_streaming_gb300 import workload

    sizes = [int(v) for v in args.sweep_slots.split(",")]
    pols = args.sweep_policies.split(",")
    L, H = w.n_layers, w.hidden
    ctx = workload.create_loaded(w, bits, max_batch=1, pool_slots=max(sizes))
    try:
        n = args.warmup + args.steps
        drift = workload.Drift(w)
        bias = np.concatenate([drift.biases()[None], drift.schedule(n - 1)])  # the bias of every step, from step 0
        n_ring = 256
        X = torch.from_numpy(np.stack([synth.tokens(w.seed, s, 1, H) for s in range(n_ring)])).cuda()
        y = torch.empty((1, H), device="cuda")
        st = torch.cuda.current_stream()
        for pol in pols:
            for S in sizes:
                moe.moe_pool_reset(ctx, S, POLICIES[pol], args.aging, st)

                def step(i):
                    moe.moe_set_router_bias_all(ctx, bias[i], st)
                    moe.moe_forward_decode_stack(ctx, 0, L, X[i % n_ring], 1, y, 1e-6, None, None, None, st)

                for i in range(args.warmup):
                    step(i)
                torch.cuda.synchronize()
                s0 = moe.moe_pool_stats(ctx)
                clk = ClockSampler(0)
                clk.start()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                for i in range(args.warmup, n):
                    step(i)
                e1.record(st)
                torch.cuda.synchronize()
                clocks = clk.stop()
                ms = e0.elapsed_time(e1)
                s1 = moe.moe_pool_stats(ctx)
                hits, misses = s1["hits"] - s0["hits"], s1["misses"] - s0["misses"]
                h2d = s1["h2d_bytes"] - s0["h2d_bytes"]
                print(json.dumps({
                    "sweep": "pool", "policy": pol, "slots": S, "n_experts": w.n_experts, "layers": L, "bits": bits,
                    "aging_period": args.aging if pol == "aged" else None, "warmup": args.warmup,
                    "steps": args.steps, "value": args.steps / (ms / 1e3), "unit": "tok/s",
                    "ms_per_step": ms / args.steps, "hit_rate_timed": hits / max(1, hits + misses),
                    "hit_rate_all": s1["hits"] / max(1, s1["hits"] + s1["misses"]),
                    "misses_per_step": misses / args.steps, "h2d_gb_per_step": h2d / args.steps / 1e9,
                    "host_link_gbs_wall": h2d / (ms / 1e3) / 1e9,
                    "h2d_copy_engine_ms": s1["h2d_ms"] - s0["h2d_ms"],
                    "host_link_probe_gbs": link_peak, "clocks": clocks}), flush=True)
    finally:
        moe.moe_destroy(ctx)


def main():
    args = parse_args()
    if not args.steps:
        args.steps = {"80b-prefill": 50, "stress": 1024}.get(args.config, 2048)
    if args.impl == "reference":
        run_reference(args)
    elif args.config == "80b-prefill":
        run_prefill(args)
    elif args.config == "stress":
        run_stress(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
