"""Benchmark of the int4 MoE layer path on B300.

Default workload: one MoE layer in decode at batch 1 (d=2048, E=256 experts,
top-8, I=512, int4 group-32 weights with fp16 scales, bf16 activations N(0,1),
fp32 router with an N(0,1) per-expert bias), a fresh seeded token every step.
A "step" is one token through the whole layer: router, top-k, grouping, the
eight expert FFNs and the combine into the residual.

Inputs larger than L2: the step cycles through 64 independently seeded copies
of the layer (29 GB of weights), so no step finds its weights in the 126 MB L2.
Timing: CUDA graph of 64 steps, replayed; CUDA events on the launching stream
around the timed replays, barrier + synchronize on both sides, max over ranks.

Other workloads (``--workload``): ``batch`` (T tokens per step, Zipf(1.1)
router skew), ``prefill`` (T=4096 chunk, Zipf skew), ``stack`` (49 layers +
RMSNorm + int4 LM head + argmax).  ``--impl reference`` times the fp64 CPU
oracle on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode tokens/s on 1 B300; achieved HBM GB/s vs ~8 TB/s roofline"
D, E, K_TOP, I_FF, V = 2048, 256, 8, 512, 131072
EXPERT_BYTES = 3 * I_FF * D * 9 // 16          # int4 + fp16 group scales of one expert (gate, up, down)
ROUTER_BYTES = E * D * 4 + E * 4               # fp32 router weight + bias
LM_BYTES = V * D * 9 // 16


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=256)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="decode", choices=["decode", "batch", "prefill", "stack"])
    p.add_argument("--T", type=int, default=None, help="tokens per step (batch / prefill / stack)")
    p.add_argument("--copies", type=int, default=64, help="independent layer copies cycled per step")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    return p.parse_args()


# ---------------------------------------------------------------- helpers


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        m = json.load(open(path))
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), float(m.get("bf16_tflops_sustained", 0)), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- device weights


def make_device_layers(n_layers, seed, bias, device="cuda"):
    """n independently seeded layers, drawn on the device and packed."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth
    layers = []
    qbuf = torch.empty(E * I_FF * D // 2, dtype=torch.uint8, device=device)
    sbuf = torch.empty(E * I_FF * D // 32, dtype=torch.float16, device=device)
    for l in range(n_layers):
        banks = {}
        for name, (rows, K) in {"gate": (I_FF, D), "up": (I_FF, D), "down": (D, I_FF)}.items():
            kq = synth.stream_key(seed, synth.TAG[name + "_q"], l)
            ks = synth.stream_key(seed, synth.TAG[name + "_s"], l)
            synth.device_fill_int4(qbuf.data_ptr(), qbuf.numel(), kq)
            synth.device_fill_scales(sbuf.data_ptr(), sbuf.numel(), ks)
            banks[name] = bm.bitmoe_pack_int4(qbuf.view(E, rows, K // 2), sbuf.view(E, rows, K // 32))
        wr = torch.from_numpy(synth.router_weight(seed, E, D, l)).to(device)
        br = torch.from_numpy(synth.router_bias(seed, E, bias, l)).to(device)
        layers.append(bm.MoeLayer(d=D, E=E, k=K_TOP, I=I_FF, gate=banks["gate"], up=banks["up"],
                                  down=banks["down"], w_router=wr, b_router=br))
    torch.cuda.synchronize()
    return layers


# ---------------------------------------------------------------- CPU oracle leg


def cpu_oracle_sample(workload, T, seconds, seed=0):
    """Time the fp64 oracle on a bounded sample of the workload; returns dict."""
    import oracle
    import synth
    bias = "normal" if workload == "decode" else "zipf"
    tensors = synth.moe_layer(seed, D, E, I_FF, bias=bias, layer=0)
    cores = oracle.num_threads()
    done, t0, step = 0, time.perf_counter(), 0
    # decode: one token per call (batch 1, as the workload), until the time budget is spent
    per_call = 1 if workload == "decode" else max(1, min(T or 1, 64))
    while time.perf_counter() - t0 < seconds:
        x = synth.activations(seed, per_call, D, step=step)
        oracle.moe_forward(x, tensors, K_TOP)
        done += per_call
        step += 1
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} tokens in {step} calls of T={per_call} on layer copy 0 ({el:.1f} s, fp64, "
                      f"OpenMP over the {per_call * K_TOP} routed rows of each call)"}


# ---------------------------------------------------------------- our decode workload


def bench_decode(args, world, rank):
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth

    T = 1 if args.workload == "decode" else (args.T or 8)
    bias = "normal" if args.workload == "decode" else "zipf"
    G = args.copies
    layers = make_device_layers(G, seed=1 + rank, bias=bias)
    ws = bm.moe_workspace(layers[0], T)
    stream = torch.cuda.current_stream()

    # fresh token(s) per step: a pool of distinct steps, cycled in chunks of G
    n_pool = max(G, min(args.steps + args.warmup, 4096))
    n_pool = (n_pool // G) * G
    xs_host = np.stack([synth.activations(rank, T, D, step=s) for s in range(n_pool)])  # [P, T, D] bf16 bits
    xs = torch.from_numpy(xs_host.view(np.int16)).view(torch.bfloat16).cuda()
    x_slots = torch.empty((G, T, D), dtype=torch.bfloat16, device="cuda")
    out_slots = torch.empty((G, T, D), dtype=torch.bfloat16, device="cuda")
    ids_slots = torch.empty((G, T, K_TOP), dtype=torch.int32, device="cuda")

    def run_chunk():
        for g in range(G):
            bm.moe_forward(x_slots[g], layers[g], ws, out=out_slots[g], ids_out=ids_slots[g])

    # warm the kernels (first launches set shared-memory attributes) then capture
    x_slots.copy_(xs[:G])
    run_chunk()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_chunk()
    torch.cuda.synchronize()
    n_kernels = count_graph_kernels(graph)
    launches_per_step = n_kernels / G if n_kernels else (1 if T <= 4 else 6)

    n_chunks_w = max(1, math.ceil(args.warmup / G))
    n_chunks = max(1, math.ceil(args.steps / G))
    steps = n_chunks * G

    def timed(nc, start_chunk=0):
        for c in range(nc):
            base = ((start_chunk + c) * G) % n_pool
            x_slots.copy_(xs[base:base + G], non_blocking=True)
            graph.replay()

    timed(n_chunks_w)
    torch.cuda.synchronize()
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        timed(n_chunks, n_chunks_w)
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world)

    # bytes actually touched per step: unique experts of each step + router + activations
    ids_all = ids_slots.cpu().numpy()
    uniq = float(np.mean([len(np.unique(ids_all[g])) for g in range(G)]))
    step_bytes = uniq * EXPERT_BYTES + ROUTER_BYTES + 2 * T * D * 2

    # e2e through the public call with host buffers: pinned x in, pinned out back, every chunk
    e2e = bench_decode_e2e(args, graph, x_slots, out_slots, xs_host, G, T, world)

    tokens = steps * T * world
    value = tokens / (ms / 1e3)
    per_step_us = ms * 1e3 / steps
    hbm, _, _, which = peaks()
    achieved = step_bytes / (per_step_us * 1e-6) / 1e9
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": n_chunks_w * G, "ms_per_step": per_step_us / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4xbf16->fp32", "data": "synthetic (seeded; weights drawn on device)",
        "config": {"workload": f"moe_layer_decode_T{T}" if T > 1 else "moe_layer_decode_batch1", "T": T, "d": D,
                   "E": E, "top_k": K_TOP, "I": I_FF, "group": 32,
                   "router_bias": bias, "layer_copies": G,
                   "l2": f"inputs larger than L2: {G} independently seeded layer copies "
                         f"({G * (E * EXPERT_BYTES + ROUTER_BYTES) / 1e9:.1f} GB) cycled per step",
                   "parallelism": f"replicas x{world}", "timing": "CUDA graph of 64 steps, events on stream"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None,
                     "kernel": "whole layer step", "bytes_per_step": int(step_bytes),
                     "unique_experts_per_step": uniq, "peak_source": which},
        "gpu_launches": int(round(launches_per_step * steps)),
        "e2e": e2e,
        "clocks": clk.summary(),
    }
    return res


def count_graph_kernels(graph):
    """Kernel nodes in a captured torch CUDA graph (0 if it cannot be read)."""
    try:
        from cuda.bindings import runtime as cudart
        g = cudart.cudaGraph_t(init_value=int(graph.raw_cuda_graph()))
        err, _, n = cudart.cudaGraphGetNodes(g, 0)
        err, nodes, n = cudart.cudaGraphGetNodes(g, n)
        cnt = 0
        for nd in nodes[:n]:
            err, t = cudart.cudaGraphNodeGetType(nd)
            if t == cudart.cudaGraphNodeType.cudaGraphNodeTypeKernel:
                cnt += 1
        return cnt
    except Exception:
        return 0


def bench_decode_e2e(args, graph, x_slots, out_slots, xs_host, G, T, world):
    import torch
    stream = torch.cuda.current_stream()
    n_chunks = max(1, min(math.ceil(args.steps / G), 64))
    hx = torch.from_numpy(xs_host[:G].view(np.int16)).view(torch.bfloat16).pin_memory()
    hout = torch.empty((G, T, D), dtype=torch.bfloat16).pin_memory()
    for _ in range(2):
        x_slots.copy_(hx, non_blocking=True)
        graph.replay()
        hout.copy_(out_slots, non_blocking=True)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(n_chunks):
        x_slots.copy_(hx, non_blocking=True)
        graph.replay()
        hout.copy_(out_slots, non_blocking=True)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    steps = n_chunks * G
    return {"value": round(steps * T * world / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 2,
            "how": f"per {G}-step chunk: pinned host x -> device, graph replay of moe_forward, out -> pinned host"}


# ---------------------------------------------------------------- prefill workload


def bench_prefill(args, world, rank):
    """T-token prefill chunk through one MoE layer (Zipf routing skew)."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth

    T = args.T or 4096
    G = min(args.copies, 4)
    layers = make_device_layers(G, seed=1 + rank, bias="zipf")
    xs = [torch.from_numpy(synth.activations(rank, T, D, step=s).view(np.int16)).view(torch.bfloat16).cuda()
          for s in range(G)]
    ws = bm.moe_workspace(layers[0], T)
    out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    steps = max(1, args.steps)
    warm = max(3, args.warmup)
    for s in range(warm):
        bm.moe_forward(xs[s % G], layers[s % G], ws, out=out)
    torch.cuda.synchronize()
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        for s in range(steps):
            bm.moe_forward(xs[s % G], layers[s % G], ws, out=out)
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1), world) / steps

    # the grouped GEMMs alone (expert FFN call on routed, grouped rows), same inputs
    ffn_ms, rows_used, active = [], [], []
    for s in range(G):
        ids, w = bm.moe_route(xs[s], layers[s], ws)
        off, rows, inv = bm.moe_permute(ids, layers[s], ws)
        for _ in range(2):
            bm.moe_expert_ffn_int4(xs[s], layers[s], off, rows, ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        reps = 5
        for _ in range(reps):
            bm.moe_expert_ffn_int4(xs[s], layers[s], off, rows, ws)
        e1.record(stream)
        torch.cuda.synchronize()
        ffn_ms.append(e0.elapsed_time(e1) / reps)
        cnt = np.diff(off.cpu().numpy())
        rows_used.append(int(cnt.sum()))
        active.append(int((cnt > 0).sum()))
    flops = 6.0 * T * K_TOP * D * I_FF
    gemm_ms = float(np.median(ffn_ms))
    _, bf16_peak, bf16_sus, which = peaks()
    achieved = flops / (gemm_ms * 1e-3) / 1e12
    tokens = steps * T * world
    return {
        "metric": "MoE-layer prefill tokens/s on 1 B300; grouped-GEMM TFLOP/s vs dense 16-bit tensor peak",
        "value": round(tokens / (ms * steps / 1e3), 1), "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4->f16 x f16 -> f32", "data": "synthetic (seeded; weights drawn on device)",
        "config": {"workload": f"moe_layer_prefill_T{T}", "T": T, "d": D, "E": E, "top_k": K_TOP, "I": I_FF,
                   "router_bias": "zipf(1.1)", "layer_copies": G,
                   "l2": f"inputs larger than L2: {G} layer copies of {E * EXPERT_BYTES / 1e6:.0f} MB cycled",
                   "active_experts_mean": float(np.mean(active)), "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": round(achieved / bf16_peak, 4), "traffic": None,
                     "kernel": "expert FFN grouped GEMMs (x->fp16, gate/up+SwiGLU, down)",
                     "flops_per_launch": flops, "ms_per_launch": gemm_ms, "peak_source": which + " burst bf16 (fp16 same rate)"},
        "gpu_launches": None,
        "clocks": clk.summary(),
    }


# ---------------------------------------------------------------- main


def main():
    args = parse()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        T = 1 if args.workload == "decode" else (args.T or 8)
        per_step_budget = max(1.0, 150.0 / max(1, args.steps + args.warmup))
        t0 = time.perf_counter()
        cb = cpu_oracle_sample(args.workload, T, min(per_step_budget * args.steps, args.cpu_seconds * 4))
        el = time.perf_counter() - t0
        res = {"metric": METRIC, "impl": "reference", "value": round(cb["value"], 3), "unit": "tokens/s",
               "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
               "config": {"workload": "moe_layer_decode_batch1" if T == 1 else f"moe_layer_decode_T{T}",
                          "T": T, "d": D, "E": E, "top_k": K_TOP, "I": I_FF},
               "ms_per_step": 1e3 / cb["value"] * T,
               "cpu_baseline": cb,
               "e2e": {"value": round(cb["value"], 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0},
               "wall_s": round(el, 1)}
        print(json.dumps(res))
        return

    import torch
    world, rank, local = dist_setup(args)
    if args.workload in ("decode", "batch"):
        res = bench_decode(args, world, rank)
    elif args.workload == "prefill":
        res = bench_prefill(args, world, rank)
    else:
        raise SystemExit(f"workload {args.workload} not wired yet")
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_oracle_sample(args.workload, res["config"]["T"], args.cpu_seconds)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
