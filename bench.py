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
K_SHARED = 6                                   # routed experts per token beside the shared expert


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=256)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="decode", choices=["decode", "batch", "prefill", "stack", "shared"],
                   help="shared: batch-1 decode with the pages' routing, top-6 of 256 plus one shared expert")
    p.add_argument("--T", type=int, default=None, help="tokens per step (batch / prefill / stack)")
    p.add_argument("--copies", type=int, default=64, help="independent layer copies cycled per step")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    return p.parse_args()


# ---------------------------------------------------------------- helpers


# Kernels whose DRAM traffic per launch is recorded under profiles/, with the
# sources that define them: a recorded figure counts only while the hash of
# those sources still matches the one written beside it.
KERNEL_SOURCES = {
    "decode_layer_kernel": ["decode.cu", "common.cuh"],
    "prefill_gemm_kernel": ["prefill.cu", "common.cuh"],
    "lmhead_kernel": ["lmhead.cu", "common.cuh"],
}


def kernel_source_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "bit_expert_ffn_warp_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, units=1.0):
    """DRAM bytes (read + write) per launch from the ncu summary of `kernel`, scaled by
    `units` (launch size / captured size), or None when absent or stale."""
    import glob
    want = kernel_source_hash(kernel)
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", f"{kernel}*.md"))):
        vals = {}
        for line in open(path):
            if line.startswith("- ") and " = " in line:
                k, v = line[2:].split(" = ", 1)
                vals[k.strip()] = v.strip().strip("`")
        if vals.get("source_sha256") == want and "dram_bytes_per_launch" in vals:
            return int(float(vals["dram_bytes_per_launch"]) * units)
    return None


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


def _reduce(v, world, op):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(v, world):
    import torch.distributed as dist
    return _reduce(v, world, dist.ReduceOp.MAX) if world > 1 else v


def sum_over_ranks(v, world):
    import torch.distributed as dist
    return _reduce(v, world, dist.ReduceOp.SUM) if world > 1 else v


def job_throughput(units, ms, world):
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return sum_over_ranks(units, world) / (max_over_ranks(ms, world) / 1e3)


# ---------------------------------------------------------------- device weights


def make_device_layers(n_layers, seed, bias, device="cuda", k=K_TOP, n_shared=0):
    """n independently seeded layers, drawn on the device and packed (with
    n_shared = 1 the banks hold E + 1 experts, the last one shared)."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth
    layers = []
    Et = E + n_shared
    qbuf = torch.empty(Et * I_FF * D // 2, dtype=torch.uint8, device=device)
    sbuf = torch.empty(Et * I_FF * D // 32, dtype=torch.float16, device=device)
    for l in range(n_layers):
        banks = {}
        for name, (rows, K) in {"gate": (I_FF, D), "up": (I_FF, D), "down": (D, I_FF)}.items():
            kq = synth.stream_key(seed, synth.TAG[name + "_q"], l)
            ks = synth.stream_key(seed, synth.TAG[name + "_s"], l)
            synth.device_fill_int4(qbuf.data_ptr(), qbuf.numel(), kq)
            synth.device_fill_scales(sbuf.data_ptr(), sbuf.numel(), ks)
            banks[name] = bm.bitmoe_pack_int4(qbuf.view(Et, rows, K // 2), sbuf.view(Et, rows, K // 32))
        wr = torch.from_numpy(synth.router_weight(seed, E, D, l)).to(device)
        br = torch.from_numpy(synth.router_bias(seed, E, bias, l)).to(device)
        layers.append(bm.MoeLayer(d=D, E=E, k=k, I=I_FF, gate=banks["gate"], up=banks["up"],
                                  down=banks["down"], w_router=wr, b_router=br, n_shared=n_shared))
    torch.cuda.synchronize()
    return layers


# ---------------------------------------------------------------- CPU oracle leg


def cpu_oracle_sample(workload, T, seconds, seed=0):
    """Time the fp64 oracle on a bounded sample of the workload; returns dict."""
    import oracle
    import synth
    one = workload in ("decode", "shared")
    bias = "normal" if one else "zipf"
    shared = workload == "shared"
    k = K_SHARED if shared else K_TOP
    tensors = (synth.moe_layer_shared if shared else synth.moe_layer)(seed, D, E, I_FF, bias=bias, layer=0)
    cores = oracle.num_threads()
    done, t0, step = 0, time.perf_counter(), 0
    # decode: one token per call (batch 1, as the workload), until the time budget is spent
    per_call = 1 if one else max(1, min(T or 1, 64))
    while time.perf_counter() - t0 < seconds:
        x = synth.activations(seed, per_call, D, step=step)
        oracle.moe_forward(x, tensors, k, n_shared=int(shared))
        done += per_call
        step += 1
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} tokens in {step} calls of T={per_call} on layer copy 0 ({el:.1f} s, fp64, "
                      f"OpenMP over the {per_call * (k + int(shared))} rows of each call)"}


# ---------------------------------------------------------------- our decode workload


def bench_decode(args, world, rank):
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth

    shared = args.workload == "shared"
    T = 1 if args.workload in ("decode", "shared") else (args.T or 8)
    bias = "normal" if args.workload in ("decode", "shared") else "zipf"
    G = args.copies
    k = K_SHARED if shared else K_TOP
    layers = make_device_layers(G, seed=1 + rank, bias=bias, k=k, n_shared=int(shared))
    ws = bm.moe_workspace(layers[0], T)
    stream = torch.cuda.current_stream()

    # fresh token(s) per step: a pool of distinct steps, cycled in chunks of G
    n_pool = max(G, min(args.steps + args.warmup, 4096))
    n_pool = (n_pool // G) * G
    xs_host = np.stack([synth.activations(rank, T, D, step=s) for s in range(n_pool)])  # [P, T, D] bf16 bits
    xs = torch.from_numpy(xs_host.view(np.int16)).view(torch.bfloat16).cuda()
    x_slots = torch.empty((G, T, D), dtype=torch.bfloat16, device="cuda")
    out_slots = torch.empty((G, T, D), dtype=torch.bfloat16, device="cuda")
    ids_slots = torch.empty((G, T, layers[0].kt), dtype=torch.int32, device="cuda")

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
    launches_per_step = count_kernels(lambda: bm.moe_forward(x_slots[0], layers[0], ws, out=out_slots[0],
                                                             ids_out=ids_slots[0]))

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
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms_local, world)

    # bytes actually touched per step: unique experts of each step + router + activations
    ids_all = ids_slots.cpu().numpy()
    uniq = float(np.mean([len(np.unique(ids_all[g])) for g in range(G)]))
    step_bytes = uniq * EXPERT_BYTES + ROUTER_BYTES + 2 * T * D * 2

    # e2e through the public call with host buffers: pinned x in, pinned out back, every chunk
    e2e = bench_decode_e2e(args, graph, x_slots, out_slots, xs_host, G, T, world)

    value = job_throughput(steps * T, ms_local, world)
    per_step_us = ms * 1e3 / steps
    hbm, _, _, which = peaks()
    achieved = step_bytes / (per_step_us * 1e-6) / 1e9
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": n_chunks_w * G, "ms_per_step": per_step_us / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4xbf16->fp32", "data": "synthetic (seeded; weights drawn on device)",
        "config": {"workload": ("moe_layer_shared_decode_batch1" if shared else
                                f"moe_layer_decode_T{T}" if T > 1 else "moe_layer_decode_batch1"), "T": T, "d": D,
                   "E": E, "top_k": k, "n_shared": int(shared), "I": I_FF, "group": 32,
                   "router_bias": bias, "layer_copies": G,
                   "l2": f"inputs larger than L2: {G} independently seeded layer copies "
                         f"({G * ((E + int(shared)) * EXPERT_BYTES + ROUTER_BYTES) / 1e9:.1f} GB) cycled per step",
                   "parallelism": f"replicas x{world}", "timing": "CUDA graph of 64 steps, events on stream"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": profiled_traffic("decode_layer_kernel") if T == 1 and not shared else None,
                     "kernel": "decode_layer_kernel (the whole layer step, one launch)" if T <= 4
                     else "whole layer step", "bytes_per_step": int(step_bytes),
                     "unique_experts_per_step": uniq, "peak_source": which},
        "gpu_launches": launches_per_step * steps if launches_per_step else None,
        "e2e": e2e,
        "clocks": clk.summary(),
    }
    return res


def count_kernels(fn):
    """Kernel launches one call of fn() makes: fn is captured once into a CUDA graph
    that is kept un-instantiated and whose kernel nodes are counted (0 if unreadable)."""
    import torch
    try:
        from cuda.bindings import runtime as cudart
        g = torch.cuda.CUDAGraph(keep_graph=True)
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        cg = cudart.cudaGraph_t(init_value=int(g.raw_cuda_graph()))
        err, _, n = cudart.cudaGraphGetNodes(cg, 0)
        err, nodes, n = cudart.cudaGraphGetNodes(cg, n)
        cnt = 0
        for nd in nodes[:n]:
            err, t = cudart.cudaGraphNodeGetType(nd)
            if t == cudart.cudaGraphNodeType.cudaGraphNodeTypeKernel:
                cnt += 1
        del g
        return cnt
    except Exception as exc:  # report, do not guess
        print(f"bench: kernel count unavailable ({exc!r})", file=sys.stderr)
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
    steps = n_chunks * G
    value = job_throughput(steps * T, ev0.elapsed_time(ev1), world)
    return {"value": round(value, 1), "unit": "tokens/s",
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
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms_local, world) / steps

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
    launches_per_step = count_kernels(lambda: bm.moe_forward(xs[0], layers[0], ws, out=out))

    # end to end through the public call: pinned host tokens in, the layer output back, every step
    x_pin = [torch.from_numpy(synth.activations(rank, T, D, step=s).view(np.int16)).view(torch.bfloat16).pin_memory()
             for s in range(G)]
    out_pin = torch.empty((T, D), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    e_steps = max(1, min(steps, 20))
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s_ in range(e_steps):
        x_dev.copy_(x_pin[s_ % G], non_blocking=True)
        bm.moe_forward(x_dev, layers[s_ % G], ws, out=out)
        out_pin.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e = {"value": round(job_throughput(e_steps * T, e0.elapsed_time(e1), world), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 2,
           "how": "per step: pinned host tokens -> device, moe_forward, layer output -> pinned host"}
    return {
        "metric": "MoE-layer prefill tokens/s on 1 B300; grouped-GEMM TFLOP/s vs dense 16-bit tensor peak",
        "value": round(job_throughput(steps * T, ms_local, world), 1), "unit": "tokens/s", "n_gpus": world,
        "steps": steps,
        "warmup": warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4->f16 x f16 -> f32", "data": "synthetic (seeded; weights drawn on device)",
        "config": {"workload": f"moe_layer_prefill_T{T}", "T": T, "d": D, "E": E, "top_k": K_TOP, "I": I_FF,
                   "router_bias": "zipf(1.1)", "layer_copies": G,
                   "l2": f"inputs larger than L2: {G} layer copies of {E * EXPERT_BYTES / 1e6:.0f} MB cycled",
                   "active_experts_mean": float(np.mean(active)), "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": round(achieved / bf16_peak, 4),
                     "traffic": profiled_traffic("prefill_gemm_kernel") if T == 4096 else None,
                     "kernel": "expert FFN grouped GEMMs (x->fp16, gate/up+SwiGLU, down)",
                     "flops_per_launch": flops, "ms_per_launch": gemm_ms, "peak_source": which + " burst bf16 (fp16 same rate)"},
        "gpu_launches": launches_per_step * steps if launches_per_step else None,
        "e2e": e2e,
        "clocks": clk.summary(),
    }


# ---------------------------------------------------------------- 49-layer stack + LM head


N_LAYERS = 49


def make_device_lm_head(seed, device="cuda"):
    """The int4 LM head [V, D] drawn on the device and packed."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth
    q = torch.empty(V * D // 2, dtype=torch.uint8, device=device)
    sc = torch.empty(V * D // 32, dtype=torch.float16, device=device)
    synth.device_fill_int4(q.data_ptr(), q.numel(), synth.stream_key(seed, synth.TAG["lm_q"], 0))
    synth.device_fill_scales(sc.data_ptr(), sc.numel(), synth.stream_key(seed, synth.TAG["lm_s"], 0))
    packed = bm.bitmoe_pack_int4(q.view(V, D // 2), sc.view(V, D // 32))
    torch.cuda.synchronize()
    return packed


def bench_stack(args, world, rank):
    """One decode step = T tokens through 49 MoE layers (RMSNorm before each, residual
    kept in bf16, attention replaced by identity), then RMSNorm, the int4 LM head and
    the arg-max."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth

    T = args.T or 1
    layers = make_device_layers(N_LAYERS, seed=1 + rank, bias="normal")
    lm = make_device_lm_head(seed=1 + rank)
    ws = bm.moe_workspace(layers[0], T)
    lm_ws = bm.lmhead_workspace(T, D, V)
    stream = torch.cuda.current_stream()

    n_pool = max(8, min(args.steps + args.warmup, 1024))
    xs_host = np.stack([synth.activations(rank, T, D, step=s) for s in range(n_pool)])
    xs = torch.from_numpy(xs_host.view(np.int16)).view(torch.bfloat16).cuda()
    x_slot = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    resid = torch.empty_like(x_slot)
    xh = torch.empty_like(x_slot)
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    ids = torch.empty((N_LAYERS, T, K_TOP), dtype=torch.int32, device="cuda")

    def step():
        resid.copy_(x_slot)
        for l in range(N_LAYERS):  # RMSNorm inside the layer step, residual updated in place
            bm.moe_forward_prenorm(resid, layers[l], ws, out=resid, ids_out=ids[l])
        bm.bitmoe_rmsnorm(resid, out=xh)
        bm.lmhead_int4_gemv(xh, lm, V, lm_ws, want_logits=False, argmax=am)

    x_slot.copy_(xs[0])
    step()
    torch.cuda.synchronize()
    launches_per_step = count_kernels(step)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()

    def run(n, first):
        for i in range(n):
            x_slot.copy_(xs[(first + i) % n_pool], non_blocking=True)
            graph.replay()

    warm = max(3, args.warmup)
    steps = max(1, args.steps)
    run(warm, 0)
    torch.cuda.synchronize()
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        run(steps, warm)
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms_local, world) / steps

    # bytes touched per step: the unique experts of every layer (last step), routers, LM head
    ids_np = ids.cpu().numpy()
    uniq = [len(np.unique(ids_np[l])) for l in range(N_LAYERS)]
    step_bytes = sum(u * EXPERT_BYTES + ROUTER_BYTES for u in uniq) + LM_BYTES + 2 * T * D * 2 * (N_LAYERS + 1)
    hbm, _, _, which = peaks()
    achieved = step_bytes / (ms * 1e-3) / 1e9

    # end to end through the public calls: pinned host tokens in, arg-max back, every step
    x_pin = torch.from_numpy(xs_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    am_pin = torch.empty(T, dtype=torch.int32).pin_memory()
    e_steps = min(steps, 256)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e_steps):
        x_slot.copy_(x_pin[i % n_pool], non_blocking=True)
        graph.replay()
        am_pin.copy_(am, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e_value = job_throughput(e_steps * T, e0.elapsed_time(e1), world)

    return {
        "metric": "49-layer MoE stack + int4 LM head decode tokens/s on 1 B300; achieved HBM GB/s",
        "value": round(job_throughput(steps * T, ms_local, world), 1), "unit": "tokens/s", "n_gpus": world,
        "steps": steps,
        "warmup": warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4xbf16->fp32", "data": "synthetic (seeded; weights drawn on device)",
        "config": {"workload": f"moe_stack49_lmhead_T{T}", "T": T, "layers": N_LAYERS, "d": D, "E": E,
                   "top_k": K_TOP, "I": I_FF, "V": V, "router_bias": "normal",
                   "l2": f"inputs larger than L2: {N_LAYERS} layers ({N_LAYERS * (E * EXPERT_BYTES + ROUTER_BYTES) / 1e9:.1f}"
                         f" GB) + LM head {LM_BYTES / 1e6:.0f} MB per step",
                   "parallelism": f"replicas x{world}", "timing": "CUDA graph of one step, events on stream"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None,
                     "kernel": "whole stack step (49 x pre-norm decode layer, RMSNorm, LM head)",
                     "bytes_per_step": int(step_bytes), "unique_experts_per_layer_mean": float(np.mean(uniq)),
                     "peak_source": which},
        "gpu_launches": launches_per_step * steps if launches_per_step else None,
        "e2e": {"value": round(e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": T * D * 2,
                "d2h_bytes_per_step": T * 4,
                "how": "per step: pinned host tokens -> device, graph replay, arg-max -> pinned host"},
        "clocks": clk.summary(),
    }


def cpu_stack_sample(T, seconds, seed=0):
    """Oracle time of one stack step, from a bounded sample: whole layers (RMSNorm, route,
    touched experts, combine) on layer copy 0 and one LM-head pass over a row sample."""
    import oracle
    import synth
    tensors = synth.moe_layer(seed, D, E, I_FF, bias="normal", layer=0)
    cores = oracle.num_threads()
    t0 = time.perf_counter()
    n_layers = 0
    resid = synth.activations(seed, T, D)
    while time.perf_counter() - t0 < seconds * 0.8 or n_layers == 0:
        xh = oracle.f64_to_bf16(oracle.rmsnorm(resid))
        res = oracle.moe_forward(xh, tensors, K_TOP, resid=resid)
        resid = oracle.f64_to_bf16(res["out"])
        n_layers += 1
    t_layer = (time.perf_counter() - t0) / n_layers
    rows = 8192
    q, sc = synth.lm_head(seed, rows, D)
    t1 = time.perf_counter()
    oracle.lmhead(oracle.f64_to_bf16(oracle.rmsnorm(resid)), q, sc, want_logits=False)
    t_lm = (time.perf_counter() - t1) * (V / rows)
    t_step = N_LAYERS * t_layer + t_lm
    return {"value": T / t_step, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_layers} layer passes of T={T} ({t_layer * 1e3:.1f} ms each) x {N_LAYERS} layers + LM head "
                      f"on {rows} of {V} rows scaled to {V} ({t_lm * 1e3:.1f} ms); fp64, OpenMP"}


# ---------------------------------------------------------------- main


def main():
    args = parse()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        if args.workload == "decode":
            T, name, metric = 1, "moe_layer_decode_batch1", METRIC
        elif args.workload == "shared":
            T, name, metric = 1, "moe_layer_shared_decode_batch1", METRIC
        elif args.workload == "batch":
            T = args.T or 8
            name, metric = f"moe_layer_decode_T{T}", METRIC
        elif args.workload == "prefill":
            T = args.T or 4096
            name = f"moe_layer_prefill_T{T}"
            metric = "MoE-layer prefill tokens/s on 1 B300; grouped-GEMM TFLOP/s vs dense 16-bit tensor peak"
        else:
            T = args.T or 1
            name = f"moe_stack49_lmhead_T{T}"
            metric = "49-layer MoE stack + int4 LM head decode tokens/s on 1 B300; achieved HBM GB/s"
        # each timed step is a bounded sample of the workload; the whole run stays within minutes
        budget = min(max(1.0, 150.0 / max(1, args.steps + args.warmup)) * args.steps, args.cpu_seconds * 4)
        t0 = time.perf_counter()
        if args.workload == "stack":
            cb = cpu_stack_sample(T, budget)
        else:
            cb = cpu_oracle_sample(args.workload, T, budget)
        el = time.perf_counter() - t0
        res = {"metric": metric, "impl": "reference", "value": round(cb["value"], 3), "unit": "tokens/s",
               "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
               "config": {"workload": name, "T": T, "d": D, "E": E,
                          "top_k": K_SHARED if args.workload == "shared" else K_TOP,
                          "n_shared": int(args.workload == "shared"), "I": I_FF},
               "ms_per_step": 1e3 / cb["value"] * T,
               "cpu_baseline": cb,
               "e2e": {"value": round(cb["value"], 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0},
               "wall_s": round(el, 1)}
        print(json.dumps(res))
        return

    import torch
    world, rank, local = dist_setup(args)
    if args.workload in ("decode", "batch", "shared"):
        res = bench_decode(args, world, rank)
    elif args.workload == "prefill":
        res = bench_prefill(args, world, rank)
    else:
        res = bench_stack(args, world, rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            if args.workload == "stack":
                res["cpu_baseline"] = cpu_stack_sample(res["config"]["T"], args.cpu_seconds)
            else:
                res["cpu_baseline"] = cpu_oracle_sample(args.workload, res["config"]["T"], args.cpu_seconds)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
