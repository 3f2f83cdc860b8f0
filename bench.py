"""Benchmark of the int4 MoE layer path on B300.

Default workload: one MoE layer in decode at batch 1 (d=2048, E=256 experts,
top-8, I=512, int4 group-32 weights with fp16 scales, bf16 activations N(0,1),
fp32 router with an N(0,1) per-expert bias), a fresh seeded token every step.
A "step" is one token through the whole layer: router, top-k, grouping, the
eight expert FFNs and the combine into the residual.

Inputs larger than L2: the steps cycle through 64 independently seeded copies
of the layer (29 GB of weights), so no step finds its weights in the 126 MB L2.

Timing.  W warm-up steps, then a timed region of exactly K steps (``--steps``),
captured as CUDA graphs.  Short regions say little on their own, so the region
is repeated back to back until at least 0.4 s of GPU time has been timed; each
repetition is bracketed by CUDA events on the launching stream and the median
repetition is reported (``timing`` in the JSON line gives the count and the
spread).  Successive repetitions replay graphs that start at different layer
copies, so a repetition never finds the previous one's weights in L2.  A barrier
and a device synchronisation bracket the whole timed part; the clock sampler runs
from before the warm-up to after the last repetition.

Other workloads (``--workload``): ``batch`` (T tokens per step, Zipf(1.1)
router skew), ``prefill`` (T=4096 chunk, Zipf skew), ``stack`` (49 layers +
RMSNorm + int4 LM head + argmax), ``shared`` (the pages' routing: top-6 of 256
plus one shared expert), ``lmhead`` (the int4 LM head alone, V = 131072).
``attn`` (one token through one attention layer beside the MoE layer: int4
q|k|v and output projections, grouped-query attention of 32 query / 4 key-value
heads of 128 over a bf16 cache of ``--ctx`` positions, whole context or a
``--window``, with sinks).
``decoder`` (one token through 49 decoder layers -- pre-norm attention at ``--ctx``
positions, 35 window layers with rotary and 14 whole-context ones, then the pre-norm
MoE block -- and RMSNorm, the int4 LM head and the arg-max).
``--format nvfp4`` runs the decode, batch, prefill and LM-head workloads with
NVFP4 weights (E2M1 codes, an E4M3 scale per 16 weights, an fp32 scale per
matrix; the same 4.5 bits per weight).  ``--impl reference`` times the fp64 CPU
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
PREFILL_METRIC = "MoE-layer prefill tokens/s on 1 B300; grouped-GEMM TFLOP/s vs dense 16-bit tensor peak"
STACK_METRIC = "49-layer MoE stack + int4 LM head decode tokens/s on 1 B300; achieved HBM GB/s"
LMHEAD_METRIC = "int4 LM-head GEMV + argmax tokens/s on 1 B300; achieved HBM GB/s"
ATTN_METRIC = "attention-layer decode tokens/s on 1 B300 (GQA 32/4 x 128, int4 projections); achieved HBM GB/s"
DECODER_METRIC = "49-layer decoder (attention + MoE) + int4 LM head decode tokens/s on 1 B300; achieved HBM GB/s"
D, E, K_TOP, I_FF, V = 2048, 256, 8, 512, 131072
EXPERT_BYTES = 3 * I_FF * D * 9 // 16          # int4 + fp16 group scales of one expert (gate, up, down)
ROUTER_BYTES = E * D * 4 + E * 4               # fp32 router weight + bias
LM_BYTES = V * D * 9 // 16
K_SHARED = 6                                   # routed experts per token beside the shared expert
NQ, NKV, HD = 32, 4, 128                       # attention heads: query, key/value, head size
WQKV_BYTES = (NQ + 2 * NKV) * HD * D * 9 // 16  # int4 + fp16 group scales of the stacked q|k|v projection
WO_BYTES = D * NQ * HD * 9 // 16
MIN_TIMED_S = 0.4                              # GPU time the repeated timed region adds up to, at least
DEFAULT_STEPS = {"decode": 2000, "shared": 2000, "batch": 500, "prefill": 20, "stack": 50, "lmhead": 500,
                 "attn": 500, "decoder": 30}
DEFAULT_WARMUP = {"decode": 200, "shared": 200, "batch": 50, "prefill": 5, "stack": 5, "lmhead": 50, "attn": 50,
                  "decoder": 3}


def parse():
    global MIN_TIMED_S
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None, help="steps in one timed region (per-workload default)")
    p.add_argument("--warmup", type=int, default=None, help="untimed warm-up steps (per-workload default, >= 3)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="decode",
                   choices=["decode", "batch", "prefill", "stack", "shared", "lmhead", "attn", "decoder"],
                   help="shared: batch-1 decode with the pages' routing, top-6 of 256 plus one shared expert")
    p.add_argument("--T", type=int, default=None, help="tokens per step (batch / prefill / stack / lmhead)")
    p.add_argument("--format", default="int4", choices=["int4", "nvfp4"],
                   help="weight format of the experts and the LM head (not the stack)")
    p.add_argument("--copies", type=int, default=64, help="independent layer copies cycled per step")
    p.add_argument("--ctx", type=int, default=None,
                   help="attn / decoder: context length, the token attends at ctx - 1 (32768 / 4096)")
    p.add_argument("--window", type=int, default=0, help="attn: sliding window (0 = whole context; 513 with rotary)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--min-timed-s", type=float, default=MIN_TIMED_S,
                   help="GPU time the repeated timed region adds up to, at least (short profiling runs)")
    a = p.parse_args()
    if a.steps is None:
        a.steps = DEFAULT_STEPS[a.workload]
    if a.warmup is None:
        a.warmup = DEFAULT_WARMUP[a.workload]
    a.steps = max(1, a.steps)
    a.warmup = max(3, a.warmup)
    MIN_TIMED_S = max(0.0, a.min_timed_s)
    if a.ctx is None:
        a.ctx = 4096 if a.workload == "decoder" else 32768
    if a.format == "nvfp4" and a.workload in ("stack", "shared", "attn", "decoder"):
        p.error("--format nvfp4 covers the decode, batch, prefill and lmhead workloads")
    return a


def fmt_suffix(fmt):
    return "_nvfp4" if fmt == "nvfp4" else ""


# ---------------------------------------------------------------- helpers


# Kernels whose DRAM traffic per launch is recorded under profiles/, with the
# sources that define them: a recorded figure counts only while the hash of
# those sources still matches the one written beside it.
KERNEL_SOURCES = {
    "decode_layer_kernel": ["decode.cu", "common.cuh"],
    "prefill_wa_kernel": ["prefill.cu", "common.cuh"],
    "lmhead_kernel": ["lmhead.cu", "common.cuh"],
    "attn_split_kernel": ["attn.cu", "common.cuh"],
}


def kernel_source_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "bit_expert_ffn_warp_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, units=1.0, workload=None):
    """DRAM bytes (read + write) per launch from the ncu summary of `kernel` (for
    `workload`, when given), scaled by `units` (launch size / captured size), or
    None when absent or stale."""
    import glob
    want = kernel_source_hash(kernel)
    pat = f"{kernel}__{workload}.md" if workload else f"{kernel}*.md"
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", pat))):
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
    """nvidia-smi clock / throttle sampling, started before the warm-up and stopped
    after the last timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        """Median SM clock over the samples taken under load (power above the idle
        draw), the maximum clock, and every throttle reason seen."""
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[3]), [n for n, v in zip(names, f[5:9])
                                                                      if v.lower() == "active"]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        pw = [r[2] for r in rows]
        cut = min(pw) + 0.25 * (max(pw) - min(pw))
        busy = [r for r in rows if r[2] >= cut] or rows
        reasons = sorted({n for r in rows for n in r[3]})
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(busy),
                "power_w_max": max(pw)}


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


def capture(fn):
    """fn() captured into a CUDA graph (its launches only; nothing runs)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def region_graphs(step, K, n_graphs):
    """n_graphs CUDA graphs of exactly K steps each; graph j runs step(j*K + i) for
    i = 0..K-1, so successive regions continue the step sequence."""
    def body(j):
        def f():
            for i in range(K):
                step(j * K + i)
        return f
    return [capture(body(j)) for j in range(n_graphs)]


def run_warmup(step, W):
    """W untimed steps (eager launches)."""
    import torch
    for i in range(W):
        step(i)
    torch.cuda.synchronize()


def time_regions(graphs, world, min_total_s=None, min_regions=5, max_regions=20000):
    """Replays the K-step region graphs (cycling through them) back to back, each
    replay between two CUDA events on the current stream, until at least
    min_total_s of GPU time is timed.  Barrier + synchronize on both sides.
    Returns the per-region times (ms)."""
    import torch
    if min_total_s is None:
        min_total_s = MIN_TIMED_S
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    barrier(world)
    times, total, batch, j = [], 0.0, min_regions, 0
    while True:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(batch + 1)]
        evs[0].record(stream)
        for i in range(batch):
            graphs[j % len(graphs)].replay()
            j += 1
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        ts = [evs[i].elapsed_time(evs[i + 1]) for i in range(batch)]
        times += ts
        total += sum(ts)
        if total >= min_total_s * 1e3 or len(times) >= max_regions:
            break
        per = total / len(times)
        batch = int(min(max_regions - len(times), max(min_regions, math.ceil((min_total_s * 1e3 - total) / per))))
    barrier(world)
    return times


def timing_record(times, K, what):
    ts = sorted(times)
    return {"regions": len(ts), "steps_per_region": K, "stat": "median region",
            "region_ms": {"min": round(ts[0], 5), "median": round(statistics.median(ts), 5), "max": round(ts[-1], 5)},
            "timed_s": round(sum(ts) / 1e3, 3), "what": what}


def n_region_graphs(K, copies):
    """Enough K-step graphs that consecutive regions start at different layer copies
    and a copy comes back only after every other one was used (at most 16 graphs)."""
    return max(1, min(16, math.ceil(copies / K)))


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


# ---------------------------------------------------------------- device weights


def make_device_layers(n_layers, seed, bias, device="cuda", k=K_TOP, n_shared=0, fmt="int4"):
    """n independently seeded layers, drawn on the device and packed (with
    n_shared = 1 the banks hold E + 1 experts, the last one shared)."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth
    layers = []
    Et = E + n_shared
    qbuf = torch.empty(Et * I_FF * D // 2, dtype=torch.uint8, device=device)
    sbuf = torch.empty(Et * I_FF * D // 32, dtype=torch.float16, device=device)
    fbuf = torch.empty(Et * I_FF * D // 16, dtype=torch.uint8, device=device)
    for l in range(n_layers):
        banks, ts = {}, {}
        for name, (rows, K) in {"gate": (I_FF, D), "up": (I_FF, D), "down": (D, I_FF)}.items():
            if fmt == "nvfp4":  # same bits as synth.moe_layer_nvfp4(seed, ..., layer=l)
                synth.device_fill_int4(qbuf.data_ptr(), qbuf.numel(), synth.stream_key(seed, synth.TAG[name + "_fq"], l))
                synth.device_fill_e4m3(fbuf.data_ptr(), fbuf.numel(), synth.stream_key(seed, synth.TAG[name + "_fs"], l))
                banks[name] = bm.bitmoe_pack_nvfp4(qbuf.view(Et, rows, K // 2), fbuf.view(Et, rows, K // 16))
                ts[name] = torch.from_numpy(
                    synth.f32_tensor_scales(synth.stream_key(seed, synth.TAG[name + "_ts"], l), 0, Et)).to(device)
                continue
            kq = synth.stream_key(seed, synth.TAG[name + "_q"], l)
            ks = synth.stream_key(seed, synth.TAG[name + "_s"], l)
            synth.device_fill_int4(qbuf.data_ptr(), qbuf.numel(), kq)
            synth.device_fill_scales(sbuf.data_ptr(), sbuf.numel(), ks)
            banks[name] = bm.bitmoe_pack_int4(qbuf.view(Et, rows, K // 2), sbuf.view(Et, rows, K // 32))
        wr = torch.from_numpy(synth.router_weight(seed, E, D, l)).to(device)
        br = torch.from_numpy(synth.router_bias(seed, E, bias, l)).to(device)
        layers.append(bm.MoeLayer(d=D, E=E, k=k, I=I_FF, gate=banks["gate"], up=banks["up"],
                                  down=banks["down"], w_router=wr, b_router=br, n_shared=n_shared,
                                  gate_ts=ts.get("gate"), up_ts=ts.get("up"), down_ts=ts.get("down")))
    torch.cuda.synchronize()
    return layers


def make_device_lm_head(seed, device="cuda", fmt="int4"):
    """The int4 LM head [V, D] drawn on the device and packed (NVFP4: the packed
    bank and its tensor scale, the bits of synth.lm_head_nvfp4)."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth
    if fmt == "nvfp4":
        q = torch.empty(V * D // 2, dtype=torch.uint8, device=device)
        sc = torch.empty(V * D // 16, dtype=torch.uint8, device=device)
        synth.device_fill_int4(q.data_ptr(), q.numel(), synth.stream_key(seed, synth.TAG["lm_fq"], 0))
        synth.device_fill_e4m3(sc.data_ptr(), sc.numel(), synth.stream_key(seed, synth.TAG["lm_fs"], 0))
        packed = bm.bitmoe_pack_nvfp4(q.view(V, D // 2), sc.view(V, D // 16))
        ts = float(synth.f32_tensor_scales(synth.stream_key(seed, synth.TAG["lm_ts"], 0), 0, 1)[0])
        torch.cuda.synchronize()
        return packed, ts
    q = torch.empty(V * D // 2, dtype=torch.uint8, device=device)
    sc = torch.empty(V * D // 32, dtype=torch.float16, device=device)
    synth.device_fill_int4(q.data_ptr(), q.numel(), synth.stream_key(seed, synth.TAG["lm_q"], 0))
    synth.device_fill_scales(sc.data_ptr(), sc.numel(), synth.stream_key(seed, synth.TAG["lm_s"], 0))
    packed = bm.bitmoe_pack_int4(q.view(V, D // 2), sc.view(V, D // 32))
    torch.cuda.synchronize()
    return packed


def token_pool(rank, n, T):
    """n distinct seeded token batches [n, T, D] as bf16 bit patterns (host)."""
    import synth
    return np.stack([synth.activations(rank, T, D, step=s) for s in range(n)])


def to_bf16(host_bits, pin=False, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(host_bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.to(device)


# ---------------------------------------------------------------- CPU oracle leg


def cpu_oracle_sample(workload, T, seconds, seed=0, fmt="int4"):
    """Time the fp64 oracle on a bounded sample of the workload; returns dict."""
    import oracle
    import synth
    one = workload in ("decode", "shared")
    bias = "normal" if one else "zipf"
    shared = workload == "shared"
    k = K_SHARED if shared else K_TOP
    if fmt == "nvfp4":
        tensors = synth.moe_layer_nvfp4(seed, D, E, I_FF, bias=bias, layer=0)
    else:
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


def cpu_lmhead_sample(T, seconds, seed=0, fmt="int4"):
    """Oracle LM head on a row sample of the V = 131072 bank, scaled to all rows."""
    import oracle
    import synth
    cores = oracle.num_threads()
    h = synth.activations(seed, T, D)
    rows, el, n = 4096, 0.0, 0
    if fmt == "nvfp4":
        q, s, ts = synth.lm_head_nvfp4(seed, rows, D)
        run = lambda: oracle.lmhead_nvfp4(h, q, s, ts, want_logits=False)  # noqa: E731
    else:
        q, s = synth.lm_head(seed, rows, D)
        run = lambda: oracle.lmhead(h, q, s, want_logits=False)  # noqa: E731
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or n == 0:
        run()
        n += 1
    el = time.perf_counter() - t0
    per_call = el / n * (V / rows)
    return {"value": T / per_call, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} passes of T={T} over {rows} of {V} rows ({el:.1f} s), scaled to {V} rows; fp64, OpenMP"}


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


# ---------------------------------------------------------------- decode workloads


def bench_decode(args, world, rank):
    import torch

    import bit_expert_ffn_warp_b300 as bm

    shared = args.workload == "shared"
    T = 1 if args.workload in ("decode", "shared") else (args.T or 8)
    bias = "normal" if args.workload in ("decode", "shared") else "zipf"
    G = args.copies
    k = K_SHARED if shared else K_TOP
    K, W = args.steps, args.warmup
    layers = make_device_layers(G, seed=1 + rank, bias=bias, k=k, n_shared=int(shared), fmt=args.format)
    ws = bm.moe_workspace(layers[0], T)
    kt = layers[0].kt

    ng = n_region_graphs(K, G)
    n_pool = min(max(K * ng, W, G), 4096)
    xs_host = token_pool(rank, n_pool, T)                      # [P, T, D] bf16 bits
    xs = to_bf16(xs_host)
    out_slots = torch.empty((G, T, D), dtype=torch.bfloat16, device="cuda")
    ids_slots = torch.zeros((G, T, kt), dtype=torch.int32, device="cuda")

    def step(s):
        g = s % G
        bm.moe_forward(xs[s % n_pool], layers[g], ws, out=out_slots[g], ids_out=ids_slots[g])

    with ClockSampler(torch.cuda.current_device()) as clk:
        run_warmup(step, W)
        graphs = region_graphs(step, K, ng)
        times = time_regions(graphs, world)
    ms_local = statistics.median(times)
    launches_per_step = count_kernels(lambda: step(0))

    # bytes actually touched per step: unique experts of each step + router + activations
    ids_all = ids_slots.cpu().numpy()
    uniq = float(np.mean([len(np.unique(ids_all[g])) for g in range(G)]))
    step_bytes = uniq * EXPERT_BYTES + ROUTER_BYTES + 2 * T * D * 2

    e2e = bench_decode_e2e(args, layers, ws, xs_host, T, world, K, ng)

    value = job_throughput(K * T, ms_local, world)
    per_step_us = max_over_ranks(ms_local, world) * 1e3 / K
    hbm, _, _, which = peaks()
    achieved = step_bytes / (per_step_us * 1e-6) / 1e9
    name = ("moe_layer_shared_decode_batch1" if shared else
            f"moe_layer_decode_T{T}" if T > 1 else "moe_layer_decode_batch1") + fmt_suffix(args.format)
    fused = T <= 8
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": per_step_us / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4xbf16->fp32" if args.format == "nvfp4" else "int4xbf16->fp32",
        "data": "synthetic (seeded; weights drawn on device)",
        "config": {"workload": name, "T": T, "d": D, "E": E, "top_k": k, "n_shared": int(shared), "I": I_FF,
                   "format": args.format, "group": 16 if args.format == "nvfp4" else 32, "router_bias": bias,
                   "layer_copies": G,
                   "l2": f"inputs larger than L2: {G} independently seeded layer copies "
                         f"({G * ((E + int(shared)) * EXPERT_BYTES + ROUTER_BYTES) / 1e9:.1f} GB) cycled step by step",
                   "parallelism": f"replicas x{world}"},
        "timing": timing_record(times, K, f"CUDA graphs of {K} moe_forward steps, {ng} graph(s) in rotation"),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": profiled_traffic("decode_layer_kernel", workload=name) if fused else None,
                     "kernel": "decode_layer_kernel (the whole layer step, one launch)" if fused
                     else "whole layer step", "bytes_per_step": int(step_bytes),
                     "unique_experts_per_step": uniq, "peak_source": which + " (copy, burst)"},
        "gpu_launches": launches_per_step * K if launches_per_step else None,
        "e2e": e2e,
        "clocks": clk.summary(),
    }


def bench_decode_e2e(args, layers, ws, xs_host, T, world, K, ng):
    """The same steps through moe_forward with host buffers: every step copies its
    token(s) from pinned host memory to the device and its output back."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    G = len(layers)
    n_pool = xs_host.shape[0]
    hx = to_bf16(xs_host, pin=True)
    hout = torch.empty((n_pool, T, D), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty((G, T, D), dtype=torch.bfloat16, device="cuda")
    od = torch.empty((G, T, D), dtype=torch.bfloat16, device="cuda")

    def step(s):
        g = s % G
        xd[g].copy_(hx[s % n_pool], non_blocking=True)
        bm.moe_forward(xd[g], layers[g], ws, out=od[g])
        hout[s % n_pool].copy_(od[g], non_blocking=True)

    run_warmup(step, 3)
    times = time_regions(region_graphs(step, K, ng), world)
    return {"value": round(job_throughput(K * T, statistics.median(times), world), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 2,
            "how": "every step: pinned host token(s) -> device, moe_forward, layer output -> pinned host "
                   "(graph-captured copies); median of repeated K-step regions",
            "regions": len(times)}


# ---------------------------------------------------------------- prefill workload


def bench_prefill(args, world, rank):
    """T-token prefill chunk through one MoE layer (Zipf routing skew)."""
    import torch

    import bit_expert_ffn_warp_b300 as bm

    T = args.T or 4096
    G = min(args.copies, 4)
    K, W = args.steps, args.warmup
    layers = make_device_layers(G, seed=1 + rank, bias="zipf", fmt=args.format)
    xs_host = token_pool(rank, G, T)
    xs = to_bf16(xs_host)
    ws = bm.moe_workspace(layers[0], T)
    out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")

    def step(s):
        bm.moe_forward(xs[s % G], layers[s % G], ws, out=out)

    # the grouped GEMMs alone: the expert-FFN call on routed, grouped rows, same inputs
    groups = []
    for s in range(G):
        ids, w = bm.moe_route(xs[s], layers[s], ws)
        off, rows, inv = bm.moe_permute(ids, layers[s], ws)
        groups.append((off, rows))
    torch.cuda.synchronize()
    y_rows = torch.empty((T * K_TOP, D), dtype=torch.float32, device="cuda")

    def ffn_step(s):
        off, rows = groups[s % G]
        (bm.moe_expert_ffn_nvfp4 if args.format == "nvfp4" else bm.moe_expert_ffn_int4)(
            xs[s % G], layers[s % G], off, rows, ws, y_out=y_rows)

    with ClockSampler(torch.cuda.current_device()) as clk:
        run_warmup(step, W)
        times = time_regions(region_graphs(step, K, 1), world)
        run_warmup(ffn_step, 3)
        ffn_times = time_regions(region_graphs(ffn_step, K, 1), world)
    ms_local = statistics.median(times)
    ms = max_over_ranks(ms_local, world) / K
    gemm_ms = max_over_ranks(statistics.median(ffn_times), world) / K
    cnt = [np.diff(g[0].cpu().numpy()) for g in groups]
    flops = 6.0 * T * K_TOP * D * I_FF
    _, bf16_peak, bf16_sus, which = peaks()
    achieved = flops / (gemm_ms * 1e-3) / 1e12
    launches_per_step = count_kernels(lambda: step(0))

    # end to end through the public call: pinned host tokens in, the layer output back, every step
    x_pin = to_bf16(xs_host, pin=True)
    out_pin = torch.empty((T, D), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")

    def e2e_step(s):
        x_dev.copy_(x_pin[s % G], non_blocking=True)
        bm.moe_forward(x_dev, layers[s % G], ws, out=out)
        out_pin.copy_(out, non_blocking=True)

    run_warmup(e2e_step, 3)
    e_times = time_regions(region_graphs(e2e_step, K, 1), world)
    e2e = {"value": round(job_throughput(K * T, statistics.median(e_times), world), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 2,
           "how": "every step: pinned host tokens -> device, moe_forward, layer output -> pinned host",
           "regions": len(e_times)}
    return {
        "metric": PREFILL_METRIC,
        "value": round(job_throughput(K * T, ms_local, world), 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("nvfp4" if args.format == "nvfp4" else "int4") + "->f16 x f16 -> f32",
        "data": "synthetic (seeded; weights drawn on device)",
        "config": {"workload": f"moe_layer_prefill_T{T}" + fmt_suffix(args.format), "T": T, "d": D, "E": E,
                   "top_k": K_TOP, "I": I_FF, "format": args.format, "router_bias": "zipf(1.1)", "layer_copies": G,
                   "l2": f"inputs larger than L2: {G} layer copies of {E * EXPERT_BYTES / 1e6:.0f} MB cycled",
                   "active_experts_mean": float(np.mean([(c > 0).sum() for c in cnt])),
                   "parallelism": f"replicas x{world}"},
        "timing": timing_record(times, K, f"CUDA graph of {K} moe_forward steps"),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": round(achieved / bf16_peak, 4),
                     "traffic": profiled_traffic("prefill_wa_kernel",
                                                 workload=f"moe_layer_prefill_T{T}" + fmt_suffix(args.format)),
                     "kernel": "expert FFN grouped GEMMs (gate/up+SwiGLU, down)",
                     "flops_per_launch": flops, "ms_per_launch": gemm_ms,
                     "launch_timing": timing_record(ffn_times, K, f"CUDA graph of {K} moe_expert_ffn_int4 calls"),
                     "peak_source": which + " burst bf16 (fp16 same rate)"},
        "gpu_launches": launches_per_step * K if launches_per_step else None,
        "e2e": e2e,
        "clocks": clk.summary(),
    }


# ---------------------------------------------------------------- 49-layer stack + LM head


N_LAYERS = 49


def bench_stack(args, world, rank):
    """One decode step = T tokens through 49 MoE layers (RMSNorm before each, residual
    kept in bf16, attention replaced by identity), then RMSNorm, the int4 LM head and
    the arg-max."""
    import torch

    import bit_expert_ffn_warp_b300 as bm

    T = args.T or 1
    K, W = args.steps, args.warmup
    layers = make_device_layers(N_LAYERS, seed=1 + rank, bias="normal")
    lm = make_device_lm_head(seed=1 + rank)
    ws = bm.moe_workspace(layers[0], T)
    lm_ws = bm.lmhead_workspace(T, D, V)

    n_pool = max(8, min(K + W, 1024))
    xs_host = token_pool(rank, n_pool, T)
    xs = to_bf16(xs_host)
    resid = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    xh = torch.empty_like(resid)
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    ids = torch.empty((N_LAYERS, T, K_TOP), dtype=torch.int32, device="cuda")

    def layer_steps():
        for l in range(N_LAYERS):  # RMSNorm inside the layer step, residual updated in place
            bm.moe_forward_prenorm(resid, layers[l], ws, out=resid, ids_out=ids[l])
        bm.bitmoe_rmsnorm(resid, out=xh)
        bm.lmhead_int4_gemv(xh, lm, V, lm_ws, want_logits=False, argmax=am)

    # the whole step in one launch where the fused decode kernel covers T
    fused = T <= 8
    ws_stack = bm.moe_stack_workspace(layers[0], T) if fused else None

    def one_launch():
        bm.moe_stack_decode(resid, layers, ws_stack, lm_w=lm, V=V, argmax=am, ids_out=ids)

    layers_and_head = one_launch if fused else layer_steps

    def step(s):
        resid.copy_(xs[s % n_pool])
        layers_and_head()

    def step_layers(s):
        resid.copy_(xs[s % n_pool])
        layer_steps()

    with ClockSampler(torch.cuda.current_device()) as clk:
        run_warmup(step, W)
        times = time_regions(region_graphs(step, K, 1), world)
    ms_local = statistics.median(times)
    ms = max_over_ranks(ms_local, world) / K
    launches_per_step = count_kernels(layers_and_head)
    compare = None
    if fused:  # the same step as 49 layer launches + RMSNorm + LM head, for comparison
        run_warmup(step_layers, 3)
        lt = time_regions(region_graphs(step_layers, K, 1), world, min_total_s=0.2)
        compare = {"ms_per_step": round(max_over_ranks(statistics.median(lt), world) / K, 5),
                   "launches_per_step": count_kernels(layer_steps), "regions": len(lt)}

    # bytes touched per step: the unique experts of every layer (last step), routers, LM head
    ids_np = ids.cpu().numpy()
    uniq = [len(np.unique(ids_np[l])) for l in range(N_LAYERS)]
    step_bytes = sum(u * EXPERT_BYTES + ROUTER_BYTES for u in uniq) + LM_BYTES + 2 * T * D * 2 * (N_LAYERS + 1)
    hbm, _, _, which = peaks()
    achieved = step_bytes / (ms * 1e-3) / 1e9

    # end to end through the public calls: pinned host tokens in, arg-max back, every step
    x_pin = to_bf16(xs_host, pin=True)
    am_pin = torch.empty((n_pool, T), dtype=torch.int32).pin_memory()

    def e2e_step(s):
        resid.copy_(x_pin[s % n_pool], non_blocking=True)
        layers_and_head()
        am_pin[s % n_pool].copy_(am, non_blocking=True)

    run_warmup(e2e_step, 3)
    e_times = time_regions(region_graphs(e2e_step, K, 1), world)
    e_value = job_throughput(K * T, statistics.median(e_times), world)

    return {
        "metric": STACK_METRIC,
        "value": round(job_throughput(K * T, ms_local, world), 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4xbf16->fp32", "data": "synthetic (seeded; weights drawn on device)",
        "config": {"workload": f"moe_stack49_lmhead_T{T}", "T": T, "layers": N_LAYERS, "d": D, "E": E,
                   "top_k": K_TOP, "I": I_FF, "V": V, "router_bias": "normal",
                   "l2": f"inputs larger than L2: {N_LAYERS} layers ({N_LAYERS * (E * EXPERT_BYTES + ROUTER_BYTES) / 1e9:.1f}"
                         f" GB) + LM head {LM_BYTES / 1e6:.0f} MB per step",
                   "parallelism": f"replicas x{world}"},
        "timing": timing_record(times, K, f"CUDA graph of {K} stack steps"),
        "per_layer_launches": compare,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None,
                     "kernel": ("decode_stack_kernel (49 pre-norm layers, RMSNorm, LM head: one launch)" if fused
                                else "whole stack step (49 x pre-norm decode layer, RMSNorm, LM head)"),
                     "bytes_per_step": int(step_bytes), "unique_experts_per_layer_mean": float(np.mean(uniq)),
                     "peak_source": which + " (copy, burst)"},
        "gpu_launches": launches_per_step * K if launches_per_step else None,
        "e2e": {"value": round(e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": T * D * 2,
                "d2h_bytes_per_step": T * 4,
                "how": "every step: pinned host tokens -> device, the stack, arg-max -> pinned host",
                "regions": len(e_times)},
        "clocks": clk.summary(),
    }


# ---------------------------------------------------------------- LM head alone


def bench_lmhead(args, world, rank):
    """T tokens through the int4 LM head (V = 131072, 151 MB) and its arg-max."""
    import torch

    import bit_expert_ffn_warp_b300 as bm

    T = args.T or 1
    K, W = args.steps, args.warmup
    n_heads = 4   # 604 MB of LM-head copies cycled: each call streams its 151 MB from HBM
    fp4 = args.format == "nvfp4"
    heads = [make_device_lm_head(seed=1 + rank + 1000 * c, fmt=args.format) for c in range(n_heads)]

    def lm_call(c, x):
        if fp4:
            bm.lmhead_nvfp4_gemv(x, heads[c][0], heads[c][1], V, lm_ws, want_logits=False, argmax=am[c])
        else:
            bm.lmhead_int4_gemv(x, heads[c], V, lm_ws, want_logits=False, argmax=am[c])
    lm_ws = bm.lmhead_workspace(T, D, V)
    n_pool = 256
    xs_host = token_pool(rank, n_pool, T)
    xs = to_bf16(xs_host)
    am = torch.empty((n_heads, T), dtype=torch.int32, device="cuda")

    def step(s):
        lm_call(s % n_heads, xs[s % n_pool])

    with ClockSampler(torch.cuda.current_device()) as clk:
        run_warmup(step, W)
        times = time_regions(region_graphs(step, K, 1), world)
    ms_local = statistics.median(times)
    ms = max_over_ranks(ms_local, world) / K
    launches_per_step = count_kernels(lambda: step(0))
    call_bytes = LM_BYTES + T * D * 2 + T * 4
    hbm, _, _, which = peaks()
    achieved = call_bytes / (ms * 1e-3) / 1e9

    x_pin = to_bf16(xs_host, pin=True)
    am_pin = torch.empty((n_pool, T), dtype=torch.int32).pin_memory()
    xd = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")

    def e2e_step(s):
        c = s % n_heads
        xd.copy_(x_pin[s % n_pool], non_blocking=True)
        lm_call(c, xd)
        am_pin[s % n_pool].copy_(am[c], non_blocking=True)

    run_warmup(e2e_step, 3)
    e_times = time_regions(region_graphs(e2e_step, K, 1), world)
    name = f"lmhead_V{V}_T{T}" + fmt_suffix(args.format)
    return {
        "metric": LMHEAD_METRIC,
        "value": round(job_throughput(K * T, ms_local, world), 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4xbf16->fp32" if fp4 else "int4xbf16->fp32",
        "data": "synthetic (seeded; weights drawn on device)",
        "config": {"workload": name, "T": T, "d": D, "V": V, "format": args.format, "group": 16 if fp4 else 32,
                   "lm_head_copies": n_heads,
                   "l2": f"inputs larger than L2: {n_heads} LM-head copies ({n_heads * LM_BYTES / 1e6:.0f} MB) cycled",
                   "parallelism": f"replicas x{world}"},
        "timing": timing_record(times, K, f"CUDA graph of {K} lmhead_int4_gemv calls"),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": profiled_traffic("lmhead_kernel", workload=name),
                     "kernel": "lmhead_kernel (+ key clear and arg-max finalise)", "bytes_per_step": call_bytes,
                     "peak_source": which + " (copy, burst)"},
        "gpu_launches": launches_per_step * K if launches_per_step else None,
        "e2e": {"value": round(job_throughput(K * T, statistics.median(e_times), world), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * 4,
                "how": "every step: pinned host tokens -> device, lmhead_int4_gemv, arg-max -> pinned host",
                "regions": len(e_times)},
        "clocks": clk.summary(),
    }


# ---------------------------------------------------------------- attention layer


def attn_name(ctx, window):
    return f"attn_decode_ctx{ctx}_" + (f"swa{window}" if window else "full")


def attn_keys(ctx, window):
    return min(ctx, window) if window else ctx


def attn_step_bytes(ctx, window):
    """Bytes one step must move: both projections' int4 banks, the attended keys and
    values, the new cache rows, and x, the residual and the output."""
    return WQKV_BYTES + WO_BYTES + attn_keys(ctx, window) * NKV * HD * 2 * 2 + NKV * HD * 2 * 2 + 3 * D * 2


def bench_attn(args, world, rank):
    """One token through one attention layer at position ctx - 1 (the cache holds ctx rows)."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth

    ctx, window = args.ctx, args.window
    if ctx < 1:
        raise SystemExit("--ctx must be >= 1")
    K, W = args.steps, args.warmup
    rope = window > 0   # rotary encoding on the sliding-window layers, none on the whole-context ones
    step_bytes = attn_step_bytes(ctx, window)
    G = max(1, min(args.copies, math.ceil(3 * 126e6 / step_bytes)))   # copies cycled: 3x L2 of inputs
    layers, kcs, vcs = [], [], []
    gen = torch.Generator(device="cuda")
    for c in range(G):
        t = synth.attn_layer(1 + rank + 1000 * c, D, NQ, NKV)
        layers.append(bm.AttnLayer.from_canonical(t, D, NQ, NKV, window=window, rope=rope))
        gen.manual_seed(7 + rank + 1000 * c)
        kcs.append(torch.randn((NKV, ctx, HD), generator=gen, device="cuda").to(torch.bfloat16))
        vcs.append(torch.randn((NKV, ctx, HD), generator=gen, device="cuda").to(torch.bfloat16))
    ws = bm.attn_workspace(layers[0], ctx)
    pos = ctx - 1
    n_pool = 256
    xs_host = token_pool(rank, n_pool, 2)   # [P, 2, D]: x and the residual of each step
    xs = to_bf16(xs_host)
    outs = torch.empty((G, D), dtype=torch.bfloat16, device="cuda")

    def step(s):
        g = s % G
        bm.attn_decode_step(xs[s % n_pool, 0], xs[s % n_pool, 1], pos, layers[g], kcs[g], vcs[g], ws, out=outs[g])

    ng = n_region_graphs(K, G)
    with ClockSampler(torch.cuda.current_device()) as clk:
        run_warmup(step, W)
        times = time_regions(region_graphs(step, K, ng), world)
    ms_local = statistics.median(times)
    per_step_us = max_over_ranks(ms_local, world) * 1e3 / K
    launches_per_step = count_kernels(lambda: step(0))
    hbm, _, _, which = peaks()
    achieved = step_bytes / (per_step_us * 1e-6) / 1e9

    x_pin = to_bf16(xs_host, pin=True)
    out_pin = torch.empty((n_pool, D), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty((G, 2, D), dtype=torch.bfloat16, device="cuda")

    def e2e_step(s):
        g = s % G
        xd[g].copy_(x_pin[s % n_pool], non_blocking=True)
        bm.attn_decode_step(xd[g, 0], xd[g, 1], pos, layers[g], kcs[g], vcs[g], ws, out=outs[g])
        out_pin[s % n_pool].copy_(outs[g], non_blocking=True)

    run_warmup(e2e_step, 3)
    e_times = time_regions(region_graphs(e2e_step, K, ng), world)
    name = attn_name(ctx, window)
    return {
        "metric": ATTN_METRIC,
        "value": round(job_throughput(K, ms_local, world), 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": per_step_us / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4xbf16->fp32; bf16 cache, fp32 softmax",
        "data": "synthetic (seeded; weights packed from host draws, caches N(0,1) drawn on device)",
        "config": {"workload": name, "T": 1, "d": D, "n_q_heads": NQ, "n_kv_heads": NKV, "head_dim": HD,
                   "ctx": ctx, "window": window, "rope": rope, "sinks": True, "keys_attended": attn_keys(ctx, window),
                   "layer_copies": G,
                   "l2": f"inputs larger than L2: {G} layer copies with their caches "
                         f"({G * (WQKV_BYTES + WO_BYTES + 2 * ctx * NKV * HD * 2) / 1e6:.0f} MB) cycled step by step",
                   "parallelism": f"replicas x{world}"},
        "timing": timing_record(times, K, f"CUDA graphs of {K} attn_decode_step calls, {ng} graph(s) in rotation"),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None,
                     "kernel": "whole attention step (q|k|v projection, split-KV attention, combine, "
                               "Wo projection + residual; 4 launches)", "bytes_per_step": step_bytes,
                     "split_kernel_dram_bytes": profiled_traffic("attn_split_kernel", workload=name),
                     "peak_source": which + " (copy, burst)"},
        "gpu_launches": launches_per_step * K if launches_per_step else None,
        "e2e": {"value": round(job_throughput(K, statistics.median(e_times), world), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * D * 2, "d2h_bytes_per_step": D * 2,
                "how": "every step: pinned host x and residual -> device, attn_decode_step, output -> pinned host",
                "regions": len(e_times)},
        "clocks": clk.summary(),
    }


def cpu_attn_sample(ctx, window, seconds, seed=0):
    """The oracle's attention step on one layer at the same context, repeated until the
    time budget is spent (the cache draw is outside the timed part)."""
    import oracle
    import synth
    from oracle import attention as A
    t = synth.attn_layer(seed, D, NQ, NKV)
    kc, vc = synth.kv_cache(seed + 1, ctx, NKV)
    cores = oracle.num_threads()
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds or n == 0:
        x = synth.activations(seed + 2, 1, D, step=n)[0]
        r = synth.activations(seed + 3, 1, D, step=n)[0]
        A.decode_step(x, r, ctx - 1, t, kc, vc, window=window, use_rope=window > 0)
        n += 1
    el = time.perf_counter() - t0
    return {"value": n / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} attention steps at position {ctx - 1} ({el:.1f} s, fp64 numpy; projections dequantised "
                      f"by the oracle's C routine)"}


# ---------------------------------------------------------------- decoder: attention + MoE per layer


def decoder_kinds(n_layers):
    """(window, rotary) of each layer: 14 of 49 attend over the whole context without
    rotary encoding (layers l with l % 7 in {3, 6}), the others over 513 tokens with it."""
    return [(0, False) if l % 7 in (3, 6) else (513, True) for l in range(n_layers)]


def make_device_attn(n_layers, seed, ctx, device="cuda"):
    """n attention layers (int4 banks drawn on the device, sinks N(0, 1)) and their
    head-major caches of ctx rows (N(0, 1) bf16)."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    import synth
    rows = (NQ + 2 * NKV) * HD
    out, gen = [], torch.Generator(device=device)
    for l, (window, rope) in enumerate(decoder_kinds(n_layers)):
        banks = {}
        for name, (r, K) in {"qkv": (rows, D), "wo": (D, NQ * HD)}.items():
            q = torch.empty(r * K // 2, dtype=torch.uint8, device=device)
            s = torch.empty(r * K // 32, dtype=torch.float16, device=device)
            synth.device_fill_int4(q.data_ptr(), q.numel(), synth.stream_key(seed, synth.TAG[name + "_q"], l))
            synth.device_fill_scales(s.data_ptr(), s.numel(), synth.stream_key(seed, synth.TAG[name + "_s"], l))
            banks[name] = bm.bitmoe_pack_int4(q.view(r, K // 2), s.view(r, K // 32))
        gen.manual_seed(seed * 1000 + l)
        sinks = torch.randn(NQ, generator=gen, device=device)
        kc = torch.randn((NKV, ctx, HD), generator=gen, device=device).to(torch.bfloat16)
        vc = torch.randn((NKV, ctx, HD), generator=gen, device=device).to(torch.bfloat16)
        out.append((bm.AttnLayer(D, NQ, NKV, banks["qkv"], banks["wo"], sinks, window=window, rope=rope), kc, vc))
    torch.cuda.synchronize()
    return out


def bench_decoder(args, world, rank):
    """One token through 49 decoder layers at position ctx - 1: per layer the pre-norm
    attention block then the pre-norm MoE block, the bf16 residual updated in place; then
    RMSNorm, the int4 LM head and the arg-max."""
    import torch

    import bit_expert_ffn_warp_b300 as bm

    ctx, K, W = args.ctx, args.steps, args.warmup
    if ctx < 1:
        raise SystemExit("--ctx must be >= 1")
    moe = make_device_layers(N_LAYERS, seed=1 + rank, bias="normal")
    attn = make_device_attn(N_LAYERS, 1 + rank, ctx)
    lm = make_device_lm_head(seed=1 + rank)
    mws = bm.moe_workspace(moe[0], 1)
    aws = bm.attn_workspace(attn[0][0], ctx)
    lm_ws = bm.lmhead_workspace(1, D, V)
    pos = ctx - 1
    n_pool = max(8, min(K + W, 1024))
    xs_host = token_pool(rank, n_pool, 1)
    xs = to_bf16(xs_host)
    resid = torch.empty((1, D), dtype=torch.bfloat16, device="cuda")
    xh = torch.empty_like(resid)
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    ids = torch.empty((N_LAYERS, 1, K_TOP), dtype=torch.int32, device="cuda")

    def layers_and_head():
        for l in range(N_LAYERS):
            lay, kc, vc = attn[l]
            bm.attn_decode_step_prenorm(resid[0], pos, lay, kc, vc, aws, out=resid[0])
            bm.moe_forward_prenorm(resid, moe[l], mws, out=resid, ids_out=ids[l])
        bm.bitmoe_rmsnorm(resid, out=xh)
        bm.lmhead_int4_gemv(xh, lm, V, lm_ws, want_logits=False, argmax=am)

    def step(s):
        resid.copy_(xs[s % n_pool])
        layers_and_head()

    with ClockSampler(torch.cuda.current_device()) as clk:
        run_warmup(step, W)
        times = time_regions(region_graphs(step, K, 1), world)
    ms_local = statistics.median(times)
    ms = max_over_ranks(ms_local, world) / K
    launches_per_step = count_kernels(layers_and_head)
    ids_np = ids.cpu().numpy()
    moe_bytes = sum(len(np.unique(ids_np[l])) * EXPERT_BYTES + ROUTER_BYTES + 2 * D * 2 for l in range(N_LAYERS))
    attn_bytes = sum(attn_step_bytes(ctx, w) for w, _ in decoder_kinds(N_LAYERS))
    step_bytes = moe_bytes + attn_bytes + LM_BYTES + D * 2 + 4
    hbm, _, _, which = peaks()
    achieved = step_bytes / (ms * 1e-3) / 1e9

    x_pin = to_bf16(xs_host, pin=True)
    am_pin = torch.empty((n_pool, 1), dtype=torch.int32).pin_memory()

    def e2e_step(s):
        resid.copy_(x_pin[s % n_pool], non_blocking=True)
        layers_and_head()
        am_pin[s % n_pool].copy_(am, non_blocking=True)

    run_warmup(e2e_step, 3)
    e_times = time_regions(region_graphs(e2e_step, K, 1), world)
    n_full = sum(1 for w, _ in decoder_kinds(N_LAYERS) if w == 0)
    return {
        "metric": DECODER_METRIC,
        "value": round(job_throughput(K, ms_local, world), 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4xbf16->fp32; bf16 cache, fp32 softmax",
        "data": "synthetic (seeded; weights drawn on device, caches N(0,1))",
        "config": {"workload": f"decoder49_lmhead_ctx{ctx}", "T": 1, "layers": N_LAYERS, "d": D, "E": E,
                   "top_k": K_TOP, "I": I_FF, "V": V, "n_q_heads": NQ, "n_kv_heads": NKV, "head_dim": HD,
                   "ctx": ctx, "whole_context_layers": n_full, "window_layers": N_LAYERS - n_full, "window": 513,
                   "l2": f"inputs larger than L2: {N_LAYERS} MoE layers ({N_LAYERS * E * EXPERT_BYTES / 1e9:.1f} GB), "
                         f"attention weights and caches, LM head {LM_BYTES / 1e6:.0f} MB per step",
                   "parallelism": f"replicas x{world}"},
        "timing": timing_record(times, K, f"CUDA graph of {K} decoder steps"),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None,
                     "kernel": "whole decoder step (49 x (attention block: 4 launches, MoE block: 1 launch), "
                               "RMSNorm, LM head)",
                     "bytes_per_step": int(step_bytes), "moe_bytes": int(moe_bytes), "attention_bytes": int(attn_bytes),
                     "peak_source": which + " (copy, burst)"},
        "gpu_launches": launches_per_step * K if launches_per_step else None,
        "e2e": {"value": round(job_throughput(K, statistics.median(e_times), world), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": D * 2, "d2h_bytes_per_step": 4,
                "how": "every step: pinned host token -> device, 49 decoder layers, LM head, arg-max -> pinned host",
                "regions": len(e_times)},
        "clocks": clk.summary(),
    }


def cpu_decoder_sample(ctx, seconds, seed=0):
    """Oracle time of one decoder step from a bounded sample: whole attention blocks (window
    and whole-context) and MoE blocks on one layer each, weighted by the layer counts, plus
    one LM-head pass over a row sample."""
    import oracle
    import synth
    from oracle import attention as A
    kinds = decoder_kinds(N_LAYERS)
    n_full = sum(1 for w, _ in kinds if w == 0)
    t = synth.attn_layer(seed, D, NQ, NKV)
    kc, vc = synth.kv_cache(seed + 1, ctx, NKV)
    tensors = synth.moe_layer(seed, D, E, I_FF, bias="normal", layer=0)
    cores = oracle.num_threads()
    resid = synth.activations(seed, 1, D)
    per = {}
    for name, (window, rope) in {"window": (513, True), "full": (0, False)}.items():
        t0, n = time.perf_counter(), 0
        while time.perf_counter() - t0 < seconds * 0.3 or n == 0:
            A.prenorm_step(resid[0], ctx - 1, t, kc, vc, window=window, use_rope=rope)
            n += 1
        per[name] = (time.perf_counter() - t0) / n
    t0, n = time.perf_counter(), 0
    while time.perf_counter() - t0 < seconds * 0.3 or n == 0:
        xh = oracle.f64_to_bf16(oracle.rmsnorm(resid))
        oracle.moe_forward(xh, tensors, K_TOP, resid=resid)
        n += 1
    t_moe = (time.perf_counter() - t0) / n
    rows = 8192
    q, sc = synth.lm_head(seed, rows, D)
    t1 = time.perf_counter()
    oracle.lmhead(oracle.f64_to_bf16(oracle.rmsnorm(resid)), q, sc, want_logits=False)
    t_lm = (time.perf_counter() - t1) * (V / rows)
    t_step = (N_LAYERS - n_full) * per["window"] + n_full * per["full"] + N_LAYERS * t_moe + t_lm
    return {"value": 1.0 / t_step, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"attention blocks at position {ctx - 1} ({per['window'] * 1e3:.0f} ms window, "
                      f"{per['full'] * 1e3:.0f} ms whole context), MoE block {t_moe * 1e3:.0f} ms, each on one layer, "
                      f"x {N_LAYERS - n_full} / {n_full} / {N_LAYERS} layers + LM head on {rows} of {V} rows scaled "
                      f"({t_lm * 1e3:.0f} ms); fp64"}


# ---------------------------------------------------------------- main


def reference_arm(args):
    """The fp64 oracle on the host cores, on this workload, a bounded sample per step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = args.workload
    if wl in ("decode", "shared"):
        T = 1
        name = "moe_layer_shared_decode_batch1" if wl == "shared" else "moe_layer_decode_batch1"
        metric = METRIC
    elif wl == "batch":
        T = args.T or 8
        name, metric = f"moe_layer_decode_T{T}", METRIC
    elif wl == "prefill":
        T = args.T or 4096
        name, metric = f"moe_layer_prefill_T{T}", PREFILL_METRIC
    elif wl == "lmhead":
        T = args.T or 1
        name, metric = f"lmhead_V{V}_T{T}", LMHEAD_METRIC
    elif wl == "attn":
        T = 1
        name, metric = attn_name(args.ctx, args.window), ATTN_METRIC
    elif wl == "decoder":
        T = 1
        name, metric = f"decoder49_lmhead_ctx{args.ctx}", DECODER_METRIC
    else:
        T = args.T or 1
        name, metric = f"moe_stack49_lmhead_T{T}", STACK_METRIC
    # each timed step is a bounded sample of the workload; the whole run stays within minutes
    budget = min(max(1.0, 150.0 / max(1, args.steps + args.warmup)) * args.steps, args.cpu_seconds * 4)
    t0 = time.perf_counter()
    if wl == "stack":
        cb = cpu_stack_sample(T, budget)
    elif wl == "lmhead":
        cb = cpu_lmhead_sample(T, budget)
    elif wl == "attn":
        cb = cpu_attn_sample(args.ctx, args.window, budget)
    elif wl == "decoder":
        cb = cpu_decoder_sample(args.ctx, budget)
    else:
        cb = cpu_oracle_sample(wl, T, budget)
    el = time.perf_counter() - t0
    cfg = {"workload": name, "T": T, "d": D}
    if wl == "lmhead":
        cfg["V"] = V
    elif wl == "attn":
        cfg.update({"n_q_heads": NQ, "n_kv_heads": NKV, "head_dim": HD, "ctx": args.ctx, "window": args.window,
                    "rope": args.window > 0, "sinks": True})
    elif wl == "decoder":
        cfg.update({"layers": N_LAYERS, "E": E, "top_k": K_TOP, "I": I_FF, "V": V, "n_q_heads": NQ,
                    "n_kv_heads": NKV, "head_dim": HD, "ctx": args.ctx})
    else:
        cfg.update({"E": E, "top_k": K_SHARED if wl == "shared" else K_TOP, "n_shared": int(wl == "shared"),
                    "I": I_FF})
    res = {"metric": metric, "impl": "reference", "value": round(cb["value"], 3), "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
           "config": cfg, "ms_per_step": 1e3 / cb["value"] * T, "cpu_baseline": cb,
           "e2e": {"value": round(cb["value"], 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "wall_s": round(el, 1)}
    print(json.dumps(res))


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
        return

    world, rank, local = dist_setup(args)
    if args.workload in ("decode", "batch", "shared"):
        res = bench_decode(args, world, rank)
    elif args.workload == "prefill":
        res = bench_prefill(args, world, rank)
    elif args.workload == "lmhead":
        res = bench_lmhead(args, world, rank)
    elif args.workload == "attn":
        res = bench_attn(args, world, rank)
    elif args.workload == "decoder":
        res = bench_decoder(args, world, rank)
    else:
        res = bench_stack(args, world, rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            T = res["config"]["T"]
            if args.workload == "stack":
                res["cpu_baseline"] = cpu_stack_sample(T, args.cpu_seconds)
            elif args.workload == "lmhead":
                res["cpu_baseline"] = cpu_lmhead_sample(T, args.cpu_seconds, fmt=args.format)
            elif args.workload == "attn":
                res["cpu_baseline"] = cpu_attn_sample(args.ctx, args.window, args.cpu_seconds)
            elif args.workload == "decoder":
                res["cpu_baseline"] = cpu_decoder_sample(args.ctx, args.cpu_seconds)
            else:
                res["cpu_baseline"] = cpu_oracle_sample(args.workload, T, args.cpu_seconds, fmt=args.format)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
