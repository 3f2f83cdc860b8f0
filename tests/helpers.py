"""Shared helpers of the GPU parity tests: seeded workloads, device upload,
error metrics and the near-tie rule."""
from __future__ import annotations

import numpy as np

import synth

# Workloads (shapes of the 256-expert, top-8 int4 layer and its tiny smoke variant).
TINY = dict(d=256, E=16, k=2, I=128, bias="zero")
FLINT = dict(d=2048, E=256, k=8, I=512)

# Tolerances on the layer output, checked on the fp32 copy before the bf16 cast.
MAX_ABS = 2e-2
REL_L2 = 1e-3
NEAR_TIE = 1e-5   # oracle k-th / (k+1)-th logit gap below which the oracle's choice is fed to both sides


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def bf16_bits_to_f64(bits):
    return synth.bf16_bits_to_f32(np.asarray(bits, np.uint16)).astype(np.float64)


def torch_bf16_from_bits(bits, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def bits_from_torch_bf16(t):
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def layer_tensors(seed, d, E, I, bias="normal", layer=0):
    return synth.moe_layer(seed, d, E, I, bias=bias, layer=layer)


def device_layer(tensors, k, renormalize=True):
    import bit_expert_ffn_warp_b300 as bm
    return bm.MoeLayer.from_canonical(tensors, k, renormalize=renormalize)


def bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (fp64)."""
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def device_drawn_layer(seed, layer, d, E, I, k, bias="normal"):
    """One MoE layer whose int4 banks are drawn on the device by the generator twin
    (same bits as ``synth.moe_layer(seed, ..., layer=layer)``) and packed there."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    banks = {}
    for name, (rows, K) in {"gate": (I, d), "up": (I, d), "down": (d, I)}.items():
        q = torch.empty(E * rows * K // 2, dtype=torch.uint8, device="cuda")
        s = torch.empty(E * rows * K // 32, dtype=torch.float16, device="cuda")
        synth.device_fill_int4(q.data_ptr(), q.numel(), synth.stream_key(seed, synth.TAG[name + "_q"], layer))
        synth.device_fill_scales(s.data_ptr(), s.numel(), synth.stream_key(seed, synth.TAG[name + "_s"], layer))
        banks[name] = bm.bitmoe_pack_int4(q.view(E, rows, K // 2), s.view(E, rows, K // 32))
    wr = torch.from_numpy(synth.router_weight(seed, E, d, layer)).cuda()
    br = torch.from_numpy(synth.router_bias(seed, E, bias, layer)).cuda()
    return bm.MoeLayer(d=d, E=E, k=k, I=I, gate=banks["gate"], up=banks["up"], down=banks["down"],
                       w_router=wr, b_router=br)


def device_drawn_lm_head(seed, V, d):
    """The int4 LM head drawn on the device (same bits as ``synth.lm_head``), packed."""
    import torch

    import bit_expert_ffn_warp_b300 as bm
    q = torch.empty(V * d // 2, dtype=torch.uint8, device="cuda")
    s = torch.empty(V * d // 32, dtype=torch.float16, device="cuda")
    synth.device_fill_int4(q.data_ptr(), q.numel(), synth.stream_key(seed, synth.TAG["lm_q"], 0))
    synth.device_fill_scales(s.data_ptr(), s.numel(), synth.stream_key(seed, synth.TAG["lm_s"], 0))
    return bm.bitmoe_pack_int4(q.view(V, d // 2), s.view(V, d // 32))


def expert_bank(seed, layer, d, I, experts, E=256):
    """Canonical gate/up/down tensors of the listed experts of one layer, in that order."""
    parts = {}
    for name, (rows, K) in {"gate": (I, d), "up": (I, d), "down": (d, I)}.items():
        qs, ss = [], []
        for e in experts:
            q, s = synth.int4_matrix(seed, name + "_q", name + "_s", layer, E, rows, K, 32, e, e + 1)
            qs.append(q)
            ss.append(s)
        parts[name + "_q"] = np.concatenate(qs)
        parts[name + "_s"] = np.concatenate(ss)
    return parts
