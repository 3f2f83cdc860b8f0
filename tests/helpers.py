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
