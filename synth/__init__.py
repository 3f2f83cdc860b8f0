"""Seeded synthetic inputs for the int4 MoE layer and the int4 LM head.

This module only draws numbers. It holds none of the layer's arithmetic (no
dequantisation, no routing, no matrix products), so the CPU oracle and the CUDA
path can both take their inputs from here without sharing any of the method.

Two generators are used:

* Uniform tensors (packed int4 weight bytes, fp16 group scales) come from a
  counter-based hash: the SplitMix64 sequence of Steele, Lea and Flood
  ("Fast splittable pseudorandom number generators", OOPSLA 2014), whose i-th
  output from state ``key`` is ``mix64(key + (i + 1) * GAMMA)``.  Element ``i``
  of a tensor depends only on (seed, tag, layer, i), so any slice (one expert,
  one layer) can be drawn on its own, and ``synth_dev.cu`` draws the same bits
  on the device for the multi-GB weight banks.
* Normal tensors (activations, router weights and biases) are drawn on the
  host with numpy's PCG64 seeded by ``SeedSequence([seed, tag, layer, step])``.

Value recipes (the workload of a 256-expert, top-8, int4 coding-model MoE
layer as described on the Flint model pages):

* int4 weights: every nibble uniform over the 16 two's-complement values
  -8..7 (one byte holds element 2b in its low nibble, 2b+1 in its high one);
* fp16 scales: ``RNE_fp16(0.005 + 0.015 * u)``, u uniform in [0, 1) with 53 bits;
* activations: N(0, 1) rounded to bf16 (nearest-even);
* router weights: N(0, 1/d) in fp32; router bias: N(0, 1) in fp32, or the
  Zipf(s) bias ``b[pi(r)] = ln(r^-s / H)`` over a seeded permutation pi;
* NVFP4 banks: E2M1 codes uniform over the 16 codes (two per byte, drawn as the
  int4 bytes are), E4M3 block scales uniform over the codes 0x58..0x67 (16..60),
  fp32 tensor scales ``RN_fp32((1 + u) * 2^-12)``, so that the weights have
  the int4 banks' magnitude (mean |w| near 0.03 against 0.05).
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1

# Tensor tags: one independent stream per tensor kind.
TAG = {
    "gate_q": 1, "gate_s": 2, "up_q": 3, "up_s": 4, "down_q": 5, "down_s": 6,
    "router_w": 7, "router_b": 8, "x": 9, "lm_q": 10, "lm_s": 11, "zipf": 12,
    # NVFP4 banks: E2M1 codes, E4M3 block scales, fp32 tensor scales
    "gate_fq": 13, "gate_fs": 14, "gate_ts": 15, "up_fq": 16, "up_fs": 17, "up_ts": 18,
    "down_fq": 19, "down_fs": 20, "down_ts": 21, "lm_fq": 22, "lm_fs": 23, "lm_ts": 24,
    # attention layer: stacked q|k|v projection, output projection, sinks, key/value cache
    "qkv_q": 25, "qkv_s": 26, "wo_q": 27, "wo_s": 28, "sinks": 29, "kcache": 30, "vcache": 31,
}

# E4M3 block scales are drawn uniformly among the 16 byte codes 0x58 .. 0x67,
# the E4M3 numbers 16, 18, ..., 30, 32, 36, ..., 60.
E4M3_SCALE_CODE0 = 0x58


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tag: int, layer: int = 0) -> int:
    """Key of the (seed, tag, layer) stream: three chained SplitMix64 steps."""
    g = 0x9E3779B97F4A7C15
    k0 = _mix64_int(seed + g)
    k1 = _mix64_int(k0 + (tag + 1) * g)
    return _mix64_int(k1 + (layer + 1) * g)


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def hash_words(key: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the SplitMix64 sequence from ``key``."""
    idx = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx + np.uint64(1)) * GAMMA
        return mix64(z)


def int4_bytes(key: int, start: int, count: int) -> np.ndarray:
    """Bytes start .. start+count-1 of a packed uniform-int4 tensor.

    Byte b is byte (b mod 8) (little-endian) of hash word b // 8.
    """
    if count == 0:
        return np.zeros(0, np.uint8)
    w0 = start // 8
    w1 = (start + count + 7) // 8
    words = hash_words(key, w0, w1 - w0)
    raw = words.view(np.uint8) if words.dtype.byteorder in ("=", "<") else words.byteswap().view(np.uint8)
    off = start - w0 * 8
    return raw[off:off + count].copy()


def f16_scales(key: int, start: int, count: int) -> np.ndarray:
    """fp16 scales (as uint16 bits): RNE_fp16(0.005 + 0.015 * u), u = (h >> 11) * 2^-53."""
    if count == 0:
        return np.zeros(0, np.uint16)
    h = hash_words(key, start, count)
    u = (h >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    v = 0.005 + 0.015 * u
    return v.astype(np.float16).view(np.uint16)


def e4m3_scale_bytes(key: int, start: int, count: int) -> np.ndarray:
    """E4M3 block-scale bytes: 0x58 + (h >> 60), one hash word per byte."""
    if count == 0:
        return np.zeros(0, np.uint8)
    h = hash_words(key, start, count)
    return (np.uint64(E4M3_SCALE_CODE0) + (h >> np.uint64(60))).astype(np.uint8)


def f32_tensor_scales(key: int, start: int, count: int) -> np.ndarray:
    """fp32 tensor scales RN_fp32((1 + u) * 2^-12), u = (h >> 11) * 2^-53."""
    if count == 0:
        return np.zeros(0, np.float32)
    h = hash_words(key, start, count)
    u = (h >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return ((1.0 + u) * 2.0 ** -12).astype(np.float32)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (nearest-even), returned as uint16 bits.

    Used only to store drawn normals in the activation format; finite inputs
    of moderate magnitude only (no overflow / subnormal handling needed here).
    """
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                      # v = m * 2^e, 0.5 <= |m| < 1
    r = np.ldexp(np.rint(m * 256.0), e - 8)  # 8 significant bits, ties to even
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, tag: int, layer: int = 0, step: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, layer, step])))


# ---------------------------------------------------------------- activations


def activations(seed: int, T: int, d: int, step: int = 0, layer: int = 0) -> np.ndarray:
    """x [T, d] ~ N(0, 1) stored as bf16 bits (uint16)."""
    return f64_to_bf16_bits(_rng(seed, TAG["x"], layer, step).standard_normal((T, d)))


def router_weight(seed: int, E: int, d: int, layer: int = 0) -> np.ndarray:
    """W_r [E, d] ~ N(0, 1/d) in fp32."""
    g = _rng(seed, TAG["router_w"], layer).standard_normal((E, d))
    return (g * (1.0 / math.sqrt(d))).astype(np.float32)


def router_bias(seed: int, E: int, kind: str = "normal", layer: int = 0, zipf_s: float = 1.1) -> np.ndarray:
    """Per-expert router bias [E] fp32: 'zero', 'normal' (N(0,1)) or 'zipf'."""
    if kind == "zero":
        return np.zeros(E, np.float32)
    if kind == "normal":
        return _rng(seed, TAG["router_b"], layer).standard_normal(E).astype(np.float32)
    if kind == "zipf":
        r = np.arange(1, E + 1, dtype=np.float64)
        w = r ** (-zipf_s)
        p = w / w.sum()
        perm = _rng(seed, TAG["zipf"], layer).permutation(E)
        b = np.empty(E, np.float64)
        b[perm] = np.log(p)
        return b.astype(np.float32)
    raise ValueError(kind)


# ---------------------------------------------------------------- int4 weights


def int4_matrix(seed: int, qtag: str, stag: str, layer: int, n_mats: int, rows: int, K: int,
                group: int = 32, mat0: int = 0, mat1: int | None = None):
    """Packed int4 bank [n_mats, rows, K] (canonical layout) and its fp16 scales.

    Returns (q [m, rows, K/2] uint8, s [m, rows, K/group] uint16) for matrices
    mat0 .. mat1-1 only; element indices are those of the full bank, so a slice
    holds exactly the bytes the full bank holds there.
    """
    if mat1 is None:
        mat1 = n_mats
    m = mat1 - mat0
    qb = rows * K // 2
    sb = rows * K // group
    kq = stream_key(seed, TAG[qtag], layer)
    ks = stream_key(seed, TAG[stag], layer)
    q = int4_bytes(kq, mat0 * qb, m * qb).reshape(m, rows, K // 2)
    s = f16_scales(ks, mat0 * sb, m * sb).reshape(m, rows, K // group)
    return q, s


def attn_layer(seed: int, d: int, n_q: int, n_kv: int, head_dim: int = 128, layer: int = 0,
               sinks: bool = True) -> dict:
    """Tensors of one attention layer: int4 banks of the stacked q | k | v projection
    [(n_q + 2 n_kv) * head_dim, d] and of the output projection [d, n_q * head_dim]
    (nibbles uniform over -8..7, fp16 scales U(0.005, 0.02)), and the sink logits
    [n_q] ~ N(0, 1) fp32 (or None)."""
    rows = (n_q + 2 * n_kv) * head_dim
    wq, ws = int4_matrix(seed, "qkv_q", "qkv_s", layer, 1, rows, d)
    oq, os_ = int4_matrix(seed, "wo_q", "wo_s", layer, 1, d, n_q * head_dim)
    sk = _rng(seed, TAG["sinks"], layer).normal(0.0, 1.0, n_q).astype(np.float32) if sinks else None
    return {"wqkv_q": wq[0], "wqkv_s": ws[0], "wo_q": oq[0], "wo_s": os_[0], "sinks": sk}


def kv_cache(seed: int, L: int, n_kv: int, head_dim: int = 128, layer: int = 0):
    """Key and value cache contents [L, n_kv, head_dim] ~ N(0, 1) as bf16 bits (keys of a
    normalised, rotated head have unit mean square as well)."""
    k = f64_to_bf16_bits(_rng(seed, TAG["kcache"], layer).normal(0.0, 1.0, (L, n_kv, head_dim)))
    v = f64_to_bf16_bits(_rng(seed, TAG["vcache"], layer).normal(0.0, 1.0, (L, n_kv, head_dim)))
    return k, v


def moe_layer(seed: int, d: int, E: int, I: int, group: int = 32, layer: int = 0,
              bias: str = "normal", experts: tuple[int, int] | None = None) -> dict:
    """All tensors of one MoE layer (or of experts [e0, e1) only)."""
    e0, e1 = experts if experts is not None else (0, E)
    gq, gs = int4_matrix(seed, "gate_q", "gate_s", layer, E, I, d, group, e0, e1)
    uq, us = int4_matrix(seed, "up_q", "up_s", layer, E, I, d, group, e0, e1)
    dq, ds = int4_matrix(seed, "down_q", "down_s", layer, E, d, I, group, e0, e1)
    return {
        "gate_q": gq, "gate_s": gs, "up_q": uq, "up_s": us, "down_q": dq, "down_s": ds,
        "w_router": router_weight(seed, E, d, layer),
        "b_router": router_bias(seed, E, bias, layer),
    }


def moe_layer_shared(seed: int, d: int, E: int, I: int, group: int = 32, layer: int = 0,
                     bias: str = "normal") -> dict:
    """A layer with E routed experts plus one shared expert: the banks hold E + 1
    experts (the last is the shared one; the first E equal those of
    moe_layer(seed, d, E, I)), the router scores the E routed experts only."""
    t = moe_layer(seed, d, E + 1, I, group, layer, bias)
    t["w_router"] = router_weight(seed, E, d, layer)
    t["b_router"] = router_bias(seed, E, bias, layer)
    return t


def dense_layer(seed: int, d: int, I: int, group: int = 32, layer: int = 0) -> dict:
    """A dense SwiGLU layer as a one-entry bank (no router): the gate/up/down
    matrices of expert 0 of moe_layer(seed, d, 1, I)."""
    t = moe_layer(seed, d, 1, I, group, layer, "zero")
    t["w_router"] = None
    t["b_router"] = None
    return t


def lm_head(seed: int, V: int, d: int, group: int = 32, rows: tuple[int, int] | None = None):
    """LM-head bank q [V, d/2], s [V, d/32] (or rows [r0, r1) of it)."""
    r0, r1 = rows if rows is not None else (0, V)
    kq = stream_key(seed, TAG["lm_q"], 0)
    ks = stream_key(seed, TAG["lm_s"], 0)
    q = int4_bytes(kq, r0 * (d // 2), (r1 - r0) * (d // 2)).reshape(r1 - r0, d // 2)
    s = f16_scales(ks, r0 * (d // group), (r1 - r0) * (d // group)).reshape(r1 - r0, d // group)
    return q, s


# ---------------------------------------------------------------- NVFP4 weights


def nvfp4_matrix(seed: int, name: str, layer: int, n_mats: int, rows: int, K: int, mat0: int = 0,
                 mat1: int | None = None):
    """NVFP4 bank [n_mats, rows, K]: codes q [m, rows, K/2] (two E2M1 codes per
    byte, uniform over all 16), E4M3 block scales s [m, rows, K/16] and fp32
    tensor scales ts [m], for matrices mat0 .. mat1-1 of the full bank."""
    if mat1 is None:
        mat1 = n_mats
    m = mat1 - mat0
    qb = rows * K // 2
    sb = rows * K // 16
    q = int4_bytes(stream_key(seed, TAG[name + "_fq"], layer), mat0 * qb, m * qb).reshape(m, rows, K // 2)
    s = e4m3_scale_bytes(stream_key(seed, TAG[name + "_fs"], layer), mat0 * sb, m * sb).reshape(m, rows, K // 16)
    ts = f32_tensor_scales(stream_key(seed, TAG[name + "_ts"], layer), mat0, m)
    return q, s, ts


def moe_layer_nvfp4(seed: int, d: int, E: int, I: int, layer: int = 0, bias: str = "normal",
                    experts: tuple[int, int] | None = None, n_shared: int = 0) -> dict:
    """An MoE layer with NVFP4 expert banks (E + n_shared entries; the router
    scores E) and the same router as moe_layer."""
    Et = E + n_shared
    e0, e1 = experts if experts is not None else (0, Et)
    t = {}
    for name, rows, K in (("gate", I, d), ("up", I, d), ("down", d, I)):
        q, s, ts = nvfp4_matrix(seed, name, layer, Et, rows, K, e0, e1)
        t[name + "_q"], t[name + "_s"], t[name + "_ts"] = q, s, ts
    t["w_router"] = router_weight(seed, E, d, layer)
    t["b_router"] = router_bias(seed, E, bias, layer)
    return t


def lm_head_nvfp4(seed: int, V: int, d: int, rows: tuple[int, int] | None = None):
    """NVFP4 LM head: q [V, d/2], s [V, d/16] (or rows [r0, r1)), ts (fp32 scalar)."""
    r0, r1 = rows if rows is not None else (0, V)
    q = int4_bytes(stream_key(seed, TAG["lm_fq"], 0), r0 * (d // 2), (r1 - r0) * (d // 2)).reshape(r1 - r0, d // 2)
    s = e4m3_scale_bytes(stream_key(seed, TAG["lm_fs"], 0), r0 * (d // 16), (r1 - r0) * (d // 16))
    ts = f32_tensor_scales(stream_key(seed, TAG["lm_ts"], 0), 0, 1)[0]
    return q, s.reshape(r1 - r0, d // 16), ts


# ---------------------------------------------------------------- device twin

_DEV = None


def _dev_lib():
    global _DEV
    if _DEV is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"device generator not built: {path} (run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        for name in ("synth_fill_int4_bytes", "synth_fill_f16_scales", "synth_fill_e4m3_scales"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p]
        _DEV = lib
    return _DEV


def device_fill_int4(dst_ptr: int, count: int, key: int, start: int = 0, stream: int = 0) -> None:
    """Write bytes start .. start+count-1 of stream ``key`` to device memory."""
    rc = _dev_lib().synth_fill_int4_bytes(dst_ptr, count, key, start, stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_int4_bytes failed: cuda error {rc}")


def device_fill_scales(dst_ptr: int, count: int, key: int, start: int = 0, stream: int = 0) -> None:
    """Write fp16 scales start .. start+count-1 of stream ``key`` to device memory."""
    rc = _dev_lib().synth_fill_f16_scales(dst_ptr, count, key, start, stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_f16_scales failed: cuda error {rc}")


def device_fill_e4m3(dst_ptr: int, count: int, key: int, start: int = 0, stream: int = 0) -> None:
    """Write E4M3 block-scale bytes start .. start+count-1 of stream ``key`` to device memory."""
    rc = _dev_lib().synth_fill_e4m3_scales(dst_ptr, count, key, start, stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_e4m3_scales failed: cuda error {rc}")
