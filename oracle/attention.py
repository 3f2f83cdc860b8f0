"""fp64 CPU oracle of one decode step of the attention layer beside the MoE layer.

TEST INFRASTRUCTURE ONLY: imported by ``tests/`` and by the CPU-baseline leg of
``bench.py``; never by the product package.  Plain numpy in fp64, one function
per step, in the order the step runs; the int4 weights are dequantised by the
oracle's own C routine (``oracle.dequant_int4``).

Sources: "Flint 40B : Best Mid Sized LLM" (video transcript) 03:05 -- grouped-query
attention with 32 query heads and 4 key/value heads of 128 dimensions; 35 of the
mixture layers attend over a sliding window of 513 tokens (the current token and
the 512 before it), the others over the whole context; rotary position encoding
on the sliding-window layers and none on the full-attention layers; 03:36 -- a
per-head RMS norm on queries and keys and learned attention sinks.  The pages give
no formula; the readings taken where they are silent (listed with the design
notes) are: int4 group-32 weights as for the experts, the q/k/v projection rows
stacked as one [(32 + 4 + 4) * 128, d] matrix, unit-gain RMS norm with eps 1e-6,
rotary encoding on pairs (i, i + 64) with base 1e6 and the token's absolute
position, scores scaled by 1/sqrt(128), a sink as one learned logit per query head
that joins the softmax denominator with a zero value, keys and values stored in
the cache as bf16 (the current token's too, before it attends), and the attention
output rounded to bf16 before the output projection, whose result is added to
the residual.
"""
from __future__ import annotations

import numpy as np

import oracle

HEAD_DIM = 128
ROPE_THETA = 1.0e6


def bf16_bits_to_f64(bits):
    """Exact values of bf16 bit patterns (the upper half of an fp32 word), for arrays
    too large for the element-wise decoder."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def project(x, w_q, w_s):
    """x [d] (fp64) times the dequantised int4 matrix [rows, d]: [rows]."""
    return oracle.dequant_int4(w_q, w_s) @ x


def rmsnorm_heads(v, eps=oracle.RMS_EPS):
    """Each row of v [heads, hd] divided by its root mean square (unit gain)."""
    return v / np.sqrt(np.mean(v * v, axis=1, keepdims=True) + eps)


def rope(v, pos, theta=ROPE_THETA):
    """Rotary encoding of the rows of v [heads, hd] at position pos: element pairs
    (i, i + hd/2) rotated by the angle pos * theta^(-2i/hd)."""
    hd = v.shape[1]
    half = hd // 2
    ang = pos * theta ** (-2.0 * np.arange(half) / hd)
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[:, :half], v[:, half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=1)


def attend(q, k_cache, v_cache, pos, window, sinks, group):
    """q [nq, hd]; caches [>pos, nkv, hd] (fp64 values); keys j in [lo, pos] with
    lo = max(0, pos - window + 1) (window 0: the whole context).  Query head h reads
    key/value head h // group.  Returns o [nq, hd]."""
    nq, hd = q.shape
    lo = max(0, pos - window + 1) if window else 0
    o = np.zeros((nq, hd))
    for h in range(nq):
        g = h // group
        K = k_cache[lo:pos + 1, g, :]
        V = v_cache[lo:pos + 1, g, :]
        s = K @ q[h] / np.sqrt(hd)
        sink = -np.inf if sinks is None else float(sinks[h])
        m = max(np.max(s), sink)
        e = np.exp(s - m)
        z = np.sum(e) + (np.exp(sink - m) if sinks is not None else 0.0)
        o[h] = (e @ V) / z
    return o


def decode_step(x_bits, resid_bits, pos, layer, k_cache_bits, v_cache_bits, window=513, use_rope=True,
                n_q=32, n_kv=4, eps=oracle.RMS_EPS, theta=ROPE_THETA):
    """One attention decode step for one token.

    x_bits, resid_bits: [d] bf16 bits.  layer: dict with wqkv_q / wqkv_s (int4 bank of
    the stacked [(n_q + 2 n_kv) * 128, d] projection), wo_q / wo_s ([d, n_q * 128]) and
    sinks ([n_q] fp32, or None).  k_cache_bits / v_cache_bits: [L, n_kv, 128] bf16 bits,
    rows 0 .. pos - 1 filled; row pos is written here (the arrays are copied).
    Returns a dict: out (fp64 [d], before the bf16 rounding), out_bits, k_bits, v_bits
    (the new cache rows), attn_bits ([n_q * 128] bf16 input of the output projection),
    q ([n_q, 128] after norm and rotation), k_cache_bits, v_cache_bits (updated)."""
    hd = HEAD_DIM
    x = oracle.bf16_to_f64(np.asarray(x_bits, np.uint16))
    qkv = project(x, layer["wqkv_q"], layer["wqkv_s"])
    q = qkv[:n_q * hd].reshape(n_q, hd)
    k = qkv[n_q * hd:(n_q + n_kv) * hd].reshape(n_kv, hd)
    v = qkv[(n_q + n_kv) * hd:].reshape(n_kv, hd)
    q = rmsnorm_heads(q, eps)
    k = rmsnorm_heads(k, eps)
    if use_rope:
        q = rope(q, pos, theta)
        k = rope(k, pos, theta)
    k_bits = oracle.f64_to_bf16(k.reshape(-1)).reshape(n_kv, hd)
    v_bits = oracle.f64_to_bf16(v.reshape(-1)).reshape(n_kv, hd)
    kc = np.array(k_cache_bits, np.uint16, copy=True)
    vc = np.array(v_cache_bits, np.uint16, copy=True)
    kc[pos] = k_bits
    vc[pos] = v_bits
    kf = bf16_bits_to_f64(kc[:pos + 1])
    vf = bf16_bits_to_f64(vc[:pos + 1])
    o = attend(q, kf, vf, pos, window, layer.get("sinks"), n_q // n_kv)
    attn_bits = oracle.f64_to_bf16(o.reshape(-1))
    y = project(oracle.bf16_to_f64(attn_bits), layer["wo_q"], layer["wo_s"])
    out = oracle.bf16_to_f64(np.asarray(resid_bits, np.uint16)) + y
    return {"out": out, "out_bits": oracle.f64_to_bf16(out), "k_bits": k_bits, "v_bits": v_bits,
            "attn_bits": attn_bits, "o": o, "q": q, "k_cache_bits": kc, "v_cache_bits": vc}


def prenorm_step(resid_bits, pos, layer, k_cache_bits, v_cache_bits, window=513, use_rope=True, n_q=32, n_kv=4,
                 eps=oracle.RMS_EPS, theta=ROPE_THETA):
    """The pre-norm attention block of a decoder layer: x = bf16(RMSNorm(residual)) (unit
    gain), then decode_step(x, residual, ...), whose out is residual + Wo attn.  The same
    norm the oracle's stack puts before each MoE block.  Returns decode_step's dict plus
    x_bits."""
    r = np.asarray(resid_bits, np.uint16)
    x = oracle.f64_to_bf16(oracle.rmsnorm(r[None, :], eps))[0]
    res = decode_step(x, r, pos, layer, k_cache_bits, v_cache_bits, window=window, use_rope=use_rope, n_q=n_q,
                      n_kv=n_kv, eps=eps, theta=theta)
    res["x_bits"] = x
    return res
