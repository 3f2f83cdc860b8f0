"""Pins of the fp64 oracle to facts outside itself.

Each test checks the oracle against something the pages or the mathematics
fix -- IEEE bit patterns, closed forms, brute force over tiny inputs, special
cases that collapse to a dense SwiGLU FFN computed with numpy, invariants of
the permutation -- so that a dropped term, a wrong sign or index, or a
transposed operand anywhere in oracle.c fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ helpers that do not use the oracle


def np_unpack_int4(q):
    """Independent nibble unpacking: low nibble first, two's complement."""
    q = np.asarray(q, np.uint8)
    lo = (q & 0x0F).astype(np.int16)
    hi = (q >> 4).astype(np.int16)
    v = np.stack([lo, hi], axis=-1).reshape(q.shape[:-1] + (q.shape[-1] * 2,))
    return np.where(v >= 8, v - 16, v).astype(np.float64)


def np_dequant(q, s, group=32):
    vals = np_unpack_int4(q)
    sc = np.asarray(s, np.uint16).view(np.float16).astype(np.float64)
    return vals * np.repeat(sc, group, axis=-1)


def np_pack_int4(vals):
    """Pack signed ints in [-8, 7] (last axis even) into bytes, low nibble first."""
    v = np.asarray(vals, np.int64) & 0xF
    return (v[..., 0::2] | (v[..., 1::2] << 4)).astype(np.uint8)


def f16_bits(values):
    return np.asarray(values, np.float64).astype(np.float16).view(np.uint16)


def bf16_to_np(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def silu(a):
    return a / (1.0 + np.exp(-a))


def layer_from_dense(gate_vals, gate_s, up_vals, up_s, down_vals, down_s, w_router, b_router=None):
    return {
        "gate_q": np_pack_int4(gate_vals), "gate_s": f16_bits(gate_s),
        "up_q": np_pack_int4(up_vals), "up_s": f16_bits(up_s),
        "down_q": np_pack_int4(down_vals), "down_s": f16_bits(down_s),
        "w_router": np.asarray(w_router, np.float32),
        "b_router": None if b_router is None else np.asarray(b_router, np.float32),
    }


# ------------------------------------------------------------------ storage formats


def test_bf16_fp16_decoding_matches_ieee_patterns():
    # bf16: 0x3F80 = 1, 0xC000 = -2, 0x7F7F = largest finite, 0x0001 = 2^-133
    assert oracle.bf16_to_f64([0x3F80, 0xC000, 0x0000, 0x8000]).tolist() == [1.0, -2.0, 0.0, -0.0]
    assert oracle.bf16_to_f64([0x7F7F])[0] == (2 - 2 ** -7) * 2.0 ** 127
    assert oracle.bf16_to_f64([0x0001])[0] == 2.0 ** -133
    # fp16: 0x3C00 = 1, 0x7BFF = 65504, 0x0001 = 2^-24, 0x0400 = 2^-14, 0xB555 = -(1+341/1024)*2^-2
    assert oracle.f16_to_f64([0x3C00, 0x7BFF, 0x0001, 0x0400]).tolist() == [1.0, 65504.0, 2.0 ** -24, 2.0 ** -14]
    assert oracle.f16_to_f64([0xB555])[0] == -(1 + 341 / 1024) * 0.25
    # agreement with numpy's fp16 on every finite pattern
    allbits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    finite = np.isfinite(allbits.view(np.float16))
    ref = allbits[finite].view(np.float16).astype(np.float64)
    got = oracle.f16_to_f64(allbits[finite])
    assert np.array_equal(got, ref)


def test_bf16_rounding_is_nearest_even():
    cases = {
        1.0: 0x3F80,
        1 + 2 ** -8: 0x3F80,           # tie -> even (down)
        1 + 3 * 2 ** -8: 0x3F82,       # tie -> even (up)
        1 + 2 ** -8 + 2 ** -30: 0x3F81,  # just above the tie
        -(1 + 2 ** -7): 0xBF81,
        (2 - 2 ** -9): 0x4000,         # rounds up into the next binade
        3.0e38 * 2: 0x7F80,            # overflow -> +inf
        2.0 ** -133: 0x0001,           # smallest subnormal
        0.0: 0x0000,
    }
    got = oracle.f64_to_bf16(np.array(list(cases.keys())))
    assert [int(g) for g in got] == list(cases.values())
    # every bf16 value is a fixed point of the rounding
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 0x7F80, 2000).astype(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16(bf16_to_np(bits)), bits)


# ------------------------------------------------------------------ dequantisation


def test_dequant_round_trip_of_representable_weights():
    rng = np.random.default_rng(2)
    rows, K = 5, 96
    vals = rng.integers(-8, 8, (rows, K))
    scales = rng.uniform(0.005, 0.02, (rows, K // 32)).astype(np.float16)
    q = np_pack_int4(vals)
    W = oracle.dequant_int4(q, scales.view(np.uint16))
    want = vals * np.repeat(scales.astype(np.float64), 32, axis=1)
    assert np.array_equal(W, want)  # exact: 4-bit x 11-bit fits fp64
    # byte 0x8F holds (low) -1 and (high) -8
    assert oracle.dequant_int4(np.array([[0x8F] * 16], np.uint8), f16_bits([[1.0]])).tolist()[0][:2] == [-1.0, -8.0]


def test_dequant_group_index_is_column_over_32():
    q = np_pack_int4(np.ones((1, 64), np.int64))
    W = oracle.dequant_int4(q, f16_bits([[2.0, -3.0]]))
    assert np.array_equal(W[0, :32], np.full(32, 2.0)) and np.array_equal(W[0, 32:], np.full(32, -3.0))


# ------------------------------------------------------------------ routing


def test_router_logits_closed_form():
    d, E = 64, 3
    x = synth.f64_to_bf16_bits(np.linspace(-1, 1, d)[None, :])
    xv = bf16_to_np(x)[0]
    Wr = np.zeros((E, d), np.float32)
    Wr[0, 5] = 1.0             # picks x[5]
    Wr[1, :] = 0.5             # half the sum
    Wr[2, 63] = -2.0           # -2 x[63]
    b = np.array([0.0, 1.0, -1.0], np.float32)
    l = oracle.router_logits(x, Wr, b)[0]
    assert l[0] == xv[5] and l[1] == 0.5 * xv.sum() + 1.0 and l[2] == -2 * xv[63] - 1.0
    assert np.array_equal(oracle.router_logits(x, Wr, None)[0], l - b)


def test_softmax_closed_forms():
    p = oracle.softmax(np.array([[0.0, 0.0, 0.0, 0.0], [3.0, 1.0, -np.inf, -np.inf]]))
    assert np.allclose(p[0], 0.25, atol=0, rtol=1e-15)
    assert abs(p[1, 0] - 1 / (1 + math.exp(-2.0))) < 1e-15  # two-way softmax = logistic
    assert p[1, 2] == 0.0 and p[1, 3] == 0.0
    rng = np.random.default_rng(3)
    l = rng.normal(0, 3, (50, 37))
    p = oracle.softmax(l)
    assert np.all(np.abs(p.sum(1) - 1) < 1e-15)
    # shift invariance and ratio law p_a / p_b = exp(l_a - l_b)
    assert np.allclose(oracle.softmax(l + 100.0), p, rtol=1e-13, atol=0)
    assert np.allclose(p[:, 0] / p[:, 1], np.exp(l[:, 0] - l[:, 1]), rtol=1e-13)


@pytest.mark.parametrize("E", [1, 2, 5, 8, 16])
def test_topk_equals_brute_force(E):
    rng = np.random.default_rng(E)
    for k in range(1, E + 1):
        l = rng.normal(size=(6, E))
        ids, gap = oracle.topk(l, k)
        for t in range(l.shape[0]):
            order = sorted(range(E), key=lambda e: (-l[t, e], e))  # python sort, not qsort
            assert ids[t].tolist() == order[:k]
            best = max(itertools.combinations(range(E), k), key=lambda c: sum(l[t, list(c)]))
            assert sorted(best) == sorted(ids[t].tolist())
            assert gap[t] == (l[t, order[k - 1]] - l[t, order[k]] if k < E else np.inf)


def test_topk_ties_go_to_the_lower_expert():
    l = np.array([[1.0, 2.0, 2.0, 0.5, 2.0, 1.0]])
    ids, gap = oracle.topk(l, 2)
    assert ids.tolist() == [[1, 2]] and gap[0] == 0.0
    ids, _ = oracle.topk(l, 4)
    assert ids.tolist() == [[1, 2, 4, 0]]


def test_gates():
    rng = np.random.default_rng(4)
    l = rng.normal(size=(7, 9))
    p = oracle.softmax(l)
    ids, _ = oracle.topk(l, 9)
    w = oracle.gates(p, ids, renorm=True)
    assert np.allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-14)  # k = E: gates are the softmax
    ids, _ = oracle.topk(l, 3)
    w = oracle.gates(p, ids, renorm=True)
    assert np.all(np.abs(w.sum(1) - 1) < 1e-15)
    sel = np.take_along_axis(l, ids, 1)
    e = np.exp(sel - sel.max(1, keepdims=True))
    assert np.allclose(w, e / e.sum(1, keepdims=True), rtol=1e-14)  # softmax restricted to the chosen logits
    w0 = oracle.gates(p, ids, renorm=False)
    assert np.array_equal(w0, np.take_along_axis(p, ids, 1))
    assert np.all(np.diff(w, axis=1) <= 0)  # descending


def test_route_composes_the_steps():
    x = synth.activations(5, 6, 128)
    Wr = synth.router_weight(5, 12, 128)
    b = synth.router_bias(5, 12, "normal")
    ids, w, l, gap = oracle.route(x, Wr, b, 3)
    xv = bf16_to_np(x)
    assert np.allclose(l, xv @ Wr.astype(np.float64).T + b, rtol=1e-12, atol=1e-12)
    ids2, gap2 = oracle.topk(l, 3)
    assert np.array_equal(ids, ids2) and np.array_equal(gap, gap2)


# ------------------------------------------------------------------ permutation


@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (5, 8, 3), (33, 16, 2), (64, 256, 8), (0, 8, 2)])
def test_permutation_invariants(T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    ids = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32).reshape(T, k)
    off, rows, inv = oracle.permute(ids, E)
    flat = ids.reshape(-1)
    assert off[0] == 0 and off[E] == T * k and np.all(np.diff(off) >= 0)
    assert np.array_equal(np.diff(off), np.bincount(flat, minlength=E))
    assert np.array_equal(rows, np.argsort(flat, kind="stable"))  # numpy's stable sort
    assert np.array_equal(rows[inv], np.arange(T * k))  # permute then unpermute = identity
    assert np.array_equal(inv[rows], np.arange(T * k))
    for e in range(E):
        assert np.all(flat[rows[off[e]:off[e + 1]]] == e)


def test_permutation_rejects_out_of_range_ids():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 9]], np.int32), 8)


# ------------------------------------------------------------------ expert FFN and combine


def test_single_expert_top1_is_a_dense_swiglu_ffn():
    rng = np.random.default_rng(6)
    d, I, T = 64, 96, 5
    gv, uv, dv = rng.integers(-8, 8, (1, I, d)), rng.integers(-8, 8, (1, I, d)), rng.integers(-8, 8, (1, d, I))
    gs, us = rng.uniform(0.005, 0.02, (1, I, d // 32)), rng.uniform(0.005, 0.02, (1, I, d // 32))
    ds = rng.uniform(0.005, 0.02, (1, d, I // 32))
    lay = layer_from_dense(gv, gs, uv, us, dv, ds, rng.normal(size=(1, d)))
    x = synth.activations(6, T, d)
    res = oracle.moe_forward(x, lay, k=1)
    assert np.all(res["ids"] == 0) and np.all(res["w"] == 1.0)
    Wg, Wu, Wd = (np_dequant(lay[n + "_q"][0], lay[n + "_s"][0]) for n in ("gate", "up", "down"))
    xv = bf16_to_np(x)
    dense = xv + (silu(xv @ Wg.T) * (xv @ Wu.T)) @ Wd.T   # numpy matmuls on independently dequantised weights
    assert np.allclose(res["out"], dense, rtol=1e-12, atol=1e-12)


def test_constant_weights_closed_form():
    d, I = 64, 32
    one = np.ones
    lay = layer_from_dense(one((1, I, d)), one((1, I, 2)), 2 * one((1, I, d)), one((1, I, 2)),
                           -one((1, d, I)), 0.5 * one((1, d, 1)), np.zeros((1, d)))
    x = synth.f64_to_bf16_bits(np.full((1, d), 0.03125))
    S = 64 * 0.03125  # sum of x = 2
    a, u = S, 2 * S
    h = a / (1 + math.exp(-a)) * u
    y = -0.5 * I * h
    out = oracle.moe_forward(x, lay, k=1)["out"]
    assert np.allclose(out, 0.03125 + y, rtol=1e-14, atol=0)


def test_one_hot_gate_selects_one_expert_and_down_scale_is_linear():
    d, E, I, T = 128, 4, 64, 3
    lay = synth.moe_layer(7, d, E, I, bias="zero")
    x = synth.activations(7, T, d)
    y = oracle.expert_ffn(x, lay, np.full((T, 1), 2, np.int32))
    res = oracle.moe_forward(x, lay, k=1, forced_ids=np.full((T, 1), 2, np.int32), forced_w=np.ones((T, 1)))
    assert np.allclose(res["out"], bf16_to_np(x) + y, rtol=1e-15, atol=1e-15)
    # doubling every fp16 scale of W_down (exact in fp16) doubles out - x
    lay2 = dict(lay)
    lay2["down_s"] = f16_bits(lay["down_s"].view(np.float16).astype(np.float64) * 2)
    res2 = oracle.moe_forward(x, lay2, k=1, forced_ids=np.full((T, 1), 2, np.int32), forced_w=np.ones((T, 1)))
    assert np.allclose(res2["out"] - bf16_to_np(x), 2 * (res["out"] - bf16_to_np(x)), rtol=1e-13, atol=1e-13)
    # swapping the expert's gate and up banks changes the result (silu is not symmetric)
    lay3 = dict(lay)
    lay3["gate_q"], lay3["up_q"], lay3["gate_s"], lay3["up_s"] = lay["up_q"], lay["gate_q"], lay["up_s"], lay["gate_s"]
    y3 = oracle.expert_ffn(x, lay3, np.full((T, 1), 2, np.int32))
    assert not np.allclose(y3, y)


def test_shared_expert_adds_its_dense_swiglu_ffn_with_weight_one():
    """Top-k routed experts plus one always-on shared expert ("Flint 40B : Best Mid
    Sized LLM", transcript 02:35): the routing of the E routed experts is that of
    the layer without the shared expert, and the output differs from that
    layer's by the shared expert's dense SwiGLU FFN (numpy on independently
    dequantised weights), added with weight 1."""
    d, E, I, T, k = 128, 6, 64, 5, 2
    lay = synth.moe_layer_shared(9, d, E, I, bias="normal")
    assert lay["gate_q"].shape[0] == E + 1 and lay["w_router"].shape[0] == E
    x = synth.activations(9, T, d)
    res = oracle.moe_forward(x, lay, k, n_shared=1)
    routed = {n: (v[:E] if n.endswith(("_q", "_s")) else v) for n, v in lay.items()}
    base = oracle.moe_forward(x, routed, k)
    assert res["ids"].shape == (T, k + 1)
    assert np.array_equal(res["ids"][:, :k], base["ids"]) and np.all(res["ids"][:, k] == E)
    assert np.array_equal(res["w"][:, :k], base["w"]) and np.all(res["w"][:, k] == 1.0)
    Wg, Wu, Wd = (np_dequant(lay[n + "_q"][E], lay[n + "_s"][E]) for n in ("gate", "up", "down"))
    xv = bf16_to_np(x)
    dense = (silu(xv @ Wg.T) * (xv @ Wu.T)) @ Wd.T
    assert np.allclose(res["out"] - base["out"], dense, rtol=1e-11, atol=1e-12)
    # feeding the same selection reproduces the routed result exactly
    fed = oracle.moe_forward(x, lay, k, n_shared=1, forced_ids=res["ids"], forced_w=res["w"])
    assert np.array_equal(fed["out"], res["out"])
    # the shared expert's weight is 1 whatever the routed gates: halving every routed gate
    # halves the routed part only
    half = oracle.moe_forward(x, lay, k, n_shared=1, forced_ids=res["ids"],
                              forced_w=np.concatenate([res["w"][:, :k] / 2, res["w"][:, k:]], axis=1))
    assert np.allclose(half["out"] - dense, bf16_to_np(x) + (base["out"] - bf16_to_np(x)) / 2, rtol=1e-11, atol=1e-12)


def test_dense_layer_is_a_swiglu_ffn_of_every_token():
    """k = 0 routed experts with the shared expert only: the stack's leading dense
    layers ("Flint 40B : Best Mid Sized LLM", transcript 02:35) as x + FFN(x),
    the FFN computed with numpy on independently dequantised weights."""
    d, I, T = 128, 96, 4
    lay = synth.dense_layer(12, d, I)
    x = synth.activations(12, T, d)
    res = oracle.moe_forward(x, lay, 0, n_shared=1)
    assert np.all(res["ids"] == 0) and np.all(res["w"] == 1.0) and res["ids"].shape == (T, 1)
    Wg, Wu, Wd = (np_dequant(lay[n + "_q"][0], lay[n + "_s"][0]) for n in ("gate", "up", "down"))
    xv = bf16_to_np(x)
    assert np.allclose(res["out"], xv + (silu(xv @ Wg.T) * (xv @ Wu.T)) @ Wd.T, rtol=1e-12, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.moe_forward(x, lay, 0, n_shared=0)


def test_expert_ffn_matches_numpy_per_row():
    d, E, I, T, k = 128, 6, 64, 4, 3
    lay = synth.moe_layer(8, d, E, I, bias="normal")
    x = synth.activations(8, T, d)
    ids, w, _, _ = oracle.route(x, lay["w_router"], lay["b_router"], k)
    y, h = oracle.expert_ffn(x, lay, ids, want_h=True)
    xv = bf16_to_np(x)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            Wg, Wu, Wd = (np_dequant(lay[n + "_q"][e], lay[n + "_s"][e]) for n in ("gate", "up", "down"))
            hh = silu(Wg @ xv[t]) * (Wu @ xv[t])
            assert np.allclose(h[t * k + j], hh, rtol=1e-12, atol=1e-12)
            assert np.allclose(y[t * k + j], Wd @ hh, rtol=1e-12, atol=1e-12)
    out = oracle.combine(y, w, x)
    want = xv + np.einsum("tj,tjc->tc", w, y.reshape(T, k, d))
    assert np.allclose(out, want, rtol=1e-14, atol=1e-14)


def test_combine_constant_rows():
    T, k, d = 3, 4, 32
    w = np.random.default_rng(9).dirichlet(np.ones(k), T)
    y = np.full((T * k, d), 0.75)
    x = synth.activations(9, T, d)
    assert np.allclose(oracle.combine(y, w, x), bf16_to_np(x) + 0.75, rtol=1e-15, atol=1e-15)


# ------------------------------------------------------------------ NVFP4


def e2m1_table():
    with open(os.path.join(GOLDEN, "nvfp4_e2m1.json")) as f:
        return np.array(json.load(f)["values"], np.float64)


def np_e4m3(b):
    """E4M3 bytes through torch's float8_e4m3fn conversion (a library routine)."""
    import torch
    return torch.from_numpy(np.asarray(b, np.uint8).copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def np_dequant_nvfp4(q, s, ts):
    """Independent NVFP4 dequantisation: low nibble first, the golden E2M1
    table, torch's E4M3 decoding, one scale per 16 columns."""
    q = np.asarray(q, np.uint8)
    codes = np.stack([q & 0x0F, q >> 4], axis=-1).reshape(q.shape[:-1] + (q.shape[-1] * 2,))
    return e2m1_table()[codes] * np.repeat(np_e4m3(s), 16, axis=-1) * float(np.float32(ts))


def np_pack_codes(codes):
    c = np.asarray(codes, np.int64) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def test_e2m1_codes_match_the_format_table():
    table = e2m1_table()
    got = oracle.e2m1_to_f64(np.arange(16))
    assert np.array_equal(got, table)
    assert np.array_equal(np.signbit(got), np.signbit(table))  # code 8 is -0
    # only the low nibble of a byte is a code
    assert np.array_equal(oracle.e2m1_to_f64(np.arange(16) + 0x30), table)


def test_e4m3_bytes_match_torch_float8_e4m3fn():
    b = np.arange(256)
    got = oracle.e4m3_to_f64(b)
    want = np_e4m3(b)
    assert np.array_equal(np.isnan(got), np.isnan(want)) and int(np.isnan(got).sum()) == 2
    fin = ~np.isnan(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(want[fin]))
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_dequant_nvfp4_matches_an_independent_decoding():
    q, s, ts = synth.nvfp4_matrix(30, "gate", 0, 1, 32, 256)
    got = oracle.dequant_nvfp4(q[0], s[0], ts[0])
    assert np.array_equal(got, np_dequant_nvfp4(q[0], s[0], ts[0]))


def test_dequant_nvfp4_block_index_is_column_over_16():
    rows, K = 3, 64
    q = np_pack_codes(np.full((rows, K), 2))  # every element 1.0
    s = (0x38 + np.arange(rows * K // 16).reshape(rows, K // 16)).astype(np.uint8)  # distinct scales 1, 1.125, ...
    got = oracle.dequant_nvfp4(q, s, 0.5)
    want = 0.5 * np.repeat(np_e4m3(s), 16, axis=1)
    assert np.array_equal(got, want)
    # the sign is bit 3 of the code, the tensor scale multiplies every element
    q = np_pack_codes(np.tile([7, 15], (rows, K // 2)))
    got = oracle.dequant_nvfp4(q, np.full((rows, K // 16), 0x38, np.uint8), 2.0)
    assert np.array_equal(got, np.tile([12.0, -12.0], (rows, K // 2)))


def test_lmhead_nvfp4_planted_row_and_ties():
    d, V = 64, 48
    rng = np.random.default_rng(31)
    codes = rng.integers(0, 16, (V, d)) & 0b1011  # magnitudes up to 1.5, either sign
    hx = synth.f64_to_bf16_bits(rng.normal(size=(2, d)))
    hv = bf16_to_np(hx)
    codes[17] = np.where(hv[0] > 0, 7, 15)  # planted: +-6 aligned with sign(h[0])
    codes[30] = np.where(hv[1] > 0, 7, 15)
    s = rng.integers(0x30, 0x40, (V, d // 16)).astype(np.uint8)
    s[17] = s[30] = 0x3F  # the largest scale drawn
    q = np_pack_codes(codes)
    ts = np.float32(0.0625)
    logits, am, gap = oracle.lmhead_nvfp4(hx, q, s, ts)
    W = np_dequant_nvfp4(q, s, ts)
    assert np.allclose(logits, hv @ W.T, rtol=1e-13, atol=1e-13)
    assert am.tolist() == [17, 30] and np.all(gap > 0)
    codes[5] = codes[17]
    s[5] = s[17]
    _, am, gap = oracle.lmhead_nvfp4(hx, np_pack_codes(codes), s, ts)
    assert am[0] == 5 and gap[0] == 0.0


def test_expert_ffn_nvfp4_matches_numpy_per_row():
    d, E, I, T, k = 128, 6, 64, 4, 3
    lay = synth.moe_layer_nvfp4(32, d, E, I, bias="normal")
    x = synth.activations(32, T, d)
    ids, w, _, _ = oracle.route(x, lay["w_router"], lay["b_router"], k)
    y, h = oracle.expert_ffn(x, lay, ids, want_h=True)
    xv = bf16_to_np(x)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            Wg, Wu, Wd = (np_dequant_nvfp4(lay[n + "_q"][e], lay[n + "_s"][e], lay[n + "_ts"][e])
                          for n in ("gate", "up", "down"))
            hh = silu(Wg @ xv[t]) * (Wu @ xv[t])
            assert np.allclose(h[t * k + j], hh, rtol=1e-12, atol=1e-12)
            assert np.allclose(y[t * k + j], Wd @ hh, rtol=1e-12, atol=1e-12)
    res = oracle.moe_forward(x, lay, k)
    assert np.array_equal(res["ids"], ids)
    want = xv + np.einsum("tj,tjc->tc", w, y.reshape(T, k, d))
    assert np.allclose(res["out"], want, rtol=1e-13, atol=1e-13)


def test_nvfp4_single_expert_top1_is_a_dense_swiglu_ffn():
    d, I, T = 64, 32, 3
    lay = synth.moe_layer_nvfp4(33, d, 1, I, bias="zero")
    x = synth.activations(33, T, d)
    res = oracle.moe_forward(x, lay, 1)
    assert np.all(res["ids"] == 0) and np.allclose(res["w"], 1.0)
    Wg, Wu, Wd = (np_dequant_nvfp4(lay[n + "_q"][0], lay[n + "_s"][0], lay[n + "_ts"][0])
                  for n in ("gate", "up", "down"))
    xv = bf16_to_np(x)
    want = xv + (silu(xv @ Wg.T) * (xv @ Wu.T)) @ Wd.T
    assert np.allclose(res["out"], want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ stack pieces


def test_rmsnorm_closed_forms():
    eps = 1e-6
    x = synth.f64_to_bf16_bits(np.full((1, 64), 0.5))
    y = oracle.rmsnorm(x, eps)
    assert np.allclose(y, 0.5 / math.sqrt(0.25 + eps), rtol=1e-15)
    x = synth.activations(10, 4, 256)
    y = oracle.rmsnorm(x, eps)
    ms = (bf16_to_np(x) ** 2).mean(1)
    assert np.allclose((y ** 2).mean(1), ms / (ms + eps), rtol=1e-13)
    assert np.all(np.sign(y) == np.sign(bf16_to_np(x)))


def test_lmhead_planted_row_and_ties():
    d, V = 64, 48
    rng = np.random.default_rng(11)
    vals = rng.integers(-3, 4, (V, d))
    hx = synth.f64_to_bf16_bits(rng.normal(size=(2, d)))
    hv = bf16_to_np(hx)
    vals[17] = np.where(hv[0] > 0, 7, -8)  # planted: aligned with sign(h[0]) at full magnitude
    vals[30] = np.where(hv[1] > 0, 7, -8)
    s = np.full((V, d // 32), 0.01)
    q = np_pack_int4(vals)
    logits, am, gap = oracle.lmhead(hx, q, f16_bits(s))
    W = np_dequant(q, f16_bits(s))
    assert np.allclose(logits, hv @ W.T, rtol=1e-13, atol=1e-13)
    assert am.tolist() == [17, 30] and np.all(gap > 0)
    # a duplicated best row ties: the lower index wins and the gap is 0
    vals[5] = vals[17]
    logits, am, gap = oracle.lmhead(hx, np_pack_int4(vals), f16_bits(s))
    assert am[0] == 5 and gap[0] == 0.0


def test_stack_equals_layer_by_layer():
    d, E, I, k, L, V = 128, 8, 64, 2, 3, 64
    layers = [synth.moe_layer(20, d, E, I, layer=l, bias="normal") for l in range(L)]
    lm_q, lm_s = synth.lm_head(20, V, d)
    x0 = synth.activations(20, 2, d)

    def expert_fn(l, ex):
        return {n: layers[l][n][ex] for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")}

    res = oracle.stack_forward(x0, lambda l: layers[l], expert_fn, L, k, lm_q, lm_s)
    r = x0
    for l in range(L):
        xh = oracle.f64_to_bf16(oracle.rmsnorm(r))
        out = oracle.moe_forward(xh, layers[l], k, resid=r)
        assert np.array_equal(res["layers"][l]["ids"], out["ids"])
        assert np.allclose(res["layers"][l]["out"], out["out"], rtol=1e-15, atol=1e-15)
        r = oracle.f64_to_bf16(out["out"])
    xh = oracle.f64_to_bf16(oracle.rmsnorm(r))
    _, am, _ = oracle.lmhead(xh, lm_q, lm_s)
    assert np.array_equal(res["argmax"], am)


# ------------------------------------------------------------------ the pages' printed size facts


def test_layer_shapes_reproduce_the_pages_size_facts():
    f = json.load(open(os.path.join(GOLDEN, "page_facts.json")))
    d, E, I, k, L, group = 2048, 256, 512, 8, f["layers"], 32
    assert E == f["experts"]
    # the pages' layout: 47 mixture layers of 256 experts (plus 2 dense ones), attention in all 49
    expert_params = 47 * E * 3 * d * I
    attn = L * (d * 32 * 128 + 2 * d * 4 * 128 + 32 * 128 * d)  # 32 query / 4 key-value heads of 128
    lm = f["lm_head_params"]["vocab"] * d
    total = expert_params + attn + 2 * lm + 47 * E * d  # + input embedding and routers
    assert abs(total / f["total_params"]["value"] - 1) < f["total_params"]["rel_tol"]
    # the 49-MoE-layer stack used for the full-stack workload has the same expert budget within 1%
    assert abs(L * E * 3 * d * I / f["total_params"]["value"] - 1) < 0.01
    active = L * k * 3 * d * I + attn + lm
    assert abs(active / f["active_params"]["value"] - 1) < f["active_params"]["rel_tol"]
    assert abs(lm / f["lm_head_params"]["value"] - 1) < f["lm_head_params"]["rel_tol"]
    assert abs(lm / active / f["lm_head_share_of_active"]["value"] - 1) < f["lm_head_share_of_active"]["rel_tol"]
    # group-32 fp16 scales give 4.5 bits per weight; that matches the ~23 GB file, groups of 16 or 64 do not
    bits = lambda g: 4 + 16 / g
    gb = lambda g: f["total_params"]["value"] * bits(g) / 8 / 1e9
    assert abs(gb(group) / f["quantised_file_gb"]["value"] - 1) < f["quantised_file_gb"]["rel_tol"]
    assert abs(gb(16) / f["quantised_file_gb"]["value"] - 1) > f["quantised_file_gb"]["rel_tol"]
    assert abs(gb(64) / f["quantised_file_gb"]["value"] - 1) > f["quantised_file_gb"]["rel_tol"]
    assert abs(f["total_params"]["value"] * 2 / 1e9 / f["full_precision_gb"]["value"] - 1) < 0.02
