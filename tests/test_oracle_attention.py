"""Pins of the attention oracle (CPU): each step against what its definition fixes,
chosen so that a dropped term, a wrong sign, index or head mapping fails one of them.

Sources: "Flint 40B : Best Mid Sized LLM", transcript 03:05 (grouped-query attention,
32 query / 4 key-value heads of 128, a 513-token sliding window on most layers,
rotary encoding there and none on full-attention layers) and 03:36 (per-head RMS norm
on queries and keys, learned attention sinks).
"""
import math

import numpy as np
import pytest

import oracle
import synth
from oracle import attention as A

HD = 128


def int4_bank(rows, K, seed):
    r = np.random.default_rng(seed)
    q = r.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    s = r.uniform(0.005, 0.02, (rows, K // 32)).astype(np.float16).view(np.uint16)
    return q, s


def small_layer(d=256, nq=4, nkv=2, seed=1, sinks=(0.5, -1.0, 2.0, 0.0)):
    wq, ws = int4_bank((nq + 2 * nkv) * HD, d, seed)
    oq, os_ = int4_bank(d, nq * HD, seed + 1)
    return dict(wqkv_q=wq, wqkv_s=ws, wo_q=oq, wo_s=os_,
                sinks=None if sinks is None else np.array(sinks[:nq], np.float32))


def caches(L, nkv, seed):
    r = np.random.default_rng(seed)
    return (synth.f64_to_bf16_bits(r.normal(0, 1, (L, nkv, HD))),
            synth.f64_to_bf16_bits(r.normal(0, 1, (L, nkv, HD))))


def test_projection_is_the_dequantised_matrix_product():
    """project() against an independent decode of the int4 bank: byte b holds element 2b
    in its low nibble and 2b + 1 in its high one, two's complement, one fp16 scale per
    32 elements of a row."""
    q, s = int4_bank(48, 256, 7)
    lo = (q & 0xF).astype(np.int64)
    hi = (q >> 4).astype(np.int64)
    vals = np.stack([lo, hi], -1).reshape(48, 256)
    vals = np.where(vals >= 8, vals - 16, vals)
    scale = np.repeat(s.view(np.float16).astype(np.float64), 32, axis=1)
    x = np.random.default_rng(8).normal(0, 1, 256)
    assert np.allclose(A.project(x, q, s), (vals * scale) @ x, rtol=1e-13, atol=1e-12)


def test_head_rmsnorm_closed_forms():
    v = np.array([np.full(HD, 3.0), np.arange(HD, dtype=np.float64) - 63.5])
    n = A.rmsnorm_heads(v, eps=1e-6)
    assert np.allclose(n[0], 1.0 / math.sqrt(1.0 + 1e-6 / 9.0), rtol=0, atol=1e-15)
    assert math.isclose(float(np.mean(n[1] ** 2)), 1.0 / (1.0 + 1e-6 / np.mean(v[1] ** 2)), rel_tol=1e-12)
    assert np.allclose(A.rmsnorm_heads(5.0 * v[1:], 0.0), A.rmsnorm_heads(v[1:], 0.0))  # scale-free


def test_rope_rotates_each_pair_by_its_angle():
    pos = 37
    for i in (0, 5, 63):
        e = np.zeros((1, HD))
        e[0, i] = 1.0
        r = A.rope(e, pos)
        ang = pos * A.ROPE_THETA ** (-2.0 * i / HD)
        want = np.zeros(HD)
        want[i], want[i + 64] = math.cos(ang), math.sin(ang)
        assert np.allclose(r[0], want, atol=1e-14)
    assert np.allclose(A.rope(np.ones((2, HD)), 0), np.ones((2, HD)))  # position 0: identity


def test_rope_keeps_norms_and_depends_on_relative_position_only():
    r = np.random.default_rng(3)
    q, k = r.normal(0, 1, (1, HD)), r.normal(0, 1, (1, HD))
    assert math.isclose(np.linalg.norm(A.rope(q, 1234)), np.linalg.norm(q), rel_tol=1e-13)
    s1 = float(np.sum(A.rope(q, 900) * A.rope(k, 650)))
    s2 = float(np.sum(A.rope(q, 900 + 77) * A.rope(k, 650 + 77)))
    s3 = float(np.sum(A.rope(q, 900) * A.rope(k, 651)))
    assert math.isclose(s1, s2, rel_tol=1e-10)
    assert not math.isclose(s1, s3, rel_tol=1e-6)


def test_single_key_returns_its_value():
    kc, vc = caches(4, 2, 5)
    kf, vf = A.bf16_bits_to_f64(kc), A.bf16_bits_to_f64(vc)
    q = np.random.default_rng(6).normal(0, 1, (4, HD))
    o = A.attend(q, kf, vf, 0, 0, None, 2)
    for h in range(4):
        assert np.array_equal(o[h], vf[0, h // 2])


def test_sink_joins_the_denominator_with_a_zero_value():
    """Equal scores (q = 0) over n keys: o = sum_j v_j / (n + e^sink)."""
    kc, vc = caches(40, 2, 9)
    kf, vf = A.bf16_bits_to_f64(kc), A.bf16_bits_to_f64(vc)
    q = np.zeros((4, HD))
    sinks = np.array([-3.0, 0.0, 1.5, 4.0])
    pos = 29
    o = A.attend(q, kf, vf, pos, 0, sinks, 2)
    for h in range(4):
        want = vf[:pos + 1, h // 2].sum(0) / (pos + 1 + math.exp(sinks[h]))
        assert np.allclose(o[h], want, rtol=1e-12, atol=1e-14)
    # a very negative sink is plain softmax attention
    assert np.allclose(A.attend(q, kf, vf, pos, 0, np.full(4, -1e4), 2), A.attend(q, kf, vf, pos, 0, None, 2))


def test_query_head_reads_its_group_kv_head():
    kc, vc = caches(30, 2, 11)
    kf, vf = A.bf16_bits_to_f64(kc), A.bf16_bits_to_f64(vc)
    vf[:, 1, :] = 0.0  # kv head 1 carries zero values
    q = np.random.default_rng(12).normal(0, 1, (4, HD))
    o = A.attend(q, kf, vf, 20, 0, None, 2)
    assert np.all(o[2:] == 0.0) and np.all(np.abs(o[:2]).max(axis=1) > 0)


def test_sliding_window_spans_the_current_token_and_512_before():
    layer = small_layer()
    kc, vc = caches(1200, 2, 13)
    x = synth.f64_to_bf16_bits(np.random.default_rng(14).normal(0, 1, 256))
    res = synth.f64_to_bf16_bits(np.random.default_rng(15).normal(0, 1, 256))
    kw = dict(n_q=4, n_kv=2)
    # below 513 tokens the window holds the whole context
    a = A.decode_step(x, res, 400, layer, kc, vc, window=513, **kw)
    b = A.decode_step(x, res, 400, layer, kc, vc, window=0, **kw)
    assert np.array_equal(a["out"], b["out"])
    # at pos = 1000 keys 488 .. 1000 count: changing key 487 changes nothing, key 488 does
    base = A.decode_step(x, res, 1000, layer, kc, vc, window=513, **kw)["o"]
    for j, moved in ((487, False), (488, True)):
        k2 = kc.copy()
        k2[j] = synth.f64_to_bf16_bits(np.full((2, HD), 3.0))
        o = A.decode_step(x, res, 1000, layer, k2, vc, window=513, **kw)["o"]
        assert (not np.array_equal(o, base)) == moved


def test_decode_step_writes_the_cache_row_and_adds_the_projection():
    layer = small_layer()
    kc, vc = caches(64, 2, 17)
    x = synth.f64_to_bf16_bits(np.random.default_rng(18).normal(0, 1, 256))
    res = synth.f64_to_bf16_bits(np.random.default_rng(19).normal(0, 1, 256))
    r = A.decode_step(x, res, 10, layer, kc, vc, window=513, n_q=4, n_kv=2)
    # v is the projection alone (no norm, no rotation), stored as bf16 at row pos
    qkv = A.project(oracle.bf16_to_f64(x), layer["wqkv_q"], layer["wqkv_s"])
    assert np.array_equal(r["v_bits"], oracle.f64_to_bf16(qkv[6 * HD:]).reshape(2, HD))
    assert np.array_equal(r["v_cache_bits"][10], r["v_bits"]) and np.array_equal(r["k_cache_bits"][10], r["k_bits"])
    assert np.array_equal(r["v_cache_bits"][:10], vc[:10])
    # k is normalised then rotated; its norm is sqrt(128) up to the bf16 rounding
    kn = np.linalg.norm(A.bf16_bits_to_f64(r["k_bits"]), axis=1)
    assert np.allclose(kn, math.sqrt(HD), rtol=1e-2)
    # a zero output projection leaves the residual
    z = dict(layer, wo_q=np.zeros_like(layer["wo_q"]))
    rz = A.decode_step(x, res, 10, z, kc, vc, window=513, n_q=4, n_kv=2)
    assert np.array_equal(rz["out"], oracle.bf16_to_f64(res))


@pytest.mark.parametrize("pos", [0, 9])
def test_rotation_applies_to_queries_and_new_keys_only_on_rope_layers(pos):
    """Without the rotary encoding q and the new key are the normalised projections; with
    it they are those rotated by the token's position (the identity at position 0)."""
    layer = small_layer(sinks=None)
    kc, vc = caches(16, 2, 21)
    x = synth.f64_to_bf16_bits(np.random.default_rng(22).normal(0, 1, 256))
    res = np.zeros(256, np.uint16)
    qkv = A.project(oracle.bf16_to_f64(x), layer["wqkv_q"], layer["wqkv_s"])
    qn = A.rmsnorm_heads(qkv[:4 * HD].reshape(4, HD))
    kn = A.rmsnorm_heads(qkv[4 * HD:6 * HD].reshape(2, HD))
    plain = A.decode_step(x, res, pos, layer, kc, vc, window=0, use_rope=False, n_q=4, n_kv=2)
    rot = A.decode_step(x, res, pos, layer, kc, vc, window=513, use_rope=True, n_q=4, n_kv=2)
    assert np.array_equal(plain["q"], qn)
    assert np.array_equal(plain["k_bits"], oracle.f64_to_bf16(kn.reshape(-1)).reshape(2, HD))
    assert np.allclose(rot["q"], A.rope(qn, pos), rtol=0, atol=0)
    assert np.array_equal(rot["q"], qn) == (pos == 0)


def test_prenorm_block_normalises_the_residual_and_adds_to_it():
    """Scaling the residual by 2 (exact in bf16) leaves the normalised input bit for bit (eps
    0: every step of the norm scales exactly), so out moves by exactly the residual; a
    constant residual normalises to ones; a zero output projection returns the residual."""
    layer = small_layer()
    kc, vc = caches(64, 2, 23)
    kw = dict(n_q=4, n_kv=2, window=0, use_rope=False)
    r = synth.f64_to_bf16_bits(np.random.default_rng(24).normal(0, 1, 256))
    r2 = synth.f64_to_bf16_bits(2.0 * A.bf16_bits_to_f64(r))
    a = A.prenorm_step(r, 20, layer, kc, vc, eps=0.0, **kw)
    b = A.prenorm_step(r2, 20, layer, kc, vc, eps=0.0, **kw)
    assert np.array_equal(a["x_bits"], b["x_bits"])
    rv, r2v = A.bf16_bits_to_f64(r), A.bf16_bits_to_f64(r2)
    assert np.array_equal(b["out"] - r2v, a["out"] - rv)
    c = A.prenorm_step(np.full(256, 0x4040, np.uint16), 20, layer, kc, vc, eps=0.0, **kw)  # 3.0
    assert np.all(c["x_bits"] == 0x3F80)  # 1.0
    z = dict(layer, wo_q=np.zeros_like(layer["wo_q"]))
    assert np.array_equal(A.prenorm_step(r, 20, z, kc, vc, **kw)["out"], rv)
    # without the norm the block would see r itself: the normalised input differs from it
    assert not np.array_equal(a["x_bits"], r)
