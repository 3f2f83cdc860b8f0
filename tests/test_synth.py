"""The seeded input generator: published SplitMix64 values, value ranges, slicing."""
import numpy as np

import synth


def test_splitmix64_matches_published_sequence():
    # SplitMix64 seeded with 0 (Steele, Lea and Flood; the reference C code by
    # Vigna): first outputs from state 0.
    expected = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = synth.hash_words(0, 0, 3)
    assert [int(v) for v in got] == expected


def test_int4_bytes_are_uniform_nibbles_and_sliceable():
    key = synth.stream_key(0, synth.TAG["gate_q"], 3)
    full = synth.int4_bytes(key, 0, 1 << 16)
    lo, hi = full & 0xF, full >> 4
    for nib in (lo, hi):
        counts = np.bincount(nib, minlength=16)
        assert counts.min() > 0.9 * len(nib) / 16 and counts.max() < 1.1 * len(nib) / 16
    for a, n in [(0, 1), (3, 17), (1001, 4096), (65535, 1)]:
        assert np.array_equal(synth.int4_bytes(key, a, n), full[a:a + n])


def test_scales_range_and_slices():
    key = synth.stream_key(1, synth.TAG["up_s"], 0)
    s = synth.f16_scales(key, 0, 50000).view(np.float16).astype(np.float64)
    # U(0.005, 0.02) rounded to fp16: within half an fp16 ulp of the interval
    assert s.min() >= 0.005 - 2 ** -19 and s.max() <= 0.02 + 2 ** -17
    assert abs(s.mean() - 0.0125) < 2e-4
    assert np.array_equal(synth.f16_scales(key, 123, 77), synth.f16_scales(key, 0, 200)[123:])


def test_layer_slices_equal_full_bank():
    full = synth.moe_layer(2, 256, 8, 128)
    part = synth.moe_layer(2, 256, 8, 128, experts=(3, 6))
    for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        assert np.array_equal(part[n], full[n][3:6])
    q, s = synth.lm_head(2, 64, 256)
    q2, s2 = synth.lm_head(2, 64, 256, rows=(16, 48))
    assert np.array_equal(q2, q[16:48]) and np.array_equal(s2, s[16:48])


def test_normals_and_bf16_storage():
    x = synth.activations(0, 64, 2048)
    v = synth.bf16_bits_to_f32(x).astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1) < 0.01
    # stored values are bf16: the low 16 bits of the fp32 pattern are zero, and rounding was to nearest
    raw = np.random.Generator(np.random.PCG64(np.random.SeedSequence([0, synth.TAG["x"], 0, 0]))).standard_normal((64, 2048))
    assert np.all(np.abs(v - raw) <= np.abs(raw) * 2.0 ** -8)
    w = synth.router_weight(0, 256, 2048)
    assert abs(w.std() * np.sqrt(2048) - 1) < 0.01


def test_zipf_bias_is_a_permuted_log_zipf_law():
    E = 256
    b = synth.router_bias(0, E, "zipf").astype(np.float64)
    p = np.sort(np.exp(b))[::-1]
    r = np.arange(1, E + 1)
    assert abs(p.sum() - 1) < 1e-5
    assert np.allclose(p[0] / p, r ** 1.1, rtol=1e-5)


def test_nvfp4_draws_codes_scales_and_tensor_scales():
    key = synth.stream_key(4, synth.TAG["down_fs"], 1)
    s = synth.e4m3_scale_bytes(key, 0, 1 << 15)
    counts = np.bincount(s, minlength=256)[0x58:0x68]
    assert counts.sum() == len(s) and counts.min() > 0.9 * len(s) / 16
    assert np.array_equal(synth.e4m3_scale_bytes(key, 100, 50), s[100:150])
    ts = synth.f32_tensor_scales(synth.stream_key(4, synth.TAG["gate_ts"], 0), 0, 4096)
    assert ts.dtype == np.float32 and ts.min() >= 2.0 ** -12 and ts.max() <= 2.0 ** -11
    full = synth.moe_layer_nvfp4(5, 256, 8, 128)
    part = synth.moe_layer_nvfp4(5, 256, 8, 128, experts=(2, 7))
    for n in ("gate_q", "gate_s", "gate_ts", "up_q", "up_s", "up_ts", "down_q", "down_s", "down_ts"):
        assert np.array_equal(part[n], full[n][2:7])
    assert full["gate_s"].shape == (8, 128, 16) and full["down_s"].shape == (8, 256, 8)
    q, s2, t = synth.lm_head_nvfp4(5, 64, 256)
    q2, s3, t2 = synth.lm_head_nvfp4(5, 64, 256, rows=(16, 48))
    assert np.array_equal(q2, q[16:48]) and np.array_equal(s3, s2[16:48]) and t == t2
