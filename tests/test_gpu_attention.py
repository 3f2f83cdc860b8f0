"""GPU parity of the attention decode step (attn_decode_step, through the C ABI)
against the fp64 oracle (oracle/attention.py) on seeded synthetic weights and caches.

Bars: the layer output within max-abs 2e-2 and rel-L2 1e-3 on the fp32 copy, whose
bf16 rounding is the bf16 output bit for bit; the cache rows other than pos untouched;
the new key and value rows (fp32 on the GPU, fp64 in the oracle, both rounded once to
bf16) equal to the oracle's except where the two sides round a value within their
difference of a bf16 rounding boundary (at most one ulp apart, at most 1% of elements).
"""
import numpy as np
import pytest

import synth
from helpers import MAX_ABS, REL_L2, bits_from_torch_bf16, max_abs, rel_l2, torch_bf16_from_bits
from oracle import attention as A

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import bit_expert_ffn_warp_b300 as bm  # noqa: E402

D, NQ, NKV, L = 2048, 32, 4, 4608


def run_step(pos, window, rope, sinks, seed=3, L=L, dims=(D, NQ, NKV)):
    d, nq, nkv = dims
    t = synth.attn_layer(seed, d, nq, nkv, sinks=sinks)
    kc, vc = synth.kv_cache(seed + 1, L, nkv)
    x = synth.activations(seed + 2, 1, d, step=pos)[0]
    res = synth.activations(seed + 3, 1, d, step=pos)[0]
    ref = A.decode_step(x, res, pos, t, kc, vc, window=window, use_rope=rope, n_q=nq, n_kv=nkv)
    lay = bm.AttnLayer.from_canonical(t, d, nq, nkv, window=window, rope=rope)
    # the oracle keeps [position, head, 128]; the library's cache is head-major
    kd = torch_bf16_from_bits(np.ascontiguousarray(kc.transpose(1, 0, 2))).contiguous()
    vd = torch_bf16_from_bits(np.ascontiguousarray(vc.transpose(1, 0, 2))).contiguous()
    ws = bm.attn_workspace(lay, L)
    out_f32 = torch.empty(d, dtype=torch.float32, device="cuda")
    out = bm.attn_decode_step(torch_bf16_from_bits(x), torch_bf16_from_bits(res), pos, lay, kd, vd, ws,
                              out_f32=out_f32)
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    return (ref, kc, vc, out, out_f32, bits_from_torch_bf16(kd).transpose(1, 0, 2),
            bits_from_torch_bf16(vd).transpose(1, 0, 2))


def close_bf16_rows(got, want):
    ulp = np.abs(A.bf16_bits_to_f64(want)) * 2.0 ** -7 + 1e-30
    diff = np.abs(A.bf16_bits_to_f64(got) - A.bf16_bits_to_f64(want))
    assert np.all(diff <= ulp * 1.01)
    assert np.mean(got != want) <= 0.01


def check_step(pos, window, rope, sinks, L=L, dims=(D, NQ, NKV)):
    ref, kc, vc, out, out_f32, kd, vd = run_step(pos, window, rope, sinks, L=L, dims=dims)
    o32 = out_f32.cpu().numpy().astype(np.float64)
    ma, rl = max_abs(o32, ref["out"]), rel_l2(o32, ref["out"])
    assert ma <= MAX_ABS and rl <= REL_L2, f"max-abs {ma:.3g} rel-L2 {rl:.3g}"
    assert np.array_equal(bits_from_torch_bf16(out), bits_from_torch_bf16(out_f32.to(torch.bfloat16)))
    keep = np.ones(L, bool)
    keep[pos] = False
    assert np.array_equal(kd[keep], kc[keep]) and np.array_equal(vd[keep], vc[keep])
    close_bf16_rows(kd[pos], ref["k_bits"])
    close_bf16_rows(vd[pos], ref["v_bits"])


@pytest.mark.parametrize("pos,window,rope,sinks", [
    (0, 513, True, True),      # one key: the current token's own
    (7, 513, True, True),
    (255, 0, False, True),     # chunk edges of the split kernel (256 positions)
    (256, 0, False, True),
    (600, 513, True, True),    # the window has left the first 88 tokens behind
    (600, 0, False, True),
    (1000, 513, True, False),  # no sinks: the plain softmax
    (4500, 0, False, True),    # 18 chunks of the whole context
])
def test_attention_decode_step_matches_the_oracle(pos, window, rope, sinks):
    check_step(pos, window, rope, sinks)


@pytest.mark.parametrize("window,rope", [(0, False), (513, True)])
def test_attention_at_long_context(window, rope):
    """40001 positions: each warp of the split kernel runs nine 16-position tiles through
    its three-stage ring (the wrap-around), and the rotation angle reaches 4e4 radians."""
    check_step(40000, window, rope, True, L=40960)


@pytest.mark.parametrize("dims,pos,window,rope", [
    ((2048, 64, 8), 3000, 0, False),  # Wo has K = 8192: each projection warp takes two batches of chunks
    ((1024, 16, 2), 2500, 513, True),  # two key/value heads: a finer split plan
])
def test_attention_other_head_counts(dims, pos, window, rope):
    check_step(pos, window, rope, True, L=3072, dims=dims)


def head_major(bits):
    return torch_bf16_from_bits(np.ascontiguousarray(bits.transpose(1, 0, 2))).contiguous()


def test_consecutive_steps_cross_the_window_edge():
    """Positions 510 .. 514 in a row with a 513-token window: each step attends over the rows
    the GPU wrote in the steps before it (the oracle chains its own cache), and the window's
    first row moves from 0 to 2.  The last step, captured in a CUDA graph and replayed,
    gives the eager result bit for bit."""
    L2 = 1024
    t = synth.attn_layer(5, D, NQ, NKV)
    kref, vref = synth.kv_cache(6, L2, NKV)
    lay = bm.AttnLayer.from_canonical(t, D, NQ, NKV, window=513, rope=True)
    kd, vd = head_major(kref), head_major(vref)
    ws = bm.attn_workspace(lay, L2)
    for pos in range(510, 515):
        x = synth.activations(7, 1, D, step=pos)[0]
        res = synth.activations(8, 1, D, step=pos)[0]
        ref = A.decode_step(x, res, pos, t, kref, vref, window=513, use_rope=True)
        kref, vref = ref["k_cache_bits"], ref["v_cache_bits"]
        xg, rg = torch_bf16_from_bits(x), torch_bf16_from_bits(res)
        out_f32 = torch.empty(D, dtype=torch.float32, device="cuda")
        out = bm.attn_decode_step(xg, rg, pos, lay, kd, vd, ws, out_f32=out_f32)
        torch.cuda.synchronize()
        o32 = out_f32.cpu().numpy().astype(np.float64)
        ma, rl = max_abs(o32, ref["out"]), rel_l2(o32, ref["out"])
        assert ma <= MAX_ABS and rl <= REL_L2, f"pos {pos}: max-abs {ma:.3g} rel-L2 {rl:.3g}"
    assert bm.bitmoe_get_device_status(ws) == 0
    eager = bits_from_torch_bf16(out)
    g = torch.cuda.CUDAGraph()
    out2 = torch.empty_like(out)
    with torch.cuda.graph(g):
        bm.attn_decode_step(xg, rg, 514, lay, kd, vd, ws, out=out2)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits_from_torch_bf16(out2), eager)


def test_attention_step_rejects_positions_outside_the_cache():
    t = synth.attn_layer(3, D, NQ, NKV)
    lay = bm.AttnLayer.from_canonical(t, D, NQ, NKV)
    kd = torch.zeros((NKV, 64, 128), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros_like(kd)
    ws = bm.attn_workspace(lay, 64)
    x = torch.zeros(D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bm.BitmoeError) as e:
        bm.attn_decode_step(x, x, 64, lay, kd, vd, ws)
    assert e.value.code == bm.ERR_INVALID_ARG
    small = bm.attn_workspace(lay, 64)[:128]
    with pytest.raises(bm.BitmoeError) as e:
        bm.attn_decode_step(x, x, 3, lay, kd, vd, small)
    assert e.value.code == bm.ERR_WORKSPACE
