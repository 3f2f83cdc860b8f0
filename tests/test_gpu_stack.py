"""GPU parity of the 49-layer decode stack (pre-norm MoE layer steps, residual in
bf16; attention replaced by identity) followed by the int4 LM head and its arg-max.

Every checked layer is teacher-forced: the oracle starts from the GPU's own bf16
residual at that layer's input, so the check measures that layer alone and not
the drift of 49 roundings.  Bars as for a single layer: RMSNorm output within one
bf16 step of the oracle's rounding, expert ids exact (the oracle's choice fed to
both sides where its k-th/(k+1)-th logit gap is below 1e-5), the fp32 copy of the
layer output within max-abs 2e-2 / rel-L2 1e-3, and the arg-max exact unless the
oracle's top-2 gap is below 1e-5.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import (FLINT, MAX_ABS, NEAR_TIE, REL_L2, bf16_bits_to_f64, bf16_ulp, bits_from_torch_bf16,
                     device_drawn_layer, device_drawn_lm_head, expert_bank, max_abs, rel_l2, torch_bf16_from_bits)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import bit_expert_ffn_warp_b300 as bm  # noqa: E402

SEED = 5
N_LAYERS = 49
V = 131072
D, E, K, I = FLINT["d"], FLINT["E"], FLINT["k"], FLINT["I"]

_STACK = {}


def stack():
    if "layers" not in _STACK:
        _STACK["layers"] = [device_drawn_layer(SEED, l, D, E, I, K) for l in range(N_LAYERS)]
        _STACK["lm"] = device_drawn_lm_head(SEED, V, D)
        torch.cuda.synchronize()
    return _STACK["layers"], _STACK["lm"]


def run_stack(x_bits):
    layers, lm = stack()
    T = x_bits.shape[0]
    ws = bm.moe_workspace(layers[0], T)
    resid = torch_bf16_from_bits(x_bits)
    xh = torch.empty_like(resid)
    rec = []
    for l in range(N_LAYERS):
        resid_in = resid.clone()
        xh_l = torch.empty_like(resid)
        o32 = torch.empty((T, D), dtype=torch.float32, device="cuda")
        ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
        bm.moe_forward_prenorm(resid, layers[l], ws, out=resid, out_f32=o32, xh_out=xh_l, ids_out=ids)
        rec.append((resid_in, xh_l, o32, ids))
    bm.bitmoe_rmsnorm(resid, out=xh)
    _, am = bm.lmhead_int4_gemv(xh, lm, V, bm.lmhead_workspace(T, D, V), want_logits=False)
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    _STACK["last_resid"] = resid.clone()
    return rec, xh.clone(), am


def check_layer(l, resid_in, xh_gpu, o32, ids_gpu):
    layers, _ = stack()
    r_bits = bits_from_torch_bf16(resid_in)
    x_bits = bits_from_torch_bf16(xh_gpu)
    # RMSNorm: the GPU's bf16 output is the oracle's rounding, or one bf16 step away at a boundary
    ref_xh = oracle.rmsnorm(r_bits)
    xv = bf16_bits_to_f64(x_bits)
    assert np.all(np.abs(xv - ref_xh) <= bf16_ulp(ref_xh)), f"layer {l}: RMSNorm"
    assert np.mean(x_bits == oracle.f64_to_bf16(ref_xh)) >= 0.99, f"layer {l}: RMSNorm rounding"
    # the layer itself, from the GPU's own input
    router = {"w_router": synth.router_weight(SEED, E, D, l), "b_router": synth.router_bias(SEED, E, "normal", l)}
    res = oracle.moe_forward_touched(x_bits, r_bits, router, lambda ex: expert_bank(SEED, l, D, I, ex, E), K)
    near = bool(np.any(res["gap"] < NEAR_TIE))
    if near:  # re-run this layer with the oracle's selection fed to the GPU
        T = x_bits.shape[0]
        ws = bm.moe_workspace(layers[l], T)
        o32 = torch.empty((T, D), dtype=torch.float32, device="cuda")
        fi = torch.from_numpy(res["ids"]).cuda()
        fw = torch.from_numpy(res["w"].astype(np.float32)).cuda()
        bm.moe_forward(xh_gpu, layers[l], ws, residual=resid_in, forced_ids=fi, forced_w=fw, out_f32=o32)
        torch.cuda.synchronize()
    else:
        assert np.array_equal(ids_gpu.cpu().numpy(), res["ids"]), f"layer {l}: expert ids"
    got = o32.cpu().numpy().astype(np.float64)
    ma, rl = max_abs(got, res["out"]), rel_l2(got, res["out"])
    assert ma <= MAX_ABS and rl <= REL_L2, f"layer {l}: max-abs {ma:.3g} rel-L2 {rl:.3g}"
    return near


@pytest.mark.parametrize("T,checked", [(1, list(range(N_LAYERS))), (16, list(range(N_LAYERS)))])
def test_stack_teacher_forced_and_lm_head(T, checked):
    x0 = synth.activations(SEED, T, D, step=T)
    rec, xh_final, am = run_stack(x0)
    near = [l for l in checked if check_layer(l, *rec[l])]
    q, s = synth.lm_head(SEED, V, D)
    _, ref_am, gap = oracle.lmhead(bits_from_torch_bf16(xh_final), q, s, want_logits=False)
    sure = gap >= NEAR_TIE
    assert np.array_equal(am.cpu().numpy()[sure], ref_am[sure])
    print(f"stack T={T}: {len(checked)} layers checked, near-tie layers {near}, "
          f"arg-max exempt tokens {int((~sure).sum())}")


@pytest.mark.parametrize("T", [1, 5, 16])
def test_prenorm_step_equals_rmsnorm_then_layer(T):
    """moe_forward_prenorm gives the bits of bitmoe_rmsnorm followed by moe_forward."""
    layers, _ = stack()
    lay = layers[3]
    x = torch_bf16_from_bits(synth.activations(SEED + 7, T, D, step=T))
    ws = bm.moe_workspace(lay, T)
    xh_a = torch.empty_like(x)
    o_a = torch.empty((T, D), dtype=torch.float32, device="cuda")
    out_a = bm.moe_forward_prenorm(x, lay, ws, out_f32=o_a, xh_out=xh_a)
    xh_b = bm.bitmoe_rmsnorm(x)
    o_b = torch.empty((T, D), dtype=torch.float32, device="cuda")
    out_b, _, _, _ = bm.moe_forward(xh_b, lay, ws, residual=x, out_f32=o_b)
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    assert torch.equal(xh_a, xh_b)
    assert torch.equal(out_a, out_b) and torch.equal(o_a, o_b)


# ------------------------------------------------------------------ one launch for the whole stack


@pytest.mark.parametrize("T", [1, 4])
def test_fused_stack_kernel_equals_layer_steps(T):
    """moe_stack_decode (49 layers + RMSNorm + LM head in one launch) gives the bits
    of the per-layer calls: every layer's expert ids, the final residual and the
    arg-max -- the per-layer path being the one checked against the oracle above."""
    layers, lm = stack()
    x0 = synth.activations(SEED + 11, T, D, step=T)
    rec, _, am_ref = run_stack(x0)
    resid_ref = _STACK["last_resid"]
    resid = torch_bf16_from_bits(x0)
    ws = bm.moe_stack_workspace(layers[0], T)
    ids = torch.full((N_LAYERS, T, K), -7, dtype=torch.int32, device="cuda")
    logits = torch.empty((T, V), dtype=torch.float32, device="cuda")
    _, am = bm.moe_stack_decode(resid, layers, ws, lm_w=lm, V=V, ids_out=ids, logits=logits)
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    for l in range(N_LAYERS):
        assert torch.equal(ids[l], rec[l][3]), f"layer {l}: expert ids"
    assert torch.equal(resid, resid_ref)
    assert torch.equal(am, am_ref)
    # the logits it wrote are the LM head's on the final normalised residual
    xh = bm.bitmoe_rmsnorm(resid_ref)
    ref_logits, _ = bm.lmhead_int4_gemv(xh, lm, V, bm.lmhead_workspace(T, D, V))
    torch.cuda.synchronize()
    assert torch.equal(logits, ref_logits)


def test_fused_stack_kernel_few_layers_repeated_without_lm_head():
    """Three layers, no LM head, two calls in a row on one workspace (the grid-barrier
    counter and the barriers' phases carry over): the residual of each call equals
    the per-layer steps'."""
    layers, _ = stack()
    sub = layers[10:13]
    T = 2
    ws = bm.moe_stack_workspace(sub[0], T)
    ws_l = bm.moe_workspace(sub[0], T)
    for call in range(2):
        x0 = synth.activations(SEED + 20 + call, T, D, step=call)
        ref = torch_bf16_from_bits(x0)
        for lay in sub:
            bm.moe_forward_prenorm(ref, lay, ws_l, out=ref)
        resid = torch_bf16_from_bits(x0)
        bm.moe_stack_decode(resid, sub, ws)
        torch.cuda.synchronize()
        assert bm.bitmoe_get_device_status(ws) == 0
        assert torch.equal(resid, ref), f"call {call}"
