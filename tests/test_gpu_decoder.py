"""GPU parity of decoder layers: the pre-norm attention block (attn_decode_step_prenorm)
followed by the pre-norm MoE block (moe_forward_prenorm), the bf16 residual updated in
place, against the oracle block by block.  Each block is teacher-forced: the oracle starts
from the GPU's own residual at the block's input.  Layer 0 is a 513-token window layer
with rotary encoding, layer 1 a whole-context layer without it.

Bars: the attention block's fp32 output and the MoE block's within the layer tolerance;
expert ids exact (the oracle's choice fed to the GPU where its k-th/(k+1)-th logit gap is
below 1e-5).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import (FLINT, MAX_ABS, NEAR_TIE, REL_L2, bits_from_torch_bf16, device_drawn_layer, expert_bank, max_abs,
                     rel_l2, torch_bf16_from_bits)
from oracle import attention as A

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import bit_expert_ffn_warp_b300 as bm  # noqa: E402

SEED = 11
D, E, K, I = FLINT["d"], FLINT["E"], FLINT["k"], FLINT["I"]
NQ, NKV, L = 32, 4, 2048
KINDS = [(513, True), (0, False)]  # (window, rotary) of layers 0 and 1


def head_major(bits):
    return torch_bf16_from_bits(np.ascontiguousarray(bits.transpose(1, 0, 2))).contiguous()


def check_moe(l, moe_layer, h_in, xh_gpu, o32, ids_gpu):
    r_bits = bits_from_torch_bf16(h_in)
    x_bits = bits_from_torch_bf16(xh_gpu)
    router = {"w_router": synth.router_weight(SEED, E, D, l), "b_router": synth.router_bias(SEED, E, "normal", l)}
    res = oracle.moe_forward_touched(x_bits, r_bits, router, lambda ex: expert_bank(SEED, l, D, I, ex, E), K)
    if np.any(res["gap"] < NEAR_TIE):  # the oracle's selection, fed to the GPU from the same input
        ws = bm.moe_workspace(moe_layer, 1)
        o32 = torch.empty((1, D), dtype=torch.float32, device="cuda")
        fi = torch.from_numpy(res["ids"]).cuda()
        fw = torch.from_numpy(res["w"].astype(np.float32)).cuda()
        bm.moe_forward(xh_gpu, moe_layer, ws, residual=h_in, forced_ids=fi, forced_w=fw, out_f32=o32)
        torch.cuda.synchronize()
    else:
        assert np.array_equal(ids_gpu.cpu().numpy(), res["ids"]), f"layer {l}: expert ids"
    got = o32.cpu().numpy().astype(np.float64)
    ma, rl = max_abs(got, res["out"]), rel_l2(got, res["out"])
    assert ma <= MAX_ABS and rl <= REL_L2, f"layer {l} MoE: max-abs {ma:.3g} rel-L2 {rl:.3g}"


@pytest.mark.parametrize("pos", [300, 1500])
def test_decoder_layers_attention_then_moe(pos):
    moe = [device_drawn_layer(SEED, l, D, E, I, K) for l in range(len(KINDS))]
    at = [synth.attn_layer(SEED, D, NQ, NKV, layer=l) for l in range(len(KINDS))]
    attn = [bm.AttnLayer.from_canonical(at[l], D, NQ, NKV, window=w, rope=r) for l, (w, r) in enumerate(KINDS)]
    caches = [synth.kv_cache(SEED + 1, L, NKV, layer=l) for l in range(len(KINDS))]
    kd = [head_major(c[0]) for c in caches]
    vd = [head_major(c[1]) for c in caches]
    aws = bm.attn_workspace(attn[0], L)
    mws = bm.moe_workspace(moe[0], 1)
    resid = torch_bf16_from_bits(synth.activations(SEED, 1, D, step=pos))  # [1, D], updated in place
    for l, (window, rope) in enumerate(KINDS):
        r_in = bits_from_torch_bf16(resid)[0]
        h32 = torch.empty(D, dtype=torch.float32, device="cuda")
        bm.attn_decode_step_prenorm(resid[0], pos, attn[l], kd[l], vd[l], aws, out=resid[0], out_f32=h32)
        torch.cuda.synchronize()
        ref = A.prenorm_step(r_in, pos, at[l], caches[l][0], caches[l][1], window=window, use_rope=rope)
        got = h32.cpu().numpy().astype(np.float64)
        ma, rl = max_abs(got, ref["out"]), rel_l2(got, ref["out"])
        assert ma <= MAX_ABS and rl <= REL_L2, f"layer {l} attention: max-abs {ma:.3g} rel-L2 {rl:.3g}"
        assert np.array_equal(bits_from_torch_bf16(resid[0]), bits_from_torch_bf16(h32.to(torch.bfloat16)))
        h_in = resid.clone()
        xh = torch.empty_like(resid)
        o32 = torch.empty((1, D), dtype=torch.float32, device="cuda")
        ids = torch.empty((1, K), dtype=torch.int32, device="cuda")
        bm.moe_forward_prenorm(resid, moe[l], mws, out=resid, out_f32=o32, xh_out=xh, ids_out=ids)
        torch.cuda.synchronize()
        check_moe(l, moe[l], h_in, xh, o32, ids)
    assert bm.bitmoe_get_device_status(aws) == 0 and bm.bitmoe_get_device_status(mws) == 0


def test_prenorm_block_equals_rmsnorm_then_block():
    """attn_decode_step_prenorm gives the result of bitmoe_rmsnorm followed by attn_decode_step
    (the same normalised bf16 input), up to the norm's fp32 summation order."""
    t = synth.attn_layer(SEED + 3, D, NQ, NKV)
    kc, vc = synth.kv_cache(SEED + 4, 1024, NKV)
    lay = bm.AttnLayer.from_canonical(t, D, NQ, NKV)
    ws = bm.attn_workspace(lay, 1024)
    r = torch_bf16_from_bits(synth.activations(SEED + 5, 1, D, step=3))
    x = bm.bitmoe_rmsnorm(r)
    a32 = torch.empty(D, dtype=torch.float32, device="cuda")
    b32 = torch.empty(D, dtype=torch.float32, device="cuda")
    bm.attn_decode_step_prenorm(r[0], 700, lay, head_major(kc), head_major(vc), ws, out_f32=a32)
    bm.attn_decode_step(x[0], r[0], 700, lay, head_major(kc), head_major(vc), ws, out_f32=b32)
    torch.cuda.synchronize()
    a, b = a32.cpu().numpy(), b32.cpu().numpy()
    assert max_abs(a, b) <= 1e-3, max_abs(a, b)
