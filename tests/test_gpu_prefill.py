"""GPU parity of the tcgen05 grouped-GEMM expert FFN (batches routing > 512 rows).

Numerics of this path: weights dequantised to fp16 RNE(q*s), activations and h
in fp16, fp32 accumulation in tensor memory.  Against the fp64 oracle the
per-row outputs agree to about 5e-4 relative (rel-L2), inside the layer
tolerance of max-abs 2e-2 and rel-L2 1e-3.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import FLINT, max_abs, rel_l2, torch_bf16_from_bits, device_layer, layer_tensors

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import bit_expert_ffn_warp_b300 as bm  # noqa: E402

_CACHE = {}


def flint(bias):
    if bias not in _CACHE:
        t = layer_tensors(11, FLINT["d"], FLINT["E"], FLINT["I"], bias=bias)
        _CACHE[bias] = (t, device_layer(t, FLINT["k"]))
    return _CACHE[bias]


U16 = 2.0 ** -11   # unit roundoff of fp16 (round to nearest)
U32 = 2.0 ** -24   # unit roundoff of fp32
F16_SUB = 2.0 ** -25  # half the spacing of fp16 subnormals


def fp16_path_error_bound(x_bits, tensors, ids):
    """First-order bound, per routed row (t, j) and output column, on |y_gpu - y_exact|
    for the fp16-operand path: every dequantised weight rounded to fp16 (relative U16),
    the tokens exact in fp16, h rounded to fp16 (relative U16, or F16_SUB absolute below
    the normal range), products exact and sums in fp32 (at most K*U32 relative to the
    sum of |terms|; taken as U16 / 4 for K = 2048 and 512).  With S(v) = sum |w_i v_i|:
      |da| <= (U16 + U16/4) S_g(x),  |du| likewise,
      |dh| <= |silu'(a) u| |da| + |silu(a)| |du| + U16 |h| + F16_SUB,
      |dy| <= sum_i |Wd_i| |dh_i| + (U16 + U16/4) S_d(|h|).
    Returned in (t, j) order; the test doubles it for higher-order terms."""
    x = oracle.bf16_to_f64(x_bits)
    T, k = ids.shape
    e_all = ids.reshape(-1)
    xr = np.repeat(x, k, axis=0)
    eps = U16 + U16 / 4
    bound = np.zeros((T * k, x.shape[1]))
    for e in np.unique(e_all):
        r = np.nonzero(e_all == e)[0]
        wg = oracle.dequant_int4(tensors["gate_q"][e], tensors["gate_s"][e])
        wu = oracle.dequant_int4(tensors["up_q"][e], tensors["up_s"][e])
        wd = oracle.dequant_int4(tensors["down_q"][e], tensors["down_s"][e])
        xe = xr[r]
        a, u = xe @ wg.T, xe @ wu.T
        da, du = eps * (np.abs(xe) @ np.abs(wg).T), eps * (np.abs(xe) @ np.abs(wu).T)
        sig = 1.0 / (1.0 + np.exp(-a))
        silu, dsilu = a * sig, sig * (1.0 + a * (1.0 - sig))
        h = silu * u
        dh = np.abs(dsilu * u) * da + np.abs(silu) * du + U16 * np.abs(h) + F16_SUB
        bound[r] = dh @ np.abs(wd).T + eps * (np.abs(h) @ np.abs(wd).T)
    return bound


@pytest.mark.parametrize("T,bias", [(65, "normal"), (300, "zipf")])
def test_grouped_gemm_expert_rows(T, bias):
    """Every y element within twice the derived first-order bound of the fp16 operand
    path (reading c.8), and rel-L2 within the layer tolerance."""
    tensors, lay = flint(bias)
    k = lay.k
    x_bits = synth.activations(70 + T, T, lay.d)
    ids, w, _, _ = oracle.route(x_bits, tensors["w_router"], tensors["b_router"], k)
    off, rows, inv = oracle.permute(ids, lay.E)
    ws = bm.moe_workspace(lay, T)
    y = bm.moe_expert_ffn_int4(torch_bf16_from_bits(x_bits), lay, torch.from_numpy(off).cuda(),
                               torch.from_numpy(rows).cuda(), ws)
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    y_ref = oracle.expert_ffn(x_bits, tensors, ids)[rows]
    yg = y.cpu().numpy().astype(np.float64)
    bound = 2.0 * fp16_path_error_bound(x_bits, tensors, ids)[rows]
    err = np.abs(yg - y_ref)
    rl, ma = rel_l2(yg, y_ref), float(err.max())
    worst = float(np.max(err / bound))
    print(f"T={T} rel-L2 {rl:.3g} max-abs {ma:.3g} worst error / bound {worst:.3g}")
    assert rl < 1e-3
    assert np.all(err <= bound), f"worst error / bound {worst:.3g}"
