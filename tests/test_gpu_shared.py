"""GPU parity of the layer with an always-on shared expert beside the routed top-k
("Flint 40B : Best Mid Sized LLM", transcript 02:35: six of 256 routed experts
per token plus one shared expert), against the fp64 oracle, through the C ABI:
the fused decode kernel (T <= 8), the streaming kernels (T*kt < 512) and the
tcgen05 grouped GEMM (T*kt >= 512), plus the separate route / permute / FFN /
combine calls.  Bars as in the other parity tests: ids (with the shared
column) and the permutation bit-exact, the oracle's choice fed at near ties,
outputs within max-abs 2e-2 / rel-L2 1e-3 on the fp32 copy."""
import numpy as np
import pytest

import oracle
import synth
from helpers import MAX_ABS, NEAR_TIE, REL_L2, bits_from_torch_bf16, max_abs, rel_l2, torch_bf16_from_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import bit_expert_ffn_warp_b300 as bm  # noqa: E402

D, E, K, I = 2048, 256, 6, 512   # the pages' routing: 6 of 256 routed experts, one shared
_CACHE = {}


def shared_layer(bias="normal", seed=21):
    key = (bias, seed)
    if key not in _CACHE:
        t = synth.moe_layer_shared(seed, D, E, I, bias=bias)
        _CACHE[key] = (t, bm.MoeLayer.from_canonical(t, K))
    return _CACHE[key]


def step(x_bits, tensors, lay):
    ref = oracle.moe_forward(x_bits, tensors, K, n_shared=1)
    T = x_bits.shape[0]
    x = torch_bf16_from_bits(x_bits)
    ws = bm.moe_workspace(lay, T)
    ids = torch.empty((T, K + 1), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K + 1), dtype=torch.float32, device="cuda")
    out_f32 = torch.empty((T, D), dtype=torch.float32, device="cuda")
    kw = {}
    if np.any(ref["gap"] < NEAR_TIE):
        kw = dict(forced_ids=torch.from_numpy(ref["ids"]).cuda(),
                  forced_w=torch.from_numpy(ref["w"].astype(np.float32)).cuda())
    out, _, _, _ = bm.moe_forward(x, lay, ws, out_f32=out_f32, ids_out=ids, w_out=w, **kw)
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    g_ids = ids.cpu().numpy()
    assert np.array_equal(g_ids, ref["ids"])
    assert np.all(g_ids[:, K] == E) and np.all(w.cpu().numpy()[:, K] == 1.0)
    assert np.allclose(w.cpu().numpy(), ref["w"], rtol=1e-5, atol=1e-6)
    o32 = out_f32.cpu().numpy().astype(np.float64)
    ma, rl = max_abs(o32, ref["out"]), rel_l2(o32, ref["out"])
    assert ma <= MAX_ABS and rl <= REL_L2, f"T={T}: max-abs {ma:.3g} rel-L2 {rl:.3g}"
    assert np.array_equal(bits_from_torch_bf16(out), bits_from_torch_bf16(out_f32.to(torch.bfloat16)))
    return ref


@pytest.mark.parametrize("T", [1, 3, 8])
def test_shared_expert_fused_decode(T):
    t, lay = shared_layer()
    assert lay.n_shared == 1 and lay.kt == K + 1 and lay.Et == E + 1
    step(synth.activations(100 + T, T, D), t, lay)


@pytest.mark.parametrize("T", [16, 40])
def test_shared_expert_streaming_kernels(T):
    t, lay = shared_layer(bias="zipf")
    step(synth.activations(200 + T, T, D), t, lay)


def test_shared_expert_grouped_gemm():
    t, lay = shared_layer(bias="zipf")
    T = 160  # 1120 routed rows, a quarter of them on the shared expert
    step(synth.activations(300, T, D), t, lay)


def test_shared_expert_separate_calls():
    t, lay = shared_layer()
    T = 12
    x_bits = synth.activations(400, T, D)
    x = torch_bf16_from_bits(x_bits)
    ws = bm.moe_workspace(lay, T)
    ids, w = bm.moe_route(x, lay, ws)
    r_ids, r_w, _, gap = oracle.route(x_bits, t["w_router"], t["b_router"], K)
    sure = gap >= NEAR_TIE
    g = ids.cpu().numpy()
    assert g.shape == (T, K + 1) and np.all(g[:, K] == E) and np.all(w.cpu().numpy()[:, K] == 1.0)
    assert np.array_equal(g[sure, :K], r_ids[sure])
    # grouping over the E + 1 bank entries: the shared expert owns T rows, last
    off, rows, inv = bm.moe_permute(ids, lay, ws)
    o_off, o_rows, o_inv = oracle.permute(g, E + 1)
    assert np.array_equal(off.cpu().numpy(), o_off) and np.array_equal(rows.cpu().numpy(), o_rows)
    assert np.array_equal(inv.cpu().numpy(), o_inv)
    assert int(o_off[E + 1] - o_off[E]) == T
    y = bm.moe_expert_ffn_int4(x, lay, off, rows, ws)
    out, out_f32 = bm.moe_combine(y, inv, w, x, lay)
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    ref = oracle.moe_forward(x_bits, t, K, n_shared=1, forced_ids=g, forced_w=w.cpu().numpy().astype(np.float64))
    o32 = out_f32.cpu().numpy().astype(np.float64)
    assert max_abs(o32, ref["out"]) <= MAX_ABS and rel_l2(o32, ref["out"]) <= REL_L2


@pytest.mark.parametrize("T", [1, 8, 16, 600])
def test_dense_layer(T):
    """k = 0 with the shared expert alone: the stack's leading dense layers, on the
    fused decode kernel (T <= 8), the streaming kernels and the grouped GEMM."""
    t = synth.dense_layer(31, D, I)
    lay = bm.MoeLayer.from_canonical(t, 0)
    assert lay.E == 0 and lay.n_shared == 1 and lay.kt == 1 and lay.w_router is None
    x_bits = synth.activations(500 + T, T, D)
    ref = oracle.moe_forward(x_bits, t, 0, n_shared=1)
    x = torch_bf16_from_bits(x_bits)
    ws = bm.moe_workspace(lay, T)
    ids = torch.empty((T, 1), dtype=torch.int32, device="cuda")
    out_f32 = torch.empty((T, D), dtype=torch.float32, device="cuda")
    bm.moe_forward(x, lay, ws, out_f32=out_f32, ids_out=ids)
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    assert np.all(ids.cpu().numpy() == 0)
    o32 = out_f32.cpu().numpy().astype(np.float64)
    ma, rl = max_abs(o32, ref["out"]), rel_l2(o32, ref["out"])
    assert ma <= MAX_ABS and rl <= REL_L2, f"T={T}: max-abs {ma:.3g} rel-L2 {rl:.3g}"


@pytest.mark.parametrize("T", [1, 16])
def test_shared_expert_prenorm_step_and_graph_replay(T):
    """A pre-norm stack step on a shared-expert layer (fused at T = 1, unfused at
    T = 16): the RMSNorm'd input and the output against the oracle fed the same
    bf16 normalised rows, then the same step replayed from a CUDA graph."""
    t, lay = shared_layer()
    x_bits = synth.activations(600 + T, T, D)
    x = torch_bf16_from_bits(x_bits)
    ws = bm.moe_workspace(lay, T)
    xh = torch.empty_like(x)
    o32 = torch.empty((T, D), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, K + 1), dtype=torch.int32, device="cuda")
    out = bm.moe_forward_prenorm(x, lay, ws, out_f32=o32, xh_out=xh, ids_out=ids)
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    xh_bits = bits_from_torch_bf16(xh)
    assert np.array_equal(xh_bits, oracle.f64_to_bf16(oracle.rmsnorm(x_bits)))
    ref = oracle.moe_forward(xh_bits, t, K, resid=x_bits, n_shared=1)
    sure = ref["gap"] >= NEAR_TIE
    assert np.array_equal(ids.cpu().numpy()[sure], ref["ids"][sure])
    if np.all(sure):
        got = o32.cpu().numpy().astype(np.float64)
        assert max_abs(got, ref["out"]) <= MAX_ABS and rel_l2(got, ref["out"]) <= REL_L2
    # graph capture and replay give the same bits
    out_g = torch.empty_like(x)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bm.moe_forward_prenorm(x, lay, ws, out=out_g)
    g.replay()
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    assert torch.equal(out_g, out)
