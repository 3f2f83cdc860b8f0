"""The fused decode kernel's phase trace: while a buffer is set, every CTA
writes its SM-clock stamps in phase order plus the global timer at its start;
a buffer below gridDim * 256 bytes, or none, turns the trace off."""
import numpy as np
import pytest

import synth
from helpers import FLINT, device_layer, layer_tensors, torch_bf16_from_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import bit_expert_ffn_warp_b300 as bm  # noqa: E402

# stamps every CTA reaches at batch 1, in the order a CTA passes them
ORDER = [0, 1, 16, 2, 22, 3, 10, 11, 4, 5, 23, 6, 7]


def test_trace_stamps_in_phase_order_and_off_switch():
    tensors = layer_tensors(5, FLINT["d"], FLINT["E"], FLINT["I"])
    lay = device_layer(tensors, FLINT["k"])
    x = torch_bf16_from_bits(synth.activations(7, 1, FLINT["d"]))
    ws = bm.moe_workspace(lay, 1)
    G = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(G * 32, dtype=torch.int64, device="cuda")
    try:
        bm.bitmoe_set_trace_buffer(buf)
        bm.moe_forward(x, lay, ws)
        torch.cuda.synchronize()
    finally:
        bm.bitmoe_set_trace_buffer(None)
    assert bm.bitmoe_get_device_status(ws) == 0
    t = buf.view(G, 32).cpu().numpy().astype(np.int64)
    assert np.all(t[:, 31] > 0)
    for cta in range(G):
        seq = t[cta, ORDER]
        assert np.all(seq > 0), (cta, seq)
        assert np.all(np.diff(seq) >= 0), (cta, seq)

    # off: nothing is written
    buf.zero_()
    bm.moe_forward(x, lay, ws)
    torch.cuda.synchronize()
    assert int(buf.abs().sum().item()) == 0
    # too small: skipped
    small = torch.zeros(G * 16, dtype=torch.int64, device="cuda")
    try:
        bm.bitmoe_set_trace_buffer(small)
        bm.moe_forward(x, lay, ws)
        torch.cuda.synchronize()
    finally:
        bm.bitmoe_set_trace_buffer(None)
    assert int(small.abs().sum().item()) == 0
