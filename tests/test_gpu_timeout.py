"""A bounded device wait that runs out reports BITMOE_ERR_TIMEOUT and leaves the
context usable.

The fused decode kernel joins its CTAs with a grid barrier on an arrival
counter in the workspace (bytes 64..67); a launch expects that counter to start
at a multiple of the grid size.  Presetting it to 1 makes one CTA's arrival aim
at a count that no CTA will ever produce (a flag that nothing sets): its wait
gives up after the kernel's limit (about 2 s), records the timeout in the
status word and the CTA leaves.  Nothing faults or traps.  Reading the status
with clear=1 resets the status and the counter, and the next launch is exact.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import FLINT, MAX_ABS, NEAR_TIE, REL_L2, device_layer, layer_tensors, max_abs, rel_l2, \
    torch_bf16_from_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import bit_expert_ffn_warp_b300 as bm  # noqa: E402

BITMOE_ERR_TIMEOUT = 5


def test_grid_barrier_wait_runs_out_and_reports_timeout():
    tensors = layer_tensors(41, FLINT["d"], FLINT["E"], FLINT["I"])
    lay = device_layer(tensors, FLINT["k"])
    x_bits = synth.activations(43, 1, FLINT["d"])
    x = torch_bf16_from_bits(x_bits)
    ws = bm.moe_workspace(lay, 1)
    assert bm.bitmoe_get_device_status(ws) == 0

    ws[64:68] = torch.tensor([1, 0, 0, 0], dtype=torch.uint8, device="cuda")  # arrival counter = 1
    bm.moe_forward(x, lay, ws)
    torch.cuda.synchronize()  # the launch ends: the stuck wait gave up
    assert bm.bitmoe_get_device_status(ws, clear=True) == BITMOE_ERR_TIMEOUT

    # status and counter are clear again; the same layer step is exact
    assert bm.bitmoe_get_device_status(ws) == 0
    ref = oracle.moe_forward(x_bits, tensors, FLINT["k"])
    forced = {}
    if np.any(ref["gap"] < NEAR_TIE):  # feed the oracle's choice at a near tie
        forced = dict(forced_ids=torch.from_numpy(ref["ids"]).cuda(),
                      forced_w=torch.from_numpy(ref["w"].astype(np.float32)).cuda())
    out_f32 = torch.empty((1, FLINT["d"]), dtype=torch.float32, device="cuda")
    bm.moe_forward(x, lay, ws, out_f32=out_f32, **forced)
    torch.cuda.synchronize()
    assert bm.bitmoe_get_device_status(ws) == 0
    got = out_f32.cpu().numpy().astype(np.float64)
    assert max_abs(got, ref["out"]) <= MAX_ABS and rel_l2(got, ref["out"]) <= REL_L2
