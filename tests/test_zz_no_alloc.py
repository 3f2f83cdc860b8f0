"""The LM head entry point that allocates nothing (lmhead_int4_gemv_static).

It serves callers that cannot allocate device memory, such as code inside
another runtime that owns all device memory through its own pool, or a
per-token loop that must not call cudaMalloc because it can synchronise the
device.  Its scratch is a fixed array inside the library, shared by every
call, so these tests check that a call does not see what the previous call
left there.  The file name makes pytest collect it after every other test.
"""
import ctypes

import numpy as np
import pytest

import synth
from tests.helpers import torch_bf16_from_bits


@pytest.fixture(scope="module")
def bm():
    import __graft_entry__
    __graft_entry__._load_build_module().build()
    import bit_expert_ffn_warp_b300 as m
    return m


def test_static_scratch_size_and_limit_without_gpu(bm):
    lib = bm._lib
    assert lib.lmhead_static_scratch_bytes() == 1024
    # T = 65 needs more scratch than the fixed array holds: rejected before any CUDA call
    rc = lib.lmhead_int4_gemv_static(ctypes.c_void_p(16), 65, 2048, 4096, 32, ctypes.c_void_p(16), None,
                                     ctypes.c_void_p(16), None)
    assert rc == 3 and b"workspace" in lib.bitmoe_status_string(rc).lower()
    assert lib.lmhead_int4_gemv_static(None, 0, 2048, 4096, 32, None, None, None, None) == 0
    assert lib.lmhead_int4_gemv_static(None, 4, 2048, 4096, 32, None, None, None, None) == 1


@pytest.mark.gpu
def test_static_lmhead_matches_workspace_lmhead_on_consecutive_calls(bm):
    import torch
    d, V = 2048, 32768
    q, s = synth.lm_head(21, V, d)
    wp = bm.bitmoe_pack_int4(torch.from_numpy(q).cuda(), torch.from_numpy(s.view(np.float16)).cuda())
    # consecutive calls of different sizes: each must ignore what the one before left in the shared array
    for call, (T, seed) in enumerate([(16, 31), (3, 32), (64, 33), (3, 34)]):
        h = torch_bf16_from_bits(synth.activations(seed, T, d))
        ref_logits, ref_am = bm.lmhead_int4_gemv(h, wp, V, bm.lmhead_workspace(T, d, V))
        logits = torch.full((T, V), float("nan"), dtype=torch.float32, device="cuda")
        am = torch.full((T,), -7, dtype=torch.int32, device="cuda")
        bm.lmhead_int4_gemv_static(h, wp, V, am, logits)
        am_only = torch.full((T,), -7, dtype=torch.int32, device="cuda")
        bm.lmhead_int4_gemv_static(h, wp, V, am_only)  # no logits output
        torch.cuda.synchronize()
        assert torch.equal(am, ref_am), f"call {call}: arg-max differs"
        assert torch.equal(am_only, ref_am), f"call {call}: arg-max without logits differs"
        err = float((logits - ref_logits).abs().max())
        assert err <= 1e-3, f"call {call}: logits max-abs {err}"
