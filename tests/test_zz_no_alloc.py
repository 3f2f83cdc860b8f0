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

import oracle
import synth
from tests.helpers import NEAR_TIE, max_abs, rel_l2, torch_bf16_from_bits


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


@pytest.mark.gpu
def test_static_lmhead_matches_the_oracle_at_full_vocabulary(bm):
    """The workspace-free LM head against the fp64 oracle directly, at the full
    V = 131072, two calls in a row (the second must not see the first's scratch)."""
    import torch
    d, V = 2048, 131072
    q, s = synth.lm_head(5, V, d)
    wp = bm.bitmoe_pack_int4(torch.from_numpy(q).cuda(), torch.from_numpy(s.view(np.float16)).cuda())
    for T, seed in [(1, 41), (16, 42)]:
        h_bits = synth.activations(seed, T, d)
        logits_ref, am_ref, gap = oracle.lmhead(h_bits, q, s)
        logits = torch.empty((T, V), dtype=torch.float32, device="cuda")
        am = torch.full((T,), -7, dtype=torch.int32, device="cuda")
        bm.lmhead_int4_gemv_static(torch_bf16_from_bits(h_bits), wp, V, am, logits)
        torch.cuda.synchronize()
        lg = logits.cpu().numpy().astype(np.float64)
        assert max_abs(lg, logits_ref) < 1e-3 and rel_l2(lg, logits_ref) < 1e-6
        ok = gap >= NEAR_TIE
        assert ok.any()
        assert np.array_equal(am.cpu().numpy()[ok], am_ref[ok])
