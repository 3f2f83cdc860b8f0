"""The C-ABI library loads, exports every symbol include/bitmoe.h declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bitmoe.h")
LIB = os.path.join(ROOT, "bit_expert_ffn_warp_b300", "libbitmoe.so")


@pytest.fixture(scope="module")
def built():
    import __graft_entry__
    __graft_entry__._load_build_module().build()
    assert os.path.exists(LIB)
    return LIB


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[a-z_][\w\s\*]*?\b([a-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_six_path_calls():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_expert_ffn_int4", "moe_combine", "moe_forward", "lmhead_int4_gemv"):
        assert n in names


def test_library_exports_every_declared_symbol(built):
    out = subprocess.run(["nm", "-D", "--defined-only", built], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(built)
    for n in declared_functions():
        assert hasattr(lib, n)


def test_binding_wraps_every_declared_symbol(built):
    import bit_expert_ffn_warp_b300 as bm
    assert sorted(bm.EXPORTED) == declared_functions()


def test_host_side_validation_without_gpu(built):
    import bit_expert_ffn_warp_b300 as bm
    lib = bm._lib
    sh = bm.MoeShape(2048, 256, 8, 512, 32, 1)
    ws = lib.moe_workspace_size(ctypes.byref(sh), 1)
    assert ws > 0
    # the workspace grows with T and covers the per-row buffers
    assert lib.moe_workspace_size(ctypes.byref(sh), 64) > ws
    assert lib.moe_workspace_size(ctypes.byref(sh), 4096) >= 4096 * 8 * 2048 * 4
    bad = [bm.MoeShape(2048, 256, 0, 512, 32, 1), bm.MoeShape(2048, 4, 8, 512, 32, 1),
           bm.MoeShape(2048, 256, 33, 512, 32, 1)]
    for b in bad:
        assert lib.moe_workspace_size(ctypes.byref(b), 1) == 0
    assert lib.moe_workspace_size(ctypes.byref(bm.MoeShape(2000, 256, 8, 512, 32, 1)), 1) == 0
    assert lib.moe_workspace_size(ctypes.byref(bm.MoeShape(2048, 256, 8, 512, 64, 1)), 1) == 0
    # the shared expert adds a bank entry and a row per token; it fills padding of the struct
    assert ctypes.sizeof(bm.MoeShape) == 48
    shared = lib.moe_workspace_size(ctypes.byref(bm.MoeShape(2048, 256, 6, 512, 32, 1, 1)), 64)
    assert shared > lib.moe_workspace_size(ctypes.byref(bm.MoeShape(2048, 256, 6, 512, 32, 1, 0)), 64)
    assert lib.moe_workspace_size(ctypes.byref(bm.MoeShape(2048, 256, 6, 512, 32, 1, 2)), 1) == 0
    assert lib.moe_workspace_size(ctypes.byref(bm.MoeShape(2048, 256, 32, 512, 32, 1, 1)), 1) == 0
    assert lib.moe_workspace_size(ctypes.byref(bm.MoeShape(2048, 1024, 8, 512, 32, 1, 1)), 1) == 0
    # a dense layer: no routed experts, the shared one alone
    assert lib.moe_workspace_size(ctypes.byref(bm.MoeShape(2048, 0, 0, 512, 32, 1, 1)), 4) > 0
    assert lib.moe_workspace_size(ctypes.byref(bm.MoeShape(2048, 0, 0, 512, 32, 1, 0)), 4) == 0
    assert lib.moe_workspace_size(ctypes.byref(bm.MoeShape(2048, 0, 2, 512, 32, 1, 1)), 4) == 0
    # null pointers -> INVALID_ARG, nothing launched
    rc = lib.moe_route(None, 1, ctypes.byref(sh), None, None, None, None, None, None, 0, None)
    assert rc == 1
    wt = bm.MoeWeights(None, None, None, None, None)
    rc = lib.moe_forward(None, None, 1, ctypes.byref(sh), ctypes.byref(wt), None, None, None, None, None, None,
                         None, 0, None)
    assert rc == 1
    # forced ids without forced gates -> INVALID_ARG
    rc = lib.moe_forward(None, None, 1, ctypes.byref(sh), ctypes.byref(wt), ctypes.c_void_p(16), None, None, None,
                         None, None, None, 0, None)
    assert rc == 1
    # unsupported shapes
    assert lib.bitmoe_packed_int4_bytes(1, 15, 2048, 32) == 0
    assert lib.bitmoe_packed_int4_bytes(1, 16, 2000, 32) == 0
    assert lib.bitmoe_packed_int4_bytes(256, 512, 2048, 32) == 256 * 512 * 2048 * 9 // 16
    assert lib.lmhead_int4_gemv(None, 65, 2048, 131072, 32, None, None, None, None, 0, None) == 2
    assert lib.lmhead_int4_gemv(None, 1, 2048, 131072, 16, None, None, None, None, 0, None) == 2
    # T = 0 is a no-op that succeeds
    assert lib.moe_forward(None, None, 0, ctypes.byref(sh), ctypes.byref(wt), None, None, None, None, None, None,
                           None, 0, None) == 0
    for code in range(7):
        assert lib.bitmoe_status_string(code)


def test_nvfp4_host_side_validation_without_gpu(built):
    import bit_expert_ffn_warp_b300 as bm
    lib = bm._lib
    assert lib.bitmoe_packed_nvfp4_bytes(256, 512, 2048) == 256 * 512 * 2048 * 9 // 16
    assert lib.bitmoe_packed_nvfp4_bytes(1, 15, 2048) == 0 and lib.bitmoe_packed_nvfp4_bytes(1, 16, 2000) == 0
    assert lib.bitmoe_pack_nvfp4(None, None, 1, 16, 128, None, None) == 1
    sh16 = bm.MoeShape(2048, 256, 8, 512, 16, 1)  # the NVFP4 block as the scale group
    sh32 = bm.MoeShape(2048, 256, 8, 512, 32, 1)
    assert lib.moe_workspace_size(ctypes.byref(sh16), 8) == lib.moe_workspace_size(ctypes.byref(sh32), 8)
    w4 = bm.MoeWeightsNvfp4(None, None, None, None, None, None, None, None)
    wi = bm.MoeWeights(None, None, None, None, None)
    args = (None, None, None, None, None, None, None, 0, None)
    # each format's calls take only their own scale group
    assert lib.moe_forward_nvfp4(None, None, 1, ctypes.byref(sh32), ctypes.byref(w4), *args) == 2
    assert lib.moe_forward(None, None, 1, ctypes.byref(sh16), ctypes.byref(wi), *args) == 2
    assert lib.moe_forward_nvfp4(None, None, 1, ctypes.byref(sh16), ctypes.byref(w4), *args) == 1
    assert lib.moe_expert_ffn_nvfp4(None, 1, ctypes.byref(sh16), ctypes.byref(w4), None, None, None, None, 0,
                                    None) == 1
    assert lib.moe_expert_ffn_int4(None, 1, ctypes.byref(sh16), ctypes.byref(wi), None, None, None, None, 0,
                                   None) == 2
    assert lib.moe_forward_nvfp4(None, None, 0, ctypes.byref(sh16), ctypes.byref(w4), *args) == 0
    # the NVFP4 LM head: T and shape limits as the int4 one, a finite tensor scale
    assert lib.lmhead_nvfp4_gemv(None, 65, 2048, 131072, None, 1.0, None, None, None, 0, None) == 2
    assert lib.lmhead_nvfp4_gemv(None, 1, 2048, 131072, None, float("nan"), None, None, None, 0, None) == 1
    assert lib.lmhead_nvfp4_gemv(None, 0, 2048, 131072, None, 1.0, None, None, None, 0, None) == 0


def test_stack_call_rejects_on_the_host_without_gpu(built):
    """moe_stack_decode: argument and shape checks that return before any launch."""
    import bit_expert_ffn_warp_b300 as bm
    lib = bm._lib
    sh = bm.MoeShape(2048, 256, 8, 512, 32, 1)
    ws_bytes = lib.moe_stack_workspace_size(ctypes.byref(sh), 1)
    assert ws_bytes == lib.moe_workspace_size(ctypes.byref(sh), 1) + 256
    fake = ctypes.c_void_p(1 << 20)  # 16-byte aligned stand-in, never dereferenced on these paths
    w = bm.MoeWeights(1 << 20, 1 << 20, 1 << 20, 1 << 20, None)
    arr = (bm.MoeWeights * 65)(*([w] * 65))
    call = lambda T, n, ws=fake, nb=ws_bytes, V=0, lm=None, am=None: lib.moe_stack_decode(
        fake, T, ctypes.byref(sh), arr, n, 1e-6, lm, V, None, am, None, ws, nb, None)
    assert call(0, 1) == 0                   # no tokens: nothing to do
    assert call(1, 0) == 1                   # no layers
    assert call(9, 2) == 2                   # T > 8: not the fused decode kernel's shapes
    assert call(1, 65) == 2                  # more layers than the launch carries
    assert call(1, 2, V=100, lm=fake, am=fake) == 2  # V % 16 != 0
    assert call(1, 2, lm=fake, am=None, V=4096) == 1  # an LM head needs the arg-max output
    assert call(1, 2, nb=ws_bytes - 1) == 3  # workspace too small
    bad = (bm.MoeWeights * 2)(w, bm.MoeWeights(1 << 20, None, 1 << 20, 1 << 20, None))
    assert lib.moe_stack_decode(fake, 1, ctypes.byref(sh), bad, 2, 1e-6, None, 0, None, None, None, fake,
                                ws_bytes, None) == 1


def test_attention_calls_reject_on_the_host_without_gpu(built):
    """attn_workspace_size / attn_decode_step / attn_decode_step_prenorm: shapes the kernels
    are not built for size no workspace, and every call below fails a check that returns
    before any launch."""
    import bit_expert_ffn_warp_b300 as bm
    lib = bm._lib
    S = lambda d=2048, nq=32, nkv=4, hd=128, L=4096, w=513, rope=1, eps=1e-6, th=1e6: bm.AttnShape(  # noqa: E731
        d, nq, nkv, hd, L, w, rope, eps, th)
    n = lib.attn_workspace_size(ctypes.byref(S()))
    assert n >= 32 * 128 * 132 * 4  # the split records of every query head
    assert lib.attn_workspace_size(ctypes.byref(S(L=131072))) == n  # independent of the cache length
    for bad in (S(hd=64), S(nq=16), S(d=2000), S(d=32768), S(w=-1), S(L=0), S(eps=-1.0), S(th=0.0),
                S(L=(1 << 31) + 1)):
        assert lib.attn_workspace_size(ctypes.byref(bad)) == 0
    assert lib.attn_workspace_size(ctypes.byref(S(rope=0, th=0.0))) == n  # no rotary: theta unused
    fake = ctypes.c_void_p(1 << 20)  # 16-byte aligned stand-in, never dereferenced on these paths
    odd = ctypes.c_void_p((1 << 20) + 2)
    w = bm.AttnWeights(1 << 20, 1 << 20, None)
    sh = S()

    def step(x=fake, r=fake, pos=10, k=fake, v=fake, out=fake, ws=fake, nb=n, shape=sh, wts=w):
        return lib.attn_decode_step(x, r, pos, ctypes.byref(shape), ctypes.byref(wts), k, v, out, None, ws, nb,
                                    None)

    def pre(r=fake, pos=10, nb=n):
        return lib.attn_decode_step_prenorm(r, pos, ctypes.byref(sh), ctypes.byref(w), fake, fake, fake, None, fake,
                                            nb, None)
    assert step(pos=4096) == 1 and step(pos=-1) == 1        # outside the cache
    assert step(x=None) == 1 and step(k=None) == 1 and step(out=None) == 1
    assert step(x=odd) == 1 and step(v=odd) == 1            # not 16-byte aligned
    assert step(nb=n - 1) == 3 and step(ws=None) == 3       # workspace too small or absent
    assert step(shape=S(hd=64)) == 2                        # a shape the kernels are not built for
    assert step(wts=bm.AttnWeights(1 << 20, None, None)) == 1
    assert pre(pos=4096) == 1 and pre(r=None) == 1 and pre(nb=n - 1) == 3
