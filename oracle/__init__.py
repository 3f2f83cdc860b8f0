"""fp64 CPU oracle of the 4-bit (int4 or NVFP4) MoE layer and LM head (ctypes front end).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the product package.
The arithmetic lives in ``oracle.c`` (plain C, fp64, one loop per formula);
this module only moves numpy arrays across and strings the steps of the
49-layer stack together.

Sources: "Flint 40B : Best Mid Sized LLM" (video transcript, 02:35 for the
256-expert router, 03:36 and 05:39 for the 4-bit output layer) and
"Recursive_SI's First Model Unveiled!" (section "Quantization").
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_LIB = None

RMS_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-Wall",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _lib():
    global _LIB
    if _LIB is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        sig = {
            "oracle_bf16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
            "oracle_f16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
            "oracle_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
            "oracle_dequant_int4": (ctypes.c_int, [P, P, I64, I64, I64, P]),
            "oracle_router_logits": (ctypes.c_int, [P, I64, I64, I64, P, P, P]),
            "oracle_softmax": (ctypes.c_int, [P, I64, I64, P]),
            "oracle_topk": (ctypes.c_int, [P, I64, I64, I64, P, P]),
            "oracle_gates": (ctypes.c_int, [P, P, I64, I64, I64, ctypes.c_int, P]),
            "oracle_route": (ctypes.c_int, [P, I64, I64, I64, I64, P, P, ctypes.c_int, P, P, P, P]),
            "oracle_permute": (ctypes.c_int, [P, I64, I64, I64, P, P, P]),
            "oracle_expert_ffn": (ctypes.c_int, [P, I64, I64, I64, I64, I64, I64, P, P, P, P, P, P, P, P, P]),
            "oracle_combine": (ctypes.c_int, [P, P, P, I64, I64, I64, P]),
            "oracle_moe_forward": (ctypes.c_int, [P, P, I64, I64, I64, I64, I64, I64, I64, ctypes.c_int, P,
                                                  P, P, P, P, P, P, P, P, P, P, P, P, P]),
            "oracle_rmsnorm": (ctypes.c_int, [P, I64, I64, ctypes.c_double, P]),
            "oracle_lmhead": (ctypes.c_int, [P, I64, I64, I64, I64, P, P, P, P, P]),
            "oracle_num_threads": (ctypes.c_int, []),
            "oracle_e2m1_to_f64": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_e4m3_to_f64": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_dequant_nvfp4": (ctypes.c_int, [P, P, ctypes.c_float, I64, I64, P]),
            "oracle_expert_ffn_nvfp4": (ctypes.c_int, [P, I64, I64, I64, I64, I64, P, P, P, P, P, P, P, P, P, P,
                                                       P, P]),
            "oracle_moe_forward_nvfp4": (ctypes.c_int, [P, P, I64, I64, I64, I64, I64, I64, ctypes.c_int, P, P,
                                                        P, P, P, P, P, P, P, P, P, P, P, P, P, P, P]),
            "oracle_lmhead_nvfp4": (ctypes.c_int, [P, I64, I64, I64, P, P, ctypes.c_float, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments (rc={rc})")


def num_threads() -> int:
    return int(_lib().oracle_num_threads())


# ---------------------------------------------------------------- formats


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    f = np.vectorize(_lib().oracle_bf16_to_f64, otypes=[np.float64])
    return f(np.asarray(bits, np.uint16))


def f16_to_f64(bits: np.ndarray) -> np.ndarray:
    f = np.vectorize(_lib().oracle_f16_to_f64, otypes=[np.float64])
    return f(np.asarray(bits, np.uint16))


def f64_to_bf16(v: np.ndarray) -> np.ndarray:
    """Nearest-even bf16 bits of fp64 values."""
    f = np.vectorize(_lib().oracle_f64_to_bf16, otypes=[np.uint16])
    return f(np.asarray(v, np.float64))


def dequant_int4(q: np.ndarray, s: np.ndarray, group: int = 32) -> np.ndarray:
    q = _c(q, np.uint8)
    s = _c(s, np.uint16)
    rows = q.shape[0] if q.ndim > 1 else 1
    K = q.shape[-1] * 2
    rows = q.size // (K // 2)
    out = np.empty((rows, K), np.float64)
    _check(_lib().oracle_dequant_int4(_p(q), _p(s), rows, K, group, _p(out)), "dequant_int4")
    return out.reshape(q.shape[:-1] + (K,))


def e2m1_to_f64(codes: np.ndarray) -> np.ndarray:
    """Values of FP4 E2M1 codes (the low nibble of each uint8)."""
    f = np.vectorize(_lib().oracle_e2m1_to_f64, otypes=[np.float64])
    return f(np.asarray(codes, np.uint8) & np.uint8(15))


def e4m3_to_f64(b: np.ndarray) -> np.ndarray:
    """Values of FP8 E4M3 bytes (NaN for the two NaN codes)."""
    f = np.vectorize(_lib().oracle_e4m3_to_f64, otypes=[np.float64])
    return f(np.asarray(b, np.uint8))


def dequant_nvfp4(q: np.ndarray, s: np.ndarray, ts: float) -> np.ndarray:
    """One NVFP4 matrix: q [rows, K/2] codes, s [rows, K/16] E4M3 bytes, ts fp32."""
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    rows, K = q.shape[0], q.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    _check(_lib().oracle_dequant_nvfp4(_p(q), _p(s), float(np.float32(ts)), rows, K, _p(out)), "dequant_nvfp4")
    return out


def is_nvfp4(layer: dict) -> bool:
    """A layer dict whose expert banks are NVFP4 (codes *_q, E4M3 *_s, fp32 tensor scales *_ts)."""
    return "gate_ts" in layer


def _nvfp4_args(layer):
    out = []
    for n in ("gate", "up", "down"):
        out += [_c(layer[n + "_q"], np.uint8), _c(layer[n + "_s"], np.uint8), _c(layer[n + "_ts"], np.float32)]
    return out


# ---------------------------------------------------------------- routing


def router_logits(x, w_router, b_router=None):
    x = _c(x, np.uint16)
    Wr = _c(w_router, np.float32)
    b = _c(b_router, np.float32)
    T, d = x.shape
    E = Wr.shape[0]
    out = np.empty((T, E), np.float64)
    _check(_lib().oracle_router_logits(_p(x), T, d, E, _p(Wr), _p(b), _p(out)), "router_logits")
    return out


def softmax(logits):
    l = _c(logits, np.float64)
    T, E = l.shape
    out = np.empty_like(l)
    _check(_lib().oracle_softmax(_p(l), T, E, _p(out)), "softmax")
    return out


def topk(logits, k):
    l = _c(logits, np.float64)
    T, E = l.shape
    ids = np.empty((T, k), np.int32)
    gap = np.empty(T, np.float64)
    _check(_lib().oracle_topk(_p(l), T, E, k, _p(ids), _p(gap)), "topk")
    return ids, gap


def gates(p, ids, renorm=True):
    p = _c(p, np.float64)
    ids = _c(ids, np.int32)
    T, E = p.shape
    k = ids.shape[1]
    w = np.empty((T, k), np.float64)
    _check(_lib().oracle_gates(_p(p), _p(ids), T, E, k, int(renorm), _p(w)), "gates")
    return w


def route(x, w_router, b_router, k, renorm=True):
    """Returns (ids [T,k] int32, w [T,k] fp64, logits [T,E] fp64, gap [T] fp64)."""
    x = _c(x, np.uint16)
    Wr = _c(w_router, np.float32)
    b = _c(b_router, np.float32)
    T, d = x.shape
    E = Wr.shape[0]
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    logits = np.empty((T, E), np.float64)
    gap = np.empty(T, np.float64)
    _check(_lib().oracle_route(_p(x), T, d, E, k, _p(Wr), _p(b), int(renorm), _p(ids), _p(w), _p(logits),
                               _p(gap)), "route")
    return ids, w, logits, gap


def permute(ids, E):
    """Returns (offsets [E+1], sorted_rows [T*k], inv [T*k]) as int32."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, np.int32)
    sorted_rows = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    _check(_lib().oracle_permute(_p(ids), T, E, k, _p(offsets), _p(sorted_rows), _p(inv)), "permute")
    return offsets, sorted_rows, inv


# ---------------------------------------------------------------- experts


def expert_ffn(x, layer, ids, group=32, want_h=False):
    """y [T*k, d] fp64 in (t, j) order (and h [T*k, I] when want_h)."""
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    T, d = x.shape
    k = ids.shape[1]
    gq = _c(layer["gate_q"], np.uint8)
    E, I = gq.shape[0], gq.shape[1]
    y = np.empty((T * k, d), np.float64)
    h = np.empty((T * k, I), np.float64) if want_h else None
    if is_nvfp4(layer):
        args = _nvfp4_args(layer)
        _check(_lib().oracle_expert_ffn_nvfp4(_p(x), T, d, I, E, k, *[_p(a) for a in args], _p(ids), _p(y), _p(h)),
               "expert_ffn_nvfp4")
        return (y, h) if want_h else y
    args = [_c(layer[n], np.uint8 if n.endswith("_q") else np.uint16)
            for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")]
    _check(_lib().oracle_expert_ffn(_p(x), T, d, I, E, k, group, *[_p(a) for a in args], _p(ids), _p(y), _p(h)),
           "expert_ffn")
    return (y, h) if want_h else y


def combine(y, w, resid):
    y = _c(y, np.float64)
    w = _c(w, np.float64)
    resid = _c(resid, np.uint16)
    T, d = resid.shape
    k = w.shape[1]
    out = np.empty((T, d), np.float64)
    _check(_lib().oracle_combine(_p(y), _p(w), _p(resid), T, d, k, _p(out)), "combine")
    return out


def moe_forward(x, layer, k, resid=None, group=32, renorm=True, forced_ids=None, forced_w=None, n_shared=0):
    """One MoE layer. Returns dict(out fp64 [T,d], ids, w, gap).

    n_shared = 1: the banks hold E + 1 experts, the last being the shared
    expert that every token uses with weight 1 after its k routed ones; ids
    and w (and forced_ids / forced_w) then have k + 1 columns.  k = 0 with
    n_shared = 1 is a dense SwiGLU layer (no router).
    """
    x = _c(x, np.uint16)
    resid = x if resid is None else _c(resid, np.uint16)
    T, d = x.shape
    gq = layer["gate_q"]
    E, I = gq.shape[0] - n_shared, gq.shape[1]
    Wr = _c(layer.get("w_router"), np.float32)
    b = _c(layer.get("b_router"), np.float32)
    if Wr is None and forced_ids is None and k > 0:
        raise ValueError("moe_forward: router weights are needed unless the selection is forced")
    fi = _c(forced_ids, np.int32)
    fw = _c(forced_w, np.float64)
    ids = np.empty((T, k + n_shared), np.int32)
    w = np.empty((T, k + n_shared), np.float64)
    gap = np.empty(T, np.float64)
    out = np.empty((T, d), np.float64)
    if is_nvfp4(layer):
        args = _nvfp4_args(layer)
        _check(_lib().oracle_moe_forward_nvfp4(_p(x), _p(resid), T, d, E, k, n_shared, I, int(renorm), _p(Wr), _p(b),
                                               *[_p(a) for a in args], _p(fi), _p(fw), _p(ids), _p(w), _p(gap),
                                               _p(out)), "moe_forward_nvfp4")
    else:
        args = [_c(layer[n], np.uint8 if n.endswith("_q") else np.uint16)
                for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")]
        _check(_lib().oracle_moe_forward(_p(x), _p(resid), T, d, E, k, n_shared, I, group, int(renorm), _p(Wr),
                                         _p(b), *[_p(a) for a in args], _p(fi), _p(fw), _p(ids), _p(w), _p(gap),
                                         _p(out)), "moe_forward")
    return {"out": out, "ids": ids, "w": w, "gap": gap}


def rmsnorm(x, eps=RMS_EPS):
    x = _c(x, np.uint16)
    T, d = x.shape
    y = np.empty((T, d), np.float64)
    _check(_lib().oracle_rmsnorm(_p(x), T, d, float(eps), _p(y)), "rmsnorm")
    return y


def lmhead(h, q, s, group=32, want_logits=True):
    """Returns (logits [T,V] fp64 or None, argmax [T] int32, gap [T] fp64)."""
    h = _c(h, np.uint16)
    q = _c(q, np.uint8)
    s = _c(s, np.uint16)
    T, d = h.shape
    V = q.shape[0]
    logits = np.empty((T, V), np.float64) if want_logits else None
    am = np.empty(T, np.int32)
    gap = np.empty(T, np.float64)
    _check(_lib().oracle_lmhead(_p(h), T, d, V, group, _p(q), _p(s), _p(logits), _p(am), _p(gap)), "lmhead")
    return logits, am, gap


def lmhead_nvfp4(h, q, s, ts, want_logits=True):
    """NVFP4 LM head: q [V, d/2] codes, s [V, d/16] E4M3, ts fp32.  Returns (logits, argmax, gap)."""
    h = _c(h, np.uint16)
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    T, d = h.shape
    V = q.shape[0]
    logits = np.empty((T, V), np.float64) if want_logits else None
    am = np.empty(T, np.int32)
    gap = np.empty(T, np.float64)
    _check(_lib().oracle_lmhead_nvfp4(_p(h), T, d, V, _p(q), _p(s), float(np.float32(ts)), _p(logits), _p(am),
                                      _p(gap)), "lmhead_nvfp4")
    return logits, am, gap


# ---------------------------------------------------------------- the stack


def moe_forward_touched(xh, resid, router, expert_fn, k, group=32, renorm=True, forced=None):
    """One MoE layer that draws only the experts its tokens select.

    ``router`` holds w_router / b_router; ``expert_fn(list_of_experts)`` returns
    gate/up/down banks holding just those experts, in that order.  The result
    equals ``moe_forward`` on the full bank (the unselected experts never enter
    the sums).  ``forced`` = (ids, w) feeds a given selection instead of routing.
    """
    if forced is None:
        ids, w, _, gap = route(xh, router["w_router"], router["b_router"], k, renorm)
    else:
        ids, w = np.asarray(forced[0], np.int32), np.asarray(forced[1], np.float64)
        gap = np.full(ids.shape[0], np.nan)
    uniq = np.unique(ids)
    bank = expert_fn([int(e) for e in uniq])
    local = np.searchsorted(uniq, ids).astype(np.int32)
    res = moe_forward(xh, bank, k, resid=resid, group=group, renorm=renorm, forced_ids=local, forced_w=w)
    return {"out": res["out"], "ids": ids, "w": w, "gap": gap}


def stack_forward(x0, router_fn, expert_fn, n_layers, k, lm_q, lm_s, group=32, renorm=True, forced=None):
    """Decode stack of MoE layers with attention replaced by identity.

    resid_0 = x0 (bf16).  For each layer l: xh = bf16(RMSNorm(resid_l));
    resid_{l+1} = bf16(resid_l + MoE_l(xh)).  Then xh = bf16(RMSNorm(resid_L)),
    logits = LM-head(xh) and the argmax.  ``router_fn(l)`` gives layer l's
    router tensors, ``expert_fn(l, experts)`` its selected experts; ``forced``
    maps a layer index to an (ids, w) selection fed to that layer.
    """
    resid = np.ascontiguousarray(x0, np.uint16)
    per_layer = []
    for l in range(n_layers):
        xh = f64_to_bf16(rmsnorm(resid))
        router = router_fn(l)
        own_ids, _, _, own_gap = route(xh, router["w_router"], router["b_router"], k, renorm)
        f = forced.get(l) if forced is not None else None
        res = moe_forward_touched(xh, resid, router, lambda ex, l=l: expert_fn(l, ex), k, group, renorm, f)
        per_layer.append({"xh": xh, "ids": own_ids, "gap": own_gap, "used_ids": res["ids"], "w": res["w"],
                          "out": res["out"], "resid_in": resid})
        resid = f64_to_bf16(res["out"])
    xh = f64_to_bf16(rmsnorm(resid))
    logits, am, gap = lmhead(xh, lm_q, lm_s, group)
    return {"layers": per_layer, "resid": resid, "xh": xh, "logits": logits, "argmax": am, "gap": gap}
