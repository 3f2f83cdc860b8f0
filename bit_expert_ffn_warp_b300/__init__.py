"""Python binding of the bitmoe C ABI (include/bitmoe.h): argument marshalling only.

Every function here takes torch CUDA tensors, checks dtypes and shapes, and
calls the entry point of the same name in ``libbitmoe.so`` on the current
torch stream.  All arithmetic runs in the library's CUDA kernels; there is no
fallback.  If the library is missing the import fails.

Tensor formats: activations bf16 ``[T, d]``; router weight fp32 ``[E, d]``,
bias fp32 ``[E]``; int4 banks are packed with :func:`bitmoe_pack_int4` from the
canonical ``q uint8 [n, rows, K/2]`` + ``scale fp16 [n, rows, K/32]``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbitmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"bitmoe CUDA library not built: {LIB_PATH} (run __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA", 5: "TIMEOUT",
                6: "DEVICE_CHECK"}
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE = 3
ERR_TIMEOUT = 5
ERR_DEVICE_CHECK = 6
GROUP = 32


class BitmoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = _lib.bitmoe_status_string(code).decode()
        extra = f" (cuda error {_lib.bitmoe_last_cuda_error()})" if code == 4 else ""
        super().__init__(f"{fn}: {STATUS_NAMES.get(code, code)}: {msg}{extra}")
        self.code = code


class MoeShape(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int64), ("E", ctypes.c_int64), ("k", ctypes.c_int64), ("I", ctypes.c_int64),
                ("group", ctypes.c_int64), ("renormalize", ctypes.c_int32), ("n_shared", ctypes.c_int32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("w_router", ctypes.c_void_p), ("b_router", ctypes.c_void_p)]


class MoeWeightsNvfp4(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("gate_scale", ctypes.c_void_p), ("up_scale", ctypes.c_void_p), ("down_scale", ctypes.c_void_p),
                ("w_router", ctypes.c_void_p), ("b_router", ctypes.c_void_p)]


FP4_BLOCK = 16


class AttnShape(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int64), ("n_q_heads", ctypes.c_int64), ("n_kv_heads", ctypes.c_int64),
                ("head_dim", ctypes.c_int64), ("max_len", ctypes.c_int64), ("window", ctypes.c_int64),
                ("rope", ctypes.c_int32), ("eps", ctypes.c_float), ("rope_theta", ctypes.c_double)]


class AttnWeights(ctypes.Structure):
    _fields_ = [("wqkv", ctypes.c_void_p), ("wo", ctypes.c_void_p), ("sinks", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_SIGS = {
    "bitmoe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "bitmoe_last_cuda_error": (ctypes.c_int, []),
    "bitmoe_version": (ctypes.c_char_p, []),
    "bitmoe_set_trace_buffer": (ctypes.c_int, [_P, _SZ]),
    "bitmoe_packed_int4_bytes": (_SZ, [_I64, _I64, _I64, _I64]),
    "bitmoe_pack_int4": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, _P, _P]),
    "bitmoe_packed_nvfp4_bytes": (_SZ, [_I64, _I64, _I64]),
    "bitmoe_pack_nvfp4": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P, _P]),
    "bitmoe_get_device_status": (ctypes.c_int, [_P, ctypes.c_int, ctypes.POINTER(ctypes.c_int32), _P]),
    "moe_workspace_size": (_SZ, [ctypes.POINTER(MoeShape), _I64]),
    "moe_route": (ctypes.c_int, [_P, _I64, ctypes.POINTER(MoeShape), _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute": (ctypes.c_int, [_P, _I64, ctypes.POINTER(MoeShape), _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_ffn_int4": (ctypes.c_int, [_P, _I64, ctypes.POINTER(MoeShape), ctypes.POINTER(MoeWeights), _P, _P,
                                           _P, _P, _SZ, _P]),
    "moe_combine": (ctypes.c_int, [_P, _P, _P, _P, _I64, ctypes.POINTER(MoeShape), _P, _P, _P]),
    "moe_forward": (ctypes.c_int, [_P, _P, _I64, ctypes.POINTER(MoeShape), ctypes.POINTER(MoeWeights), _P, _P, _P,
                                   _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_nvfp4": (ctypes.c_int, [_P, _P, _I64, ctypes.POINTER(MoeShape), ctypes.POINTER(MoeWeightsNvfp4), _P,
                                         _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_ffn_nvfp4": (ctypes.c_int, [_P, _I64, ctypes.POINTER(MoeShape), ctypes.POINTER(MoeWeightsNvfp4), _P,
                                            _P, _P, _P, _SZ, _P]),
    "moe_forward_prenorm": (ctypes.c_int, [_P, _I64, _P, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                           _P]),
    "moe_stack_workspace_size": (_SZ, [ctypes.POINTER(MoeShape), _I64]),
    "moe_stack_decode": (ctypes.c_int, [_P, _I64, ctypes.POINTER(MoeShape), _P, _I64, ctypes.c_float, _P, _I64, _P,
                                        _P, _P, _P, _SZ, _P]),
    "lmhead_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "lmhead_int4_gemv": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _SZ, _P]),
    "lmhead_nvfp4_gemv": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, ctypes.c_float, _P, _P, _P, _SZ, _P]),
    "lmhead_static_scratch_bytes": (_SZ, []),
    "lmhead_int4_gemv_static": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _P, _P, _P, _P]),
    "bitmoe_rmsnorm": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_float, _P, _P]),
    "attn_workspace_size": (_SZ, [ctypes.POINTER(AttnShape)]),
    "attn_decode_step": (ctypes.c_int, [_P, _P, _I64, ctypes.POINTER(AttnShape), ctypes.POINTER(AttnWeights), _P,
                                        _P, _P, _P, _P, _SZ, _P]),
    "attn_decode_step_prenorm": (ctypes.c_int, [_P, _I64, ctypes.POINTER(AttnShape), ctypes.POINTER(AttnWeights),
                                                _P, _P, _P, _P, _P, _SZ, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


def _check(fn: str, rc: int) -> None:
    if rc != OK:
        raise BitmoeError(fn, rc)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t, dtype, shape, name):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def version() -> str:
    return _lib.bitmoe_version().decode()


def bitmoe_set_trace_buffer(buf) -> None:
    """Turn the fused-decode phase trace on (a uint64 CUDA tensor) or off (None)."""
    if buf is None:
        _check("bitmoe_set_trace_buffer", _lib.bitmoe_set_trace_buffer(None, 0))
    else:
        _check("bitmoe_set_trace_buffer", _lib.bitmoe_set_trace_buffer(_ptr(buf), buf.numel() * buf.element_size()))


# ---------------------------------------------------------------- weights


def bitmoe_packed_int4_bytes(n_mats: int, rows: int, K: int, group: int = GROUP) -> int:
    return int(_lib.bitmoe_packed_int4_bytes(n_mats, rows, K, group))


def bitmoe_pack_int4(q: torch.Tensor, scale: torch.Tensor, group: int = GROUP) -> torch.Tensor:
    """Canonical bank q uint8 [n, rows, K/2] + scale fp16 [n, rows, K/group] -> packed uint8 tiles."""
    if q.dim() == 2:
        q, scale = q.unsqueeze(0), scale.unsqueeze(0)
    n, rows, kh = q.shape
    K = kh * 2
    _need(q, torch.uint8, (n, rows, kh), "q")
    _need(scale, torch.float16, (n, rows, K // group), "scale")
    nbytes = bitmoe_packed_int4_bytes(n, rows, K, group)
    if nbytes == 0:
        raise BitmoeError("bitmoe_pack_int4", 2)
    out = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check("bitmoe_pack_int4", _lib.bitmoe_pack_int4(_ptr(q), _ptr(scale), n, rows, K, group, _ptr(out), _stream()))
    return out


def bitmoe_pack_nvfp4(q: torch.Tensor, scale: torch.Tensor) -> torch.Tensor:
    """Canonical NVFP4 bank q uint8 [n, rows, K/2] (E2M1 codes) + scale uint8
    [n, rows, K/16] (E4M3 bytes) -> packed uint8 tiles."""
    if q.dim() == 2:
        q, scale = q.unsqueeze(0), scale.unsqueeze(0)
    n, rows, kh = q.shape
    K = kh * 2
    _need(q, torch.uint8, (n, rows, kh), "q")
    _need(scale, torch.uint8, (n, rows, K // 16), "scale")
    nbytes = int(_lib.bitmoe_packed_nvfp4_bytes(n, rows, K))
    if nbytes == 0:
        raise BitmoeError("bitmoe_pack_nvfp4", 2)
    out = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check("bitmoe_pack_nvfp4", _lib.bitmoe_pack_nvfp4(_ptr(q), _ptr(scale), n, rows, K, _ptr(out), _stream()))
    return out


@dataclass
class MoeLayer:
    """Device-resident weights of one MoE layer (packed banks + fp32 router).

    E routed experts, k of them per token; with n_shared = 1 the banks hold one
    more expert (entry E), the shared expert every token uses with weight 1, and
    the per-token arrays have kt = k + 1 entries, the shared one last.  k = 0
    (with n_shared = 1) is a dense SwiGLU layer: no router, w_router None.
    """
    d: int
    E: int
    k: int
    I: int
    gate: torch.Tensor
    up: torch.Tensor
    down: torch.Tensor
    w_router: torch.Tensor | None
    b_router: torch.Tensor | None
    renormalize: bool = True
    n_shared: int = 0
    # NVFP4 banks: fp32 tensor scales [Et] (device); None for int4 banks
    gate_ts: torch.Tensor | None = None
    up_ts: torch.Tensor | None = None
    down_ts: torch.Tensor | None = None

    @property
    def nvfp4(self) -> bool:
        return self.gate_ts is not None

    @property
    def kt(self) -> int:
        """Rows per token: the routed experts, then the shared one."""
        return self.k + self.n_shared

    @property
    def Et(self) -> int:
        """Bank entries: the routed experts, then the shared one."""
        return self.E + self.n_shared

    @property
    def shape(self) -> MoeShape:
        return MoeShape(self.d, self.E, self.k, self.I, FP4_BLOCK if self.nvfp4 else GROUP, int(self.renormalize),
                        int(self.n_shared))

    @property
    def weights(self):
        wr = None if self.w_router is None else self.w_router.data_ptr()
        br = None if self.b_router is None else self.b_router.data_ptr()
        if self.nvfp4:
            return MoeWeightsNvfp4(self.gate.data_ptr(), self.up.data_ptr(), self.down.data_ptr(),
                                   self.gate_ts.data_ptr(), self.up_ts.data_ptr(), self.down_ts.data_ptr(), wr, br)
        return MoeWeights(self.gate.data_ptr(), self.up.data_ptr(), self.down.data_ptr(), wr, br)

    @classmethod
    def from_canonical(cls, tensors: dict, k: int, device="cuda", renormalize: bool = True) -> "MoeLayer":
        """Build from host/device canonical tensors (gate_q/gate_s/.../w_router/b_router);
        NVFP4 banks when the tensors carry gate_ts/up_ts/down_ts (then *_s are E4M3 bytes)."""
        if "gate_ts" in tensors:
            return cls._from_canonical_nvfp4(tensors, k, device, renormalize)

        def dev(name, dtype):
            t = tensors[name]
            if not isinstance(t, torch.Tensor):
                t = torch.from_numpy(t)
            if dtype == torch.float16 and t.dtype != torch.float16:
                t = t.view(torch.float16) if t.dtype in (torch.int16, torch.uint16) else t.to(torch.float16)
            return t.to(device=device).contiguous()
        gq, gs = dev("gate_q", torch.uint8), dev("gate_s", torch.float16)
        Et, I, dh = gq.shape
        d = dh * 2
        if k == 0:  # dense layer: the bank's one entry is the shared expert
            E = Et - 1
        else:
            E = tensors["w_router"].shape[0] if tensors.get("w_router") is not None else Et
        if Et - E not in (0, 1):
            raise ValueError("the banks hold the routed experts plus at most one shared expert")
        b = tensors.get("b_router")
        wr = tensors.get("w_router")
        return cls(
            d=d, E=E, k=k, I=I, n_shared=Et - E,
            gate=bitmoe_pack_int4(gq, gs),
            up=bitmoe_pack_int4(dev("up_q", torch.uint8), dev("up_s", torch.float16)),
            down=bitmoe_pack_int4(dev("down_q", torch.uint8), dev("down_s", torch.float16)),
            w_router=None if wr is None else dev("w_router", torch.float32),
            b_router=None if b is None else dev("b_router", torch.float32),
            renormalize=renormalize)

    @classmethod
    def _from_canonical_nvfp4(cls, tensors: dict, k: int, device, renormalize: bool) -> "MoeLayer":
        def dev(name, dtype):
            t = tensors[name]
            if not isinstance(t, torch.Tensor):
                t = torch.as_tensor(t)
            return t.to(device=device, dtype=dtype).contiguous()
        packed, ts = {}, {}
        for n in ("gate", "up", "down"):
            packed[n] = bitmoe_pack_nvfp4(dev(n + "_q", torch.uint8), dev(n + "_s", torch.uint8))
            ts[n] = dev(n + "_ts", torch.float32)
        Et, I, dh = tensors["gate_q"].shape
        wr, b = tensors.get("w_router"), tensors.get("b_router")
        E = Et - 1 if k == 0 else (wr.shape[0] if wr is not None else Et)
        if Et - E not in (0, 1):
            raise ValueError("the banks hold the routed experts plus at most one shared expert")
        return cls(d=dh * 2, E=E, k=k, I=I, n_shared=Et - E, gate=packed["gate"], up=packed["up"],
                   down=packed["down"], w_router=None if wr is None else dev("w_router", torch.float32),
                   b_router=None if b is None else dev("b_router", torch.float32), renormalize=renormalize,
                   gate_ts=ts["gate"], up_ts=ts["up"], down_ts=ts["down"])


def moe_workspace_size(layer_or_shape, T: int) -> int:
    sh = layer_or_shape.shape if isinstance(layer_or_shape, MoeLayer) else layer_or_shape
    return int(_lib.moe_workspace_size(ctypes.byref(sh), T))


def moe_workspace(layer: MoeLayer, T: int) -> torch.Tensor:
    """A zero-filled workspace for calls on up to T tokens (its status word starts clear)."""
    n = moe_workspace_size(layer, T)
    if n == 0:
        raise BitmoeError("moe_workspace_size", 2)
    return torch.zeros(n, dtype=torch.uint8, device=layer.gate.device)


def bitmoe_get_device_status(workspace: torch.Tensor, clear: bool = False) -> int:
    out = ctypes.c_int32(0)
    _check("bitmoe_get_device_status",
           _lib.bitmoe_get_device_status(_ptr(workspace), int(clear), ctypes.byref(out), _stream()))
    return out.value


# ---------------------------------------------------------------- MoE layer entry points


def moe_route(x, layer: MoeLayer, workspace, want_logits: bool = False):
    T = x.shape[0]
    _need(x, torch.bfloat16, (T, layer.d), "x")
    ids = torch.empty((T, layer.kt), dtype=torch.int32, device=x.device)
    w = torch.empty((T, layer.kt), dtype=torch.float32, device=x.device)
    logits = torch.empty((T, layer.E), dtype=torch.float32, device=x.device) if want_logits else None
    sh = layer.shape
    _check("moe_route", _lib.moe_route(_ptr(x), T, ctypes.byref(sh), _ptr(layer.w_router), _ptr(layer.b_router),
                                       _ptr(ids), _ptr(w), _ptr(logits), _ptr(workspace), workspace.numel(),
                                       _stream()))
    return (ids, w, logits) if want_logits else (ids, w)


def moe_permute(ids, layer: MoeLayer, workspace):
    T = ids.shape[0]
    _need(ids, torch.int32, (T, layer.kt), "ids")
    dev = ids.device
    offsets = torch.empty(layer.Et + 1, dtype=torch.int32, device=dev)
    rows = torch.empty(T * layer.kt, dtype=torch.int32, device=dev)
    inv = torch.empty(T * layer.kt, dtype=torch.int32, device=dev)
    sh = layer.shape
    _check("moe_permute", _lib.moe_permute(_ptr(ids), T, ctypes.byref(sh), _ptr(offsets), _ptr(rows), _ptr(inv),
                                           _ptr(workspace), workspace.numel(), _stream()))
    return offsets, rows, inv


def moe_expert_ffn_int4(x, layer: MoeLayer, offsets, sorted_rows, workspace, y_out=None):
    """Expert FFNs of the grouped rows (int4 banks; NVFP4 layers go to moe_expert_ffn_nvfp4)."""
    return _expert_ffn(x, layer, offsets, sorted_rows, workspace, y_out, False)


def moe_expert_ffn_nvfp4(x, layer: MoeLayer, offsets, sorted_rows, workspace, y_out=None):
    """Expert FFNs of the grouped rows over NVFP4 banks."""
    return _expert_ffn(x, layer, offsets, sorted_rows, workspace, y_out, True)


def _expert_ffn(x, layer, offsets, sorted_rows, workspace, y_out, nvfp4):
    if layer.nvfp4 != nvfp4:
        raise ValueError("the layer's banks are " + ("NVFP4" if layer.nvfp4 else "int4"))
    T = x.shape[0]
    _need(x, torch.bfloat16, (T, layer.d), "x")
    _need(offsets, torch.int32, (layer.Et + 1,), "offsets")
    _need(sorted_rows, torch.int32, (T * layer.kt,), "sorted_rows")
    if y_out is None:
        y = torch.empty((T * layer.kt, layer.d), dtype=torch.float32, device=x.device)
    else:
        y = _need(y_out, torch.float32, (T * layer.kt, layer.d), "y_out")
    sh, wt = layer.shape, layer.weights
    name = "moe_expert_ffn_nvfp4" if layer.nvfp4 else "moe_expert_ffn_int4"
    _check(name, getattr(_lib, name)(_ptr(x), T, ctypes.byref(sh), ctypes.byref(wt), _ptr(offsets),
                                     _ptr(sorted_rows), _ptr(y), _ptr(workspace), workspace.numel(), _stream()))
    return y


def moe_combine(y_rows, inv_rows, topk_w, residual, layer: MoeLayer, out=None, want_f32: bool = True):
    T = residual.shape[0]
    _need(residual, torch.bfloat16, (T, layer.d), "residual")
    out = torch.empty_like(residual) if out is None else out
    out_f32 = torch.empty((T, layer.d), dtype=torch.float32, device=residual.device) if want_f32 else None
    sh = layer.shape
    _check("moe_combine", _lib.moe_combine(_ptr(y_rows), _ptr(inv_rows), _ptr(topk_w), _ptr(residual), T,
                                           ctypes.byref(sh), _ptr(out), _ptr(out_f32), _stream()))
    return out, out_f32


def moe_forward_nvfp4(x, layer: MoeLayer, workspace, **kw):
    """moe_forward of a layer with NVFP4 banks (moe_forward itself dispatches on the layer)."""
    if not layer.nvfp4:
        raise ValueError("the layer's banks are int4")
    return moe_forward(x, layer, workspace, **kw)


def moe_forward(x, layer: MoeLayer, workspace, residual=None, forced_ids=None, forced_w=None, out=None,
                out_f32=None, ids_out=None, w_out=None):
    """One MoE layer: returns (out bf16 [T,d], out_f32 or None, ids or None, w or None).
    Calls moe_forward_nvfp4 of the C ABI for a layer with NVFP4 banks."""
    T = x.shape[0]
    _need(x, torch.bfloat16, (T, layer.d), "x")
    residual = x if residual is None else residual
    _need(residual, torch.bfloat16, (T, layer.d), "residual")
    if forced_ids is not None:
        _need(forced_ids, torch.int32, (T, layer.kt), "forced_ids")
        _need(forced_w, torch.float32, (T, layer.kt), "forced_w")
    out = torch.empty_like(x) if out is None else out
    sh, wt = layer.shape, layer.weights
    name = "moe_forward_nvfp4" if layer.nvfp4 else "moe_forward"
    _check(name, getattr(_lib, name)(_ptr(x), _ptr(residual), T, ctypes.byref(sh), ctypes.byref(wt),
                                     _ptr(forced_ids), _ptr(forced_w), _ptr(ids_out), _ptr(w_out), _ptr(out),
                                     _ptr(out_f32), _ptr(workspace), workspace.numel(), _stream()))
    return out, out_f32, ids_out, w_out


def moe_forward_prenorm(residual, layer: MoeLayer, workspace, eps: float = 1e-6, out=None, out_f32=None,
                        xh_out=None, ids_out=None, w_out=None, forced_ids=None, forced_w=None):
    """out = residual + MoE(RMSNorm(residual)); out may be residual itself (in place)."""
    if layer.nvfp4:
        raise ValueError("moe_forward_prenorm takes int4 banks")
    T = residual.shape[0]
    _need(residual, torch.bfloat16, (T, layer.d), "residual")
    out = torch.empty_like(residual) if out is None else out
    wts = layer.weights
    sh = layer.shape
    _check("moe_forward_prenorm",
           _lib.moe_forward_prenorm(_ptr(residual), T, ctypes.byref(sh), ctypes.byref(wts), float(eps),
                                    _ptr(forced_ids), _ptr(forced_w), _ptr(ids_out), _ptr(w_out), _ptr(xh_out),
                                    _ptr(out), _ptr(out_f32), _ptr(workspace), workspace.numel(), _stream()))
    return out


def moe_stack_workspace(layer: MoeLayer, T: int) -> torch.Tensor:
    """A zero-filled workspace for moe_stack_decode on T tokens of this layer shape."""
    n = int(_lib.moe_stack_workspace_size(ctypes.byref(layer.shape), T))
    if n == 0:
        raise BitmoeError("moe_stack_workspace_size", 2)
    return torch.zeros(n, dtype=torch.uint8, device=layer.gate.device)


def moe_stack_decode(residual, layers, workspace, eps: float = 1e-6, lm_w=None, V: int = 0, argmax=None,
                     logits=None, ids_out=None):
    """One decode step of a stack of pre-norm MoE layers (and, with lm_w, the LM head's
    arg-max) in a single launch.  residual [T, d] bf16 is updated in place."""
    T = residual.shape[0]
    lay0 = layers[0]
    _need(residual, torch.bfloat16, (T, lay0.d), "residual")
    if any(l.shape.d != lay0.d or l.k != lay0.k or l.E != lay0.E or l.I != lay0.I or l.n_shared != lay0.n_shared
           for l in layers):
        raise ValueError("every layer of a stack shares one shape")
    if any(l.nvfp4 for l in layers):
        raise ValueError("moe_stack_decode takes int4 banks")
    arr = (MoeWeights * len(layers))(*[l.weights for l in layers])
    if lm_w is not None:
        argmax = torch.empty(T, dtype=torch.int32, device=residual.device) if argmax is None else argmax
        _need(argmax, torch.int32, (T,), "argmax")
        if logits is not None:
            _need(logits, torch.float32, (T, V), "logits")
    if ids_out is not None:
        _need(ids_out, torch.int32, (len(layers), T, lay0.kt), "ids_out")
    sh = lay0.shape
    _check("moe_stack_decode", _lib.moe_stack_decode(_ptr(residual), T, ctypes.byref(sh), arr, len(layers),
                                                     float(eps), _ptr(lm_w), V, _ptr(logits), _ptr(argmax),
                                                     _ptr(ids_out), _ptr(workspace), workspace.numel(), _stream()))
    return residual, argmax


# ---------------------------------------------------------------- LM head and norm


def lmhead_workspace(T: int, d: int, V: int, device="cuda") -> torch.Tensor:
    return torch.zeros(int(_lib.lmhead_workspace_size(T, d, V)), dtype=torch.uint8, device=device)


def lmhead_int4_gemv(h, w_packed, V: int, workspace, want_logits: bool = True, logits=None, argmax=None):
    T, d = h.shape
    _need(h, torch.bfloat16, (T, d), "h")
    logits = (torch.empty((T, V), dtype=torch.float32, device=h.device) if want_logits else None) \
        if logits is None else logits
    argmax = torch.empty(T, dtype=torch.int32, device=h.device) if argmax is None else argmax
    _check("lmhead_int4_gemv", _lib.lmhead_int4_gemv(_ptr(h), T, d, V, GROUP, _ptr(w_packed), _ptr(logits),
                                                     _ptr(argmax), _ptr(workspace), workspace.numel(), _stream()))
    return logits, argmax


def lmhead_nvfp4_gemv(h, w_packed, tensor_scale: float, V: int, workspace, want_logits: bool = True, logits=None,
                      argmax=None):
    """LM head over a packed NVFP4 [V, d] bank with its fp32 tensor scale."""
    T, d = h.shape
    _need(h, torch.bfloat16, (T, d), "h")
    logits = (torch.empty((T, V), dtype=torch.float32, device=h.device) if want_logits else None) \
        if logits is None else logits
    argmax = torch.empty(T, dtype=torch.int32, device=h.device) if argmax is None else argmax
    _check("lmhead_nvfp4_gemv", _lib.lmhead_nvfp4_gemv(_ptr(h), T, d, V, _ptr(w_packed), float(tensor_scale),
                                                       _ptr(logits), _ptr(argmax), _ptr(workspace), workspace.numel(),
                                                       _stream()))
    return logits, argmax


def lmhead_int4_gemv_static(h, w_packed, V: int, argmax, logits=None):
    """LM head that allocates nothing: the caller passes every output buffer
    (``logits`` may be None) and the scratch is the library's fixed array."""
    T, d = h.shape
    _need(h, torch.bfloat16, (T, d), "h")
    _need(argmax, torch.int32, (T,), "argmax")
    if logits is not None:
        _need(logits, torch.float32, (T, V), "logits")
    _check("lmhead_int4_gemv_static", _lib.lmhead_int4_gemv_static(_ptr(h), T, d, V, GROUP, _ptr(w_packed),
                                                                   _ptr(logits), _ptr(argmax), _stream()))
    return logits, argmax


def bitmoe_rmsnorm(x, eps: float = 1e-6, out=None):
    T, d = x.shape
    _need(x, torch.bfloat16, (T, d), "x")
    out = torch.empty_like(x) if out is None else out
    _check("bitmoe_rmsnorm", _lib.bitmoe_rmsnorm(_ptr(x), T, d, eps, _ptr(out), _stream()))
    return out


# ------------------------------------------------------------------ attention decode step

@dataclass
class AttnLayer:
    """Device-resident weights of one attention layer: the packed int4 banks of the stacked
    q | k | v projection [(nq + 2 nkv) * 128, d] and of the output projection [d, nq * 128],
    the fp32 sink logits [nq] (or None), and the layer's kind (window 0 = whole context,
    rope 0 / 1)."""
    d: int
    n_q: int
    n_kv: int
    wqkv: torch.Tensor
    wo: torch.Tensor
    sinks: torch.Tensor | None
    window: int = 513
    rope: bool = True
    eps: float = 1e-6
    theta: float = 1.0e6

    def shape(self, max_len: int) -> AttnShape:
        return AttnShape(self.d, self.n_q, self.n_kv, 128, int(max_len), int(self.window), int(self.rope),
                         float(self.eps), float(self.theta))

    @property
    def weights(self) -> AttnWeights:
        return AttnWeights(self.wqkv.data_ptr(), self.wo.data_ptr(),
                           None if self.sinks is None else self.sinks.data_ptr())

    @classmethod
    def from_canonical(cls, t: dict, d: int, n_q: int, n_kv: int, window: int = 513, rope: bool = True,
                       device="cuda") -> "AttnLayer":
        """t: numpy canonical banks wqkv_q / wqkv_s, wo_q / wo_s (int4 bytes, fp16 scale bits)
        and sinks (fp32 or None)."""
        def pack(q, sc):
            return bitmoe_pack_int4(torch.from_numpy(q).to(device), torch.from_numpy(sc.view("float16")).to(device))
        sinks = None if t.get("sinks") is None else torch.from_numpy(t["sinks"].astype("float32")).to(device)
        return cls(d, n_q, n_kv, pack(t["wqkv_q"], t["wqkv_s"]), pack(t["wo_q"], t["wo_s"]), sinks, window, rope)


def attn_workspace(layer: AttnLayer, max_len: int) -> torch.Tensor:
    n = int(_lib.attn_workspace_size(ctypes.byref(layer.shape(max_len))))
    if n == 0:
        raise BitmoeError("attn_workspace_size", ERR_UNSUPPORTED)
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def _attn_caches(layer: AttnLayer, k_cache, v_cache):
    _need(k_cache, torch.bfloat16, None, "k_cache")
    _need(v_cache, torch.bfloat16, tuple(k_cache.shape), "v_cache")
    if k_cache.dim() != 3 or k_cache.shape[0] != layer.n_kv or k_cache.shape[2] != 128:
        raise ValueError("caches must be [n_kv, max_len, 128] (head-major)")


def attn_decode_step_prenorm(residual, pos: int, layer: AttnLayer, k_cache, v_cache, workspace, out=None,
                             out_f32=None):
    """The pre-norm attention block: out = residual + Attn(bf16(RMSNorm(residual))) (eps =
    layer.eps).  out may be residual itself.  Returns out [d] bf16."""
    d = layer.d
    _need(residual, torch.bfloat16, (d,), "residual")
    _attn_caches(layer, k_cache, v_cache)
    if out is None:
        out = torch.empty(d, dtype=torch.bfloat16, device="cuda")
    sh = layer.shape(k_cache.shape[1])
    wts = layer.weights
    _check("attn_decode_step_prenorm",
           _lib.attn_decode_step_prenorm(_ptr(residual), int(pos), ctypes.byref(sh), ctypes.byref(wts),
                                         _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(out_f32), _ptr(workspace),
                                         workspace.numel(), _stream()))
    return out


def attn_decode_step(x, residual, pos: int, layer: AttnLayer, k_cache, v_cache, workspace, out=None, out_f32=None):
    """One token: x, residual [d] bf16; caches [n_kv, max_len, 128] bf16, head-major (row pos
    of every head is written).
    Returns out [d] bf16."""
    d = layer.d
    _need(x, torch.bfloat16, (d,), "x")
    _need(residual, torch.bfloat16, (d,), "residual")
    _attn_caches(layer, k_cache, v_cache)
    if out is None:
        out = torch.empty(d, dtype=torch.bfloat16, device="cuda")
    sh = layer.shape(k_cache.shape[1])
    wts = layer.weights
    _check("attn_decode_step",
           _lib.attn_decode_step(_ptr(x), _ptr(residual), int(pos), ctypes.byref(sh), ctypes.byref(wts),
                                 _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(out_f32), _ptr(workspace),
                                 workspace.numel(), _stream()))
    return out
