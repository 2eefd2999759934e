"""ctypes binding of libmoe_gb300 (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. PyTorch provides device memory and the current stream. The library
must have been built (``python -m bit_moe_expert_route_gb300.build``); if it
is missing, the first call raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from .synth import LayerShape

_PKG = os.path.dirname(os.path.abspath(__file__))
SO_PATH = os.path.join(_PKG, "libmoe_gb300.so")

EPI_NONE, EPI_SWIGLU, EPI_COMBINE = 0, 1, 2
OPERAND_BF16, OPERAND_F16 = 0, 1
DEV_OK, DEV_BAD_TILE, DEV_BAD_ROW, DEV_TIMEOUT, DEV_BAD_EXPERT = 0, 1, 2, 3, 4


class MoeError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {code} ({status_string(code)})")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "d_model", "n_experts", "top_k", "d_ff", "d_ff_shared", "group")]

    @classmethod
    def of(cls, shape: LayerShape, T: int):
        return cls(T, shape.d_model, shape.n_experts, shape.top_k, shape.d_ff,
                   shape.d_ff_shared, shape.group)


class W4(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class Weights(ctypes.Structure):
    _fields_ = [(n, W4) for n in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")] + [
        ("router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
        ("shared_gate", ctypes.c_void_p)]


class ForwardViews(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "logits", "gate_logit", "topk_ids", "topk_w", "counts", "offsets", "perm", "inv_perm",
        "row_token", "row_weight", "block_map", "num_tiles", "x16", "h", "out_acc", "status")] + [
        ("max_tiles", ctypes.c_int32), ("block_n", ctypes.c_int32),
        ("down_block_map", ctypes.c_void_p), ("down_num_tiles", ctypes.c_void_p),
        ("down_max_tiles", ctypes.c_int32), ("down_block_n", ctypes.c_int32),
        ("y", ctypes.c_void_p), ("down_window", ctypes.c_int32)]


class DecodeViews(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("logits", "gate_logit", "topk_ids", "topk_w", "h", "status")]


_lib = None


def lib():
    """Load the CUDA library (no fallback: a missing library is an error)."""
    global _lib
    if _lib is None:
        if not os.path.exists(SO_PATH):
            raise RuntimeError(
                f"{SO_PATH} is missing; build it with `python -m bit_moe_expert_route_gb300.build`")
        L = ctypes.CDLL(SO_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [i32]
        L.moe_version.restype = i32
        L.moe_pick_block_n.argtypes = [i32, i32, i32]
        L.moe_max_tiles.argtypes = [i32, i32, i32, i32, i32]
        L.moe_route_workspace_bytes.restype = sz
        L.moe_route_workspace_bytes.argtypes = [i32, i32]
        L.moe_route.argtypes = [vp, vp, i32, i32, i32, i32, i32] + [vp] * 10 + [i32, vp, sz, vp]
        L.moe_gemm_workspace_bytes.restype = sz
        L.moe_grouped_gemm_w4a16.argtypes = [vp, i64, i32, vp, i64, vp, i32, i32, vp, vp, vp, i32,
                                             i32, i32, i32, vp, vp, vp, i64, i64, vp, sz, vp]
        L.moe_workspace_bytes.restype = sz
        L.moe_workspace_bytes.argtypes = [vp, i32]
        L.moe_forward_views.argtypes = [vp, sz, vp, i32, vp]
        L.moe_forward.argtypes = [vp, vp, vp, i32, vp, vp, sz, vp]
        L.moe_workspace_bytes_ex.restype = sz
        L.moe_workspace_bytes_ex.argtypes = [vp, i32, i32]
        L.moe_forward_views_ex.argtypes = [vp, sz, vp, i32, i32, vp]
        L.moe_forward_ex.argtypes = [vp, vp, vp, i32, i32, vp, vp, sz, vp]
        L.moe_gdn_scan.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
        L.moe_gdn_scan_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, vp]
        L.moe_decode_attention_workspace_bytes.restype = sz
        L.moe_decode_attention_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.moe_decode_attention.argtypes = [vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, vp, vp,
                                           sz, vp]
        L.moe_decode_workspace_bytes.restype = sz
        L.moe_decode_workspace_bytes.argtypes = [vp]
        L.moe_decode_views.argtypes = [vp, sz, vp, vp]
        L.moe_decode_gemv_w4.argtypes = [vp, vp, vp, vp, vp, sz, vp]
        L.moe_decode_gemv_w4_noalloc.argtypes = [vp, vp, vp, vp, vp]
        L.moe_decode_noalloc_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        L.moe_decode_noalloc_reset.argtypes = [vp]
        L.moe_decode_batch_workspace_bytes.restype = sz
        L.moe_decode_batch_workspace_bytes.argtypes = [vp]
        L.moe_decode_batch_views.argtypes = [vp, sz, vp, vp]
        L.moe_decode_batch_w4.argtypes = [vp, vp, vp, vp, vp, sz, vp]
        L.moe_get_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
        L.moe_debug_decode_fault.argtypes = [ctypes.c_uint64, i32]
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def _check(fn, rc):
    if rc != 0:
        raise MoeError(fn, rc)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled device workspace (the decode call requires a zeroed one)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def device_status(ws: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(0)
    rc = lib().moe_get_device_status(_p(ws), _stream(stream), ctypes.byref(v))
    if rc not in (0, -6):
        raise MoeError("moe_get_device_status", rc)
    return int(v.value)


# ------------------------------------------------------------------ weights on the device
def to_device(a, device="cuda") -> torch.Tensor | None:
    """numpy -> device tensor with the same bytes (uint16 -> int16, uint32 -> int32)."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(device)


class DeviceLayer:
    """One layer's weights resident on the GPU plus the moe_weights_t that points at them."""

    def __init__(self, host: dict, shape: LayerShape, device="cuda"):
        self.shape = shape
        self.t = {}
        for name in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
            w = host.get(name)
            self.t[name] = None if w is None else tuple(to_device(a, device) for a in w)
        for name in ("router", "router_bias", "shared_gate"):
            self.t[name] = to_device(host.get(name), device)
        W = Weights()
        for name in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
            w = self.t[name]
            if w is not None:
                setattr(W, name, W4(w[0].data_ptr(), w[1].data_ptr(), w[2].data_ptr()))
        W.router = self.t["router"].data_ptr()
        W.router_bias = None if self.t["router_bias"] is None else self.t["router_bias"].data_ptr()
        W.shared_gate = None if self.t["shared_gate"] is None else self.t["shared_gate"].data_ptr()
        self.weights = W

    @property
    def nbytes(self) -> int:
        n = 0
        for v in self.t.values():
            if v is None:
                continue
            for a in (v if isinstance(v, tuple) else (v,)):
                n += a.numel() * a.element_size()
        return n


# ------------------------------------------------------------------ entry points
def max_tiles(T, n_experts, top_k, block_n, with_shared=True) -> int:
    return lib().moe_max_tiles(T, n_experts, top_k, block_n, int(with_shared))


def pick_block_n(T, n_experts, top_k) -> int:
    return lib().moe_pick_block_n(T, n_experts, top_k)


def route(logits: torch.Tensor, top_k: int, block_n: int, with_shared: bool = True,
          bias: torch.Tensor | None = None, stream=None) -> dict:
    """moe_route on fp32 logits [T, E]; returns the routing arrays as device tensors."""
    T, E = logits.shape
    dev = logits.device
    mt = max_tiles(T, E, top_k, block_n, with_shared)
    i32 = dict(dtype=torch.int32, device=dev)
    r = dict(
        topk_ids=torch.empty(T, top_k, **i32),
        topk_w=torch.empty(T, top_k, dtype=torch.float32, device=dev),
        counts=torch.empty(E, **i32),
        offsets=torch.empty(E + 1, **i32),
        perm=torch.empty(T * top_k, **i32),
        inv_perm=torch.empty(T * top_k, **i32),
        row_token=torch.empty(T * top_k + (T if with_shared else 0), **i32),
        row_weight=torch.empty(T * top_k, dtype=torch.float32, device=dev),
        block_map=torch.zeros(max(mt, 1), 4, **i32),
        num_tiles=torch.zeros(1, **i32),
    )
    ws = workspace(lib().moe_route_workspace_bytes(T, E), dev)
    rc = lib().moe_route(
        _p(logits), _p(bias), T, E, top_k, block_n, int(with_shared), _p(r["topk_ids"]),
        _p(r["topk_w"]), _p(r["counts"]), _p(r["offsets"]), _p(r["perm"]), _p(r["inv_perm"]),
        _p(r["row_token"]), _p(r["row_weight"]), _p(r["block_map"]), _p(r["num_tiles"]), mt,
        _p(ws), ws.numel(), _stream(stream))
    _check("moe_route", rc)
    r["max_tiles"] = mt
    r["ws"] = ws
    return r


def grouped_gemm_w4a16(A, W, n_groups, N, block_map, num_tiles, max_tiles_, block_n, epilogue,
                       row_index=None, n_rows=None, W_extra=None, row_scale=None, out_row=None,
                       C=None, C_rows=None, operand=None, stream=None):
    """moe_grouped_gemm_w4a16. W / W_extra: list of (q, scale, bias) device tensors.
    operand: OPERAND_F16 / OPERAND_BF16; by default taken from A's dtype (float16 -> f16)."""
    if operand is None:
        operand = OPERAND_F16 if A.dtype == torch.float16 else OPERAND_BF16
    A_rows, K = A.shape
    if n_rows is None:
        n_rows = row_index.numel() if row_index is not None else A_rows
    Ws = (W4 * len(W))(*[W4(q.data_ptr(), s.data_ptr(), b.data_ptr()) for q, s, b in W])
    Wx = None
    if W_extra is not None:
        Wx = (W4 * len(W_extra))(*[W4(q.data_ptr(), s.data_ptr(), b.data_ptr())
                                  for q, s, b in W_extra])
    if C is None:
        dt = torch.float32
        if epilogue == EPI_SWIGLU:
            dt = torch.float16 if operand == OPERAND_F16 else torch.bfloat16
        C = torch.zeros(C_rows if C_rows is not None else n_rows, N, dtype=dt, device=A.device)
    ws = workspace(lib().moe_gemm_workspace_bytes(), A.device)
    rc = lib().moe_grouped_gemm_w4a16(
        _p(A), A_rows, K, _p(row_index), n_rows, ctypes.cast(Ws, ctypes.c_void_p), n_groups, N,
        None if Wx is None else ctypes.cast(Wx, ctypes.c_void_p), _p(block_map), _p(num_tiles),
        max_tiles_, block_n, epilogue, operand, _p(row_scale), _p(out_row), _p(C), C.shape[0],
        C.stride(0), _p(ws), ws.numel(), _stream(stream))
    _check("moe_grouped_gemm_w4a16", rc)
    return C, ws


GDN_STATE_EARLY = 1


def gdn_scan(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor,
             beta: torch.Tensor, state: torch.Tensor, out: torch.Tensor | None = None,
             stream=None, state_early: bool = False) -> torch.Tensor:
    """moe_gdn_scan_ex (include/gdn.h): q, k bf16 [T, Hk, dk]; v bf16 [T, Hv, dv]; alpha,
    beta fp32 [T, Hv]; state fp32 [Hv, dv, dk], advanced in place over the T tokens.
    state_early (MOE_GDN_STATE_EARLY): the previous launch on the stream does not write
    this state, so it is read before waiting for that launch. Returns out fp32 [T, Hv, dv]."""
    T, Hk, dk = k.shape
    Hv, dv = v.shape[1], v.shape[2]
    if out is None:
        out = torch.empty(T, Hv, dv, dtype=torch.float32, device=state.device)
    rc = lib().moe_gdn_scan_ex(_p(q), _p(k), _p(v), _p(alpha), _p(beta), T, Hk, Hv, dk, dv,
                               _p(state), _p(out), GDN_STATE_EARLY if state_early else 0,
                               _stream(stream))
    _check("moe_gdn_scan_ex", rc)
    return out


def decode_attention(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scale: float = 0.0,
                     out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """moe_decode_attention (include/attn.h): q bf16 [Hq, d]; K, V bf16 [L, Hkv, d];
    scale <= 0 means 1/sqrt(d). Returns out fp32 [Hq, d]."""
    Hq, d = q.shape
    L, Hkv = K.shape[0], K.shape[1]
    nbytes = lib().moe_decode_attention_workspace_bytes(L, Hq, Hkv, d)
    if nbytes == 0:
        raise MoeError("moe_decode_attention_workspace_bytes", -3)
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty(Hq, d, dtype=torch.float32, device=q.device)
    rc = lib().moe_decode_attention(_p(q), _p(K), _p(V), L, Hq, Hkv, d, float(scale), _p(out),
                                    _p(ws), ws.numel(), _stream(stream))
    _check("moe_decode_attention", rc)
    return out


FWD_DETERMINISTIC = 1
FWD_DOWN_WINDOWS = 2
FWD_FUSED = 4


class Forward:
    """moe_forward_ex with a reusable workspace for one (shape, T, block_n, flags);
    deterministic=True sets MOE_FWD_DETERMINISTIC (fixed-order combine),
    down_windows=True MOE_FWD_DOWN_WINDOWS (down tiles ordered by token window),
    fused=True MOE_FWD_FUSED (gate/up, SwiGLU and down per 64-row tile in one kernel)."""

    def __init__(self, layer: DeviceLayer, T: int, block_n: int = 0, device="cuda",
                 deterministic: bool = False, down_windows: bool = False, fused: bool = False):
        self.layer = layer
        self.T = T
        self.shape = Shape.of(layer.shape, T)
        self.flags = ((FWD_DETERMINISTIC if deterministic else 0) | (FWD_DOWN_WINDOWS if down_windows else 0)
                      | (FWD_FUSED if fused else 0))
        self.block_n = block_n or (64 if fused else pick_block_n(T, layer.shape.n_experts, layer.shape.top_k))
        nbytes = lib().moe_workspace_bytes_ex(ctypes.byref(self.shape), self.block_n, self.flags)
        if nbytes == 0:
            raise MoeError("moe_workspace_bytes_ex", -3)
        self.ws = workspace(nbytes, device)
        self.views = ForwardViews()
        _check("moe_forward_views_ex", lib().moe_forward_views_ex(
            _p(self.ws), self.ws.numel(), ctypes.byref(self.shape), self.block_n, self.flags,
            ctypes.byref(self.views)))

    def __call__(self, x: torch.Tensor, out: torch.Tensor | None = None, stream=None):
        if out is None:
            out = torch.empty(self.T, self.layer.shape.d_model, dtype=torch.bfloat16,
                              device=x.device)
        rc = lib().moe_forward_ex(_p(x), ctypes.byref(self.layer.weights),
                                  ctypes.byref(self.shape), self.block_n, self.flags, _p(out),
                                  _p(self.ws), self.ws.numel(), _stream(stream))
        _check("moe_forward_ex", rc)
        return out

    def view(self, name: str, shape, dtype) -> torch.Tensor:
        """A device tensor aliasing one of the workspace intermediates."""
        base = self.ws.data_ptr()
        off = getattr(self.views, name) - base
        n = int(np.prod(shape))
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(*shape)


class DecodeBatch:
    """moe_decode_batch_w4 (1 <= T <= 8 tokens) with a reusable workspace."""

    def __init__(self, layer: DeviceLayer, T: int, device="cuda"):
        self.layer, self.T = layer, T
        self.shape = Shape.of(layer.shape, T)
        nbytes = lib().moe_decode_batch_workspace_bytes(ctypes.byref(self.shape))
        if nbytes == 0:
            raise MoeError("moe_decode_batch_workspace_bytes", -3)
        self.ws = workspace(nbytes, device)
        self.views = DecodeViews()
        _check("moe_decode_batch_views", lib().moe_decode_batch_views(
            _p(self.ws), self.ws.numel(), ctypes.byref(self.shape), ctypes.byref(self.views)))

    def view(self, name: str, shape, dtype) -> torch.Tensor:
        """A workspace array (logits [T][E], gate_logit [T], topk_ids [T][k],
        topk_w [T][k+1] with the shared gate last, h fp32 [T][k+1][d_ff])."""
        off = getattr(self.views, name) - self.ws.data_ptr()
        n = int(np.prod(shape))
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(*shape)

    def __call__(self, x: torch.Tensor, out: torch.Tensor | None = None, stream=None):
        if out is None:
            out = torch.empty(self.T, self.layer.shape.d_model, dtype=torch.bfloat16, device=x.device)
        rc = lib().moe_decode_batch_w4(_p(x), ctypes.byref(self.layer.weights),
                                       ctypes.byref(self.shape), _p(out), _p(self.ws),
                                       self.ws.numel(), _stream(stream))
        _check("moe_decode_batch_w4", rc)
        return out


class Decode:
    """moe_decode_gemv_w4 (T = 1) with a reusable workspace."""

    def __init__(self, layer: DeviceLayer, device="cuda"):
        self.layer = layer
        self.shape = Shape.of(layer.shape, 1)
        nbytes = lib().moe_decode_workspace_bytes(ctypes.byref(self.shape))
        if nbytes == 0:
            raise MoeError("moe_decode_workspace_bytes", -3)
        self.ws = workspace(nbytes, device)
        self.views = DecodeViews()
        _check("moe_decode_views", lib().moe_decode_views(
            _p(self.ws), self.ws.numel(), ctypes.byref(self.shape), ctypes.byref(self.views)))

    def __call__(self, x: torch.Tensor, out: torch.Tensor | None = None, stream=None):
        if out is None:
            out = torch.empty(self.layer.shape.d_model, dtype=torch.bfloat16, device=x.device)
        rc = lib().moe_decode_gemv_w4(_p(x), ctypes.byref(self.layer.weights),
                                      ctypes.byref(self.shape), _p(out), _p(self.ws),
                                      self.ws.numel(), _stream(stream))
        _check("moe_decode_gemv_w4", rc)
        return out

    def view(self, name: str, shape, dtype) -> torch.Tensor:
        off = getattr(self.views, name) - self.ws.data_ptr()
        n = int(np.prod(shape))
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(*shape)
