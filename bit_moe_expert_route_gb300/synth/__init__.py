"""Seeded synthetic inputs for the 4-bit MoE layer.

This module produces inputs only: token activations, router weights, the
shared-expert gate vector and groupwise affine 4-bit expert weights.  It holds
none of the layer's arithmetic (no dequantisation, routing or expert math), so
both the CUDA path and the CPU oracle can be fed from it.

Distributions (the Qwen3.6-35B-A3B-style layer this library targets):
  x       bf16 ~ N(0, 1)
  router  fp32 ~ N(0, 0.02), shape [d_model, n_experts]
  w_sg    fp32 ~ N(0, 0.02), shape [d_model]
  q       uniform codes 0..15, eight per uint32, low nibble = lowest k
  scale   bf16 ~ U[0.005, 0.02] per group of `group` along K
  bias    bf16 = -8 * scale + N(0, 0.001)
Every element is a pure function of (seed, layer, tensor id, element index).
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")

# tensor ids inside one (seed, layer)
X = 1
ROUTER = 2
SHARED_GATE = 3
X_DECODE = 4
PROJ = ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")


def _proj_ids(p: int):
    base = 16 + 4 * p
    return base, base + 1, base + 2  # q, scale, bias-noise


def build(force: bool = False) -> str:
    """Compile the generator into libsynth.so beside its source."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        L.synth_key.restype = u64
        L.synth_key.argtypes = [u64, u64, u64]
        L.synth_normal_f32.argtypes = [u64, i64, i64, dbl, vp]
        L.synth_normal_bf16.argtypes = [u64, i64, i64, dbl, vp]
        L.synth_q4.argtypes = [u64, i64, i64, vp]
        L.synth_scale_bias.argtypes = [u64, u64, i64, i64, dbl, dbl, dbl, vp, vp]
        L.synth_uniform_int.argtypes = [u64, i64, i64, ctypes.c_uint32, vp]
        _lib = L
    return _lib


def key(seed: int, layer: int, tensor: int) -> int:
    return lib().synth_key(seed, layer, tensor)


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def normal_f32(k: int, n: int, sigma: float, off: int = 0) -> np.ndarray:
    out = np.empty(n, np.float32)
    lib().synth_normal_f32(k, off, n, sigma, _ptr(out))
    return out


def normal_bf16(k: int, n: int, sigma: float, off: int = 0) -> np.ndarray:
    out = np.empty(n, np.uint16)
    lib().synth_normal_bf16(k, off, n, sigma, _ptr(out))
    return out


def q4(k: int, nwords: int, off: int = 0) -> np.ndarray:
    out = np.empty(nwords, np.uint32)
    lib().synth_q4(k, off, nwords, _ptr(out))
    return out


def scale_bias(ks: int, kb: int, n: int, off: int = 0, lo=0.005, hi=0.02, noise=0.001):
    s = np.empty(n, np.uint16)
    b = np.empty(n, np.uint16)
    lib().synth_scale_bias(ks, kb, off, n, lo, hi, noise, _ptr(s), _ptr(b))
    return s, b


def uniform_int(k: int, n: int, n_range: int, off: int = 0) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().synth_uniform_int(k, off, n, n_range, _ptr(out))
    return out


@dataclasses.dataclass(frozen=True)
class LayerShape:
    d_model: int = 2048
    n_experts: int = 256
    top_k: int = 8
    d_ff: int = 512
    d_ff_shared: int = 512
    group: int = 64


def proj_dims(shape: LayerShape, p: int):
    """(groups stacked, N rows, K) of projection p."""
    d, f, fs, E = shape.d_model, shape.d_ff, shape.d_ff_shared, shape.n_experts
    return [(E, f, d), (E, f, d), (E, d, f), (1, fs, d), (1, fs, d), (1, d, fs)][p]


def w4_projection(shape: LayerShape, seed: int, layer: int, p: int):
    """(q [G,N,K/8] uint32, scale [G,N,K/group] bf16 bits, bias [G,N,K/group] bf16 bits)."""
    g, n, kdim = proj_dims(shape, p)
    kq, ks, kb = (key(seed, layer, t) for t in _proj_ids(p))
    q = q4(kq, g * n * kdim // 8).reshape(g, n, kdim // 8)
    s, b = scale_bias(ks, kb, g * n * kdim // shape.group)
    return q, s.reshape(g, n, kdim // shape.group), b.reshape(g, n, kdim // shape.group)


def zipf_router_bias(n_experts: int, alpha: float = 1.5) -> np.ndarray:
    """Per-expert logit offset alpha*log(1/rank), rank(e) = e+1 (expert 0 most popular)."""
    return np.array([-alpha * math.log(e + 1) for e in range(n_experts)], np.float32)


def layer_weights(shape: LayerShape, seed: int = 0, layer: int = 0, shared: bool = True,
                  router_bias: np.ndarray | None = None) -> dict:
    """All weights of one layer as host numpy arrays (bf16 stored as uint16 bits)."""
    d, E = shape.d_model, shape.n_experts
    w = {
        "router": normal_f32(key(seed, layer, ROUTER), d * E, 0.02).reshape(d, E),
        "router_bias": router_bias,
        "shared_gate": normal_f32(key(seed, layer, SHARED_GATE), d, 0.02) if shared else None,
    }
    for p, name in enumerate(PROJ):
        if p >= 3 and not shared:
            w[name] = None
            continue
        w[name] = w4_projection(shape, seed, layer, p)
    return w


def tokens(shape: LayerShape, T: int, seed: int = 0, layer: int = 0, off: int = 0,
           tensor: int = X) -> np.ndarray:
    """x [T, d_model] bf16 bits; rows off..off+T-1 of the layer's token stream."""
    d = shape.d_model
    return normal_bf16(key(seed, layer, tensor), T * d, 1.0, off=off * d).reshape(T, d)


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bits (finite inputs)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
