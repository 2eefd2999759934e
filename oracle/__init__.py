"""ctypes front end of the CPU oracle (oracle/moe_ref.cpp).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library neither
imports nor links this module, and this module imports nothing from the CUDA
package.

All arrays are numpy; bf16 values travel as uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_ref.cpp")


def so_path(mutant: int = 0) -> str:
    name = "libmoe_ref.so" if mutant == 0 else f"libmoe_ref_mutant{mutant}.so"
    return os.path.join(_HERE, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (optionally with one planted mistake) beside its source."""
    so = so_path(mutant)
    if force or not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(_SRC):
        tmp = so + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c++17", _SRC, "-o", tmp]
        if mutant:
            cmd.insert(1, f"-DORACLE_MUTANT={mutant}")
        subprocess.check_call(cmd)
        os.replace(tmp, so)
    return so


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "contiguous numpy array expected"
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        L = ctypes.CDLL(build(mutant))
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        L.oracle_dequant.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.oracle_router.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
        L.oracle_topk.argtypes = [vp, vp, i32, i32, i32, vp, vp]
        L.oracle_route_meta.argtypes = [vp, i32, i32, i32, i32, i32] + [vp] * 7 + [i32]
        L.oracle_expert.argtypes = [vp, i32, i32, i32, i32, i32] + [vp] * 10
        L.oracle_moe_forward.argtypes = [i32] * 7 + [vp] * 27
        self.L = L

    # w = scale*q + bias, exact (fp64) for `rows` rows of K codes
    def dequant(self, q, s, b, group):
        q = np.ascontiguousarray(q, np.uint32)
        s = np.ascontiguousarray(s, np.uint16)
        b = np.ascontiguousarray(b, np.uint16)
        rows = q.size // q.shape[-1]
        K = q.shape[-1] * 8
        out = np.empty((rows, K), np.float64)
        rc = self.L.oracle_dequant(_p(q), _p(s), _p(b), rows, K, group, _p(out))
        assert rc == 0
        return out.reshape(q.shape[:-1] + (K,))

    def router(self, x, Wr, wsg=None):
        x = np.ascontiguousarray(x, np.uint16)
        Wr = np.ascontiguousarray(Wr, np.float32)
        T, d = x.shape
        E = Wr.shape[1]
        logits = np.empty((T, E), np.float32)
        gl = np.empty(T, np.float32) if wsg is not None else None
        wsg = None if wsg is None else np.ascontiguousarray(wsg, np.float32)
        assert self.L.oracle_router(_p(x), _p(Wr), _p(wsg), T, d, E, _p(logits), _p(gl)) == 0
        return logits, gl

    def topk(self, logits, k, bias=None):
        logits = np.ascontiguousarray(logits, np.float32)
        T, E = logits.shape
        ids = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        bias = None if bias is None else np.ascontiguousarray(bias, np.float32)
        assert self.L.oracle_topk(_p(logits), _p(bias), T, E, k, _p(ids), _p(w)) == 0
        return ids, w

    @staticmethod
    def max_tiles(T, k, E, block_n, with_shared=True):
        return -(-T * k // block_n) + E + (-(-T // block_n) if with_shared else 0)

    def route_meta(self, ids, E, block_n, with_shared=True):
        ids = np.ascontiguousarray(ids, np.int32)
        T, k = ids.shape
        A = T * k
        mt = self.max_tiles(T, k, E, block_n, with_shared)
        r = dict(
            counts=np.empty(E, np.int32),
            offsets=np.empty(E + 1, np.int32),
            perm=np.empty(A, np.int32),
            inv_perm=np.empty(A, np.int32),
            row_token=np.empty(A + (T if with_shared else 0), np.int32),
            block_map=np.zeros((mt, 4), np.int32),
            num_tiles=np.zeros(1, np.int32),
        )
        rc = self.L.oracle_route_meta(
            _p(ids), T, k, E, block_n, int(with_shared), _p(r["counts"]), _p(r["offsets"]),
            _p(r["perm"]), _p(r["inv_perm"]), _p(r["row_token"]), _p(r["block_map"]),
            _p(r["num_tiles"]), mt)
        assert rc == 0, rc
        r["num_tiles"] = int(r["num_tiles"][0])
        r["block_map"] = r["block_map"][: r["num_tiles"]]
        return r

    def expert(self, x, gate, up, down, group, g=0):
        """One SwiGLU expert (index g of the stacked projections) on x [T,d]."""
        x = np.ascontiguousarray(x, np.uint16)
        T, d = x.shape
        f = gate[0].shape[1]
        y = np.empty((T, d), np.float64)
        args = []
        for q, s, b in (gate, up, down):
            args += [_p(np.ascontiguousarray(q)), _p(np.ascontiguousarray(s)),
                     _p(np.ascontiguousarray(b))]
        assert self.L.oracle_expert(_p(x), T, d, f, group, g, *args, _p(y)) == 0
        return y

    def moe_forward(self, x, w, shape, logits_in=None):
        """Whole layer. w: dict from synth.layer_weights. Returns dict of outputs."""
        x = np.ascontiguousarray(x, np.uint16)
        T, d = x.shape
        E, k, f, fs, G = shape.n_experts, shape.top_k, shape.d_ff, shape.d_ff_shared, shape.group
        shared = w.get("shared_gate") is not None
        out = np.empty((T, d), np.float32)
        logits = np.empty((T, E), np.float32)
        ids = np.empty((T, k), np.int32)
        wt = np.empty((T, k), np.float32)
        gate = np.empty(T, np.float32)
        projs = []
        for name in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
            t = w.get(name)
            projs += [None, None, None] if t is None else [_p(np.ascontiguousarray(a)) for a in t]
        li = None if logits_in is None else np.ascontiguousarray(logits_in, np.float32)
        rb = w.get("router_bias")
        rb = None if rb is None else np.ascontiguousarray(rb, np.float32)
        rc = self.L.oracle_moe_forward(
            T, d, E, k, f, fs, G, _p(x), _p(np.ascontiguousarray(w["router"], np.float32)),
            _p(rb), _p(None if not shared else np.ascontiguousarray(w["shared_gate"], np.float32)),
            *projs, _p(li), _p(out), _p(logits), _p(ids), _p(wt), _p(gate))
        assert rc == 0, rc
        return dict(out=out, logits=logits, ids=ids, w=wt, gate=gate)
