"""The C ABI without a GPU: the library loads, exports every function that
include/*.h declares, and rejects bad arguments before touching a device."""
import ctypes
import glob
import os
import re

import pytest

from bit_moe_expert_route_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    from bit_moe_expert_route_gb300 import ops
    return ops.lib()


def declared_functions():
    src = "".join(open(h).read() for h in sorted(glob.glob(os.path.join(os.path.dirname(HEADER), "*.h"))))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z0-9_]+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("moe_route", "moe_grouped_gemm_w4a16", "moe_forward", "moe_decode_gemv_w4"):
        assert fn in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings(L):
    from bit_moe_expert_route_gb300 import ops
    assert ops.status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5, -6, -7, 101, 102, 103, 104):
        assert ops.status_string(code) not in ("", "unknown status")
    assert ops.status_string(12345) == "unknown status"


def test_block_n_and_tile_bounds(L):
    from bit_moe_expert_route_gb300 import ops
    assert ops.pick_block_n(64, 256, 8) == 16
    assert ops.pick_block_n(512, 256, 8) == 64
    assert ops.pick_block_n(128, 256, 8) == 16
    assert ops.pick_block_n(2048, 256, 8) == 64
    assert ops.pick_block_n(4096, 256, 8) == 128
    assert ops.pick_block_n(32768, 256, 8) == 128
    assert ops.max_tiles(3, 4, 2, 2, True) == 3 + 4 + 2
    assert ops.max_tiles(32768, 256, 8, 128, True) == 2048 + 256 + 256


def test_workspace_sizes(L):
    from bit_moe_expert_route_gb300 import ops
    from bit_moe_expert_route_gb300.synth import LayerShape
    sh = ops.Shape.of(LayerShape(), 4096)
    n = L.moe_workspace_bytes(ctypes.byref(sh), 128)
    T, E, k, d, f = 4096, 256, 8, 2048, 512
    assert n >= T * E * 4 + (T * k + T) * f * 2 + T * d * 4
    assert n % 256 == 0
    bad = ops.Shape(4096, 2048, 256, 8, 512, 512, 32)  # group 32 unsupported
    assert L.moe_workspace_bytes(ctypes.byref(bad), 128) == 0
    assert L.moe_workspace_bytes(ctypes.byref(sh), 48) == 0  # block_n 48 unsupported
    assert L.moe_decode_workspace_bytes(ctypes.byref(ops.Shape.of(LayerShape(), 1))) > 0
    for T, ok in ((1, True), (4, True), (8, True), (9, False), (0, False)):
        n = L.moe_decode_batch_workspace_bytes(ctypes.byref(ops.Shape.of(LayerShape(), T)))
        assert (n > 0) == ok, T
        if ok:  # logits, gate, ids, weights, h of every token
            assert n >= T * (256 * 4 + 4 + 8 * 4 + 9 * 4 + 9 * 512 * 4)
    assert L.moe_route_workspace_bytes(32768, 256) >= 256 * 256 * 4
    # the deterministic mode adds the down projection's rows, fp32 [9T][d]
    n_det = L.moe_workspace_bytes_ex(ctypes.byref(sh), 128, 1)
    assert n_det >= L.moe_workspace_bytes(ctypes.byref(sh), 128) + (T * k + T) * d * 4
    assert L.moe_workspace_bytes_ex(ctypes.byref(sh), 128, 0) == L.moe_workspace_bytes(
        ctypes.byref(sh), 128)
    assert L.moe_workspace_bytes_ex(ctypes.byref(sh), 128, 8) == 0  # unknown flag
    # the fused chain: 64-row tiles only, not with the other flags, d/f multiples of 512
    assert L.moe_workspace_bytes_ex(ctypes.byref(sh), 0, 4) == L.moe_workspace_bytes(ctypes.byref(sh), 64)
    assert L.moe_workspace_bytes_ex(ctypes.byref(sh), 128, 4) == 0
    assert L.moe_workspace_bytes_ex(ctypes.byref(sh), 0, 4 | 1) == 0
    small = ops.Shape(64, 256, 32, 4, 256, 256, 64)
    assert L.moe_workspace_bytes_ex(ctypes.byref(small), 0, 4) == 0


def test_forward_views_pick_the_down_tile_map(L):
    """The down projection gets a second, 256-row block map only when gate/up runs
    128-row tiles and the experts average 256 or more rows; otherwise both
    projections share one map. (The views only carve a workspace: host memory
    serves here.)"""
    from bit_moe_expert_route_gb300 import ops
    from bit_moe_expert_route_gb300.synth import LayerShape
    for T, bn, separate in ((32768, 128, True), (8192, 128, True), (8191, 128, False),
                            (32768, 64, False), (4096, 128, False)):
        sh = ops.Shape.of(LayerShape(), T)
        n = L.moe_workspace_bytes(ctypes.byref(sh), bn)
        buf = ctypes.create_string_buffer(n + 256)
        base = (ctypes.addressof(buf) + 255) // 256 * 256
        v = ops.ForwardViews()
        assert L.moe_forward_views(ctypes.c_void_p(base), n, ctypes.byref(sh), bn,
                                   ctypes.byref(v)) == 0
        assert v.block_n == bn and not v.y
        if separate:
            assert v.down_block_n == 256 and v.down_block_map != v.block_map
            assert v.down_window == 0
            assert v.down_max_tiles == L.moe_max_tiles(T, 256, 8, 256, 1)
            assert base <= v.down_block_map and v.down_num_tiles + 4 <= base + n
            # with MOE_FWD_DOWN_WINDOWS, above 8192 tokens the down map is cut per
            # 8192-token window: every (window, expert) and (window, shared) piece
            # may end in a partial tile
            nw = L.moe_workspace_bytes_ex(ctypes.byref(sh), bn, 2)
            bufw = ctypes.create_string_buffer(nw + 256)
            basew = (ctypes.addressof(bufw) + 255) // 256 * 256
            vw = ops.ForwardViews()
            assert L.moe_forward_views_ex(ctypes.c_void_p(basew), nw, ctypes.byref(sh), bn, 2,
                                          ctypes.byref(vw)) == 0
            W = 8192 if T > 8192 else 0
            assert vw.down_window == W
            nW = -(-T // W) if W else 1
            assert vw.down_max_tiles == -(-T * 8 // 256) + nW * 256 + -(-T // 256) + nW - 1
            assert vw.down_max_tiles >= v.down_max_tiles
        else:
            assert (v.down_block_n, v.down_max_tiles) == (bn, v.max_tiles)
            assert (v.down_block_map, v.down_num_tiles) == (v.block_map, v.num_tiles)
            assert v.down_window == 0


def test_deterministic_views(L):
    """The deterministic workspace keeps every other intermediate where moe_forward
    puts it and adds y [T*k + T][d] fp32 at its end."""
    from bit_moe_expert_route_gb300 import ops
    from bit_moe_expert_route_gb300.synth import LayerShape
    T, k, d = 512, 8, 2048
    sh = ops.Shape.of(LayerShape(), T)
    n = L.moe_workspace_bytes_ex(ctypes.byref(sh), 0, 1)
    buf = ctypes.create_string_buffer(n + 256)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    v0, v1 = ops.ForwardViews(), ops.ForwardViews()
    assert L.moe_forward_views_ex(ctypes.c_void_p(base), n, ctypes.byref(sh), 0, 0,
                                  ctypes.byref(v0)) == 0
    assert L.moe_forward_views_ex(ctypes.c_void_p(base), n, ctypes.byref(sh), 0, 1,
                                  ctypes.byref(v1)) == 0
    for name in ("logits", "h", "out_acc", "block_map", "inv_perm", "row_weight"):
        assert getattr(v0, name) == getattr(v1, name), name
    assert not v0.y and v1.y >= v1.out_acc + T * d * 4
    assert v1.y + (T * k + T) * d * 4 <= base + n
    assert L.moe_forward_views_ex(ctypes.c_void_p(base), n - 256, ctypes.byref(sh), 0, 1,
                                  ctypes.byref(v1)) == -4  # too small for y


def test_gdn_scan_arguments_are_checked_on_the_host(L):
    vp = ctypes.c_void_p
    buf = ctypes.create_string_buffer(1 << 16)
    a = (ctypes.addressof(buf) + 255) // 256 * 256
    ok = dict(q=a, k=a, v=a, al=a, be=a, T=4, Hk=2, Hv=4, dk=128, dv=128, st=a, out=a)

    def call(**kw):
        c = dict(ok, **kw)
        return L.moe_gdn_scan(vp(c["q"]), vp(c["k"]), vp(c["v"]), vp(c["al"]), vp(c["be"]),
                              c["T"], c["Hk"], c["Hv"], c["dk"], c["dv"], vp(c["st"]),
                              vp(c["out"]), None)
    assert call(T=-1) == -3
    assert call(dk=96) == -3 and call(dv=12) == -3 and call(Hv=3) == -3 and call(Hk=0) == -3
    assert call(st=None) == -1 and call(q=None) == -1 and call(out=None) == -1
    assert call(q=a + 8) == -2 and call(v=a + 8) == -2 and call(st=a + 8) == -2
    assert call(dk=64, st=a + 8) != -2  # an 8-byte aligned state suffices at d_k 64
    assert call(T=0, q=None, k=None, v=None, al=None, be=None, out=None) == 0  # no work

    def call_ex(flags, **kw):
        c = dict(ok, **kw)
        return L.moe_gdn_scan_ex(vp(c["q"]), vp(c["k"]), vp(c["v"]), vp(c["al"]), vp(c["be"]),
                                 c["T"], c["Hk"], c["Hv"], c["dk"], c["dv"], vp(c["st"]),
                                 vp(c["out"]), flags, None)
    assert call_ex(2) == -3 and call_ex(-1) == -3  # unknown flag bits
    assert call_ex(1, T=-1) == -3 and call_ex(1, st=None) == -1 and call_ex(1, st=a + 8) == -2
    assert call_ex(1, T=0, q=None, k=None, v=None, al=None, be=None, out=None) == 0


def test_decode_attention_arguments_are_checked_on_the_host(L):
    vp = ctypes.c_void_p
    ws_n = L.moe_decode_attention_workspace_bytes(4096, 16, 2, 256)
    # partials: (m, l, 256 outputs) per query head, one per 64-position slice at most
    assert ws_n == 16 * (4096 // 64) * (2 + 256) * 4
    for args in ((0, 16, 2, 256), (10, 16, 2, 96), (10, 16, 3, 256), (10, 32, 2, 128)):
        assert L.moe_decode_attention_workspace_bytes(*args) == 0, args  # 16 per KV head > 8
    buf = ctypes.create_string_buffer(1 << 20)
    a = (ctypes.addressof(buf) + 255) // 256 * 256
    ok = dict(q=a, K=a, V=a, L=64, Hq=8, Hkv=1, d=128, out=a, ws=a, n=1 << 19)

    def call(**kw):
        c = dict(ok, **kw)
        return L.moe_decode_attention(vp(c["q"]), vp(c["K"]), vp(c["V"]), c["L"], c["Hq"],
                                      c["Hkv"], c["d"], ctypes.c_float(0.0), vp(c["out"]),
                                      vp(c["ws"]), c["n"], None)
    assert call(L=0) == -3 and call(d=48) == -3 and call(Hq=9) == -3
    assert call(q=None) == -1 and call(V=None) == -1
    assert call(K=a + 8) == -2 and call(q=a + 4) == -2
    assert call(ws=None) == -4 and call(n=16) == -4


def test_bad_arguments_are_rejected_on_the_host(L):
    vp = ctypes.c_void_p
    fake = vp(0x10000)  # never dereferenced: every call below fails validation first
    # unsupported top_k
    assert L.moe_route(fake, None, 8, 16, 17, 16, 1, *([fake] * 10), 100, fake, 1 << 20,
                       None) == -3
    # unsupported block_n
    assert L.moe_route(fake, None, 8, 16, 2, 24, 1, *([fake] * 10), 100, fake, 1 << 20,
                       None) == -3
    # max_tiles below the bound
    assert L.moe_route(fake, None, 8, 16, 2, 16, 1, *([fake] * 10), 1, fake, 1 << 20,
                       None) == -3
    # NULL output
    assert L.moe_route(fake, None, 8, 16, 2, 16, 1, *([fake] * 9), None, 100, fake, 1 << 20,
                       None) == -1
    # workspace too small
    assert L.moe_route(fake, None, 8, 16, 2, 16, 1, *([fake] * 10), 100, fake, 16, None) == -4
    # misaligned workspace
    assert L.moe_route(fake, None, 8, 16, 2, 16, 1, *([fake] * 10), 100, vp(0x10004), 1 << 20,
                       None) == -4
    # grouped GEMM: N not a multiple of 128, bad epilogue, misaligned A
    W = (ctypes.c_void_p * 3)(0x10000, 0x10000, 0x10000)
    args = lambda A, N, epi, fmt=1: (A, 10, 128, None, 10, ctypes.cast(W, vp), 4, N, None, fake,
                                     fake, 10, 16, epi, fmt, fake, fake, fake, 10, N, fake,
                                     1 << 20, None)
    assert L.moe_grouped_gemm_w4a16(*args(fake, 100, 0)) == -3
    assert L.moe_grouped_gemm_w4a16(*args(fake, 128, 7)) == -3
    assert L.moe_grouped_gemm_w4a16(*args(fake, 128, 0, 5)) == -3  # unknown operand format
    assert L.moe_grouped_gemm_w4a16(*args(vp(0x10002), 128, 0)) == -2
    # forward: NULL weights, bad shape
    from bit_moe_expert_route_gb300 import ops
    sh = ops.Shape(4, 2048, 256, 8, 512, 512, 64)
    assert L.moe_forward(fake, None, ctypes.byref(sh), 0, fake, fake, 1 << 30, None) == -1
    sh_bad = ops.Shape(4, 2000, 256, 8, 512, 512, 64)
    assert L.moe_forward(fake, None, ctypes.byref(sh_bad), 0, fake, fake, 1 << 30, None) == -3
    # decode requires T == 1
    sh2 = ops.Shape(2, 2048, 256, 8, 512, 512, 64)
    assert L.moe_decode_gemv_w4(fake, None, ctypes.byref(sh2), fake, fake, 1 << 20, None) == -3


def test_max_tiles_bounds_every_routing(L, orc):
    """The device block map is sized by moe_max_tiles before the routing is known:
    the exact tile count the oracle builds for any routing must stay within it
    (uniform, fully concentrated and round-robin routings, every tile height)."""
    import numpy as np
    rng = np.random.default_rng(0)
    for T, E, k in ((1, 8, 1), (7, 8, 8), (64, 72, 4), (1000, 256, 8), (4096, 256, 8)):
        routings = {
            "uniform": np.argsort(rng.random((T, E)), axis=1)[:, :k],
            "concentrated": np.tile(np.arange(k), (T, 1)),
            "round-robin": (np.arange(T)[:, None] * k + np.arange(k)[None, :]) % E,
        }
        for name, ids in routings.items():
            ids = ids.astype(np.int32)
            for bn in (16, 32, 64, 128, 256):
                m = orc.route_meta(ids, E, bn, True)
                assert m["num_tiles"] <= L.moe_max_tiles(T, E, k, bn, 1), (T, E, k, name, bn)
