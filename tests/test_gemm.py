"""moe_grouped_gemm_w4a16 against references built from the oracle's
dequantisation and a library matmul, for both tensor-core operand formats
(f16, used by moe_forward, and bf16).

* integer-exact: x in {-2..2}, scale 1, bias -8 -> every product and partial
  sum is an integer below 2^24, so the fp32 result is exact: bit-exact.
* one-hot readout: A rows are unit vectors, so C reads back the weight the
  tensor core saw, which must be RNE(scale*q + bias) in the operand format,
  bit for bit; this pins the on-chip dequantisation and the operand layouts.
* SwiGLU and combine epilogues on random data, against fp64 references on the
  same operands (fp32 accumulation order and the rounding of h are the only
  differences).
* block maps with ragged tiles, every block_n, an extra group (shared expert),
  empty work, and out-of-range entries that the kernel must reject.
"""
import numpy as np
import pytest

from bit_moe_expert_route_gb300 import synth
from bit_moe_expert_route_gb300.synth import LayerShape
from gpu_util import to_np

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

FMTS = {"f16": 1, "bf16": 0}


def dev(a):
    from bit_moe_expert_route_gb300 import ops
    return ops.to_device(a)


def to_fmt(a, fmt):
    """float array -> operand bit patterns (uint16), RNE."""
    a = np.asarray(a, np.float32)
    return a.astype(np.float16).view(np.uint16) if fmt == "f16" else synth.f32_to_bf16(a)


def from_fmt(bits, fmt):
    bits = np.asarray(bits, np.uint16)
    if fmt == "f16":
        return bits.view(np.float16).astype(np.float64)
    return synth.bf16_to_f32(bits).astype(np.float64)


def round_fmt(a, fmt):
    return from_fmt(to_fmt(a, fmt), fmt)


def c_np(C, fmt):
    return from_fmt(to_np(C.view(torch.int16)).view(np.uint16), fmt)


def routing(orc, T, E, k, bn, seed, with_shared=True):
    keys = synth.normal_f32(synth.key(seed, 0, 200), T * E, 1.0).reshape(T, E)
    ids = np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)
    return ids, orc.route_meta(ids, E, bn, with_shared)


def deq(orc, proj, g, fmt):
    """Weights of expert g as the tensor core sees them: RNE(scale*q + bias) in fmt."""
    q, s, b = proj
    return round_fmt(orc.dequant(q[g], s[g], b[g], 64), fmt)


def gemm_call(A, projs, n_groups, N, m, bn, epi, fmt, row_index=None, extra=None, **kw):
    from bit_moe_expert_route_gb300 import ops
    bm = torch.zeros(max(len(m["block_map"]), 1), 4, dtype=torch.int32, device="cuda")
    if len(m["block_map"]):
        bm[: len(m["block_map"])] = torch.from_numpy(m["block_map"]).cuda()
    nt = torch.tensor([m["num_tiles"]], dtype=torch.int32, device="cuda")
    W = [tuple(dev(a) for a in p) for p in projs]
    Wx = None if extra is None else [tuple(dev(a) for a in p) for p in extra]
    C, ws = ops.grouped_gemm_w4a16(A, W, n_groups, N, bm, nt, bm.shape[0], bn, epi,
                                   row_index=row_index, W_extra=Wx, operand=FMTS[fmt], **kw)
    torch.cuda.synchronize()
    return C, ws


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("bn,K", [(16, 512), (32, 512), (64, 512), (128, 512), (256, 512),
                                  (32, 192), (128, 320), (256, 192)])
def test_integer_exact_none_epilogue(orc, bn, K, fmt):
    """K = 192 and 320: an odd number of 64-wide k-blocks per tile."""
    from bit_moe_expert_route_gb300 import ops
    E, N, T, k = 8, 256, 150, 2
    q = synth.q4(synth.key(1, 0, 300), E * N * K // 8).reshape(E, N, K // 8)
    s = np.full((E, N, K // 64), 0x3F80, np.uint16)   # 1.0
    b = np.full((E, N, K // 64), 0xC100, np.uint16)   # -8.0
    xi = synth.uniform_int(synth.key(1, 0, 301), T * K, 5).reshape(T, K) - 2
    x = to_fmt(xi.astype(np.float32), fmt)
    ids, m = routing(orc, T, E, k, bn, seed=bn, with_shared=False)
    rt = torch.from_numpy(m["row_token"]).cuda()
    C, ws = gemm_call(dev(x), [(q, s, b)], E, N, m, bn, ops.EPI_NONE, fmt, row_index=rt)
    assert ops.device_status(ws) == 0
    got = to_np(C)
    for e in range(E):
        W = orc.dequant(q[e], s[e], b[e], 64).astype(np.int64)
        rows = np.arange(m["offsets"][e], m["offsets"][e + 1])
        ref = xi[m["row_token"][rows]].astype(np.int64) @ W.T
        assert np.array_equal(got[rows], ref.astype(np.float32)), f"expert {e}"


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_one_hot_reads_back_dequantised_weights(orc, fmt):
    """C[r, n] = W_g[n, r % K] exactly: every (row, k) of two experts' gate weights."""
    from bit_moe_expert_route_gb300 import ops
    full = LayerShape()
    K, N, G = full.d_model, full.d_ff, 2
    q, s, b = synth.w4_projection(LayerShape(n_experts=G), seed=3, layer=0, p=0)
    A = np.zeros((K, K), np.uint16)
    A[np.arange(K), np.arange(K)] = to_fmt(np.ones(1), fmt)[0]
    bn = 128
    bmap = [[g, g * K + r0, min(bn, K - r0), 0] for g in range(G) for r0 in range(0, K, bn)]
    m = dict(block_map=np.array(bmap, np.int32), num_tiles=len(bmap))
    row_index = torch.from_numpy(np.tile(np.arange(K, dtype=np.int32), G)).cuda()
    C, ws = gemm_call(dev(A), [(q, s, b)], G, N, m, bn, ops.EPI_NONE, fmt, row_index=row_index)
    assert ops.device_status(ws) == 0
    got = to_np(C).reshape(G, K, N)
    for g in range(G):
        assert np.array_equal(got[g].T, deq(orc, (q, s, b), g, fmt).astype(np.float32)), g


@pytest.mark.parametrize("fmt,bn,T,E,k,K", [
    ("f16", 16, 333, 16, 4, 1024), ("f16", 128, 333, 16, 4, 1024), ("bf16", 64, 333, 16, 4, 1024),
    # experts with 2-3 tiles and ragged last tiles (the MMA's N follows the
    # tile's rows); K/64 not a multiple of 4 (one k-block per packed-code stage)
    ("f16", 128, 700, 8, 3, 1024), ("f16", 128, 333, 16, 4, 320),
    # 256-row tiles: both accumulators fill tensor memory (one buffer)
    ("f16", 256, 700, 8, 3, 1024), ("bf16", 256, 333, 16, 4, 320)])
def test_swiglu_epilogue_with_shared_group(orc, bn, fmt, T, E, k, K):
    from bit_moe_expert_route_gb300 import ops
    shape = LayerShape(d_model=K, n_experts=16, top_k=4, d_ff=256, d_ff_shared=256)
    N = 256
    w = synth.layer_weights(shape, seed=9)
    X = round_fmt(synth.bf16_to_f32(synth.tokens(shape, T, seed=9)), fmt)
    ids, m = routing(orc, T, E, k, bn, seed=9 + bn)
    rt = torch.from_numpy(m["row_token"]).cuda()
    C, ws = gemm_call(dev(to_fmt(X, fmt)), [w["gate"], w["up"]], E, N, m, bn, ops.EPI_SWIGLU,
                      fmt, row_index=rt, extra=[w["sh_gate"], w["sh_up"]])
    assert ops.device_status(ws) == 0
    got = c_np(C, fmt)
    ref = np.zeros_like(got)
    for g in range(E + 1):
        if g < E:
            rows = np.arange(m["offsets"][g], m["offsets"][g + 1])
            Wg, Wu = deq(orc, w["gate"], g, fmt), deq(orc, w["up"], g, fmt)
        else:
            rows = np.arange(T * k, T * k + T)
            Wg, Wu = deq(orc, w["sh_gate"], 0, fmt), deq(orc, w["sh_up"], 0, fmt)
        xr = X[m["row_token"][rows]]
        gg, uu = xr @ Wg.T, xr @ Wu.T
        ref[rows] = gg / (1 + np.exp(-gg)) * uu
    err = got - ref
    tol = 1e-3 if fmt == "f16" else 4e-3  # rounding of h to the operand format dominates
    assert np.linalg.norm(err) / np.linalg.norm(ref) < tol
    assert np.max(np.abs(err) / (np.abs(ref) + 1e-2 * np.sqrt(np.mean(ref ** 2)))) < 5 * tol


@pytest.mark.parametrize("K", [1024, 320])
def test_swiglu_tile_height_leaves_h_unchanged(orc, K):
    """Each output row is the same sum over K whatever tile it sits in: the
    gate/up products on 256-row tiles equal those on 128-row tiles bit for bit."""
    from bit_moe_expert_route_gb300 import ops
    T, E, k, N = 1500, 8, 3, 256
    shape = LayerShape(d_model=K, n_experts=16, top_k=4, d_ff=256, d_ff_shared=256)
    w = synth.layer_weights(shape, seed=11)
    X = round_fmt(synth.bf16_to_f32(synth.tokens(shape, T, seed=11)), "f16")
    outs = []
    for bn in (128, 256):
        ids, m = routing(orc, T, E, k, bn, seed=11)
        rt = torch.from_numpy(m["row_token"]).cuda()
        C, ws = gemm_call(dev(to_fmt(X, "f16")), [w["gate"], w["up"]], E, N, m, bn, ops.EPI_SWIGLU,
                          "f16", row_index=rt, extra=[w["sh_gate"], w["sh_up"]])
        assert ops.device_status(ws) == 0
        outs.append(C.view(torch.int16).cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("fmt,bn", [("f16", 32), ("bf16", 64), ("f16", 256)])
def test_combine_epilogue(orc, bn, fmt):
    from bit_moe_expert_route_gb300 import ops
    shape = LayerShape(d_model=512, n_experts=8, top_k=3, d_ff=256, d_ff_shared=256)
    T, E, k, d, f = 200, 8, 3, 512, 256
    w = synth.layer_weights(shape, seed=13)
    ids, m = routing(orc, T, E, k, bn, seed=13 + bn)
    rows = T * k + T
    H = round_fmt(synth.normal_f32(synth.key(13, 0, 400), rows * f, 1.0).reshape(rows, f), fmt)
    scale = synth.normal_f32(synth.key(13, 0, 401), rows, 0.5)
    out = torch.zeros(T, d, dtype=torch.float32, device="cuda")
    C, ws = gemm_call(dev(to_fmt(H, fmt)), [w["down"]], E, d, m, bn, ops.EPI_COMBINE, fmt,
                      extra=[w["sh_down"]], row_scale=torch.from_numpy(scale).cuda(),
                      out_row=torch.from_numpy(m["row_token"]).cuda(), C=out)
    assert ops.device_status(ws) == 0
    ref = np.zeros((T, d))
    for g in range(E + 1):
        r = (np.arange(m["offsets"][g], m["offsets"][g + 1]) if g < E
             else np.arange(T * k, rows))
        Wd = deq(orc, w["down"], g, fmt) if g < E else deq(orc, w["sh_down"], 0, fmt)
        np.add.at(ref, m["row_token"][r], scale[r, None] * (H[r] @ Wd.T))
    got = to_np(out).astype(np.float64)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-5
    assert np.max(np.abs(got - ref)) < 1e-4 * np.max(np.abs(ref))


def test_empty_work_leaves_output_untouched(orc):
    from bit_moe_expert_route_gb300 import ops
    K, N = 256, 128
    q, s, b = synth.w4_projection(LayerShape(d_model=K, d_ff=N, n_experts=2), 4, 0, 0)
    m = dict(block_map=np.zeros((0, 4), np.int32), num_tiles=0)
    A = dev(synth.tokens(LayerShape(d_model=K), 4, seed=4))
    C = torch.full((4, N), 7.0, device="cuda")
    C, ws = gemm_call(A, [(q, s, b)], 2, N, m, 16, ops.EPI_NONE, "bf16", C=C)
    assert ops.device_status(ws) == 0 and bool((C == 7.0).all())


def test_bad_block_map_and_rows_are_rejected_on_device(orc):
    """Out-of-range entries are refused by the kernel's own checks (no access)."""
    from bit_moe_expert_route_gb300 import ops
    K, N = 256, 128
    q, s, b = synth.w4_projection(LayerShape(d_model=K, d_ff=N, n_experts=2), 4, 0, 0)
    A = dev(synth.tokens(LayerShape(d_model=K), 8, seed=4))
    bad_group = dict(block_map=np.array([[5, 0, 4, 0]], np.int32), num_tiles=1)
    C, ws = gemm_call(A, [(q, s, b)], 2, N, bad_group, 16, ops.EPI_NONE, "bf16", n_rows=8)
    assert ops.device_status(ws) == ops.DEV_BAD_TILE
    bad_rows = dict(block_map=np.array([[0, 6, 4, 0]], np.int32), num_tiles=1)  # 6+4 > 8
    C, ws = gemm_call(A, [(q, s, b)], 2, N, bad_rows, 16, ops.EPI_NONE, "bf16", n_rows=8)
    assert ops.device_status(ws) == ops.DEV_BAD_TILE
    ri = torch.tensor([0, 1, 99, 3], dtype=torch.int32, device="cuda")  # row 99 of 8
    ok_map = dict(block_map=np.array([[1, 0, 4, 0]], np.int32), num_tiles=1)
    C = torch.full((4, N), 7.0, device="cuda")
    C, ws = gemm_call(A, [(q, s, b)], 2, N, ok_map, 16, ops.EPI_NONE, "bf16", row_index=ri, C=C)
    assert ops.device_status(ws) == ops.DEV_BAD_ROW
    assert bool((C[2] == 0).all()) and bool((C[0] != 7.0).any())  # refused row reads as zeros
