"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin compares the oracle with one of
  * values worked by hand (tests/golden/*.json, each with its source),
  * an independent numpy formulation (vectorised bit unpacking, BLAS matmuls,
    a stable library sort, a dense evaluation of every expert masked by a
    one-hot top-k mask with softmax-then-renormalise weights),
  * closed forms and special cases (unit-vector inputs read back weight rows,
    all-zero weights give a zero output, E=1/k=1 is a plain SwiGLU MLP,
    k=E is a dense softmax mixture),
  * invariants of the routing metadata.
`test_planted_mistakes_are_caught` rebuilds the oracle with one known mistake
at a time and requires every one of them to fail at least one pin.
"""
import json
import os

import numpy as np
import pytest

from bit_moe_expert_route_gb300 import synth
from bit_moe_expert_route_gb300.synth import LayerShape

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TINY = LayerShape(d_model=128, n_experts=16, top_k=4, d_ff=64, d_ff_shared=64, group=64)


# ---------------------------------------------------------------- numpy side
def bf(a):
    return synth.bf16_to_f32(np.asarray(a, np.uint16)).astype(np.float64)


def np_codes(q):
    """[..., K/8] uint32 -> [..., K] codes, low nibble first."""
    q = np.asarray(q, np.uint32)
    c = (q[..., :, None] >> (np.uint32(4) * np.arange(8, dtype=np.uint32))) & np.uint32(15)
    return c.reshape(q.shape[:-1] + (q.shape[-1] * 8,)).astype(np.float64)


def np_dequant(q, s, b, group):
    c = np_codes(q)
    return c * np.repeat(bf(s), group, axis=-1) + np.repeat(bf(b), group, axis=-1)


def np_swiglu(X, gate, up, down, group, e):
    Wg = np_dequant(gate[0][e], gate[1][e], gate[2][e], group)
    Wu = np_dequant(up[0][e], up[1][e], up[2][e], group)
    Wd = np_dequant(down[0][e], down[1][e], down[2][e], group)
    g = X @ Wg.T
    return ((g / (1.0 + np.exp(-g))) * (X @ Wu.T)) @ Wd.T


def np_dense_layer(x, w, shape, logits):
    """Every expert on every token, masked by a one-hot top-k mask."""
    X = bf(x)
    T, E, k = X.shape[0], shape.n_experts, shape.top_k
    z = logits.astype(np.float32)
    if w.get("router_bias") is not None:
        z = (z + w["router_bias"][None, :]).astype(np.float32)
    zz = z.astype(np.float64)
    beats = (zz[:, None, :] > zz[:, :, None]) | (
        (zz[:, None, :] == zz[:, :, None]) & (np.arange(E)[None, None, :] < np.arange(E)[None, :, None]))
    rank = beats.sum(axis=2)  # rank[t, e]
    sel = rank < k
    p = np.exp(zz - zz.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    m = np.where(sel, p, 0.0)
    m /= m.sum(axis=1, keepdims=True)
    out = np.zeros((T, shape.d_model))
    for e in range(E):
        out += m[:, e:e + 1] * np_swiglu(X, w["gate"], w["up"], w["down"], shape.group, e)
    if w.get("shared_gate") is not None:
        s = (X @ w["shared_gate"].astype(np.float64)).astype(np.float32).astype(np.float64)
        out += (1.0 / (1.0 + np.exp(-s)))[:, None] * np_swiglu(
            X, w["sh_gate"], w["sh_up"], w["sh_down"], shape.group, 0)
    return out


def rel_err(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ---------------------------------------------------------------- the pins
def pin_dequant_golden(orc):
    with open(os.path.join(GOLDEN, "dequant_known.json")) as f:
        g = json.load(f)
    for row in g["rows"]:
        q = np.array([[int(h, 16) for h in row["words_hex"]]], np.uint32)
        s = np.array([[int(row["scale_bf16_hex"], 16)]], np.uint16)
        b = np.array([[int(row["bias_bf16_hex"], 16)]], np.uint16)
        got = orc.dequant(q, s, b, g["group"])[0]
        assert np.array_equal(got, np.array(row["expect"], np.float64)), got


def pin_dequant_random_vs_numpy(orc):
    q, s, b = synth.w4_projection(LayerShape(d_model=256, d_ff=32, n_experts=3), 7, 0, 0)
    got = orc.dequant(q, s, b, 64)
    assert np.array_equal(got, np_dequant(q, s, b, 64))


def pin_router_unit_vectors(orc):
    # x_t = e_{k_t} reads back row k_t of W_r and entry k_t of w_sg exactly
    d, E = 96, 40
    Wr = synth.normal_f32(synth.key(3, 0, 2), d * E, 0.02).reshape(d, E)
    wsg = synth.normal_f32(synth.key(3, 0, 3), d, 0.02)
    ks = np.array([0, 5, 95, 17])
    x = np.zeros((len(ks), d), np.uint16)
    x[np.arange(len(ks)), ks] = 0x3F80  # bf16 1.0
    logits, gl = orc.router(x, Wr, wsg)
    assert np.array_equal(logits, Wr[ks]) and np.array_equal(gl, wsg[ks])


def pin_router_vs_blas(orc):
    d, E, T = 2048, 64, 5
    Wr = synth.normal_f32(synth.key(4, 0, 2), d * E, 0.02).reshape(d, E)
    x = synth.tokens(LayerShape(d_model=d), T, seed=4)
    logits, _ = orc.router(x, Wr)
    ref = bf(x) @ Wr.astype(np.float64)
    bound = 1e-6 * (np.abs(bf(x)) @ np.abs(Wr.astype(np.float64)))
    assert np.all(np.abs(logits - ref) <= bound + 1e-30)


def pin_topk_vs_stable_sort(orc):
    T, E, k = 300, 64, 8
    logits = synth.normal_f32(synth.key(5, 0, 9), T * E, 1.0).reshape(T, E)
    logits[:, 7] = logits[:, 9]  # exact ties between two experts on every token
    bias = synth.normal_f32(synth.key(5, 0, 10), E, 0.3)
    ids, w = orc.topk(logits, k, bias)
    z = (logits + bias[None, :]).astype(np.float32)
    ref_ids = np.argsort(-z, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref_ids)
    p = np.exp(z.astype(np.float64) - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, ref_ids, axis=1)
    assert np.allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-6, atol=0)


def pin_topk_ties_and_sums(orc):
    E, k = 32, 8
    ids, w = orc.topk(np.zeros((2, E), np.float32), k)
    assert np.array_equal(ids, np.tile(np.arange(k), (2, 1)))
    assert np.all(w == np.float32(1.0 / k))
    logits = synth.normal_f32(synth.key(6, 0, 9), 50 * E, 2.0).reshape(50, E)
    ids, w = orc.topk(logits, k)
    assert np.allclose(w.sum(axis=1, dtype=np.float64), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)


def pin_route_golden(orc):
    with open(os.path.join(GOLDEN, "route_tiny.json")) as f:
        g = json.load(f)
    r = orc.route_meta(np.array(g["ids"], np.int32), g["E"], g["block_n"], True)
    for key in ("counts", "offsets", "perm", "inv_perm", "row_token", "block_map"):
        assert np.array_equal(r[key], np.array(g[key])), key
    assert r["num_tiles"] == g["num_tiles"]


def check_route_invariants(ids, E, block_n, r, with_shared=True):
    T, k = ids.shape
    A = T * k
    c, off, perm = r["counts"], r["offsets"], r["perm"]
    assert c.sum() == A and off[0] == 0 and off[E] == A and np.all(np.diff(off) == c)
    assert np.array_equal(np.sort(perm), np.arange(A))
    flat = ids.reshape(-1)
    e_of = flat[perm]
    assert np.all(np.diff(e_of) >= 0)
    same = np.diff(e_of) == 0
    assert np.all(np.diff(perm)[same] > 0)  # stable inside an expert
    assert np.array_equal(r["inv_perm"][perm], np.arange(A))
    assert np.array_equal(r["row_token"][:A], perm // k)
    if with_shared:
        assert np.array_equal(r["row_token"][A:], np.arange(T))
    covered = np.zeros(A + (T if with_shared else 0), np.int32)
    for g, start, rows, _ in r["block_map"]:
        assert 1 <= rows <= block_n
        if g < E:
            assert off[g] <= start and start + rows <= off[g + 1]
            assert rows == block_n or start + rows == off[g + 1]
        else:
            assert g == E and with_shared and A <= start and start + rows <= A + T
        covered[start:start + rows] += 1
    assert np.all(covered == 1)
    n_exp = int(np.sum(-(-c // block_n))) + (-(-T // block_n) if with_shared else 0)
    assert r["num_tiles"] == n_exp


def pin_route_invariants_and_lexsort(orc):
    T, E, k, bn = 1000, 64, 8, 16
    keys = synth.normal_f32(synth.key(8, 0, 11), T * E, 1.0).reshape(T, E)
    ids = np.argsort(keys, axis=1)[:, :k].astype(np.int32)  # distinct experts per token
    ids[:5] = np.arange(k)  # a few identical rows
    r = orc.route_meta(ids, E, bn, True)
    check_route_invariants(ids, E, bn, r)
    flat = ids.reshape(-1)
    assert np.array_equal(r["perm"], np.lexsort((np.arange(T * k), flat)))
    assert np.array_equal(r["counts"], np.bincount(flat, minlength=E))


def pin_expert_is_plain_swiglu(orc):
    shape = LayerShape(d_model=256, n_experts=2, d_ff=128, group=64)
    gate = synth.w4_projection(shape, 9, 0, 0)
    up = synth.w4_projection(shape, 9, 0, 1)
    down = synth.w4_projection(shape, 9, 0, 2)
    x = synth.tokens(shape, 6, seed=9)
    for e in (0, 1):
        got = orc.expert(x, gate, up, down, 64, g=e)
        ref = np_swiglu(bf(x), gate, up, down, 64, e)
        assert rel_err(got, ref) < 1e-12


def _tiny_layer(seed, shape=TINY, bias=False):
    w = synth.layer_weights(shape, seed=seed, layer=0)
    if bias:
        w["router_bias"] = synth.zipf_router_bias(shape.n_experts, 0.5)
    x = synth.tokens(shape, 24, seed=seed)
    return x, w


def pin_layer_dense_bruteforce(orc, k=4, bias=False):
    shape = LayerShape(**{**TINY.__dict__, "top_k": k})
    x, w = _tiny_layer(11 + k, shape, bias)
    ref_logits = bf(x) @ w["router"].astype(np.float64)
    o = orc.moe_forward(x, w, shape)
    assert np.allclose(o["logits"], ref_logits, rtol=1e-6, atol=1e-7)
    o = orc.moe_forward(x, w, shape, logits_in=ref_logits.astype(np.float32))
    ref = np_dense_layer(x, w, shape, ref_logits.astype(np.float32))
    assert rel_err(o["out"], ref) < 1e-6


def pin_layer_dense_k_eq_E(orc):
    pin_layer_dense_bruteforce(orc, k=TINY.n_experts)


def pin_layer_dense_bias(orc):
    pin_layer_dense_bruteforce(orc, k=2, bias=True)


def pin_zero_weights_give_zero(orc):
    x, w = _tiny_layer(21)
    for name in synth.PROJ:
        q, s, b = w[name]
        q[:] = 0x88888888
        b[:] = synth.f32_to_bf16(-8.0 * synth.bf16_to_f32(s))  # exact: -8*s is a bf16
    o = orc.moe_forward(x, w, TINY)
    assert np.all(o["out"] == 0.0)


def pin_single_expert_top1(orc):
    shape = LayerShape(d_model=128, n_experts=1, top_k=1, d_ff=64, d_ff_shared=64, group=64)
    w = synth.layer_weights(shape, seed=23, shared=False)
    x = synth.tokens(shape, 5, seed=23)
    o = orc.moe_forward(x, w, shape)
    assert np.all(o["w"] == 1.0)
    assert rel_err(o["out"], np_swiglu(bf(x), w["gate"], w["up"], w["down"], 64, 0)) < 1e-6


def pin_shared_gate(orc):
    x, w = _tiny_layer(25)
    for name in ("gate", "up", "down"):  # routed experts contribute nothing
        q, s, b = w[name]
        q[:] = 0x88888888
        b[:] = synth.f32_to_bf16(-8.0 * synth.bf16_to_f32(s))
    o = orc.moe_forward(x, w, TINY)
    X = bf(x)
    s = (X @ w["shared_gate"].astype(np.float64)).astype(np.float32).astype(np.float64)
    ref = (1 / (1 + np.exp(-s)))[:, None] * np_swiglu(X, w["sh_gate"], w["sh_up"], w["sh_down"], 64, 0)
    assert rel_err(o["out"], ref) < 1e-6
    assert np.allclose(o["gate"], 1 / (1 + np.exp(-s)), rtol=1e-6)


PINS = [
    pin_dequant_golden, pin_dequant_random_vs_numpy, pin_router_unit_vectors, pin_router_vs_blas,
    pin_topk_vs_stable_sort, pin_topk_ties_and_sums, pin_route_golden,
    pin_route_invariants_and_lexsort, pin_expert_is_plain_swiglu, pin_layer_dense_bruteforce,
    pin_layer_dense_k_eq_E, pin_layer_dense_bias, pin_zero_weights_give_zero,
    pin_single_expert_top1, pin_shared_gate,
]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


MUTANTS = {
    1: "nibble order reversed",
    2: "bias term dropped",
    3: "silu on the up projection",
    4: "weights not renormalised over the top k",
    5: "ties go to the higher expert id",
    6: "shared expert gate without sigmoid",
    7: "scale/bias read with a transposed layout",
    8: "router weight read transposed",
    9: "scatter not stable within an expert",
    10: "last tile of an expert not ragged",
    11: "routing weights not applied in the combine",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_planted_mistakes_are_caught(mutant):
    from oracle import Oracle
    bad = Oracle(mutant)
    failed = []
    for pin in PINS:
        try:
            pin(bad)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake '{MUTANTS[mutant]}' passed every pin"


def test_route_invariants_hold_for_random_shapes(orc):
    """Property test of the routing invariants (counts, offsets, stable
    permutation and its inverse, row tokens, block map covering every row once
    with the exact tile count) over random token counts (including none),
    expert counts, top-k, tile heights and with or without the shared rows."""
    pytest.importorskip("hypothesis")
    from hypothesis import given, settings, strategies as st

    @settings(max_examples=80, deadline=None)
    @given(T=st.integers(0, 300), E=st.sampled_from([8, 16, 72, 256]), k=st.integers(1, 8),
           bn=st.sampled_from([16, 32, 64, 128, 256]), shared=st.booleans(),
           seed=st.integers(0, 2 ** 31 - 1))
    def prop(T, E, k, bn, shared, seed):
        rng = np.random.default_rng(seed)
        ids = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
        r = orc.route_meta(ids, E, bn, shared)
        check_route_invariants(ids, E, bn, r, shared)

    prop()
