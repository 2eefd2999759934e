"""Pins of the decode-attention oracle (oracle/attn.py), CPU only.

A1  one cached position: the output is that position's value, whatever q is.
A2  all keys equal: every position gets the same weight, the output is the
    mean of the values.
A3  one key aligned with q and the others orthogonal to it, with a score gap
    of s: the weights are e^s / (e^s + L - 1) and 1 / (e^s + L - 1) (closed
    form of the softmax), so o = (e^s v_m + sum of the others) / (e^s + L - 1).
A4  grouped heads: query head h equals a one-head call on KV head
    h // (Hq / Hkv); heads of one group with the same query agree.
A5  permuting the cache positions (keys and values together) changes nothing,
    and the output is linear in the values.
A6  all-one values give an all-one output (the weights sum to one).
Each planted mistake (the oracle's `mutant`) fails at least one pin.
"""
import math

import numpy as np
import pytest

from oracle.attn import decode_attention


def rand(L, Hq, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((Hq, d)), rng.standard_normal((L, Hkv, d)),
            rng.standard_normal((L, Hkv, d)))


def pin_single_position(mutant=0):
    q, K, V = rand(1, 4, 2, 8, 1)
    o = decode_attention(q, K, V, mutant=mutant)
    return np.allclose(o, V[0][np.arange(4) // 2], rtol=0, atol=1e-15)


def pin_equal_keys(mutant=0):
    q, K, V = rand(9, 4, 2, 8, 2)
    K[:] = K[0]
    o = decode_attention(q, K, V, mutant=mutant)
    ref = V.mean(axis=0)[np.arange(4) // 2]
    return np.allclose(o, ref, rtol=1e-13, atol=1e-14)


def pin_aligned_key(mutant=0):
    L, d, m, gap = 7, 4, 3, 2.0
    rng = np.random.default_rng(3)
    q = np.zeros((1, d))
    q[0, 0] = 1.0
    K = np.zeros((L, 1, d))
    K[:, 0, 1] = rng.standard_normal(L)  # orthogonal to q: score 0
    K[m, 0] = 0.0
    K[m, 0, 0] = gap * math.sqrt(d)      # scaled score = gap
    V = rng.standard_normal((L, 1, d))
    o = decode_attention(q, K, V, mutant=mutant)
    e = math.exp(gap)
    ref = (e * V[m, 0] + V[:, 0].sum(axis=0) - V[m, 0]) / (e + L - 1)
    return np.allclose(o[0], ref, rtol=1e-13, atol=1e-14)


def pin_grouped_heads(mutant=0):
    L, Hq, Hkv, d = 11, 8, 2, 6
    q, K, V = rand(L, Hq, Hkv, d, 4)
    q[1] = q[0]
    o = decode_attention(q, K, V, mutant=mutant)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        o1 = decode_attention(q[h:h + 1], K[:, g:g + 1], V[:, g:g + 1])
        if not np.allclose(o[h], o1[0], rtol=1e-13, atol=1e-15):
            return False
    return np.allclose(o[0], o[1], rtol=0, atol=1e-15)


def pin_permutation_and_linearity(mutant=0):
    L, Hq, Hkv, d = 13, 4, 1, 5
    q, K, V = rand(L, Hq, Hkv, d, 5)
    o = decode_attention(q, K, V, mutant=mutant)
    perm = np.random.default_rng(6).permutation(L)
    op = decode_attention(q, K[perm], V[perm], mutant=mutant)
    V2 = np.random.default_rng(7).standard_normal(V.shape)
    lin = decode_attention(q, K, 2.0 * V - 3.0 * V2, mutant=mutant)
    ref = 2.0 * o - 3.0 * decode_attention(q, K, V2, mutant=mutant)
    return np.allclose(o, op, rtol=1e-13, atol=1e-14) and np.allclose(lin, ref, rtol=1e-12,
                                                                       atol=1e-13)


def pin_values_all_one(mutant=0):
    """The output is a convex combination of value rows: all-one values give ones."""
    q, K, _ = rand(23, 8, 2, 16, 8)
    o = decode_attention(q, K, np.ones((23, 2, 16)), mutant=mutant)
    return np.allclose(o, 1.0, rtol=0, atol=1e-13)


PINS = [pin_single_position, pin_equal_keys, pin_aligned_key, pin_grouped_heads,
        pin_permutation_and_linearity, pin_values_all_one]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin_holds(pin):
    assert pin()


@pytest.mark.parametrize("mutant", [1, 2, 3, 4])
def test_planted_mistake_is_caught(mutant):
    assert not all(pin(mutant) for pin in PINS), f"mutant {mutant} passed every pin"


def test_pins_for_random_shapes():
    """A4-A6 over random cache lengths, head counts, group sizes and head dims."""
    pytest.importorskip("hypothesis")
    from hypothesis import given, settings, strategies as st

    @settings(max_examples=60, deadline=None)
    @given(L=st.integers(1, 40), Hkv=st.integers(1, 3), group=st.integers(1, 8),
           d=st.integers(1, 12), seed=st.integers(0, 2 ** 31 - 1))
    def prop(L, Hkv, group, d, seed):
        Hq = Hkv * group
        q, K, V = rand(L, Hq, Hkv, d, seed)
        o = decode_attention(q, K, V)
        assert np.allclose(decode_attention(q, K, np.ones_like(V)), 1.0, rtol=0, atol=1e-12)
        perm = np.random.default_rng(seed + 1).permutation(L)
        assert np.allclose(decode_attention(q, K[perm], V[perm]), o, rtol=1e-12, atol=1e-13)
        for h in range(Hq):
            g = h // group
            o1 = decode_attention(q[h:h + 1], K[:, g:g + 1], V[:, g:g + 1])
            assert np.allclose(o[h], o1[0], rtol=1e-13, atol=1e-14)

    prop()

