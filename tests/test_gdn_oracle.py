"""Pins of the gated delta rule oracle (oracle/gdn.py), CPU only.

G1  beta = 0: nothing is written, the state only decays:
    o_t = (alpha_1 ... alpha_t) S_0 q_t.
G2  alpha = 1, beta = 1 and unit-vector keys e_j: the delta rule overwrites
    column j of the state with v_t and leaves the others; a unit-vector query
    e_m reads column m back.
G3  the product form, evaluated with explicit d_k x d_k matrices:
    S_t = S_{t-1} A_t + beta_t v_t k_t^T, A_t = alpha_t (I - beta_t k_t k_t^T),
    and o_t = S_t q_t (a different formula from the oracle's update).
G4  grouped heads: value head h of a multi-head scan equals a one-head scan on
    key head h // (Hv / Hk).
Each planted mistake (the oracle's `mutant`) fails at least one pin.
"""
import numpy as np
import pytest

from oracle.gdn import gdn_scan


def rand_inputs(T, Hk, Hv, dk, dv, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, Hk, dk))
    k = rng.standard_normal((T, Hk, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, Hv, dv))
    alpha = rng.uniform(0.8, 1.0, (T, Hv))
    beta = rng.uniform(0.0, 1.0, (T, Hv))
    S0 = 0.1 * rng.standard_normal((Hv, dv, dk))
    return q, k, v, alpha, beta, S0


def pin_beta_zero(mutant=0):
    q, k, v, alpha, _, S0 = rand_inputs(7, 2, 4, 8, 6, 1)
    o, S = gdn_scan(q, k, v, alpha, np.zeros_like(alpha), S0, mutant)
    decay = np.cumprod(alpha, axis=0)  # [T, Hv]
    for t in range(7):
        for h in range(4):
            ref = decay[t, h] * S0[h] @ q[t, h // 2]
            if not np.allclose(o[t, h], ref, rtol=1e-12, atol=1e-14):
                return False
    return np.allclose(S, decay[-1][:, None, None] * S0, rtol=1e-12, atol=1e-14)


def pin_overwrite(mutant=0):
    T, dk, dv = 9, 5, 3
    rng = np.random.default_rng(2)
    cols = [0, 3, 1, 3, 4, 0, 2, 2, 1]
    k = np.zeros((T, 1, dk))
    k[np.arange(T), 0, cols] = 1.0
    reads = [4, 3, 1, 0, 2, 0, 2, 3, 1]
    q = np.zeros((T, 1, dk))
    q[np.arange(T), 0, reads] = 1.0
    v = rng.standard_normal((T, 1, dv))
    S0 = rng.standard_normal((1, dv, dk))
    o, S = gdn_scan(q, k, v, np.ones((T, 1)), np.ones((T, 1)), S0, mutant)
    ref = S0[0].copy()
    for t in range(T):
        ref[:, cols[t]] = v[t, 0]  # column j now holds the latest value written at key e_j
        if not np.allclose(o[t, 0], ref[:, reads[t]], rtol=0, atol=1e-14):
            return False
    return np.allclose(S[0], ref, rtol=0, atol=1e-14)


def pin_product_form(mutant=0):
    T, Hk, Hv, dk, dv = 6, 1, 1, 4, 3
    q, k, v, alpha, beta, S0 = rand_inputs(T, Hk, Hv, dk, dv, 3)
    o, S = gdn_scan(q, k, v, alpha, beta, S0, mutant)
    St = S0[0]
    for t in range(T):
        kt = k[t, 0][:, None]
        A = alpha[t, 0] * (np.eye(dk) - beta[t, 0] * kt @ kt.T)
        St = St @ A + beta[t, 0] * v[t, 0][:, None] @ kt.T
        if not np.allclose(o[t, 0], St @ q[t, 0], rtol=1e-11, atol=1e-13):
            return False
    return np.allclose(S[0], St, rtol=1e-11, atol=1e-13)


def pin_grouped_heads(mutant=0):
    T, Hk, Hv, dk, dv = 5, 2, 6, 4, 3
    q, k, v, alpha, beta, S0 = rand_inputs(T, Hk, Hv, dk, dv, 4)
    o, S = gdn_scan(q, k, v, alpha, beta, S0, mutant)
    for h in range(Hv):
        hk = h // (Hv // Hk)
        o1, S1 = gdn_scan(q[:, hk:hk + 1], k[:, hk:hk + 1], v[:, h:h + 1], alpha[:, h:h + 1],
                          beta[:, h:h + 1], S0[h:h + 1])
        if not (np.allclose(o[:, h], o1[:, 0], rtol=1e-13, atol=1e-15)
                and np.allclose(S[h], S1[0], rtol=1e-13, atol=1e-15)):
            return False
    return True


PINS = [pin_beta_zero, pin_overwrite, pin_product_form, pin_grouped_heads]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin_holds(pin):
    assert pin()


@pytest.mark.parametrize("mutant", [1, 2, 3, 4])
def test_planted_mistake_is_caught(mutant):
    assert not all(pin(mutant) for pin in PINS), f"mutant {mutant} passed every pin"


def test_decay_only_state_matches_closed_form_over_long_scan():
    """A long scan with beta = 0 and constant alpha: S_T = alpha^T S_0 exactly up to
    rounding (no drift from the update's other terms)."""
    q, k, v, _, _, S0 = rand_inputs(200, 1, 1, 4, 4, 5)
    o, S = gdn_scan(q, k, v, np.full((200, 1), 0.99), np.zeros((200, 1)), S0)
    assert np.allclose(S, 0.99 ** 200 * S0, rtol=1e-12)


def test_product_form_for_random_shapes():
    """The product-form pin (G3) over random sequence lengths, head sizes, grouped
    heads, decays and write strengths (including alpha = 1 and beta = 0 or 1)."""
    pytest.importorskip("hypothesis")
    from hypothesis import given, settings, strategies as st

    @settings(max_examples=60, deadline=None)
    @given(T=st.integers(1, 12), Hk=st.integers(1, 3), group=st.integers(1, 3),
           dk=st.integers(1, 7), dv=st.integers(1, 5), seed=st.integers(0, 2 ** 31 - 1),
           edge=st.sampled_from(["none", "alpha1", "beta0", "beta1"]))
    def prop(T, Hk, group, dk, dv, seed, edge):
        Hv = Hk * group
        q, k, v, alpha, beta, S0 = rand_inputs(T, Hk, Hv, dk, dv, seed)
        if edge == "alpha1":
            alpha[:] = 1.0
        elif edge == "beta0":
            beta[:] = 0.0
        elif edge == "beta1":
            beta[:] = 1.0
        o, S = gdn_scan(q, k, v, alpha, beta, S0)
        for h in range(Hv):
            hk = h // group
            St = S0[h]
            for t in range(T):
                kt = k[t, hk][:, None]
                A = alpha[t, h] * (np.eye(dk) - beta[t, h] * kt @ kt.T)
                St = St @ A + beta[t, h] * v[t, h][:, None] @ kt.T
                assert np.allclose(o[t, h], St @ q[t, hk], rtol=1e-10, atol=1e-12)
            assert np.allclose(S[h], St, rtol=1e-10, atol=1e-12)

    prop()
