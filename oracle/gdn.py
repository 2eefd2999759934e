"""Gated DeltaNet recurrence (the gated delta rule), float64 on the CPU.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers. The CUDA library neither
imports nor links this module, and this module imports nothing from the CUDA
package.

Source: "Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple
Silicon", section "What Lily actually does" (30 of the model's 40 layers are
Gated DeltaNet layers: linear attention with a fixed-size recurrent state) and
section "Prefill optimizations", third bullet (the scan carries the state
through every token, one state column per SIMD group, in registers). The page
gives no formula; this module follows the published gated delta rule (Yang,
Kautz and Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta
Rule", 2024). Per value head h, with state S in R^{d_v x d_k}:

    S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
    o_t = S_t q_t

which is S_t = S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T.
Key and query heads are shared by groups of value heads: value head h reads
key/query head h // (Hv / Hk). alpha_t (decay, in (0, 1]) and beta_t (write
strength, in [0, 1]) are per token and value head; q, k, v are given (any
normalisation or gate activation happens before the scan).

mutant (tests only) plants one mistake, so the pins can show they catch it:
  1 the correction term forgets the decay: (v_t - S_{t-1} k_t)
  2 the output reads the state before the update: o_t = S_{t-1} q_t
  3 the output uses the key instead of the query: o_t = S_t k_t
  4 value head h reads key head h % Hk instead of h // (Hv / Hk)
"""
from __future__ import annotations

import numpy as np


def gdn_scan(q, k, v, alpha, beta, S0, mutant: int = 0):
    """q, k [T, Hk, dk]; v [T, Hv, dv]; alpha, beta [T, Hv]; S0 [Hv, dv, dk].
    Returns (o [T, Hv, dv], S_T [Hv, dv, dk]), float64."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    alpha = np.asarray(alpha, np.float64)
    beta = np.asarray(beta, np.float64)
    S = np.array(S0, np.float64, copy=True)
    T, Hk, _ = k.shape
    Hv = v.shape[1]
    group = Hv // Hk
    o = np.zeros((T, Hv, v.shape[2]))
    for t in range(T):
        for h in range(Hv):
            hk = h % Hk if mutant == 4 else h // group
            kt, qt = k[t, hk], q[t, hk]
            a, b = alpha[t, h], beta[t, h]
            prev = S[h].copy()
            pred = prev @ kt                               # S_{t-1} k_t
            corr = v[t, h] - (pred if mutant == 1 else a * pred)
            S[h] = a * prev + b * np.outer(corr, kt)
            if mutant == 2:
                o[t, h] = prev @ qt
            elif mutant == 3:
                o[t, h] = S[h] @ kt
            else:
                o[t, h] = S[h] @ qt
    return o, S
