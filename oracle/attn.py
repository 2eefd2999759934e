"""Batch-1 decode attention with grouped KV heads, float64 on the CPU.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers. The CUDA library neither
imports nor links this module, and this module imports nothing from the CUDA
package.

Source: "Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple
Silicon", section "What Lily actually does" (10 of the model's 40 layers are
full attention) and section "Decode optimizations", the paragraph on GQA
packing (eight query heads share one KV head; packing four query heads into
one threadgroup lets them share the KV loads). The page gives no formula; this
is scaled dot-product attention for one new token over a cache of L positions:

    o_h = sum_j softmax_j(scale * q_h . k_{g(h), j}) v_{g(h), j},
    g(h) = h // (Hq / Hkv),

softmax over j = 0 .. L-1 (every cached position is visible to the new
token), scale given (1 / sqrt(d) when the caller passes none).

mutant (tests only) plants one mistake, so the pins can show they catch it:
  1 the scale is left out
  2 query head h reads KV head h % Hkv instead of h // (Hq / Hkv)
  3 the weights are normalised by L instead of by their sum
  4 the keys stand in for the values
"""
from __future__ import annotations

import math

import numpy as np


def decode_attention(q, K, V, scale: float | None = None, mutant: int = 0):
    """q [Hq, d]; K, V [L, Hkv, d]. Returns o [Hq, d], float64."""
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    Hq, d = q.shape
    L, Hkv, _ = K.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    group = Hq // Hkv
    o = np.zeros((Hq, d))
    for h in range(Hq):
        g = h % Hkv if mutant == 2 else h // group
        s = K[:, g] @ q[h]                      # [L] dot products
        if mutant != 1:
            s = s * scale
        w = np.exp(s - s.max())
        w = w / (L if mutant == 3 else w.sum())
        vals = K[:, g] if mutant == 4 else V[:, g]
        o[h] = w @ vals
    return o
