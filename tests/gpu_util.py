"""Helpers shared by the GPU tests: inputs come from the seeded generators,
expected values from the oracle; nothing here computes the layer."""
import numpy as np

from bit_moe_expert_route_gb300 import synth
from bit_moe_expert_route_gb300.synth import LayerShape

FULL = LayerShape()  # d 2048, 256 experts, top-8, d_ff 512, shared 512, group 64


def logits_like_router(T, E, seed, zipf=False):
    """fp32 logits with the router's spread (x ~ N(0,1), W_r ~ N(0, 0.02), d = 2048)."""
    lg = synth.normal_f32(synth.key(seed, 0, 100), T * E, 0.02 * np.sqrt(2048)).reshape(T, E)
    bias = synth.zipf_router_bias(E) if zipf else None
    return lg, bias


def to_np(t):
    return t.detach().cpu().numpy()


def bf16_np(t):
    """bf16 device tensor -> float32 numpy."""
    return synth.bf16_to_f32(to_np(t.view(__import__("torch").int16)).view(np.uint16))


def bf16_half_ulp(v):
    """Half the bf16 spacing at |v| (the most a round-to-nearest bf16 store can move v)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 8)


def tolerance_check(got, ref, bf16_output=False):
    """Layer-output bar: max|err| <= 2e-2 * rms(ref) and ||err|| / ||ref|| <= 5e-3.

    bf16_output: `got` went through a final round-to-nearest bf16 store; that
    store alone may move an element by half a bf16 spacing (0.125 at |v| >= 32,
    above the bar whenever rms(ref) < 6.25), so the per-element bound is the bar
    plus half a bf16 spacing at that element. rel-L2 keeps the plain bar."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = got - ref
    rms = np.sqrt(np.mean(ref ** 2))
    bound = 2e-2 * rms + (bf16_half_ulp(np.maximum(np.abs(got), np.abs(ref))) if bf16_output else 0.0)
    worst = float(np.max(np.abs(err) - bound))
    rel_l2 = float(np.linalg.norm(err) / np.linalg.norm(ref))
    return worst <= 0 and rel_l2 <= 5e-3, dict(max_err=float(np.max(np.abs(err))), rms=rms,
                                              rel_l2=rel_l2, worst_over_bound=worst)
