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


def tolerance_check(got, ref):
    """Layer-output bar: max|err| <= 2e-2 * rms(ref) and ||err|| / ||ref|| <= 5e-3."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = got - ref
    rms = np.sqrt(np.mean(ref ** 2))
    max_err = float(np.max(np.abs(err)))
    rel_l2 = float(np.linalg.norm(err) / np.linalg.norm(ref))
    return max_err <= 2e-2 * rms and rel_l2 <= 5e-3, dict(max_err=max_err, rms=rms,
                                                          rel_l2=rel_l2)
