"""moe_decode_attention against the float64 oracle (oracle/attn.py).

Inputs: bf16 q [Hq, d] and K, V caches [L, Hkv, d] drawn N(0, 1); the oracle
sees the same values exactly. The kernel computes the scores and the softmax
in fp32 (two positions per warp step, a lone last one masked), merges the
warps' partial softmaxes inside each block and then the blocks'; the output is a convex
combination of value rows. Bar: |err| <= 1e-4 * (rms(ref) + |ref|) per element.
"""
import numpy as np
import pytest

from oracle.attn import decode_attention

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def bf16_round(a):
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).view(np.float32)


def close(got, ref):
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    assert np.all(err <= 1e-4 * (rms + np.abs(ref))), float(np.max(err / (rms + np.abs(ref))))


def run(L, Hq, Hkv, d, seed, scale=0.0):
    from bit_moe_expert_route_gb300 import ops
    rng = np.random.default_rng(seed)
    q = bf16_round(rng.standard_normal((Hq, d)))
    K = bf16_round(rng.standard_normal((L, Hkv, d)))
    V = bf16_round(rng.standard_normal((L, Hkv, d)))

    def dev(a):
        return torch.from_numpy(a).cuda().to(torch.bfloat16)
    out = ops.decode_attention(dev(q), dev(K), dev(V), scale=scale)
    torch.cuda.synchronize()
    return out.cpu().numpy(), decode_attention(q, K, V, scale if scale > 0 else None)


@pytest.mark.parametrize("L,Hq,Hkv,d", [(1, 16, 2, 256), (37, 16, 2, 256), (1000, 16, 2, 128),
                                        (300, 4, 4, 64), (4097, 8, 1, 256), (129, 6, 2, 64),
                                        (12, 8, 2, 128)])
def test_matches_oracle(L, Hq, Hkv, d):
    got, ref = run(L, Hq, Hkv, d, seed=L + d)
    close(got, ref)


def test_long_context_and_explicit_scale():
    """32768 cached positions (many slices, many partials per head), and a scale
    other than 1/sqrt(d)."""
    got, ref = run(32768, 16, 2, 256, seed=3)
    close(got, ref)
    got, ref = run(2048, 16, 2, 128, seed=4, scale=0.25)
    close(got, ref)


def test_late_large_scores_move_the_max():
    """Keys planted late in the cache give query head 0 (and its group) scores
    far above the rest, twice, so the running max moves mid-sequence and the
    partial outputs are rescaled; the result is still the oracle's softmax."""
    from bit_moe_expert_route_gb300 import ops
    L, Hq, Hkv, d = 3001, 16, 2, 128
    rng = np.random.default_rng(11)
    q = bf16_round(rng.standard_normal((Hq, d)))
    K = bf16_round(rng.standard_normal((L, Hkv, d)))
    V = bf16_round(rng.standard_normal((L, Hkv, d)))
    u = q[0] / np.linalg.norm(q[0])
    for j, c in ((1500, 60.0), (2900, 120.0), (2901, 121.0)):
        K[j, 0] = bf16_round(c * u)  # head 0's score about c * |q0| / sqrt(d)

    def dev(a):
        return torch.from_numpy(a).cuda().to(torch.bfloat16)
    got = ops.decode_attention(dev(q), dev(K), dev(V))
    torch.cuda.synchronize()
    close(got.cpu().numpy(), decode_attention(q, K, V, None))
