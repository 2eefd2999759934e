"""moe_gdn_scan (the Gated DeltaNet scan) against the float64 oracle.

Inputs are bf16 q, k, v (unit-norm q and k rows, as the layer feeds them),
fp32 decay alpha in [0.8, 1) and write strength beta in [0, 1), fp32 initial
state; the oracle sees the same values exactly. The kernel runs the recurrence
in fp32: every dot product has dk terms and the state update is a contraction
(|alpha| <= 1, ||I - beta k k^T|| <= 1 for unit k), so rounding does not grow
along the scan. Bar: |err| <= 1e-4 * (rms(ref) + |ref|) per element, on the
outputs and on the final state.
"""
import numpy as np
import pytest

from oracle.gdn import gdn_scan

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def bf16_round(a):
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).view(np.float32)


def inputs(T, Hk, Hv, dk, dv, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, Hk, dk))
    k = rng.standard_normal((T, Hk, dk))
    q = bf16_round(q / np.linalg.norm(q, axis=-1, keepdims=True))
    k = bf16_round(k / np.linalg.norm(k, axis=-1, keepdims=True))
    v = bf16_round(rng.standard_normal((T, Hv, dv)))
    alpha = rng.uniform(0.8, 1.0, (T, Hv)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (T, Hv)).astype(np.float32)
    S0 = (0.1 * rng.standard_normal((Hv, dv, dk))).astype(np.float32)
    return q, k, v, alpha, beta, S0


def to_dev(q, k, v, alpha, beta, S0):
    def b16(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(torch.bfloat16)
    return (b16(q), b16(k), b16(v), torch.from_numpy(alpha).cuda(), torch.from_numpy(beta).cuda(),
            torch.from_numpy(S0.copy()).cuda())


def close(got, ref):
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    assert np.all(err <= 1e-4 * (rms + np.abs(ref))), float(np.max(err / (rms + np.abs(ref))))


@pytest.mark.parametrize("T,Hk,Hv,dk,dv", [(1, 2, 4, 128, 128), (5, 2, 4, 128, 64),
                                           (64, 2, 4, 64, 128), (64, 1, 3, 128, 8),
                                           (300, 4, 8, 128, 128),
                                           # 2 rows per warp (dv % 32 != 0); chunk edges at 32, 64
                                           (65, 2, 2, 64, 48), (33, 1, 2, 128, 16)])
def test_scan_matches_oracle(T, Hk, Hv, dk, dv):
    from bit_moe_expert_route_gb300 import ops
    host = inputs(T, Hk, Hv, dk, dv, seed=T + dk)
    q, k, v, al, be, S = to_dev(*host)
    out = ops.gdn_scan(q, k, v, al, be, S)
    torch.cuda.synchronize()
    ref_o, ref_S = gdn_scan(*host)
    close(out.cpu().numpy(), ref_o)
    close(S.cpu().numpy(), ref_S)


def test_scan_at_layer_size_sampled_heads():
    """T = 4096 tokens, 16 key heads, 32 value heads, d_k = d_v = 128 (the layer the
    benchmark times): heads 0, 17 and 31 against one-head oracle scans on their key
    heads (value head h reads key head h // 2)."""
    from bit_moe_expert_route_gb300 import ops
    T, Hk, Hv, dk, dv = 4096, 16, 32, 128, 128
    q, k, v, alpha, beta, S0 = inputs(T, Hk, Hv, dk, dv, seed=7)
    dq, dk_, dv_, dal, dbe, dS = to_dev(q, k, v, alpha, beta, S0)
    out = ops.gdn_scan(dq, dk_, dv_, dal, dbe, dS)
    torch.cuda.synchronize()
    out, S = out.cpu().numpy(), dS.cpu().numpy()
    for h in (0, 17, 31):
        hk = h // 2
        ro, rS = gdn_scan(q[:, hk:hk + 1], k[:, hk:hk + 1], v[:, h:h + 1], alpha[:, h:h + 1],
                          beta[:, h:h + 1], S0[h:h + 1])
        close(out[:, h], ro[:, 0])
        close(S[h], rS[0])


def test_split_sequence_equals_one_scan():
    """Two calls over the halves (the state carried in memory between them) give
    the same bits as one call over the whole sequence, outputs and final state."""
    from bit_moe_expert_route_gb300 import ops
    T, Hk, Hv, dk, dv = 96, 2, 4, 128, 128
    host = inputs(T, Hk, Hv, dk, dv, seed=11)
    q, k, v, al, be, S = to_dev(*host)
    S2 = S.clone()
    whole = ops.gdn_scan(q, k, v, al, be, S)
    a = ops.gdn_scan(q[:40], k[:40], v[:40], al[:40], be[:40], S2)
    b = ops.gdn_scan(q[40:], k[40:], v[40:], al[40:], be[40:], S2)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([a, b]), whole)
    assert torch.equal(S2, S)


def test_empty_sequence_and_graph_replay():
    from bit_moe_expert_route_gb300 import ops
    T, Hk, Hv, dk, dv = 16, 1, 2, 64, 64
    host = inputs(T, Hk, Hv, dk, dv, seed=13)
    q, k, v, al, be, S = to_dev(*host)
    S_before = S.clone()
    ops.gdn_scan(q[:0], k[:0], v[:0], al[:0], be[:0], S)
    torch.cuda.synchronize()
    assert torch.equal(S, S_before)
    eager_S = S.clone()
    eager = ops.gdn_scan(q, k, v, al, be, eager_S)
    out = torch.empty_like(eager)
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    work = S.clone()
    with torch.cuda.graph(g, stream=st):
        ops.gdn_scan(q, k, v, al, be, work, out=out)
    work.copy_(S_before)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager) and torch.equal(work, eager_S)


def test_state_read_early_in_a_chain_of_layers():
    """A chain of single-token scans over distinct states (decode through several
    layers), each launch marked MOE_GDN_STATE_EARLY (its state is read before it waits
    for the previous launch, which writes another layer's state), captured in one
    graph: the same bits as the chain run eagerly without the flag."""
    from bit_moe_expert_route_gb300 import ops
    Hk, Hv, dk, dv, n_layers = 2, 4, 128, 128, 6
    layers = [to_dev(*inputs(1, Hk, Hv, dk, dv, seed=40 + i)) for i in range(n_layers)]
    ref_S = [lay[5].clone() for lay in layers]
    ref_out = [ops.gdn_scan(*lay[:5], ref_S[i]) for i, lay in enumerate(layers)]
    work_S = [lay[5].clone() for lay in layers]
    outs = [torch.empty_like(o) for o in ref_out]
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for i, lay in enumerate(layers):
            ops.gdn_scan(*lay[:5], work_S[i], out=outs[i], state_early=True)
    for i, lay in enumerate(layers):
        work_S[i].copy_(lay[5])
    g.replay()
    torch.cuda.synchronize()
    for i in range(n_layers):
        assert torch.equal(outs[i], ref_out[i]) and torch.equal(work_S[i], ref_S[i]), i
