"""moe_decode_batch_w4 (1 to 8 tokens) against the oracle.

As for the batch-1 decode: the GPU's fp32 router logits are checked against
the oracle's, then the oracle runs the layer on the GPU's logits so both take
the same top-k decision; ids must match exactly, routing weights within 2 ulp,
and the bf16 output must satisfy max|err| <= 2e-2 rms(ref) and rel-L2 <= 5e-3. Batches with repeated tokens, and a router bias
that concentrates the selection, make tokens share experts (each shared
expert's rows are computed once for all of its tokens)."""
import numpy as np
import pytest

from bit_moe_expert_route_gb300 import synth
from gpu_util import FULL, bf16_np, to_np, tolerance_check

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def layer():
    from bit_moe_expert_route_gb300 import ops
    host = synth.layer_weights(FULL, seed=0, layer=0)
    return host, ops.DeviceLayer(host, FULL)


def check_batch(orc, host, shape, dec, x):
    from bit_moe_expert_route_gb300 import ops
    T, E, k = x.shape[0], shape.n_experts, shape.top_k
    out = dec(torch.from_numpy(x.view(np.int16)).cuda())
    torch.cuda.synchronize()
    assert ops.device_status(dec.ws) == 0
    lg = to_np(dec.view("logits", (T, E), torch.float32))
    ref_free = orc.moe_forward(x, host, shape)
    np.testing.assert_allclose(lg, ref_free["logits"], rtol=1e-5, atol=2e-5)
    ref = orc.moe_forward(x, host, shape, logits_in=lg)
    assert np.array_equal(to_np(dec.view("topk_ids", (T, k), torch.int32)), ref["ids"])
    w = to_np(dec.view("topk_w", (T, k + 1), torch.float32))
    np.testing.assert_allclose(w[:, :k], ref["w"], rtol=2e-6)
    if host["shared_gate"] is not None:
        np.testing.assert_allclose(w[:, k], ref["gate"], rtol=2e-6)
    ok, info = tolerance_check(bf16_np(out).reshape(T, -1), ref["out"])
    assert ok, info
    return ref


@pytest.mark.parametrize("T", [1, 2, 4, 5, 8])
def test_batch_matches_oracle(orc, layer, T):
    from bit_moe_expert_route_gb300 import ops
    host, dl = layer
    dec = ops.DecodeBatch(dl, T)
    for step in range(2):
        x = synth.tokens(FULL, T, seed=3, layer=0, off=16 * step + T, tensor=synth.X_DECODE)
        check_batch(orc, host, FULL, dec, x)


def test_batch_with_repeated_tokens_shares_experts(orc, layer):
    from bit_moe_expert_route_gb300 import ops
    host, dl = layer
    x = synth.tokens(FULL, 4, seed=4, tensor=synth.X_DECODE)
    x[2] = x[0]
    x[3] = x[0]
    ref = check_batch(orc, host, FULL, ops.DecodeBatch(dl, 4), x)
    assert np.array_equal(ref["ids"][0], ref["ids"][2])


def test_batch_with_concentrated_routing(orc):
    """A Zipf router bias: most tokens pick the same few experts."""
    from bit_moe_expert_route_gb300 import ops
    host = synth.layer_weights(FULL, seed=0, layer=0, router_bias=synth.zipf_router_bias(FULL.n_experts))
    dec = ops.DecodeBatch(ops.DeviceLayer(host, FULL), 6)
    x = synth.tokens(FULL, 6, seed=6, tensor=synth.X_DECODE)
    ref = check_batch(orc, host, FULL, dec, x)
    assert len(np.unique(ref["ids"])) < 6 * FULL.top_k  # experts shared across tokens


def test_batch_small_shapes(orc):
    """No shared expert; a router width with a partial last 8-expert block; k = E."""
    from bit_moe_expert_route_gb300 import ops
    from bit_moe_expert_route_gb300.synth import LayerShape
    cases = [(LayerShape(d_model=256, n_experts=72, top_k=5, d_ff=128, d_ff_shared=128), 3, False),
             (LayerShape(d_model=384, n_experts=16, top_k=16, d_ff=256, d_ff_shared=256), 2, True),
             (LayerShape(d_model=128, n_experts=8, top_k=2, d_ff=128, d_ff_shared=128), 8, True)]
    for shape, T, shared in cases:
        host = synth.layer_weights(shape, seed=T, shared=shared)
        dec = ops.DecodeBatch(ops.DeviceLayer(host, shape), T)
        check_batch(orc, host, shape, dec, synth.tokens(shape, T, seed=T))


def test_batch_graph_replay_matches_eager(layer):
    from bit_moe_expert_route_gb300 import ops
    host, dl = layer
    dec = ops.DecodeBatch(dl, 4)
    x = torch.from_numpy(synth.tokens(FULL, 4, seed=9).view(np.int16)).cuda()
    eager = dec(x).clone()
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dec(x, out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dec(x, out)
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
