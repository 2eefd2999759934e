"""moe_decode_gemv_w4 (T = 1) against the oracle.

The GPU's fp32 router logits are checked against the oracle's (they differ
only in summation order), then the oracle runs the layer on the GPU's logits
so both sides take the same top-k decision; ids must match exactly and the
bf16 output must satisfy max|err| <= 2e-2 rms(ref) and rel-L2 <= 5e-3.

The chained test runs several layers as a model does: each layer's bf16
output is the next layer's input, the layers captured in one CUDA graph with
programmatic-dependent-launch edges (each layer's weight prefetch runs
before its dependency wait, while the previous layer still runs)."""
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


def check_one(orc, host, dec, x):
    out = dec(torch.from_numpy(x.view(np.int16)).cuda().view(-1))
    torch.cuda.synchronize()
    from bit_moe_expert_route_gb300 import ops
    assert ops.device_status(dec.ws) == 0
    lg = to_np(dec.view("logits", (1, FULL.n_experts), torch.float32))
    ids = to_np(dec.view("topk_ids", (1, FULL.top_k), torch.int32))
    ref_free = orc.moe_forward(x, host, FULL)
    np.testing.assert_allclose(lg, ref_free["logits"], rtol=1e-5, atol=2e-5)
    ref = orc.moe_forward(x, host, FULL, logits_in=lg)
    assert np.array_equal(ids, ref["ids"])
    w = to_np(dec.view("topk_w", (1, FULL.top_k + 1), torch.float32))
    np.testing.assert_allclose(w[:, :FULL.top_k], ref["w"], rtol=2e-6)
    np.testing.assert_allclose(w[0, FULL.top_k], ref["gate"][0], rtol=2e-6)
    ok, info = tolerance_check(bf16_np(out).reshape(1, -1), ref["out"])
    assert ok, info


def test_decode_matches_oracle(orc, layer):
    from bit_moe_expert_route_gb300 import ops
    host, dl = layer
    dec = ops.Decode(dl)
    for step in range(3):
        x = synth.tokens(FULL, 1, seed=0, layer=0, off=step, tensor=synth.X_DECODE)
        check_one(orc, host, dec, x)


def test_decode_graph_replay_matches_eager(layer):
    from bit_moe_expert_route_gb300 import ops
    host, dl = layer
    dec = ops.Decode(dl)
    x = torch.from_numpy(synth.tokens(FULL, 1, seed=1).view(np.int16)).cuda().view(-1)
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


def test_decode_without_shared_expert(orc):
    from bit_moe_expert_route_gb300 import ops
    from bit_moe_expert_route_gb300.synth import LayerShape
    shape = LayerShape(d_model=256, n_experts=32, top_k=4, d_ff=256, d_ff_shared=256)
    host = synth.layer_weights(shape, seed=5, shared=False)
    dl = ops.DeviceLayer(host, shape)
    dec = ops.Decode(dl)
    x = synth.tokens(shape, 1, seed=5)
    out = dec(torch.from_numpy(x.view(np.int16)).cuda().view(-1))
    torch.cuda.synchronize()
    lg = to_np(dec.view("logits", (1, 32), torch.float32))
    ref = orc.moe_forward(x, host, shape, logits_in=lg)
    ok, info = tolerance_check(bf16_np(out).reshape(1, -1), ref["out"])
    assert ok, info


def test_decode_chain_in_graph_matches_oracle(orc):
    """Layers of distinct weights chained through their outputs inside one
    captured graph (the decode step's schedule): every layer's output is held
    to the bar against the oracle run on that layer's own input (the previous
    layer's bf16 output as the GPU produced it) and logits, and the graph's
    outputs equal an eager run of the same chain bit for bit.

    Bare MoE layers (no normalisation between them, unlike a model) map an
    input of rms r to an output of rms about 4.4 r^2 with these weights, so a
    chain of them grows or dies out within a few layers. The first input is
    N(0,1) scaled by 0.1, which keeps the six outputs' rms between 0.006 and
    44 (measured with the oracle), inside the 16-bit formats' normal range."""
    from bit_moe_expert_route_gb300 import ops
    NL = 6
    hosts = [synth.layer_weights(FULL, seed=11, layer=l) for l in range(NL)]
    decs = [ops.Decode(ops.DeviceLayer(h, FULL)) for h in hosts]
    xs = synth.f32_to_bf16(0.1 * synth.bf16_to_f32(synth.tokens(FULL, 1, seed=11, tensor=synth.X_DECODE)))
    x0 = torch.from_numpy(xs.view(np.int16)).cuda().view(-1)
    outs = torch.zeros(NL, FULL.d_model, dtype=torch.bfloat16, device="cuda")

    def chain():
        for l in range(NL):
            decs[l](x0 if l == 0 else outs[l - 1].view(torch.int16), outs[l])

    chain()
    torch.cuda.synchronize()
    eager = outs.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for _ in range(3):
        outs.zero_()
        g.replay()
    torch.cuda.synchronize()
    for d in decs:
        assert ops.device_status(d.ws) == 0
    assert torch.equal(outs.view(torch.int16), eager.view(torch.int16))
    xin = to_np(x0.view(1, -1)).view(np.uint16)
    for l in range(NL):
        lg = to_np(decs[l].view("logits", (1, FULL.n_experts), torch.float32))
        ref_free = orc.moe_forward(xin, hosts[l], FULL)
        np.testing.assert_allclose(lg, ref_free["logits"], rtol=1e-5, atol=2e-5)
        ref = orc.moe_forward(xin, hosts[l], FULL, logits_in=lg)
        ids = to_np(decs[l].view("topk_ids", (1, FULL.top_k), torch.int32))
        assert np.array_equal(ids, ref["ids"]), l
        ok, info = tolerance_check(bf16_np(outs[l]).reshape(1, -1), ref["out"])
        assert ok, (l, info)
        xin = to_np(outs[l].view(torch.int16)).view(np.uint16).reshape(1, -1)


def test_decode_timeout_is_reported_and_recovers(orc, layer):
    """Failure detection without a GPU fault: with a 1 ms wait limit and one
    block withholding its router partial sums (moe_debug_decode_fault), every
    other block's bounded poll runs out, the call records MOE_DEV_TIMEOUT in
    the workspace status word and still ends; after the documented recovery
    (the workspace zeroed) the next call matches the oracle again."""
    from bit_moe_expert_route_gb300 import ops
    host, dl = layer
    dec = ops.Decode(dl)
    L = ops.lib()
    x = synth.tokens(FULL, 1, seed=0, layer=0, off=9, tensor=synth.X_DECODE)
    xt = torch.from_numpy(x.view(np.int16)).cuda().view(-1)
    dec(xt)
    torch.cuda.synchronize()
    assert ops.device_status(dec.ws) == ops.DEV_OK
    try:
        assert L.moe_debug_decode_fault(1_000_000, 3) == 0
        dec(xt)
        torch.cuda.synchronize()
        assert ops.device_status(dec.ws) == ops.DEV_TIMEOUT
    finally:
        L.moe_debug_decode_fault(0, -1)
    dec.ws.zero_()
    check_one(orc, host, dec, x)
