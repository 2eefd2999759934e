"""moe_route on the GPU against the oracle's routing on identical logits.

Bar: ids, counts, offsets, perm, inv_perm, row_token, row_weight order,
block map and tile count bit-exact; routing weights (expf) within 2e-6
relative. Sizes: the layer's T = 64 / 512 / 4096 / 32768 (Zipf-biased),
plus crafted ties, T = 1, empty input and small expert counts."""
import numpy as np
import pytest

from gpu_util import logits_like_router, to_np
from test_oracle_pins import check_route_invariants

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def run_and_compare(orc, logits, bias, k, bn, with_shared=True):
    from bit_moe_expert_route_gb300 import ops
    T, E = logits.shape
    dl = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    db = None if bias is None else torch.from_numpy(bias).cuda()
    r = ops.route(dl, k, bn, with_shared=with_shared, bias=db)
    torch.cuda.synchronize()
    assert ops.device_status(r["ws"]) == 0
    ids, w = orc.topk(logits, k, bias)
    m = orc.route_meta(ids, E, bn, with_shared)
    assert np.array_equal(to_np(r["topk_ids"]), ids)
    np.testing.assert_allclose(to_np(r["topk_w"]), w, rtol=2e-6, atol=0)
    for key in ("counts", "offsets", "perm", "inv_perm", "row_token"):
        assert np.array_equal(to_np(r[key]), m[key]), key
    nt = int(to_np(r["num_tiles"])[0])
    assert nt == m["num_tiles"]
    assert np.array_equal(to_np(r["block_map"])[:nt], m["block_map"])
    # row_weight is topk_w gathered through perm, bit for bit
    gw = to_np(r["topk_w"]).reshape(-1)
    assert np.array_equal(to_np(r["row_weight"]), gw[m["perm"]])
    check_route_invariants(ids, E, bn, m, with_shared)
    return m


@pytest.mark.parametrize("T,bn", [(64, 16), (512, 16), (4096, 128), (4096, 32)])
def test_route_layer_sizes(orc, T, bn):
    logits, _ = logits_like_router(T, 256, seed=T)
    run_and_compare(orc, logits, None, 8, bn)


def test_route_32768_zipf(orc):
    logits, bias = logits_like_router(32768, 256, seed=7, zipf=True)
    m = run_and_compare(orc, logits, bias, 8, 128)
    c = m["counts"]
    assert c.max() > 10 * c.mean() and (c == 0).sum() >= 2  # the stressed load imbalance


def test_route_ties_and_degenerate(orc):
    E, k = 256, 8
    eq = np.zeros((40, E), np.float32)  # every logit equal: ids 0..7, w = 1/8
    run_and_compare(orc, eq, None, k, 16)
    lg, _ = logits_like_router(300, E, seed=3)
    lg[:, 10:20] = lg[:, 5:6]  # runs of exact ties
    lg = np.round(lg * 4) / 4  # many coincident values
    run_and_compare(orc, lg.astype(np.float32), None, k, 64)
    one, _ = logits_like_router(1, E, seed=4)
    run_and_compare(orc, one, None, k, 16)


@pytest.mark.parametrize("E,k,bn,shared", [(16, 4, 16, True), (64, 1, 32, False), (1024, 32, 256, True),
                                           (8, 8, 16, True)])
def test_route_other_shapes(orc, E, k, bn, shared):
    logits, _ = logits_like_router(777, E, seed=E + k)
    run_and_compare(orc, logits, None, k, bn, shared)


def test_route_empty():
    from bit_moe_expert_route_gb300 import ops
    r = ops.route(torch.empty(0, 256, device="cuda"), 8, 16)
    torch.cuda.synchronize()
    assert int(r["num_tiles"].item()) == 0
    assert int(r["counts"].sum().item()) == 0 and int(r["offsets"].abs().sum().item()) == 0


def test_route_graph_capture_matches_eager(orc):
    """The routing launches capture into a CUDA graph (no host round trip)."""
    from bit_moe_expert_route_gb300 import ops
    logits, _ = logits_like_router(4096, 256, seed=11)
    dl = torch.from_numpy(logits).cuda()
    eager = ops.route(dl, 8, 128)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ops.route(dl, 8, 128)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = ops.route(dl, 8, 128)
    g.replay()
    torch.cuda.synchronize()
    for key in ("topk_ids", "perm", "block_map", "num_tiles", "offsets"):
        assert torch.equal(eager[key], cap[key]), key
