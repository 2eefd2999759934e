"""moe_decode_gemv_w4_noalloc: the decode entry point for callers that may not
allocate device memory (plug-ins inside a framework that owns the GPU's
memory pool, serving loops that cannot afford an allocation). It runs on a
scratch array built into the library instead of a caller workspace.

Checked through the C ABI on two calls in a row (the built-in scratch keeps
the previous call's contents): each output equals moe_decode_gemv_w4's
(caller workspace) bit for bit, since both run the same kernel on the same
inputs, and both are held to the layer bar against the oracle. The scratch's
status word reads clean through moe_decode_noalloc_device_status, and a
reset followed by a call still gives the same bits. Shapes the kernel does
not support are refused as by moe_decode_gemv_w4, and supported shapes too
large for the 256 KB scratch with MOE_ERR_WORKSPACE. This file is collected
last so that a failure here does not stop the other tests."""
import ctypes

import numpy as np
import pytest

from bit_moe_expert_route_gb300 import synth
from gpu_util import FULL, bf16_np, to_np, tolerance_check

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(L, x, layer, shape, out):
    from bit_moe_expert_route_gb300 import ops
    rc = L.moe_decode_gemv_w4_noalloc(_ptr(x), ctypes.byref(layer.weights), ctypes.byref(shape),
                                      _ptr(out), ops._stream())
    assert rc == 0, ops.status_string(rc)


def _noalloc_status(L):
    from bit_moe_expert_route_gb300 import ops
    v = ctypes.c_int32(-1)
    rc = L.moe_decode_noalloc_device_status(ops._stream(), ctypes.byref(v))
    assert rc in (0, -6), ops.status_string(rc)
    return v.value


def test_noalloc_decode_matches_workspace_decode(orc):
    from bit_moe_expert_route_gb300 import ops
    host = synth.layer_weights(FULL, seed=7, layer=3)
    layer = ops.DeviceLayer(host, FULL)
    dec = ops.Decode(layer)
    shape = ops.Shape.of(FULL, 1)
    L = ops.lib()
    for step in range(3):
        if step == 2:
            assert L.moe_decode_noalloc_reset(ops._stream()) == 0
        xs = synth.tokens(FULL, 1, seed=7, layer=3, off=step, tensor=synth.X_DECODE)
        x = torch.from_numpy(xs.view(np.int16)).cuda().view(-1)
        ref = dec(x)
        out = torch.full_like(ref, float("nan"))
        _noalloc(L, x, layer, shape, out)
        torch.cuda.synchronize()
        assert _noalloc_status(L) == 0
        assert ops.device_status(dec.ws) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), step
        lg = to_np(dec.view("logits", (1, FULL.n_experts), torch.float32))
        want = orc.moe_forward(xs, host, FULL, logits_in=lg)
        ok, info = tolerance_check(bf16_np(out).reshape(1, -1), want["out"])
        assert ok, info


def test_noalloc_refuses_shapes_beyond_its_scratch():
    from bit_moe_expert_route_gb300 import ops
    L = ops.lib()
    host = synth.layer_weights(FULL, seed=7, layer=3)
    layer = ops.DeviceLayer(host, FULL)
    x = torch.zeros(8192, dtype=torch.int16, device="cuda")
    out = torch.zeros(8192, dtype=torch.int16, device="cuda")
    s = ops._stream()
    # a shape the decode kernel runs whose workspace is above 256 KB: refused
    # before anything is read (the weights above are never dereferenced)
    big = ops.Shape(1, 2048, 256, 16, 2048, 2048, 64)
    assert L.moe_decode_workspace_bytes(ctypes.byref(big)) > 256 * 1024
    assert L.moe_decode_gemv_w4_noalloc(_ptr(x), ctypes.byref(layer.weights), ctypes.byref(big),
                                        _ptr(out), s) == -4
    # shapes the kernel does not support: the same code as moe_decode_gemv_w4
    for bad in (ops.Shape(2, 2048, 256, 8, 512, 512, 64),
                ops.Shape(1, 2048, 64, 32, 2048, 2048, 64)):
        assert L.moe_decode_gemv_w4_noalloc(_ptr(x), ctypes.byref(layer.weights),
                                            ctypes.byref(bad), _ptr(out), s) == -3


def test_noalloc_timeout_status_and_reset():
    """A call on the built-in scratch whose bounded waits run out (one block
    withholds its router partials under moe_debug_decode_fault) is visible
    through moe_decode_noalloc_device_status; after moe_decode_noalloc_reset
    the next call equals moe_decode_gemv_w4's output bit for bit."""
    from bit_moe_expert_route_gb300 import ops
    host = synth.layer_weights(FULL, seed=7, layer=3)
    layer = ops.DeviceLayer(host, FULL)
    dec = ops.Decode(layer)
    shape = ops.Shape.of(FULL, 1)
    L = ops.lib()
    xs = synth.tokens(FULL, 1, seed=7, layer=3, off=5, tensor=synth.X_DECODE)
    x = torch.from_numpy(xs.view(np.int16)).cuda().view(-1)
    out = torch.empty(FULL.d_model, dtype=torch.bfloat16, device="cuda")
    try:
        assert L.moe_debug_decode_fault(1_000_000, 5) == 0
        _noalloc(L, x, layer, shape, out)
        torch.cuda.synchronize()
        assert _noalloc_status(L) == ops.DEV_TIMEOUT
    finally:
        L.moe_debug_decode_fault(0, -1)
    assert L.moe_decode_noalloc_reset(ops._stream()) == 0
    ref = dec(x)
    _noalloc(L, x, layer, shape, out)
    torch.cuda.synchronize()
    assert _noalloc_status(L) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
