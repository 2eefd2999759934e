"""moe_decode_gemv_w4_noalloc: the decode entry point for callers that may not
allocate device memory (plug-ins inside a framework that owns the GPU's
memory pool, serving loops that cannot afford an allocation). It runs on a
scratch array built into the library instead of a caller workspace.

Checked through the C ABI against moe_decode_gemv_w4 (caller workspace) on
two calls in a row, since the built-in scratch keeps the previous call's
contents; and shapes too large for the 256 KB scratch are refused. This file
is collected last so that a failure here does not stop the other tests."""
import ctypes

import numpy as np
import pytest

from bit_moe_expert_route_gb300 import synth
from gpu_util import FULL, bf16_np, tolerance_check

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_decode_matches_workspace_decode():
    from bit_moe_expert_route_gb300 import ops
    host = synth.layer_weights(FULL, seed=7, layer=3)
    layer = ops.DeviceLayer(host, FULL)
    dec = ops.Decode(layer)
    shape = ops.Shape.of(FULL, 1)
    L = ops.lib()
    for step in range(2):
        xs = synth.tokens(FULL, 1, seed=7, layer=3, off=step, tensor=synth.X_DECODE)
        x = torch.from_numpy(xs.view(np.int16)).cuda().view(-1)
        ref = dec(x)
        out = torch.full_like(ref, float("nan"))
        rc = L.moe_decode_gemv_w4_noalloc(_ptr(x), ctypes.byref(layer.weights),
                                          ctypes.byref(shape), _ptr(out), ops._stream())
        assert rc == 0, ops.status_string(rc)
        torch.cuda.synchronize()
        got = bf16_np(out).reshape(1, -1).astype(np.float64)
        want = bf16_np(ref).reshape(1, -1).astype(np.float64)
        ok, info = tolerance_check(got, want, bf16_output=True)
        assert ok, info


def test_noalloc_refuses_shapes_beyond_its_scratch():
    from bit_moe_expert_route_gb300 import ops
    L = ops.lib()
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the call is refused first
    big = ops.Shape(1, 2048, 64, 32, 2048, 2048, 64)  # (32 + 1) * 2048 fp32 activations > 256 KB
    assert L.moe_decode_gemv_w4_noalloc(fake, fake, ctypes.byref(big), fake, None) == -4
    two_tokens = ops.Shape(2, 2048, 256, 8, 512, 512, 64)
    assert L.moe_decode_gemv_w4_noalloc(fake, fake, ctypes.byref(two_tokens), fake, None) == -3
