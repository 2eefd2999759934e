"""GB300-native 4-bit sparse MoE layer: GPU-resident routing, fused-dequant
grouped GEMM on tcgen05 tensor cores, and a batch-1 W4 decode GEMV.

The compute lives in the CUDA library `libmoe_gb300.so` (C ABI, see
include/moe.h); `bit_moe_expert_route_gb300.ops` is a thin ctypes binding
over it.  Importing this package does not load the library; the first call
into `ops` does, and fails loudly if it has not been built.
"""
__all__ = ["synth", "ops"]
