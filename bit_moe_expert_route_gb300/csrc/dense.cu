// Router GEMM and the fp32 -> bf16 output conversion.
//
// The router is the linear map that scores every token against every routed
// expert ("Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple
// Silicon", section "What Lily actually does": 8 of 256 experts per token).
// Its weights are fp32, so it runs on the fp32 FMA pipes: x (bf16, widened
// exactly) times W_r with fp32 accumulation.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRM = 64;   // tokens per CTA
constexpr int kRN = 128;  // experts per CTA
constexpr int kRK = 32;   // K step

// logits[t][e] = sum_k x[t][k] * Wr[k][e]. 256 threads: thread (ty, tx)
// owns tokens ty*8..ty*8+7 and experts tx*4..tx*4+3 of the CTA tile.
__global__ void __launch_bounds__(256) router_gemm_kernel(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ Wr, int T,
                                                          int d, int E, float* __restrict__ logits,
                                                          uint16_t* __restrict__ x16) {
  __shared__ __align__(16) float xs[kRK][kRM];
  __shared__ __align__(16) float ws[kRK][kRN];
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int m0 = blockIdx.y * kRM, n0 = blockIdx.x * kRN;
  float acc[8][4] = {};
  for (int k0 = 0; k0 < d; k0 += kRK) {
    {  // x tile: 64 tokens x 32 k, one 16-byte load (8 bf16) per thread
      const int r = tid >> 2, c = (tid & 3) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (m0 + r < T) v = *reinterpret_cast<const uint4*>(x + (size_t)(m0 + r) * d + k0 + c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      if (x16 && blockIdx.x == 0 && m0 + r < T) {  // f16 copy of x for the tensor-core path
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = fminf(fmaxf(__uint_as_float(u[i] << 16), -65504.f), 65504.f);
          const float hi = fminf(fmaxf(__uint_as_float(u[i] & 0xFFFF0000u), -65504.f), 65504.f);
          const __half2 h2 = __floats2half2_rn(lo, hi);
          o[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(x16 + (size_t)(m0 + r) * d + k0 + c) = make_uint4(o[0], o[1], o[2], o[3]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xs[c + 2 * i][r] = __uint_as_float(u[i] << 16);
        xs[c + 2 * i + 1][r] = __uint_as_float(u[i] & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // W tile: 32 k x 128 experts
      const int idx = tid + i * 256;
      const int r = idx >> 5, c = (idx & 31) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (n0 + c < E) v = *reinterpret_cast<const float4*>(Wr + (size_t)(k0 + r) * E + n0 + c);
      *reinterpret_cast<float4*>(&ws[r][c]) = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&xs[kk][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&xs[kk][ty * 8 + 4]);
      const float4 b = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = m0 + ty * 8 + i;
    const int e = n0 + tx * 4;
    if (t < T && e < E)
      *reinterpret_cast<float4*>(logits + (size_t)t * E + e) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
}

__global__ void f32_to_bf16_kernel(const float4* __restrict__ in, uint2* __restrict__ out,
                                   int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = in[i];
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    out[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                        *reinterpret_cast<const uint32_t*>(&hi));
  }
}

}  // namespace

cudaError_t router_gemm_launch(const uint16_t* x, const float* Wr, int T, int d, int E,
                               float* logits, uint16_t* x16, cudaStream_t s) {
  dim3 grid((E + kRN - 1) / kRN, (T + kRM - 1) / kRM);
  router_gemm_kernel<<<grid, 256, 0, s>>>(x, Wr, T, d, E, logits, x16);
  return cudaGetLastError();
}

cudaError_t f32_to_bf16_launch(const float* in, uint16_t* out, int64_t n, cudaStream_t s) {
  const int64_t n4 = n / 4;  // n is a multiple of 128
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = std::min<int64_t>((n4 + 255) / 256, (int64_t)sms * 8);
  f32_to_bf16_kernel<<<(int)std::max<int64_t>(blocks, 1), 256, 0, s>>>(
      reinterpret_cast<const float4*>(in), reinterpret_cast<uint2*>(out), n4);
  return cudaGetLastError();
}

}  // namespace moe
