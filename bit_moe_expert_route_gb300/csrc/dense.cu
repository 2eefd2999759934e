// Router GEMM on the tensor cores, and the fp32 -> bf16 output conversion.
//
// The router is the linear map that scores every token against every routed
// expert ("Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple
// Silicon", section "What Lily actually does": 8 of 256 experts per token);
// the shared expert's gate vector w_sg is one more column of the same map.
//
// The router weights are fp32 and x is bf16. Every fp32 weight is the exact
// sum of three bf16 numbers,
//   hi = bf16(w),  lo = bf16(w - hi),  lo2 = bf16(w - hi - lo)
// (each residual is exact in fp32, and the last one has at most 8
// significant bits), and the product of two bf16 numbers is exact in fp32.
// So x . hi, x . lo and x . lo2 are three exact-product bf16 dot products
// with fp32 accumulation; their sum is x . w up to the rounding of fp32
// accumulation, as in an fp32 dot product. The three weight tiles of a K
// step are stacked along N (N = 3 x the tile's experts), so one tcgen05 MMA
// per 16-wide K step reads the x tile once for all three.
//
//   router_split_kernel  Wr [d][E] (+ w_sg) -> planes [3][Ep][d] bf16, K-major
//   router_tc_kernel     one CTA per (128-token tile, expert tile):
//                          warp 0     TMA producer (x tile + 3 weight tiles
//                                     per 64-wide K step, 4-stage ring)
//                          warp 1     TMEM allocation, tcgen05.mma issue
//                                     (three accumulators side by side)
//                          warps 2-5  during the main loop, in the CTAs of
//                                     expert tile 0: the f16 copy of x read
//                                     back from the staged x tiles; then the
//                                     epilogue: tcgen05.ld of the three
//                                     accumulators, hi + lo + lo2 per logit,
//                                     and the gate logit (sigmoid weight of
//                                     the shared rows)
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRTM = 128;                   // tokens per tile (MMA M)
constexpr int kRKB = 64;                    // K per stage: one 128-byte swizzled row
constexpr int kRStages = 4;
constexpr int kRThreads = 192;
constexpr uint32_t kRATile = kRTM * kRKB * 2;  // 16 KB of x per stage
constexpr int kRBn = 64;                    // experts per tile (the last tile may differ)

// ---------------------------------------------------------------- weight split
// planes[j][e][k] for j = 0, 1, 2 (hi, lo, lo2); row e = E holds w_sg, rows
// past it (up to Ep) are zero.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ Wr,
                                                           const float* __restrict__ wsg, int d,
                                                           int E, int Ep,
                                                           uint16_t* __restrict__ planes) {
  __shared__ float tile[32][33];  // [k][e]
  const int e0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int i = ty; i < 32; i += 8) {
    const int k = k0 + i, e = e0 + tx;
    float v = 0.f;
    if (k < d) {
      if (e < E) v = Wr[(size_t)k * E + e];
      else if (e == E && wsg) v = wsg[k];
    }
    tile[i][tx] = v;
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int e = e0 + i, k = k0 + tx;
    if (e >= Ep || k >= d) continue;
    const float w = tile[tx][i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(lo);
    const __nv_bfloat16 lo2 = __float2bfloat16_rn(r2);
    const size_t plane = (size_t)Ep * d, at = (size_t)e * d + k;
    planes[at] = __bfloat16_as_ushort(hi);
    planes[plane + at] = __bfloat16_as_ushort(lo);
    planes[2 * plane + at] = __bfloat16_as_ushort(lo2);
  }
}

// ---------------------------------------------------------------- tensor-core router
struct RouterKParams {
  CUtensorMap tm_x;     // x [T][d] bf16, box 64 x 128
  CUtensorMap tm_w;     // planes [3*Ep][d] bf16, box 64 x kRBn
  CUtensorMap tm_wl;    // same, box 64 x n_last (the last expert tile)
  RouterParams p;
  int Ep;               // rows per plane
  int n_tiles;          // expert tiles
  int n_last;           // MMA N of the last tile (16..80, a multiple of 16)
  uint32_t stage_bytes;
  uint32_t tmem_cols;
};

// Bounded wait that ignores the abort flag: used only to let this CTA's own
// asynchronous work finish before its shared and tensor memory are released.
MOE_DEVINL bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

__global__ void __launch_bounds__(kRThreads, 1)
    router_tc_kernel(const __grid_constant__ RouterKParams kp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const RouterParams& p = kp.p;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRStages * kp.stage_bytes);
  uint64_t* empty = full + kRStages;
  uint64_t* acc_full = empty + kRStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x, m0 = blockIdx.y * kRTM;
  const bool last = nt == kp.n_tiles - 1;
  const int n0 = nt * kRBn;
  const int n_mma = last ? kp.n_last : kRBn;   // experts (+ gate) of this tile
  const uint32_t b_stride = (uint32_t)n_mma * 128u;  // one plane's tile: n_mma rows of 128 B
  const bool convert = p.x16 != nullptr && nt == 0;
  const int KB = p.d / kRKB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], convert ? 5 : 1);  // the MMA commit (+ 4 converting warps)
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kp.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      tma_prefetch_desc(&kp.tm_x);
      tma_prefetch_desc(last ? &kp.tm_wl : &kp.tm_w);
      const uint64_t pol_w = l2_policy_evict_last();  // every token tile reads the planes
      const uint64_t pol_x = l2_policy_evict_normal();
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % kRStages;
        if (kb >= kRStages &&
            !mbar_wait(&empty[s], ((kb / kRStages) & 1) ^ 1, abort_flag, p.status, 40))
          break;
        uint8_t* st = smem + (size_t)s * kp.stage_bytes;
        mbar_arrive_expect_tx(&full[s], kRATile + 3 * (uint32_t)n_mma * 128u);
        tma_load_2d(st, &kp.tm_x, kb * kRKB, m0, &full[s], pol_x);
        for (int j = 0; j < 3; ++j)
          tma_load_2d(st + kRATile + j * b_stride, last ? &kp.tm_wl : &kp.tm_w, kb * kRKB,
                      j * kp.Ep + n0, &full[s], pol_w);
        ++issued;
      }
      // the copies still in flight land before the CTA releases its memory
      for (int kb = max(0, issued - kRStages); kb < issued; ++kb)
        drain_wait(&full[kb % kRStages], (kb / kRStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issue
      const uint32_t idesc = idesc_bf16_f32(kRTM, 3 * n_mma);  // planes stacked along N
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % kRStages;
        if (!mbar_wait(&full[s], (kb / kRStages) & 1, abort_flag, p.status, 41)) break;
        tc_fence_after();
        const uint32_t a = smem_u32(smem + (size_t)s * kp.stage_bytes);
        const uint32_t b = a + kRATile;
#pragma unroll
        for (int kk = 0; kk < kRKB / 16; ++kk)
          tc_mma_bf16(tmem, smem_desc_sw128(a + kk * 32), smem_desc_sw128(b + kk * 32), idesc,
                      (kb | kk) != 0);
        tc_commit(&empty[s]);
      }
      tc_commit(acc_full);  // also issued after an abort: tracks every MMA issued
      drain_wait(acc_full, 0);
    }
  } else {
    const int et = threadIdx.x - 64;  // 0..127
    if (convert) {  // f16 copy of x (saturated to the f16 range) from the staged tiles
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % kRStages;
        if (!mbar_wait(&full[s], (kb / kRStages) & 1, abort_flag, p.status, 42)) break;
        const uint8_t* a = smem + (size_t)s * kp.stage_bytes;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int idx = i * 128 + et, r = idx >> 3, c = idx & 7;
          if (m0 + r < p.T) {
            const uint4 v = *reinterpret_cast<const uint4*>(a + sw128_offset(r, c));
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float lo = fminf(fmaxf(__uint_as_float(u[q] << 16), -65504.f), 65504.f);
              const float hi = fminf(fmaxf(__uint_as_float(u[q] & 0xFFFF0000u), -65504.f), 65504.f);
              const __half2 h2 = __floats2half2_rn(lo, hi);
              o[q] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(p.x16 + (size_t)(m0 + r) * p.d + kb * kRKB + c * 8) =
                make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        mbar_arrive_warp(&empty[s]);
      }
    }
    // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (its tokens)
    const int quarter = warp & 3;
    if (mbar_wait(acc_full, 0, abort_flag, p.status, 43)) {
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
      const int t = m0 + quarter * 32 + lane;
      float* row = p.logits + (size_t)t * p.E;
      const int gcol = last && p.wsg ? p.E - n0 : -1;  // the gate column follows the last expert
#pragma unroll 1
      for (int c0 = 0; c0 < n_mma; c0 += 16) {
        uint32_t hi[16], lo[16], lo2[16];
        tmem_ld_32x32b_x16(taddr + c0, hi);
        tmem_ld_32x32b_x16(taddr + n_mma + c0, lo);
        tmem_ld_32x32b_x16(taddr + 2 * n_mma + c0, lo2);
        tc_wait_ld();
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          v[j] = (__uint_as_float(hi[j]) + __uint_as_float(lo[j])) + __uint_as_float(lo2[j]);
        if (t < p.T) {
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const int e = n0 + c0 + j;  // E - n0 is a multiple of 8
            if (e < p.E)
              *reinterpret_cast<float4*>(row + e) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          }
          if (gcol >= c0 && gcol < c0 + 16) {
            float g = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j == gcol) g = v[j];
            p.gate_logit[t] = g;
            if (p.row_weight) p.row_weight[(size_t)p.T * p.k + t] = 1.f / (1.f + expf(-g));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kp.tmem_cols);
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

// Deterministic combine of the down projection's per-row outputs y [rows][d]
// (unweighted; rows in expert order, the shared rows last): for every token t
// and output column, acc = 0, then acc = w * y[row] + acc (one fused
// multiply-add) for the token's routed rows in slot order j = 0..k-1 (row
// inv_perm[t*k + j], weight row_weight[row]) and last for its shared row
// T*k + t (weight = the sigmoid gate). The order is fixed, so the result does
// not depend on how the GEMM scheduled its tiles. Writes the fp32 sum and its
// bf16 rounding. One float4 of one token per thread, d/4 threads per token.
__global__ void combine_rows_kernel(const float4* __restrict__ y, const int32_t* __restrict__ inv_perm,
                                    const float* __restrict__ row_weight, int T, int k, int d4,
                                    int shared, float4* __restrict__ acc_out,
                                    uint2* __restrict__ out, int32_t* status) {
  const int64_t n = (int64_t)T * d4, rows_routed = (int64_t)T * k;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / d4), c = (int)(i - (int64_t)t * d4);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j <= k; ++j) {
      int64_t r;
      if (j < k) {
        r = __ldg(inv_perm + (int64_t)t * k + j);
        if (r < 0 || r >= rows_routed) {
          report(status, MOE_DEV_BAD_ROW, 60, (int)r);
          continue;
        }
      } else {
        if (!shared) break;
        r = rows_routed + t;
      }
      const float w = __ldg(row_weight + r);
      const float4 v = __ldcs(y + r * d4 + c);  // read once: stream past L2
      a.x = fmaf(w, v.x, a.x);
      a.y = fmaf(w, v.y, a.y);
      a.z = fmaf(w, v.z, a.z);
      a.w = fmaf(w, v.w, a.w);
    }
    acc_out[i] = a;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
    out[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                        *reinterpret_cast<const uint32_t*>(&hi));
  }
}

// bf16 tensor [rows][cols] (row stride cols), box 64 columns x box_rows, 128-byte swizzle.
bool make_bf16_map(CUtensorMap* tm, const uint16_t* base, int64_t rows, int cols, int box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn || rows < 1) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kRKB, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t router_launch(const RouterParams& p, cudaStream_t s) {
  if (p.T < 1) return cudaSuccess;
  if (p.d % kRKB || p.E % 8) return cudaErrorInvalidValue;
  const bool gate = p.wsg != nullptr;
  const int Ep = router_split_rows(p.E, gate);
  const dim3 sgrid((Ep + 31) / 32, (p.d + 31) / 32);
  router_split_kernel<<<sgrid, 256, 0, s>>>(p.Wr, p.wsg, p.d, p.E, Ep, p.wsplit);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  RouterKParams kp;
  memset(&kp, 0, sizeof kp);
  kp.p = p;
  kp.Ep = Ep;
  kp.n_tiles = (p.E + kRBn - 1) / kRBn;
  const int rem = p.E - (kp.n_tiles - 1) * kRBn;  // experts in the last tile (8..64)
  kp.n_last = ((rem + (gate ? 1 : 0)) + 15) / 16 * 16;
  const int n_max = std::max(kp.n_tiles > 1 ? kRBn : 0, kp.n_last);
  kp.stage_bytes = kRATile + 3 * (uint32_t)n_max * 128u;
  kp.tmem_cols = 3 * n_max > 128 ? 256 : 3 * n_max > 64 ? 128 : 64;
  if (!make_bf16_map(&kp.tm_x, p.x, p.T, p.d, kRTM)) return cudaErrorInvalidValue;
  if (!make_bf16_map(&kp.tm_wl, p.wsplit, 3LL * Ep, p.d, kp.n_last)) return cudaErrorInvalidValue;
  if (kp.n_tiles > 1 && !make_bf16_map(&kp.tm_w, p.wsplit, 3LL * Ep, p.d, kRBn))
    return cudaErrorInvalidValue;
  const int smem = kRStages * (int)kp.stage_bytes + 1024 + 128;
  err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  const dim3 grid(kp.n_tiles, (p.T + kRTM - 1) / kRTM);
  router_tc_kernel<<<grid, kRThreads, smem, s>>>(kp);
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

cudaError_t combine_rows_launch(const float* y, const int32_t* inv_perm, const float* row_weight,
                                int T, int k, int d, bool shared, float* acc, uint16_t* out,
                                int32_t* status, cudaStream_t s) {
  if (T < 1) return cudaSuccess;
  if (d % 4) return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n = (int64_t)T * (d / 4);
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)sms * 8);
  combine_rows_kernel<<<(int)std::max<int64_t>(blocks, 1), 256, 0, s>>>(
      reinterpret_cast<const float4*>(y), inv_perm, row_weight, T, k, d / 4, shared ? 1 : 0,
      reinterpret_cast<float4*>(acc), reinterpret_cast<uint2*>(out), status);
  return cudaGetLastError();
}

}  // namespace moe
