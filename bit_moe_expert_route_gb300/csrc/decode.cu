// Batch-1 decode: one token through the MoE layer with matrix-vector kernels
// that stream only the router, the shared expert and the top-k selected
// experts' packed 4-bit weights. ("Perplexity's Lily Beats MLX-LM by 1.35x
// Running Qwen3.6 on Apple Silicon", section "Why prefill and decode get
// different treatment": batch-1 decode is bound by reading the weights, and
// uses matrix-vector kernels on the vector ALUs.)
//
// Three launches:
//   1. decode_router_kernel   split-K router GEMV (+ shared gate logit) into
//                             per-block partial sums; the last block to finish
//                             reduces them in a fixed order, selects the top k
//                             and writes the routing weights and the gate.
//   2. decode_gateup_kernel   one warp per (expert slot, row): gate and up rows
//                             of the selected experts, h = silu(g) * u.
//   3. decode_down_kernel     one warp per output column: the down rows of all
//                             selected experts and the shared expert, weighted
//                             and summed in slot order, rounded once to bf16.
//
// Dot products use the affine form per group: sum_k (s*q_k + b) v_k =
// s * sum_k q_k v_k + b * sum_k v_k, with the activation chunk sums taken once.
// Weights are read as 16-byte chunks (32 codes); lanes read consecutive chunks
// of a row so a warp's loads are fully coalesced.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kRouterRows = 16;  // K rows of W_r per router block

// Activation vector staged in shared memory as fp32 chunks of 32 values
// (8 float4 each). float4 j of chunk c lives at c*8 + (j ^ (c & 7)), so eight
// lanes reading eight consecutive chunks hit distinct banks.
MOE_DEVINL int chunk_slot(int c, int j) { return c * 8 + (j ^ (c & 7)); }

// sum over the 32 codes of a 16-byte chunk of q_k * v_k (v: swizzled smem chunk).
MOE_DEVINL float chunk_dot(const uint4 q, const float4* __restrict__ v, int c) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v0 = v[chunk_slot(c, 2 * i)];
    const float4 v1 = v[chunk_slot(c, 2 * i + 1)];
    const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      // exact code -> float: 2^23 + q has q in its low mantissa bits
      const float qf = __uint_as_float(0x4B000000u | ((w[i] >> (4 * n)) & 0xFu)) - 8388608.f;
      acc = fmaf(qf, vv[n], acc);
    }
  }
  return acc;
}

template <int NPL>
__global__ void __launch_bounds__(256) decode_router_kernel(DecodeParams p, int nsplit) {
  __shared__ float s_logit[1025];
  __shared__ int s_last;
  const int E = p.E;
  const int k0 = blockIdx.x * kRouterRows;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
#pragma unroll
    for (int r = 0; r < kRouterRows; ++r)
      acc = fmaf(bf16_bits_to_f32(p.x[k0 + r]), p.w.router[(size_t)(k0 + r) * E + e], acc);
    p.part[(size_t)blockIdx.x * (E + 1) + e] = acc;
  }
  if (threadIdx.x < 32) {
    float acc = 0.f;
    if (p.shared && threadIdx.x < kRouterRows)
      acc = bf16_bits_to_f32(p.x[k0 + threadIdx.x]) * p.w.shared_gate[k0 + threadIdx.x];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
    if (threadIdx.x == 0) p.part[(size_t)blockIdx.x * (E + 1) + E] = acc;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(p.counter, 1u) == (uint32_t)(nsplit - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    float acc = 0.f;
    for (int b = 0; b < nsplit; ++b) acc += __ldcg(p.part + (size_t)b * (E + 1) + e);
    s_logit[e] = acc;
    if (e < E) p.logits[e] = acc;
    else p.gate_logit[0] = acc;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float z[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = i * 32 + lane;
      z[i] = e < E ? (p.w.router_bias ? s_logit[e] + p.w.router_bias[e] : s_logit[e]) : 0.f;
    }
    uint32_t taken = 0;
    float my_z = 0.f;
    int my_e = 0;
    for (int j = 0; j < p.k; ++j) {
      float bv = 0.f;
      int be = INT_MAX;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = i * 32 + lane;
        if (e < E && !((taken >> i) & 1u) && (be == INT_MAX || z[i] > bv)) {
          bv = z[i];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, off);
        const int oe = __shfl_xor_sync(kFull, be, off);
        if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == j) {
        my_z = bv;
        my_e = be;
      }
    }
    const float zmax = __shfl_sync(kFull, my_z, 0);
    const float ex = lane < p.k ? expf(my_z - zmax) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (lane < p.k) {
      p.ids[lane] = my_e;
      p.wts[lane] = ex / sum;
    }
    if (lane == 0) {
      p.wts[p.k] = p.shared ? 1.f / (1.f + expf(-s_logit[E])) : 0.f;
      *p.counter = 0u;  // ready for the next call
    }
  }
}

// Stage a bf16 activation vector of n values (n % 32 == 0) as swizzled fp32
// chunks in shared memory, with per-chunk sums.
MOE_DEVINL void stage_bf16_vector(const uint16_t* __restrict__ src, int n, float4* v,
                                  float* csum) {
  const int nch = n / 32;
  for (int i = threadIdx.x; i < n / 4; i += blockDim.x) {  // i: float4 index
    const uint2 b = *reinterpret_cast<const uint2*>(src + 4 * i);
    const float4 f = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u),
                                 __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xFFFF0000u));
    v[chunk_slot(i >> 3, i & 7)] = f;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nch; c += blockDim.x) {
    float s = 0.f;
    for (int j = 0; j < 8; ++j) {
      const float4 f = v[chunk_slot(c, j)];
      s += (f.x + f.y) + (f.z + f.w);
    }
    csum[c] = s;
  }
  __syncthreads();
}

// Row dot of one 4-bit row (K codes, group 64) with a staged vector:
// lanes take consecutive 16-byte chunks; returns the warp-reduced sum.
MOE_DEVINL float w4_row_dot(const uint32_t* __restrict__ q, const uint16_t* __restrict__ sc,
                            const uint16_t* __restrict__ bi, int K, const float4* v,
                            const float* csum) {
  const int lane = threadIdx.x & 31;
  const uint4* q4 = reinterpret_cast<const uint4*>(q);
  float acc = 0.f;
  for (int c = lane; c < K / 32; c += 32) {
    const uint4 w = __ldcs(q4 + c);  // streamed once: evict-first
    const float s = bf16_bits_to_f32(sc[c >> 1]);
    const float b = bf16_bits_to_f32(bi[c >> 1]);
    acc = fmaf(s, chunk_dot(w, v, c), fmaf(b, csum[c], acc));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
  return acc;
}

// grid: ceil((k + shared) * f / 8) blocks of 8 warps; warp -> (slot, row).
__global__ void __launch_bounds__(256) decode_gateup_kernel(DecodeParams p) {
  extern __shared__ float4 smem4[];
  float4* v = smem4;                                   // d/4 float4
  float* csum = reinterpret_cast<float*>(smem4 + p.d / 4);  // d/32
  stage_bf16_vector(p.x, p.d, v, csum);
  const int nslots = p.k + (p.shared ? 1 : 0);
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (gw >= nslots * p.f) return;
  const int slot = gw / p.f, row = gw % p.f;
  const int64_t qrow = p.d / 8, grow = p.d / 64;
  const moe_w4_t *G, *U;
  int64_t e = 0;
  if (slot < p.k) {
    e = p.ids[slot];
    if (e < 0 || e >= p.E) {
      report(p.status, MOE_DEV_BAD_EXPERT, 21, (int)e);
      return;
    }
    G = &p.w.gate;
    U = &p.w.up;
  } else {
    G = &p.w.sh_gate;
    U = &p.w.sh_up;
  }
  const int64_t r = e * p.f + row;
  const float g = w4_row_dot(G->q + r * qrow, G->scale + r * grow, G->bias + r * grow, p.d, v, csum);
  const float u = w4_row_dot(U->q + r * qrow, U->scale + r * grow, U->bias + r * grow, p.d, v, csum);
  if ((threadIdx.x & 31) == 0) p.h[(size_t)slot * p.f + row] = g / (1.f + expf(-g)) * u;
}

// grid: d / 8 blocks of 8 warps; warp -> output column j.
__global__ void __launch_bounds__(256) decode_down_kernel(DecodeParams p) {
  extern __shared__ float4 smem4[];
  const int nslots = p.k + (p.shared ? 1 : 0);
  const int fch = p.f / 32;                  // chunks per h row
  float4* hv = smem4;                        // nslots * f / 4 float4
  float* hsum = reinterpret_cast<float*>(smem4 + nslots * p.f / 4);  // nslots * fch
  float* coef = hsum + nslots * fch;         // nslots
  int* eid = reinterpret_cast<int*>(coef + nslots);
  for (int i = threadIdx.x; i < nslots * p.f / 4; i += blockDim.x)
    hv[chunk_slot(i >> 3, i & 7)] = reinterpret_cast<const float4*>(p.h)[i];
  if (threadIdx.x < nslots) {
    coef[threadIdx.x] = p.wts[threadIdx.x];
    eid[threadIdx.x] = threadIdx.x < p.k ? p.ids[threadIdx.x] : 0;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nslots * fch; c += blockDim.x) {
    float s = 0.f;
    for (int j = 0; j < 8; ++j) {
      const float4 f = hv[chunk_slot(c, j)];
      s += (f.x + f.y) + (f.z + f.w);
    }
    hsum[c] = s;
  }
  __syncthreads();
  const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (j >= p.d) return;
  const int lane = threadIdx.x & 31;
  const int64_t qrow = p.f / 8, grow = p.f / 64;
  float acc = 0.f;
  for (int idx = lane; idx < nslots * fch; idx += 32) {
    const int slot = idx / fch, c = idx % fch;
    const moe_w4_t* D = slot < p.k ? &p.w.down : &p.w.sh_down;
    const int64_t e = slot < p.k ? eid[slot] : 0;
    if (e < 0 || e >= p.E) continue;
    const int64_t r = e * p.d + j;
    const uint4 w = __ldcs(reinterpret_cast<const uint4*>(D->q + r * qrow) + c);
    const float s = bf16_bits_to_f32(D->scale[r * grow + (c >> 1)]);
    const float b = bf16_bits_to_f32(D->bias[r * grow + (c >> 1)]);
    const float part = fmaf(s, chunk_dot(w, hv, idx), b * hsum[idx]);
    acc = fmaf(coef[slot], part, acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
  if (lane == 0) {
    const __nv_bfloat16 o = __float2bfloat16_rn(acc);
    p.out[j] = *reinterpret_cast<const uint16_t*>(&o);
  }
}

}  // namespace

int decode_router_splits(int d) { return d / kRouterRows; }

cudaError_t decode_launch(const DecodeParams& p, cudaStream_t s) {
  const int nsplit = decode_router_splits(p.d);
  const int npl = (p.E + 31) / 32;
  if (npl <= 1) decode_router_kernel<1><<<nsplit, 256, 0, s>>>(p, nsplit);
  else if (npl <= 2) decode_router_kernel<2><<<nsplit, 256, 0, s>>>(p, nsplit);
  else if (npl <= 4) decode_router_kernel<4><<<nsplit, 256, 0, s>>>(p, nsplit);
  else if (npl <= 8) decode_router_kernel<8><<<nsplit, 256, 0, s>>>(p, nsplit);
  else if (npl <= 16) decode_router_kernel<16><<<nsplit, 256, 0, s>>>(p, nsplit);
  else decode_router_kernel<32><<<nsplit, 256, 0, s>>>(p, nsplit);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int nslots = p.k + (p.shared ? 1 : 0);
  const size_t gu_smem = (size_t)p.d * 4 + (size_t)(p.d / 32) * 4;
  if (gu_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(decode_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)gu_smem);
    if (err != cudaSuccess) return err;
  }
  decode_gateup_kernel<<<(nslots * p.f + 7) / 8, 256, gu_smem, s>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t dn_smem = (size_t)nslots * p.f * 4 + (size_t)nslots * (p.f / 32) * 4 + nslots * 8;
  if (dn_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)dn_smem);
    if (err != cudaSuccess) return err;
  }
  decode_down_kernel<<<(p.d + 7) / 8, 256, dn_smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
