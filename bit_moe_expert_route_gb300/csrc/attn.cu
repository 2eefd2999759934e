// Batch-1 decode attention with grouped KV heads (GQA packing).
//
// "Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple Silicon",
// section "Decode optimizations", the GQA paragraph: eight query heads share
// one KV head, and packing the query heads of a group into one threadgroup lets
// them share the KV loads. Here one block takes one KV head and one slice of
// the cache for all of that head's query heads (up to 8): every K and V row
// the block reads serves every query head of the group.
//
//   o_h = sum_j softmax_j(scale * q_h . k_{g,j}) v_{g,j},   g = h / (Hq / Hkv)
//
// Split kernel: grid (Hkv, splits); 8 warps per block, warp w takes positions
// j = j0 + w, j0 + w + 8, ... of its slice. Lane l holds elements
// l*E .. l*E+E-1 (E = d / 32) of q (pre-scaled), of the current k and v rows
// and of the running output of every query head. Per position: the group's
// scores (E-term partial dots, butterfly warp sums), then the online softmax
// update per head (running max m, running sum l, output rescaled when the max
// grows). Each warp writes its (m, l, unnormalised output) per head as one
// partial. Combine kernel: per query head, all partials merged with weights
// exp(m_part - max m) and divided by the merged sum.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kAttnWarps = 8;
constexpr int kAttnMaxGroup = 8;

template <int E>
MOE_DEVINL void load_row(const uint16_t* p, float (&f)[E]) {
  if constexpr (E == 8) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(u[i] << 16);
      f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  } else if constexpr (E == 4) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  } else {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(p));
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xFFFF0000u);
  }
}

MOE_DEVINL float attn_warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

template <int E>
__global__ void __launch_bounds__(32 * kAttnWarps, 1) attn_split_kernel(const AttnParams p) {
  const int g = blockIdx.x, split = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv, d = 32 * E;
  const int per = (p.L + gridDim.y - 1) / gridDim.y;
  const int j0 = split * per, j1 = min(p.L, j0 + per);
  float q[kAttnMaxGroup][E], acc[kAttnMaxGroup][E], m[kAttnMaxGroup], l[kAttnMaxGroup];
#pragma unroll
  for (int h = 0; h < kAttnMaxGroup; ++h) {
    float f[E];
    if (h < G) {
      load_row<E>(p.q + (int64_t)(g * G + h) * d + lane * E, f);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) f[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      q[h][e] = f[e] * p.scale;
      acc[h][e] = 0.f;
    }
    m[h] = -INFINITY;
    l[h] = 0.f;
  }
#pragma unroll 1
  for (int j = j0 + warp; j < j1; j += kAttnWarps) {
    float k[E], v[E];
    const int64_t row = ((int64_t)j * p.Hkv + g) * d + lane * E;
    load_row<E>(p.K + row, k);
    load_row<E>(p.V + row, v);
#pragma unroll
    for (int h = 0; h < kAttnMaxGroup; ++h) {
      if (h >= G) break;
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) s = fmaf(q[h][e], k[e], s);
      s = attn_warp_sum(s);
      const float m_new = fmaxf(m[h], s);
      const float c = __expf(m[h] - m_new);  // 0 while m is still -inf
      const float w = __expf(s - m_new);
      l[h] = fmaf(l[h], c, w);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[h][e] = fmaf(acc[h][e], c, w * v[e]);
      m[h] = m_new;
    }
  }
  // one partial per (warp, query head): running max, running sum, output
  const int P = gridDim.y * kAttnWarps, part = split * kAttnWarps + warp;
#pragma unroll
  for (int h = 0; h < kAttnMaxGroup; ++h) {
    if (h >= G) break;
    const int qh = g * G + h;
    if (lane == 0) {
      p.part_m[(int64_t)qh * P + part] = m[h];
      p.part_l[(int64_t)qh * P + part] = l[h];
    }
    float* o = p.part_o + ((int64_t)qh * P + part) * d + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = acc[h][e];
  }
}

// One block per query head; thread t merges element t of every partial.
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnParams p, int P) {
  const int qh = blockIdx.x, d = p.d;
  const float* pm = p.part_m + (int64_t)qh * P;
  const float* pl = p.part_l + (int64_t)qh * P;
  float M = -INFINITY;
  for (int i = 0; i < P; ++i) M = fmaxf(M, pm[i]);
  float L = 0.f;
  for (int i = 0; i < P; ++i)
    if (pm[i] > -INFINITY) L = fmaf(pl[i], __expf(pm[i] - M), L);
  const float inv = 1.f / L;
  for (int t = threadIdx.x; t < d; t += blockDim.x) {
    float o = 0.f;
    for (int i = 0; i < P; ++i)
      if (pm[i] > -INFINITY) o = fmaf(p.part_o[((int64_t)qh * P + i) * d + t], __expf(pm[i] - M), o);
    p.out[(int64_t)qh * d + t] = o * inv;
  }
}

}  // namespace

bool attn_shape_supported(int L, int Hq, int Hkv, int d) {
  return L >= 1 && (d == 64 || d == 128 || d == 256) && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 &&
         Hq / Hkv <= kAttnMaxGroup;
}

int attn_splits(int L, int Hkv, int sms) {
  const int by_len = (L + 255) / 256;           // at least 32 positions per warp
  const int by_grid = std::max(1, 2 * sms / Hkv);  // about two blocks per SM
  return std::max(1, std::min(by_len, by_grid));
}

size_t attn_workspace_floats(int L, int Hq, int Hkv, int d, int sms) {
  const size_t P = (size_t)attn_splits(L, Hkv, sms) * kAttnWarps;
  return (size_t)Hq * P * (2 + (size_t)d);
}

cudaError_t attn_decode_launch(const AttnParams& pin, int sms, cudaStream_t s) {
  if (!attn_shape_supported(pin.L, pin.Hq, pin.Hkv, pin.d) || !pin.ws) return cudaErrorInvalidValue;
  const int splits = attn_splits(pin.L, pin.Hkv, sms);
  const size_t P = (size_t)splits * kAttnWarps;  // partials per query head
  AttnParams p = pin;
  p.part_m = p.ws;
  p.part_l = p.ws + (size_t)p.Hq * P;
  p.part_o = p.ws + 2 * (size_t)p.Hq * P;
  const dim3 grid(p.Hkv, splits);
  if (p.d == 256)
    attn_split_kernel<8><<<grid, 32 * kAttnWarps, 0, s>>>(p);
  else if (p.d == 128)
    attn_split_kernel<4><<<grid, 32 * kAttnWarps, 0, s>>>(p);
  else
    attn_split_kernel<2><<<grid, 32 * kAttnWarps, 0, s>>>(p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  attn_combine_kernel<<<p.Hq, 256, 0, s>>>(p, splits * kAttnWarps);
  return cudaGetLastError();
}

}  // namespace moe
