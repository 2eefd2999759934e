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
// j = j0 + w, j0 + w + 8, ... of its slice, two per step. Lane l holds
// elements l*E .. l*E+E-1 (E = d / 32) of q (pre-scaled), of the current k and
// v rows and of the running output of every query head. Per position: the
// group's scores (E-term partial dots, one transpose reduction for all
// heads), then the online softmax update per head (running max m, running sum
// l; the output is scaled by exp(m_old - m_new), exactly 1 when the max
// stays, with no branch). The block's 8 warp
// states merge (in warp order) into one partial (m, l, unnormalised output)
// per query head. Combine kernel: per query head and 64 output elements, the
// blocks' partials merged with weights exp(m_part - max m) and divided by the
// merged sum (block-wide reductions in a fixed order).
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

constexpr int kRing = 16;  // positions in flight per warp

// 16-, 8- or 4-byte cp.async global -> shared (the lane's own elements of a row)
template <int B>
MOE_DEVINL void cp_async_bytes(uint32_t dst, const void* src) {
  if constexpr (B == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(dst), "l"(src), "n"(B) : "memory");
}

template <int E>
MOE_DEVINL void load_row_smem(const uint8_t* p, float (&f)[E]) {
  if constexpr (E == 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(u[i] << 16);
      f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  } else if constexpr (E == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xFFFF0000u);
  }
}

// The group's 8 scores from each lane's partial dots x[h]: a transpose
// reduction (at the step across lane bit b, a lane keeps half of its values
// and adds the partner's copies of them: 4 + 2 + 1 shuffles), the remaining
// two steps of a butterfly, then each head's sum broadcast from a lane that
// holds it: 17 shuffles instead of 8 butterflies of 5. x[h] becomes head h's
// full sum on every lane.
MOE_DEVINL void group_scores(float (&x)[kAttnMaxGroup], int lane) {
  constexpr unsigned kAll = 0xffffffffu;
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float y[4], z[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // heads 4 b4 + i
    const float send = b4 ? x[i] : x[i + 4], keep = b4 ? x[i + 4] : x[i];
    y[i] = keep + __shfl_xor_sync(kAll, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {  // heads 4 b4 + 2 b3 + i
    const float send = b3 ? y[i] : y[i + 2], keep = b3 ? y[i + 2] : y[i];
    z[i] = keep + __shfl_xor_sync(kAll, send, 8);
  }
  float w = (b2 ? z[1] : z[0]) + __shfl_xor_sync(kAll, b2 ? z[0] : z[1], 4);  // head 4 b4 + 2 b3 + b2
  w += __shfl_xor_sync(kAll, w, 2);
  w += __shfl_xor_sync(kAll, w, 1);
#pragma unroll
  for (int h = 0; h < kAttnMaxGroup; ++h)
    x[h] = __shfl_sync(kAll, w, ((h >> 2) << 4) | (((h >> 1) & 1) << 3) | ((h & 1) << 2));
}

template <int E>
__global__ void __launch_bounds__(32 * kAttnWarps, 1) attn_split_kernel(const AttnParams p) {
  const int g = blockIdx.x, split = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv, d = 32 * E;
  const int per = (p.L + gridDim.y - 1) / gridDim.y;
  const int j0 = split * per, j1 = min(p.L, j0 + per);
  // K and V rows of the warp's next kRing positions in flight: each lane
  // copies (cp.async) exactly the E elements of each row it later reads, into
  // its own slots of a per-warp shared-memory ring, so the ring needs no
  // synchronisation beyond the lane's own wait_group
  extern __shared__ __align__(16) uint8_t attn_ring[];
  uint8_t* ring = attn_ring + (size_t)warp * kRing * 2 * (32 * E * 2);
  auto slot = [&](int r, int kv) { return smem_u32(ring + ((size_t)(r * 2 + kv) * 32 + lane) * (E * 2)); };
  auto issue = [&](int j, int r) {
    if (j < j1) {
      const int64_t row = ((int64_t)j * p.Hkv + g) * d + lane * E;
      cp_async_bytes<E * 2>(slot(r, 0), p.K + row);
      cp_async_bytes<E * 2>(slot(r, 1), p.V + row);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int r = 0; r < kRing; ++r) issue(j0 + warp + r * kAttnWarps, r);
  // q and the running state (after the first copies are on their way)
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
  // Two positions per step (j and j + 8, ring slots r and r + 1): their
  // score reductions and softmax updates are independent chains that
  // overlap. A second position past the slice's end counts as score -inf
  // with its v taken as zero (its ring slot was never filled).
  int r = 0;
#pragma unroll 1
  for (int j = j0 + warp; j < j1; j += 2 * kAttnWarps, r = (r + 2) % kRing) {
    const bool two = j + kAttnWarps < j1;
    cp_async_wait<kRing - 2>();
    float k[2][E], v[2][E];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      load_row_smem<E>(ring + ((size_t)((r + t) * 2 + 0) * 32 + lane) * (E * 2), k[t]);
      load_row_smem<E>(ring + ((size_t)((r + t) * 2 + 1) * 32 + lane) * (E * 2), v[t]);
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) issue(j + (kRing + t) * kAttnWarps, r + t);  // the slots are read: refill them
    if (!two) {
#pragma unroll
      for (int e = 0; e < E; ++e) v[1][e] = 0.f;
    }
    float sc[2][kAttnMaxGroup];  // (q of the heads past G is zero)
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int h = 0; h < kAttnMaxGroup; ++h) {
        sc[t][h] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) sc[t][h] = fmaf(q[h][e], k[t][e], sc[t][h]);
      }
    group_scores(sc[0], lane);
    group_scores(sc[1], lane);
#pragma unroll
    for (int h = 0; h < kAttnMaxGroup; ++h) {
      if (h >= G) break;
      const float s0 = sc[0][h], s1 = two ? sc[1][h] : -INFINITY;
      const float mn = fmaxf(m[h], fmaxf(s0, s1));
      const float c = __expf(m[h] - mn);  // 1 when the max stays; 0 while m is -inf
      m[h] = mn;
      const float w0 = __expf(s0 - mn), w1 = __expf(s1 - mn);
      l[h] = fmaf(l[h], c, w0 + w1);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[h][e] = fmaf(w1, v[1][e], fmaf(w0, v[0][e], acc[h][e] * c));
    }
  }
  // the warps' states merge into one partial per (block, query head): each
  // warp's (m, l, output) goes to shared memory (the ring, once every copy
  // has landed), then each (head, element) is merged over the warps in order
  cp_async_wait<0>();
  __syncthreads();
  float* st = reinterpret_cast<float*>(attn_ring);  // [warp][head][2 + d]
#pragma unroll
  for (int h = 0; h < kAttnMaxGroup; ++h) {
    if (h >= G) break;
    float* w = st + (size_t)(warp * G + h) * (2 + d);
    if (lane == 0) {
      w[0] = m[h];
      w[1] = l[h];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) w[2 + lane * E + e] = acc[h][e];
  }
  __syncthreads();
  const int P = gridDim.y;
  for (int i = threadIdx.x; i < G * d; i += blockDim.x) {
    const int h = i / d, e = i - h * d;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, st[(size_t)(w * G + h) * (2 + d)]);
    float sl = 0.f, so = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float* ws = st + (size_t)(w * G + h) * (2 + d);
      const float c = ws[0] > -INFINITY ? __expf(ws[0] - M) : 0.f;
      sl = fmaf(ws[1], c, sl);
      so = fmaf(ws[2 + e], c, so);
    }
    const int qh = g * G + h;
    if (e == 0) {
      p.part_m[(int64_t)qh * P + split] = M;
      p.part_l[(int64_t)qh * P + split] = sl;
    }
    p.part_o[((int64_t)qh * P + split) * d + e] = so;
  }
}

// Merge of the partials: one block per (query head, 64 output elements).
// The merged max over the P partials and the weights w_i = exp(m_i - max)
// come from block-wide reductions in a fixed order (each thread's share in
// index order, then the warps' butterfly, then warps in order), so the result
// does not depend on timing; then each output element is summed over the
// partials by 4 threads (quarters of the index range, added in order).
constexpr int kCombThreads = 256;
MOE_DEVINL float block_reduce(float v, bool is_max, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  __syncthreads();  // red is free
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < kCombThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  return r;
}

__global__ void __launch_bounds__(kCombThreads) attn_combine_kernel(const AttnParams p, int P) {
  extern __shared__ float s_w[];  // [P] merge weights, then [4][64] quarter sums, then [8] reduction slots
  float* quart = s_w + P;
  float* red = quart + 4 * 64;
  const int qh = blockIdx.x, e0 = blockIdx.y * 64, d = p.d;
  const float* pm = p.part_m + (int64_t)qh * P;
  const float* pl = p.part_l + (int64_t)qh * P;
  float m = -INFINITY;
  for (int i = threadIdx.x; i < P; i += kCombThreads) m = fmaxf(m, pm[i]);
  const float M = block_reduce(m, true, red);
  float l = 0.f;
  for (int i = threadIdx.x; i < P; i += kCombThreads) {
    const float mi = pm[i];
    const float w = mi > -INFINITY ? __expf(mi - M) : 0.f;
    s_w[i] = w;
    l = fmaf(pl[i], w, l);
  }
  const float inv = 1.f / block_reduce(l, false, red);  // also orders the s_w writes before the reads
  const int t = threadIdx.x & 63, q = threadIdx.x >> 6;  // element, quarter of the partials
  const int i0 = P * q / 4, i1 = P * (q + 1) / 4;
  float o = 0.f;
  if (e0 + t < d) {
    const float* po = p.part_o + ((int64_t)qh * P) * d + e0 + t;
#pragma unroll 4
    for (int i = i0; i < i1; ++i) o = fmaf(po[(int64_t)i * d], s_w[i], o);
  }
  quart[q * 64 + t] = o;
  __syncthreads();
  if (threadIdx.x < 64 && e0 + t < d)
    p.out[(int64_t)qh * d + e0 + t] = (((quart[t] + quart[64 + t]) + quart[128 + t]) + quart[192 + t]) * inv;
}

}  // namespace

bool attn_shape_supported(int L, int Hq, int Hkv, int d) {
  return L >= 1 && (d == 64 || d == 128 || d == 256) && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 &&
         Hq / Hkv <= kAttnMaxGroup;
}

// slots: blocks resident at once on the GPU (blocks per SM x SMs).
int attn_splits(int L, int Hkv, int slots) {
  const int by_len = (L + 63) / 64;                // at least 8 positions per warp
  const int by_grid = std::max(1, slots / Hkv);    // one wave of resident blocks
  return std::max(1, std::min(by_len, by_grid));
}

size_t attn_workspace_floats(int L, int Hq, int Hkv, int d, int slots) {
  const size_t P = (size_t)attn_splits(L, Hkv, slots);
  return (size_t)Hq * P * (2 + (size_t)d);
}

template <int E>
cudaError_t split_setup(size_t ring, int sms, int* slots) {
  cudaError_t err = cudaFuncSetAttribute(attn_split_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_split_kernel<E>, 32 * kAttnWarps, ring);
  *slots = std::max(1, per_sm) * sms;
  return err;
}

cudaError_t attn_decode_launch(const AttnParams& pin, int sms, cudaStream_t s) {
  if (!attn_shape_supported(pin.L, pin.Hq, pin.Hkv, pin.d) || !pin.ws) return cudaErrorInvalidValue;
  const size_t ring = (size_t)kAttnWarps * kRing * 2 * pin.d * 2;  // bf16 K and V rows per warp slot
  int slots = sms;
  cudaError_t err = pin.d == 256 ? split_setup<8>(ring, sms, &slots)
                    : pin.d == 128 ? split_setup<4>(ring, sms, &slots)
                                   : split_setup<2>(ring, sms, &slots);
  if (err != cudaSuccess) return err;
  const int splits = attn_splits(pin.L, pin.Hkv, slots);
  const size_t P = (size_t)splits;  // partials per query head: one per block
  AttnParams p = pin;
  p.part_m = p.ws;
  p.part_l = p.ws + (size_t)p.Hq * P;
  p.part_o = p.ws + 2 * (size_t)p.Hq * P;
  const dim3 grid(p.Hkv, splits);
  if (p.d == 256)
    attn_split_kernel<8><<<grid, 32 * kAttnWarps, ring, s>>>(p);
  else if (p.d == 128)
    attn_split_kernel<4><<<grid, 32 * kAttnWarps, ring, s>>>(p);
  else
    attn_split_kernel<2><<<grid, 32 * kAttnWarps, ring, s>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int P2 = splits;
  const size_t comb_smem = ((size_t)P2 + 4 * 64 + kCombThreads / 32) * sizeof(float);
  if (comb_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(attn_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)comb_smem);
    if (err != cudaSuccess) return err;
  }
  attn_combine_kernel<<<dim3(p.Hq, (p.d + 63) / 64), kCombThreads, comb_smem, s>>>(p, P2);
  return cudaGetLastError();
}

}  // namespace moe
