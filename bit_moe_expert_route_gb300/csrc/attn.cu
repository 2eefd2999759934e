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
// Split kernel: grid (Hkv, splits); 8 position sets per block, each walked by
// one warp per group of 4 query heads (8 or 16 warps): the warps of set w take
// positions j = j0 + w, j0 + w + 8, ... of the slice, two per step. Lane l
// holds elements l*E .. l*E+E-1 (E = d / 32) of q (its bf16 pairs), of the
// current k and v rows and of the running output of each of its 4 query
// heads. Per position: the heads' scores (E-term partial dots of bf16 pairs
// in mixed-precision FMAs, exact products; one transpose reduction for the 4
// heads; then the scale), then the online softmax update per head (reference
// max m, running sum l: m moves, and the output and l are rescaled by
// exp(m_old - m_new), only when a score exceeds m by more than 8, so the
// weights exp(s - m) stay below e^8 and rescales are rare). Each head's 8 position-set
// states merge (in set order) into one partial (m, l, unnormalised output)
// per block and query head. Combine kernel: per query head and 64 output elements, the
// blocks' partials merged with weights exp(m_part - max m) and divided by the
// merged sum (block-wide reductions in a fixed order).
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "gemv_dot.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kAttnWarps = 8;     // position sets per block (one warp per set and head group)
constexpr int kAttnMaxGroup = 8;  // query heads per KV head

constexpr int kRing = 16;  // positions in flight per position set (per warp: 16 / head groups)

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

// Four heads' scores from each lane's partial dots x[h]: a transpose
// reduction over lane bits 4 and 3 (2 + 1 shuffles), a butterfly over bits
// 2..0, then each head's sum broadcast from a lane that holds it.
MOE_DEVINL void group_scores4(float (&x)[4], int lane) {
  constexpr unsigned kAll = 0xffffffffu;
  const bool b4 = lane & 16, b3 = lane & 8;
  float y[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {  // heads 2 b4 + i
    const float send = b4 ? x[i] : x[i + 2], keep = b4 ? x[i + 2] : x[i];
    y[i] = keep + __shfl_xor_sync(kAll, send, 16);
  }
  float w = (b3 ? y[1] : y[0]) + __shfl_xor_sync(kAll, b3 ? y[0] : y[1], 8);  // head 2 b4 + b3
  w += __shfl_xor_sync(kAll, w, 4);
  w += __shfl_xor_sync(kAll, w, 2);
  w += __shfl_xor_sync(kAll, w, 1);
#pragma unroll
  for (int h = 0; h < 4; ++h) x[h] = __shfl_sync(kAll, w, ((h >> 1) << 4) | ((h & 1) << 3));
}

constexpr int kHeadsPerWarp = 4;
// a head's reference max m moves only when a score exceeds it by more than
// this (natural-log units): the weights exp(s - m) stay below e^8
constexpr float kLazy = 8.f;

// Block: 8 position sets x HG head groups of 4 (HG = 1 for up to 4 query
// heads per KV head, else 2): warp w walks positions j0 + (w % 8) + 8 i for
// heads 4 (w / 8) .. 4 (w / 8) + 3, with a ring of R = 16 / HG positions.
template <int E>
__global__ void __launch_bounds__(32 * kAttnWarps * 2, 1) attn_split_kernel(const AttnParams p) {
  const int g = blockIdx.x, split = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pw = warp % kAttnWarps, hg = warp / kAttnWarps;
  const int HG = blockDim.x / (32 * kAttnWarps), R = kRing / HG;
  const int G = p.Hq / p.Hkv, d = 32 * E;
  const int per = (p.L + gridDim.y - 1) / gridDim.y;
  const int j0 = split * per, j1 = min(p.L, j0 + per);
  extern __shared__ __align__(16) uint8_t attn_ring[];
  uint8_t* ring = attn_ring + (size_t)warp * R * 2 * (32 * E * 2);
  auto slot = [&](int r, int kv) { return smem_u32(ring + ((size_t)(r * 2 + kv) * 32 + lane) * (E * 2)); };
  auto issue = [&](int j, int r) {
    if (j < j1) {
      const int64_t row = ((int64_t)j * p.Hkv + g) * d + lane * E;
      cp_async_bytes<E * 2>(slot(r, 0), p.K + row);
      cp_async_bytes<E * 2>(slot(r, 1), p.V + row);
    }
    cp_async_commit();
  };
  for (int r = 0; r < R; ++r) issue(j0 + pw + r * kAttnWarps, r);
  constexpr int NH = kHeadsPerWarp;
  // q as the lane's bf16 pairs (exact: the scale multiplies the reduced score)
  uint32_t qp[NH][E / 2];
  float acc[NH][E], m[NH], l[NH];
#pragma unroll
  for (int hh = 0; hh < NH; ++hh) {
    const int h = hg * NH + hh;
#pragma unroll
    for (int i = 0; i < E / 2; ++i)
      qp[hh][i] = h < G ? __ldg(reinterpret_cast<const uint32_t*>(p.q + (int64_t)(g * G + h) * d + lane * E) + i) : 0u;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[hh][e] = 0.f;
    m[hh] = -INFINITY;
    l[hh] = 0.f;
  }
  int r = 0;
#pragma unroll 1
  for (int j = j0 + pw; j < j1; j += 2 * kAttnWarps, r = (r + 2 == R) ? 0 : r + 2) {
    const bool two = j + kAttnWarps < j1;
    if (R == kRing) cp_async_wait<kRing - 2>(); else cp_async_wait<kRing / 2 - 2>();
    float sc[2][NH];  // (q of the heads past G is zero)
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      uint32_t kw[E / 2];
      const uint8_t* kr = ring + ((size_t)((r + t) * 2 + 0) * 32 + lane) * (E * 2);
#pragma unroll
      for (int i = 0; i < E / 2; ++i) kw[i] = reinterpret_cast<const uint32_t*>(kr)[i];
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < E / 2; ++i) fma_pair<true>(a0, a1, qp[hh][i], kw[i]);
        sc[t][hh] = a0 + a1;
      }
    }
    float v[2][E];
#pragma unroll
    for (int t = 0; t < 2; ++t) load_row_smem<E>(ring + ((size_t)((r + t) * 2 + 1) * 32 + lane) * (E * 2), v[t]);
#pragma unroll
    for (int t = 0; t < 2; ++t) issue(j + (R + t) * kAttnWarps, r + t);  // the slots are read: refill them
    if (!two) {
#pragma unroll
      for (int e = 0; e < E; ++e) v[1][e] = 0.f;
    }
    group_scores4(sc[0], lane);
    group_scores4(sc[1], lane);
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) sc[t][hh] *= p.scale;
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      const float s0 = sc[0][hh], s1 = two ? sc[1][hh] : -INFINITY;
      const float smax = fmaxf(s0, s1);
      if (smax > m[hh] + kLazy) {  // same on every lane; rare once the max has settled
        const float c = __expf(m[hh] - smax);  // 0 while m is -inf
        l[hh] *= c;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[hh][e] *= c;
        m[hh] = smax;
      }
      const float w0 = __expf(s0 - m[hh]), w1 = __expf(s1 - m[hh]);
      l[hh] += w0 + w1;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[hh][e] = fmaf(w1, v[1][e], fmaf(w0, v[0][e], acc[hh][e]));
    }
  }
  // the warps' states merge into one partial per (block, query head): each
  // warp's (m, l, output) goes to shared memory (the ring, once every copy
  // has landed), then each (head, element) is merged over the 8 position
  // sets in order
  cp_async_wait<0>();
  __syncthreads();
  float* st = reinterpret_cast<float*>(attn_ring);  // [head][position set][2 + d]
#pragma unroll
  for (int hh = 0; hh < NH; ++hh) {
    const int h = hg * NH + hh;
    if (h >= G) break;
    float* w = st + (size_t)(h * kAttnWarps + pw) * (2 + d);
    if (lane == 0) {
      w[0] = m[hh];
      w[1] = l[hh];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) w[2 + lane * E + e] = acc[hh][e];
  }
  __syncthreads();
  const int P = gridDim.y;
  for (int i = threadIdx.x; i < G * d; i += blockDim.x) {
    const int h = i / d, e = i - h * d;
    const float* sh = st + (size_t)h * kAttnWarps * (2 + d);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, sh[(size_t)w * (2 + d)]);
    float sl = 0.f, so = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float* ws = sh + (size_t)w * (2 + d);
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

// Merge of the partials: one block per (query head, 32 output elements).
// The merged max over the P partials and the weights w_i = exp(m_i - max)
// come from block-wide reductions in a fixed order (each thread's share in
// index order, then the warps' butterfly, then warps in order), so the result
// does not depend on timing; then each output element is summed over the
// partials by 8 threads, one per warp (eighths of the index range, added in
// order). A thread loads its first 16 partial outputs before the reductions
// (they do not depend on the weights), so those loads overlap them.
constexpr int kCombThreads = 256;
constexpr int kCombCols = 32;                          // output elements per block
constexpr int kCombSlices = kCombThreads / kCombCols;  // partial ranges per element
constexpr int kCombAhead = 16;                         // partial outputs loaded early
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
  extern __shared__ float s_w[];  // [P] merge weights, [8][32] slice sums, [8] reduction slots
  float* slice = s_w + P;
  float* red = slice + kCombSlices * kCombCols;
  const int qh = blockIdx.x, e0 = blockIdx.y * kCombCols, d = p.d;
  const int t = threadIdx.x % kCombCols, q = threadIdx.x / kCombCols;  // element, slice of the partials
  const int i0 = P * q / kCombSlices, i1 = P * (q + 1) / kCombSlices;
  const bool col = e0 + t < d;
  const float* po = p.part_o + ((int64_t)qh * P) * d + e0 + t;
  float ahead[kCombAhead];
#pragma unroll
  for (int k = 0; k < kCombAhead; ++k) ahead[k] = col && i0 + k < i1 ? po[(int64_t)(i0 + k) * d] : 0.f;
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
  float o = 0.f;
#pragma unroll
  for (int k = 0; k < kCombAhead; ++k)
    if (i0 + k < i1) o = fmaf(ahead[k], s_w[i0 + k], o);
  if (col)
    for (int i = i0 + kCombAhead; i < i1; ++i) o = fmaf(po[(int64_t)i * d], s_w[i], o);
  slice[q * kCombCols + t] = o;
  __syncthreads();
  if (threadIdx.x < kCombCols && col) {
    float r = slice[t];
#pragma unroll
    for (int k = 1; k < kCombSlices; ++k) r += slice[k * kCombCols + t];
    p.out[(int64_t)qh * d + e0 + t] = r * inv;
  }
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
cudaError_t split_setup(size_t ring, int threads, int sms, int* slots) {
  cudaError_t err = cudaFuncSetAttribute(attn_split_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_split_kernel<E>, threads, ring);
  *slots = std::max(1, per_sm) * sms;
  return err;
}

cudaError_t attn_decode_launch(const AttnParams& pin, int sms, cudaStream_t s) {
  if (!attn_shape_supported(pin.L, pin.Hq, pin.Hkv, pin.d) || !pin.ws) return cudaErrorInvalidValue;
  // bf16 K and V rows: kRing slots per position set (shared out among its warps)
  const size_t ring = (size_t)kAttnWarps * kRing * 2 * pin.d * 2;
  const int HG = pin.Hq / pin.Hkv > kHeadsPerWarp ? 2 : 1;         // head groups of 4 per block
  const int threads = 32 * kAttnWarps * HG;
  int slots = sms;
  cudaError_t err = pin.d == 256 ? split_setup<8>(ring, threads, sms, &slots)
                    : pin.d == 128 ? split_setup<4>(ring, threads, sms, &slots)
                                   : split_setup<2>(ring, threads, sms, &slots);
  if (err != cudaSuccess) return err;
  const int splits = attn_splits(pin.L, pin.Hkv, slots);
  const size_t P = (size_t)splits;  // partials per query head: one per block
  AttnParams p = pin;
  p.part_m = p.ws;
  p.part_l = p.ws + (size_t)p.Hq * P;
  p.part_o = p.ws + 2 * (size_t)p.Hq * P;
  const dim3 grid(p.Hkv, splits);
  if (p.d == 256)
    attn_split_kernel<8><<<grid, threads, ring, s>>>(p);
  else if (p.d == 128)
    attn_split_kernel<4><<<grid, threads, ring, s>>>(p);
  else
    attn_split_kernel<2><<<grid, threads, ring, s>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int P2 = splits;
  const size_t comb_smem = ((size_t)P2 + kCombSlices * kCombCols + kCombThreads / 32) * sizeof(float);
  if (comb_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(attn_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)comb_smem);
    if (err != cudaSuccess) return err;
  }
  attn_combine_kernel<<<dim3(p.Hq, (p.d + kCombCols - 1) / kCombCols), kCombThreads, comb_smem, s>>>(p, P2);
  return cudaGetLastError();
}

}  // namespace moe
