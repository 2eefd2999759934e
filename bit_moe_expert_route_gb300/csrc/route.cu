// GPU-resident expert routing: top-k selection and weights, per-block
// histograms, a scan that yields per-expert offsets and the block map, and a
// stable, atomics-free scatter of the (token, slot) assignments into expert
// order. ("Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple
// Silicon", section "Prefill optimizations", second bullet: histogram,
// prefix scan, scatter and block-map build all stay on the GPU.)
//
// Three launches, no host round trip:
//   1. route_topk_kernel    one warp per token (32 warps per block, the next
//                           token's logits loaded while the current one is
//                           ranked): top-k by warp argmax (value descending,
//                           ties to the lower id) with two warp reductions per
//                           round, softmax over the selected logits, per-block
//                           expert histogram (shared-memory counts).
//   2. route_scan_kernel    one CTA: per-(block, expert) bases, counts,
//                           offsets, tile offsets and the block map.
//   3. route_scatter_kernel per block: stable rank of each assignment inside
//                           its warp slice by __match_any_sync + popc, then
//                           perm / inv_perm / row_token / row_weight.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kFull = 0xFFFFFFFFu;

// Threads per top-k block: 32 warps (4 tokens each) while the per-lane
// logit registers stay small, 8 warps for very wide routers.
template <int NPL>
constexpr int topk_threads() { return NPL <= 8 ? 1024 : 256; }

template <int NPL>  // logits per lane: E <= 32 * NPL
__global__ void __launch_bounds__(topk_threads<NPL>()) route_topk_kernel(RouteParams p) {
  constexpr int kW = topk_threads<NPL>() / 32;
  constexpr bool kPrefetch = NPL <= 8;
  extern __shared__ int hist[];  // [E]
  for (int e = threadIdx.x; e < p.E; e += kW * 32) hist[e] = 0;
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t_begin = blockIdx.x * kRouteTPB;
  const int t_end = min(p.T, t_begin + kRouteTPB);
  // keys of z = logit + bias (fp32 add, the decision precision) for one token
  auto load_keys = [&](int t, uint32_t (&key)[NPL]) {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = i * 32 + lane;
      uint32_t kv = 0u;
      if (e < p.E) {
        float v = p.logits[(size_t)t * p.E + e];
        if (p.bias) v = v + p.bias[e];
        kv = order_key(v);
      }
      key[i] = kv;
    }
  };
  uint32_t next[NPL];
  if (kPrefetch && t_begin + warp < t_end) load_keys(t_begin + warp, next);
  for (int t = t_begin + warp; t < t_end; t += kW) {
    uint32_t key[NPL];
    if (kPrefetch) {
#pragma unroll
      for (int i = 0; i < NPL; ++i) key[i] = next[i];
      if (t + kW < t_end) load_keys(t + kW, next);
    } else {
      load_keys(t, key);
    }
    // k rounds of a warp argmax: the largest key, then among the lanes that
    // hold it the lowest expert id (ties go to the lower id)
    uint32_t taken = 0;
    float my_z = 0.f;
    int my_e = 0;
    for (int j = 0; j < p.k; ++j) {
      uint32_t bk = 0u, be = 0xFFFFFFFFu;
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (!((taken >> i) & 1u) && key[i] > bk) {
          bk = key[i];
          be = (uint32_t)(i * 32 + lane);
        }
      const uint32_t m = __reduce_max_sync(kFull, bk);
      const uint32_t e = __reduce_min_sync(kFull, bk == m ? be : 0xFFFFFFFFu);
      if ((int)(e & 31u) == lane) taken |= 1u << (e >> 5);
      if (lane == j) {
        my_z = key_value(m);
        my_e = (int)e;
      }
    }
    const float zmax = __shfl_sync(kFull, my_z, 0);
    const float ex = lane < p.k ? expf(my_z - zmax) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (lane < p.k) {
      const size_t a = (size_t)t * p.k + lane;
      p.ids[a] = my_e;
      p.w[a] = ex / sum;
      atomicAdd(&hist[my_e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < p.E; e += kW * 32) p.blk[(size_t)blockIdx.x * p.E + e] = hist[e];
}

// Exclusive scan over the CTA (blockDim.x == 1024). Returns the exclusive
// prefix of `v`; *total (shared memory) receives the sum of all values.
__device__ int block_exclusive_scan_1024(int v, int* total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFull, si, off);
      if (lane >= off) si += o;
    }
    warp_sums[lane] = si - s;  // exclusive prefix of the warp totals
    if (lane == 31) *total = si;
  }
  __syncthreads();
  const int r = incl - v + warp_sums[warp];
  __syncthreads();  // warp_sums is reused by the next call
  return r;
}

// Block map of the routed rows (expert after expert) and the shared rows in
// tiles of bn rows: {group, first row, rows, 0} per tile, num_tiles on the
// device. Every thread of the 1024-thread block calls it; `total` is the
// thread's expert's row count, s_off / s_cnt the experts' offsets and counts.
__device__ void build_block_map(const RouteParams& p, int bn, int total, const int* s_off,
                                const int* s_cnt, int* s_toff, int* s_tiles, int32_t* block_map,
                                int32_t* num_tiles, int max_tiles, int where) {
  const int e = threadIdx.x;
  const int nt = e < p.E ? (total + bn - 1) / bn : 0;
  const int toff = block_exclusive_scan_1024(nt, s_tiles);
  if (e < p.E) s_toff[e] = toff;
  if (e == 0) s_toff[p.E] = *s_tiles;
  __syncthreads();
  const int routed_tiles = *s_tiles;
  const int shared_tiles = p.with_shared ? (p.T + bn - 1) / bn : 0;
  int num = routed_tiles + shared_tiles;
  if (num > max_tiles) {
    if (e == 0) report(p.status, MOE_DEV_BAD_TILE, where, num);
    num = max_tiles;
  }
  if (e == 0) *num_tiles = num;
  const int kT = p.T * p.k;
  for (int i = e; i < num; i += blockDim.x) {
    int4 m;
    if (i < routed_tiles) {
      // last expert g with s_toff[g] <= i (experts without tiles share offsets)
      int lo = 0, hi = p.E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_toff[mid] <= i) lo = mid; else hi = mid - 1;
      }
      const int j = i - s_toff[lo];
      m.x = lo;
      m.y = s_off[lo] + j * bn;
      m.z = min(bn, s_cnt[lo] - j * bn);
    } else {
      const int j = i - routed_tiles;
      m.x = p.E;
      m.y = kT + j * bn;
      m.z = min(bn, p.T - j * bn);
    }
    m.w = 0;
    reinterpret_cast<int4*>(block_map)[i] = m;
  }
  __syncthreads();  // s_toff and s_tiles are reused by a second call
}

// The same rows cut per token window of W tokens (W a multiple of
// kRouteTPB): for each window, the tiles of every expert's rows whose tokens
// lie in the window (experts in order; those rows are contiguous in expert
// order because the scatter is stable), then the window's shared rows. A
// GEMM that walks the map in order then finishes one window's tokens before
// the next: the output rows it adds into stay in L2 while all of their
// contributions arrive. p.blk holds the per-(block, expert) bases here.
__device__ void build_windowed_map(const RouteParams& p, int bn, int W, int nblk, const int* s_off,
                                   const int* s_cnt, int* s_tiles, int32_t* block_map,
                                   int32_t* num_tiles, int max_tiles, int where) {
  const int e = threadIdx.x;
  const int bw = W / kRouteTPB;
  const int nW = (p.T + W - 1) / W;
  const int kT = p.T * p.k;
  int written = 0;  // the same in every thread
  for (int w = 0; w < nW; ++w) {
    int lo = 0, n = 0, nt = 0;
    if (e < p.E) {
      const int b0 = w * bw, b1 = (w + 1) * bw;
      lo = p.blk[(size_t)b0 * p.E + e];
      const int hi = b1 < nblk ? p.blk[(size_t)b1 * p.E + e] : s_cnt[e];
      n = hi - lo;
      nt = (n + bn - 1) / bn;
    }
    const int toff = block_exclusive_scan_1024(nt, s_tiles);
    const int routed = *s_tiles;
    for (int j = 0; j < nt; ++j) {
      const int i = written + toff + j;
      if (i < max_tiles)
        reinterpret_cast<int4*>(block_map)[i] = make_int4(e, s_off[e] + lo + j * bn, min(bn, n - j * bn), 0);
    }
    const int t0 = w * W, t1 = min(p.T, t0 + W);
    const int ns = p.with_shared ? (t1 - t0 + bn - 1) / bn : 0;
    for (int j = e; j < ns; j += blockDim.x) {
      const int i = written + routed + j;
      if (i < max_tiles)
        reinterpret_cast<int4*>(block_map)[i] = make_int4(p.E, kT + t0 + j * bn, min(bn, t1 - t0 - j * bn), 0);
    }
    written += routed + ns;
    __syncthreads();  // *s_tiles is rewritten by the next window's scan
  }
  if (e == 0) {
    if (written > max_tiles) report(p.status, MOE_DEV_BAD_TILE, where, written);
    *num_tiles = min(written, max_tiles);
  }
}

__global__ void __launch_bounds__(1024) route_scan_kernel(RouteParams p, int nblk) {
  __shared__ int s_off[1025];
  __shared__ int s_cnt[1024];
  __shared__ int s_toff[1025];
  __shared__ int s_total;
  __shared__ int s_tiles;
  const int e = threadIdx.x;
  int total = 0;
  if (e < p.E) {
    // 16 blocks' counts are loaded before any base is stored back (a store
    // to the same array would otherwise hold every next load behind it: one
    // L2 round trip per block)
    constexpr int kB = 16;
    for (int b0 = 0; b0 < nblk; b0 += kB) {
      int c[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) c[j] = b0 + j < nblk ? p.blk[(size_t)(b0 + j) * p.E + e] : 0;
#pragma unroll
      for (int j = 0; j < kB; ++j)
        if (b0 + j < nblk) {
          p.blk[(size_t)(b0 + j) * p.E + e] = total;  // exclusive base of block b inside expert e
          total += c[j];
        }
    }
    p.counts[e] = total;
    s_cnt[e] = total;
  }
  const int off = block_exclusive_scan_1024(e < p.E ? total : 0, &s_total);
  if (e < p.E) {
    p.offsets[e] = off;
    s_off[e] = off;
  }
  if (e == 0) {
    p.offsets[p.E] = s_total;
    s_off[p.E] = s_total;
  }
  __syncthreads();
  build_block_map(p, p.block_n, total, s_off, s_cnt, s_toff, &s_tiles, p.block_map, p.num_tiles,
                  p.max_tiles, 11);
  if (p.block_map2 && p.window2 > 0)  // a second GEMM's tiles, ordered by token window
    build_windowed_map(p, p.block_n2, p.window2, nblk, s_off, s_cnt, &s_tiles, p.block_map2,
                       p.num_tiles2, p.max_tiles2, 13);
  else if (p.block_map2)  // the same rows in tiles of block_n2 (a second GEMM's tile height)
    build_block_map(p, p.block_n2, total, s_off, s_cnt, s_toff, &s_tiles, p.block_map2,
                    p.num_tiles2, p.max_tiles2, 13);
}

__global__ void __launch_bounds__(kThreads) route_scatter_kernel(RouteParams p) {
  extern __shared__ int wbase[];  // [kWarps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t a0 = (int64_t)blockIdx.x * kRouteTPB * p.k;
  const int64_t a1 = min((int64_t)p.T, (int64_t)(blockIdx.x + 1) * kRouteTPB) * p.k;
  const int64_t span = (a1 - a0 + kWarps - 1) / kWarps;
  const int64_t w0 = a0 + warp * span;
  const int64_t w1 = min(a1, w0 + span);

  for (int i = threadIdx.x; i < kWarps * p.E; i += kThreads) wbase[i] = 0;
  __syncthreads();
  int* mine = wbase + warp * p.E;
  for (int64_t a = w0 + lane; a < w1; a += 32) {
    const int e = p.ids[a];
    if (e >= 0 && e < p.E) atomicAdd(&mine[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < p.E; e += kThreads) {
    int base = p.offsets[e] + p.blk[(size_t)blockIdx.x * p.E + e];
    for (int w = 0; w < kWarps; ++w) {
      const int c = wbase[w * p.E + e];
      wbase[w * p.E + e] = base;
      base += c;
    }
  }
  __syncthreads();
  for (int64_t c0 = w0; c0 < w1; c0 += 32) {
    const int64_t a = c0 + lane;
    const bool valid = a < w1;
    int e = valid ? p.ids[a] : -1 - lane;
    if (valid && (e < 0 || e >= p.E)) {
      report(p.status, MOE_DEV_BAD_EXPERT, 12, (int)a);
      e = -100 - lane;
    }
    const uint32_t m = __match_any_sync(kFull, e);
    int pos = 0;
    if (e >= 0) {
      pos = mine[e] + __popc(m & lanemask_lt());
      p.perm[pos] = (int32_t)a;
      p.inv_perm[a] = pos;
      p.row_token[pos] = (int32_t)((uint32_t)a / (uint32_t)p.k);  // a < T * k < 2^31
      if (p.row_weight) p.row_weight[pos] = p.w[a];
    }
    __syncwarp();
    if (e >= 0 && lane == 31 - __clz(m)) mine[e] += __popc(m);
    __syncwarp();
  }
  if (p.with_shared) {
    const int t_begin = blockIdx.x * kRouteTPB;
    const int t_end = min(p.T, t_begin + kRouteTPB);
    for (int t = t_begin + threadIdx.x; t < t_end; t += kThreads)
      p.row_token[(size_t)p.T * p.k + t] = t;
  }
}

}  // namespace

cudaError_t route_launch(const RouteParams& p, cudaStream_t s) {
  const int nblk = route_nblk(p.T);
  const size_t hist_bytes = (size_t)p.E * sizeof(int);
  const int npl = (p.E + 31) / 32;
  if (npl <= 1) route_topk_kernel<1><<<nblk, topk_threads<1>(), hist_bytes, s>>>(p);
  else if (npl <= 2) route_topk_kernel<2><<<nblk, topk_threads<2>(), hist_bytes, s>>>(p);
  else if (npl <= 4) route_topk_kernel<4><<<nblk, topk_threads<4>(), hist_bytes, s>>>(p);
  else if (npl <= 8) route_topk_kernel<8><<<nblk, topk_threads<8>(), hist_bytes, s>>>(p);
  else if (npl <= 16) route_topk_kernel<16><<<nblk, topk_threads<16>(), hist_bytes, s>>>(p);
  else route_topk_kernel<32><<<nblk, topk_threads<32>(), hist_bytes, s>>>(p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  route_scan_kernel<<<1, 1024, 0, s>>>(p, nblk);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t wb_bytes = (size_t)kWarps * p.E * sizeof(int);
  if (wb_bytes > 48 * 1024) {
    err = cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)wb_bytes);
    if (err != cudaSuccess) return err;
  }
  route_scatter_kernel<<<nblk, kThreads, wb_bytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
