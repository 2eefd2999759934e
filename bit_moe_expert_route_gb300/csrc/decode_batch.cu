// Small-batch decode: 1 to 8 tokens (e.g. a speculative-decoding verification
// batch) through the MoE layer with matrix-vector work that reads the router,
// the shared expert and each selected expert's packed 4-bit rows once per
// call (an expert two tokens both select, and the shared expert, are read
// again for the second token, mostly from L2). ("Perplexity's Lily Beats MLX-LM by 1.35x
// Running Qwen3.6 on Apple Silicon", section "Why prefill and decode get
// different treatment": decode is bound by reading the weights, and uses
// matrix-vector work on the vector ALUs; the same page names small
// verification batches whose rows hit different experts as the case its
// tensor-core kernels did not help.)
//
// Three launches chained by programmatic dependent launch; each waits
// (griddepcontrol.wait) before it reads what the previous one wrote:
//   1. batch_router_kernel   one block per 8 experts (one more for the shared
//        gate vector w_sg) and K slice (kBatchKS of them): its router columns
//        over its rows, applied to every token; fp32 partial logits, summed
//        in a fixed order by the next kernel.
//   2. batch_gateup_kernel   every block ranks each token's logits (one warp
//        per token: value descending, ties to the lower id; softmax over the
//        selected), block 0 stores ids and weights; then the row pairs of
//        gate/up, each (row, token) a task: h = silu(x . g) * (x . u) in fp32,
//        each warp streaming its tasks' rows through its own shared-memory
//        ring (cp.async, four tasks ahead).
// The gate/up and down kernels also have an instantiation for the standard
// layer shape (d_model 2048, d_ff 512, top-8) with those sizes as constants.
//   3. batch_down_kernel     output columns split over the blocks; for each
//        column and token, every slot's down row weighted by its routing
//        weight (the shared expert's by sigmoid of the gate logit), summed in
//        a fixed order and rounded once to bf16.
// Dot products as in the batch-1 decode (gemv_dot.cuh): codes become exact
// 16-bit floats f = 1 + q/16 and meet the bf16 activations in mixed-precision
// FMAs; for a group with scale s and bias b,
//   sum_k (s*q_k + b) v_k = 16 s * sum_k f_k v_k + (b - 16 s) * sum_k v_k,
// with the activation group sums taken once per token.
#include <algorithm>

#include "common.cuh"
#include "gemv_dot.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr uint32_t kFullMask = 0xFFFFFFFFu;
constexpr int kBThreads = 256;
constexpr int kBWarps = kBThreads / 32;

MOE_DEVINL void pdl_wait_b() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEVINL void pdl_launch_b() { asm volatile("griddepcontrol.launch_dependents;" :::); }

MOE_DEVINL float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Activations in shared memory: 64-value groups of eight 16-byte pieces,
// each piece the four pairs (v_i, v_{i+4}) of its 8 bf16 values (pair_up);
// piece p of group g is stored at position p ^ (g % 8), so that lanes
// reading the same piece of consecutive groups hit different banks.

// sum over the 64 codes of a group (8 packed words, low nibble first) of
// f_k * v_k; v is the group's 8 pieces (layout as above, group g).
MOE_DEVINL float group_fdot(const uint32_t (&w)[8], const uint16_t* v, int g) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int pc = 0; pc < 8; ++pc)  // piece pc = word pc = codes 8pc .. 8pc+7
    word_fdot<true>(w[pc], reinterpret_cast<const uint4*>(v)[(pc ^ g) & 7], a0, a1);
  return a0 + a1;
}

// Sum of the 64 bf16 values of one group (any order of the values inside
// it): the 32 words start at a lane-dependent word, so that the lanes of a
// warp, each summing its own group, read 32 different banks.
MOE_DEVINL float group_sum64(const uint16_t* v) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(v);
  const int r = threadIdx.x & 31;
  float a = 0.f, b = 0.f;
#pragma unroll 8
  for (int j = 0; j < 32; ++j) {
    const uint32_t u = w[(j + r) & 31];
    a += __uint_as_float(u << 16);
    b += __uint_as_float(u & 0xFFFF0000u);
  }
  return a + b;
}

// ---------------------------------------------------------------- 1. router
template <int TB>  // token capacity: T <= TB
__global__ void __launch_bounds__(kBThreads) batch_router_kernel(const __grid_constant__ BatchParams p) {
  extern __shared__ __align__(16) uint8_t bsm[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(bsm);                       // [T][d]
  float* red = reinterpret_cast<float*>(bsm + (size_t)p.T * p.d * 2);    // [warps][T * 8]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, d = p.d, E = p.E;
  const int ncol = E / 8 + (p.shared ? 1 : 0);  // column blocks: 8 experts each, then w_sg
  const int cb = blockIdx.x % ncol, ks = blockIdx.x / ncol;
  const bool gate_block = cb == E / 8;
  const int e0 = cb * 8;
  const int rs = (d + kBatchKS - 1) / kBatchKS, r_lo = ks * rs, r_hi = min(d, r_lo + rs);
  // the weight columns do not depend on the previous kernel: pull them toward L2
  for (int r = r_lo + tid; r < r_hi; r += kBThreads) {
    const float* w = gate_block ? p.w.shared_gate + r : p.w.router + (size_t)r * E + e0;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(w));
  }
  pdl_wait_b();
  pdl_launch_b();
  if (blockIdx.x == 0 && tid < 4) p.status[tid] = 0;
  for (int i = tid; i < T * d / 8; i += kBThreads)
    reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(p.x)[i];
  __syncthreads();
  float acc[TB][8];
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[t][c] = 0.f;
  constexpr int kRB = 4;  // rows per thread per batch: all loads issued before the arithmetic
  for (int r0 = r_lo + tid; r0 < r_hi; r0 += kRB * kBThreads) {
    float wv[kRB][8];
#pragma unroll
    for (int b = 0; b < kRB; ++b) {
      const int r = r0 + b * kBThreads;
#pragma unroll
      for (int c = 0; c < 8; ++c) wv[b][c] = 0.f;
      if (r < r_hi) {
        if (gate_block) {
          wv[b][0] = p.w.shared_gate[r];
        } else {
          const float4* w = reinterpret_cast<const float4*>(p.w.router + (size_t)r * E + e0);
          const float4 a = w[0], c4 = w[1];
          wv[b][0] = a.x; wv[b][1] = a.y; wv[b][2] = a.z; wv[b][3] = a.w;
          wv[b][4] = c4.x; wv[b][5] = c4.y; wv[b][6] = c4.z; wv[b][7] = c4.w;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kRB; ++b) {
      const int r = r0 + b * kBThreads;
      if (r >= r_hi) break;
#pragma unroll
      for (int t = 0; t < TB; ++t)
        if (t < T) {
          const float xv = bf16f(xs[(size_t)t * d + r]);
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[t][c] = fmaf(xv, wv[b][c], acc[t][c]);
        }
    }
  }
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float v = acc[t][c];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
      if (lane == 0 && t < T) red[warp * (kBatchMaxT * 8) + t * 8 + c] = v;
    }
  __syncthreads();
  if (tid < T * 8) {
    float v = 0.f;
    for (int w = 0; w < kBWarps; ++w) v += red[w * (kBatchMaxT * 8) + tid];  // fixed order
    const int t = tid / 8, c = tid % 8;
    float* part = p.part + ((size_t)ks * T + t) * (E + 1);  // the K slice's partial logits
    if (gate_block) {
      if (c == 0) part[E] = v;
    } else {
      part[e0 + c] = v;
    }
  }
}

// ---------------------------------------------------------------- 2. top-k, gate/up
constexpr int kRD = 4;  // gate/up tasks in flight per warp (the ring path)

// The gate/up kernel's task ring: after x, its group sums and the ids, 16-byte
// aligned, over the top-k keys (dead once the tasks start).
MOE_DEVINL uint8_t* gateup_ring(uint8_t* base, int T, int d, int k) {
  const size_t off = (size_t)T * d * 2 + (size_t)T * (d / 64) * 4 + (size_t)T * k * 4;
  return base + ((off + 15) & ~(size_t)15);
}

// SD: the standard layer shape (d_model 2048, d_ff 512, top-8) as compile-time
// constants, so that the task and item indices split with shifts and
// multiplications instead of divisions by run-time values; otherwise 0.
template <int TB, int SD>
__global__ void __launch_bounds__(kBThreads, 2) batch_gateup_kernel(const __grid_constant__ BatchParams p) {
  extern __shared__ __align__(16) uint8_t bsm[];
  const int T = p.T, d = SD ? 2048 : p.d, E = p.E, k = SD ? 8 : p.k, f = SD ? 512 : p.f, S = k + 1;
  const int ng = d / 64;  // groups per row
  uint16_t* xs = reinterpret_cast<uint16_t*>(bsm);                                 // [T][d]
  float* xsum = reinterpret_cast<float*>(bsm + (size_t)T * d * 2);                 // [T][ng]
  int* s_ids = reinterpret_cast<int*>(xsum + (size_t)T * ng);                      // [T][k]
  uint32_t* keys = reinterpret_cast<uint32_t*>(s_ids + T * k);                     // [T][E] order keys
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int kKB = 8;  // experts per lane per batch of the top-k, all partials loaded first
  // the router bias of this lane's first batch of experts (weights, not
  // written by the previous kernel): loaded before the dependency wait
  float bias0[kKB];
#pragma unroll
  for (int m = 0; m < kKB; ++m) {
    const int e = lane + m * 32;
    bias0[m] = p.w.router_bias && warp < T && e < E ? p.w.router_bias[e] : 0.f;
  }
  pdl_wait_b();
  pdl_launch_b();
  for (int i = tid; i < T * d / 8; i += kBThreads) {  // piece i: row i / (d/8), group (i % (d/8)) / 8
    const int g = (i % (d / 8)) >> 3;
    reinterpret_cast<uint4*>(xs)[(i & ~7) | (((i & 7) ^ g) & 7)] =
        pair_up(reinterpret_cast<const uint4*>(p.x)[i]);
  }
  // top k of each token (warp t), its softmax weights and the shared gate
  if (warp < T) {
    const int t = warp;
    uint32_t* kr = keys + (size_t)t * E;  // order keys of this token's experts
    for (int e0 = lane; e0 < E; e0 += kKB * 32) {
      float z[kKB][kBatchKS];
#pragma unroll
      for (int m = 0; m < kKB; ++m)
#pragma unroll
        for (int q = 0; q < kBatchKS; ++q) {
          const int e = e0 + m * 32;
          z[m][q] = e < E ? p.part[((size_t)q * T + t) * (E + 1) + e] : 0.f;
        }
#pragma unroll
      for (int m = 0; m < kKB; ++m) {
        const int e = e0 + m * 32;
        if (e >= E) break;
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < kBatchKS; ++q) v += z[m][q];  // fixed order
        if (blockIdx.x == 0) p.logits[(size_t)t * E + e] = v;
        if (p.w.router_bias) v = v + (e0 == lane ? bias0[m] : p.w.router_bias[e]);
        kr[e] = order_key(v);
      }
    }
    __syncwarp();
    uint32_t taken = 0;
    float my_z = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
      uint32_t bk = 0u, be = 0xFFFFFFFFu;
      for (int i = 0; i * 32 < E; ++i) {
        const uint32_t kv = i * 32 + lane < E ? kr[i * 32 + lane] : 0u;
        if (!((taken >> i) & 1u) && kv > bk) {
          bk = kv;
          be = (uint32_t)(i * 32 + lane);
        }
      }
      const uint32_t m = __reduce_max_sync(kFullMask, bk);
      const uint32_t e = __reduce_min_sync(kFullMask, bk == m ? be : 0xFFFFFFFFu);
      if ((int)(e & 31u) == lane) taken |= 1u << (e >> 5);
      if (lane == j) {
        my_z = key_value(m);
        my_e = (int)e;
      }
    }
    const float zmax = __shfl_sync(kFullMask, my_z, 0);
    const float ex = lane < k ? expf(my_z - zmax) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFullMask, sum, off);
    if (lane < k) s_ids[t * k + lane] = my_e;
    if (blockIdx.x == 0) {
      if (lane < k) {
        p.ids[t * k + lane] = my_e;
        p.wts[t * S + lane] = ex / sum;
      }
      if (lane == 0) {
        float gl = 0.f;
        for (int q = 0; q < kBatchKS; ++q) gl += p.part[((size_t)q * T + t) * (E + 1) + E];
        if (p.shared) p.gate_logit[t] = gl;
        p.wts[t * S + k] = p.shared ? 1.f / (1.f + expf(-gl)) : 0.f;
      }
    }
  }
  __syncthreads();
  const int n_routed = T * k * f, n_tasks = n_routed + (p.shared ? T * f : 0);
  const int gw = blockIdx.x * kBWarps + warp, nw = gridDim.x * kBWarps;
  const int per = (n_tasks + nw - 1) / nw;
  const int i_lo = min(n_tasks, gw * per), i_hi = min(n_tasks, i_lo + per);
  // group sums of x per token
  for (int i = tid; i < T * ng; i += kBThreads) xsum[i] = group_sum64(xs + (size_t)(i / ng) * d + (i % ng) * 64);
  __syncthreads();
  // tasks: (slot i of T*k, row r): token i / k times its expert's row r;
  // then (shared row r, token t) at T*k*f + t*f + r. Each warp takes a
  // contiguous run of tasks. Rows of an expert that two tokens select are
  // read once per token (the second read mostly from L2).
  auto task_of = [&](int it, int& tk_, int& row_, bool& sh_) {
    sh_ = it >= n_routed;
    tk_ = sh_ ? (it - n_routed) / f : (it / f) / k;
    row_ = sh_ ? (it - n_routed) % f : s_ids[it / f] * f + it % f;
  };
  if (d % 512 == 0) {
    // Each warp streams its tasks' gate and up rows (codes, then scale and
    // bias rows) into its own shared-memory ring, kRD tasks ahead, with
    // 16-byte cp.async, so the copies of the next tasks are in flight while
    // two are computed; a lane reads its group (64 codes of each matrix)
    // from the ring.
    const int rb = d + d / 8;  // bytes per task: two code rows, four scale/bias rows
    uint8_t* ring = gateup_ring(bsm, T, d, k) + (size_t)warp * kRD * rb;
    const int nq = d / 32, ns = d / 512;  // 16-byte chunks of a code row / of a scale row
    auto issue = [&](int it, int slot) {
      if (it < i_hi) {
        int tk_, row_;
        bool sh_;
        task_of(it, tk_, row_, sh_);
        const moe_w4_t& G = sh_ ? p.w.sh_gate : p.w.gate;
        const moe_w4_t& U = sh_ ? p.w.sh_up : p.w.up;
        uint8_t* dst = ring + (size_t)slot * rb;
        const uint8_t* gq = reinterpret_cast<const uint8_t*>(G.q) + (size_t)row_ * (d / 2);
        const uint8_t* uq = reinterpret_cast<const uint8_t*>(U.q) + (size_t)row_ * (d / 2);
        for (int c = lane; c < nq; c += 32) {
          cp_async_16(smem_u32(dst + c * 16), gq + c * 16, 16);
          cp_async_16(smem_u32(dst + d / 2 + c * 16), uq + c * 16, 16);
        }
        for (int c = lane; c < 4 * ns; c += 32) {
          const int a = c / ns, o = c - a * ns;  // gate scale, gate bias, up scale, up bias
          const uint16_t* src = a == 0 ? G.scale : a == 1 ? G.bias : a == 2 ? U.scale : U.bias;
          cp_async_16(smem_u32(dst + d + a * (d / 32) + o * 16),
                      reinterpret_cast<const uint8_t*>(src + (size_t)row_ * ng) + o * 16, 16);
        }
      }
      cp_async_commit();
    };
#pragma unroll 1
    for (int r = 0; r < kRD; ++r) issue(i_lo + r, r);
#pragma unroll 1
    for (int it = i_lo; it < i_hi; it += 2) {  // two tasks per step: two independent chains
      const bool two = it + 1 < i_hi;
      cp_async_wait<kRD - 2>();
      __syncwarp();  // every lane's copies of these tasks have landed
      int tk_[2], row_[2];
      bool sh_[2];
      float ag[2] = {0.f, 0.f}, au[2] = {0.f, 0.f};
      const uint8_t* src[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        task_of(t == 0 || two ? it + t : it, tk_[t], row_[t], sh_[t]);
        src[t] = ring + (size_t)((it - i_lo + t) % kRD) * rb;
      }
      for (int g = lane; g < ng; g += 32) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (t == 1 && !two) break;
          const uint8_t* sr = src[t];
          const uint16_t* sb = reinterpret_cast<const uint16_t*>(sr + d);
          const uint4 g0 = reinterpret_cast<const uint4*>(sr + g * 32)[0];
          const uint4 g1 = reinterpret_cast<const uint4*>(sr + g * 32)[1];
          const uint4 u0 = reinterpret_cast<const uint4*>(sr + d / 2 + g * 32)[0];
          const uint4 u1 = reinterpret_cast<const uint4*>(sr + d / 2 + g * 32)[1];
          const uint32_t wg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          const uint32_t wu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          const float gs = bf16f(sb[g]), gb = bf16f(sb[ng + g]), us = bf16f(sb[2 * ng + g]),
                      ub = bf16f(sb[3 * ng + g]);
          const uint16_t* v = xs + (size_t)tk_[t] * d + g * 64;
          const float xsm = xsum[tk_[t] * ng + g];
          ag[t] = fmaf(16.f * gs, group_fdot(wg, v, g), fmaf(gb - 16.f * gs, xsm, ag[t]));
          au[t] = fmaf(16.f * us, group_fdot(wu, v, g), fmaf(ub - 16.f * us, xsm, au[t]));
        }
      }
      __syncwarp();  // every lane is done with the two slots
#pragma unroll
      for (int t = 0; t < 2; ++t) issue(it + kRD + t, (it - i_lo + t) % kRD);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          ag[t] += __shfl_xor_sync(kFullMask, ag[t], off);
          au[t] += __shfl_xor_sync(kFullMask, au[t], off);
        }
      }
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (lane == 0 && (t == 0 || two)) {
          const float hv = ag[t] / (1.f + expf(-ag[t])) * au[t];
          const int slot_h = sh_[t] ? k : ((it + t) / f) % k;  // routed: slot of the token's selection
          p.h[((size_t)tk_[t] * S + slot_h) * f + row_[t] % f] = hv;
        }
    }
    cp_async_wait<0>();
    return;
  }
  // other row lengths: batches of kIB tasks, every load of a batch issued
  // before its arithmetic (a lane holds 64 codes of each matrix per pass)
  constexpr int kIB = 3;
  for (int i0 = i_lo; i0 < i_hi; i0 += kIB) {
    int tok[kIB], srow[kIB];
    bool live[kIB], shr[kIB];
#pragma unroll
    for (int b = 0; b < kIB; ++b) {
      const int it = i0 + b;
      live[b] = it < i_hi;
      shr[b] = it >= n_routed;
      tok[b] = 0;
      srow[b] = 0;
      if (live[b]) {
        if (!shr[b]) {
          tok[b] = (it / f) / k;
          srow[b] = s_ids[it / f] * f + it % f;
        } else {
          tok[b] = (it - n_routed) / f;
          srow[b] = (it - n_routed) % f;
        }
      }
    }
    float ag[kIB], au[kIB];
#pragma unroll
    for (int b = 0; b < kIB; ++b) ag[b] = au[b] = 0.f;
    for (int g = lane; g < ng; g += 32) {
      uint4 qg[kIB][2], qu[kIB][2];
      float gs[kIB], gb[kIB], us[kIB], ub[kIB];
#pragma unroll
      for (int b = 0; b < kIB; ++b) {
        if (!live[b]) continue;
        const moe_w4_t& G = shr[b] ? p.w.sh_gate : p.w.gate;
        const moe_w4_t& U = shr[b] ? p.w.sh_up : p.w.up;
        const uint4* gq = reinterpret_cast<const uint4*>(G.q + (size_t)srow[b] * (d / 8) + g * 8);
        const uint4* uq = reinterpret_cast<const uint4*>(U.q + (size_t)srow[b] * (d / 8) + g * 8);
        qg[b][0] = gq[0]; qg[b][1] = gq[1]; qu[b][0] = uq[0]; qu[b][1] = uq[1];
        const size_t si = (size_t)srow[b] * ng + g;
        gs[b] = bf16f(G.scale[si]); gb[b] = bf16f(G.bias[si]);
        us[b] = bf16f(U.scale[si]); ub[b] = bf16f(U.bias[si]);
      }
#pragma unroll
      for (int b = 0; b < kIB; ++b) {
        if (!live[b]) continue;
        const uint32_t wg[8] = {qg[b][0].x, qg[b][0].y, qg[b][0].z, qg[b][0].w,
                                qg[b][1].x, qg[b][1].y, qg[b][1].z, qg[b][1].w};
        const uint32_t wu[8] = {qu[b][0].x, qu[b][0].y, qu[b][0].z, qu[b][0].w,
                                qu[b][1].x, qu[b][1].y, qu[b][1].z, qu[b][1].w};
        const uint16_t* v = xs + (size_t)tok[b] * d + g * 64;
        const float xsm = xsum[tok[b] * ng + g];
        ag[b] = fmaf(16.f * gs[b], group_fdot(wg, v, g), fmaf(gb[b] - 16.f * gs[b], xsm, ag[b]));
        au[b] = fmaf(16.f * us[b], group_fdot(wu, v, g), fmaf(ub[b] - 16.f * us[b], xsm, au[b]));
      }
    }
#pragma unroll
    for (int b = 0; b < kIB; ++b) {
      if (!live[b]) continue;
      float g = ag[b], u = au[b];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        g += __shfl_xor_sync(kFullMask, g, off);
        u += __shfl_xor_sync(kFullMask, u, off);
      }
      if (lane == 0) {
        const int it = i0 + b;
        const float hv = g / (1.f + expf(-g)) * u;
        const int slot = shr[b] ? k : (it / f) % k;  // routed: slot of the token's selection
        p.h[((size_t)tok[b] * S + slot) * f + srow[b] % f] = hv;
      }
    }
  }
}

// ---------------------------------------------------------------- 3. down + combine
template <int TB, int SD>  // SD: as for the gate/up kernel
__global__ void __launch_bounds__(kBThreads, 2) batch_down_kernel(const __grid_constant__ BatchParams p) {
  extern __shared__ __align__(16) uint8_t bsm[];
  const int T = p.T, d = SD ? 2048 : p.d, k = SD ? 8 : p.k, f = SD ? 512 : p.f, S = k + 1;
  const int nslots = p.shared ? S : k, ngf = f / 64;
  uint16_t* hs = reinterpret_cast<uint16_t*>(bsm);                                   // bf16 [T][S][f]
  float* hsum = reinterpret_cast<float*>(bsm + (size_t)T * S * f * 2);              // [T][S][ngf]
  float* s_w = hsum + (size_t)T * S * ngf;                                          // [T][S]
  int* s_ids = reinterpret_cast<int*>(s_w + T * S);                                 // [T][k]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gw = blockIdx.x * kBWarps + warp, nw = gridDim.x * kBWarps;
  pdl_wait_b();
  pdl_launch_b();
  // h as bf16 (the operand precision of the down projection; swizzled like
  // x above), group sums, routing weights and ids
  {
    constexpr int kHB = 6;  // pieces (8 values, two float4) per thread per batch, loads first
    const int n8 = T * S * f / 8;
    for (int i0 = tid; i0 < n8; i0 += kHB * kBThreads) {
      float4 v[kHB][2];
#pragma unroll
      for (int m = 0; m < kHB; ++m) {
        const int i = i0 + m * kBThreads;
        v[m][0] = v[m][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < n8 && ((i * 8) / f) % S < nslots) {
          v[m][0] = reinterpret_cast<const float4*>(p.h)[2 * i];
          v[m][1] = reinterpret_cast<const float4*>(p.h)[2 * i + 1];
        }
      }
#pragma unroll
      for (int m = 0; m < kHB; ++m) {
        const int i = i0 + m * kBThreads;
        if (i >= n8) break;
        const int e8 = i * 8, ts = e8 / f, c = e8 % f, g = c >> 6, pc = (c & 63) >> 3;
        const float f8[8] = {v[m][0].x, v[m][0].y, v[m][0].z, v[m][0].w,
                             v[m][1].x, v[m][1].y, v[m][1].z, v[m][1].w};
        uint32_t raw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(f8[2 * q], f8[2 * q + 1]);
          raw[q] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        reinterpret_cast<uint4*>(hs + (size_t)ts * f + g * 64)[(pc ^ g) & 7] =
            pair_up(make_uint4(raw[0], raw[1], raw[2], raw[3]));
      }
    }
  }
  for (int i = tid; i < T * S; i += kBThreads) s_w[i] = p.wts[i];
  for (int i = tid; i < T * k; i += kBThreads) s_ids[i] = p.ids[i];
  __syncthreads();
  for (int i = tid; i < T * S * ngf; i += kBThreads) hsum[i] = group_sum64(hs + (size_t)i * 64);
  __syncthreads();
  // one warp per output column; its lanes share the (token, slot, group)
  // items of the routed rows, then the groups of the shared expert's row
  // (which serves every token)
  const int n_routed = T * k * ngf;
  constexpr int kDB = 8;  // routed items per lane per batch, loads issued first
  for (int j = gw; j < d; j += nw) {
    float acc[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[t] = 0.f;
    for (int u0 = lane; u0 < n_routed; u0 += kDB * 32) {
      uint4 qa[kDB], qb[kDB];
      float sc[kDB], bi[kDB];
      int tk[kDB];  // the item's token, found once
#pragma unroll
      for (int m = 0; m < kDB; ++m) {
        const int u = u0 + m * 32;
        if (u >= n_routed) break;
        const int ts0 = u / ngf, g = u - ts0 * ngf, t = ts0 / k, s = ts0 - t * k;
        tk[m] = t;
        const size_t row = (size_t)s_ids[ts0] * d + j;
        const uint4* q = reinterpret_cast<const uint4*>(p.w.down.q + row * (f / 8) + g * 8);
        qa[m] = q[0];
        qb[m] = q[1];
        const size_t si = row * ngf + g;
        sc[m] = bf16f(p.w.down.scale[si]);
        bi[m] = bf16f(p.w.down.bias[si]);
      }
#pragma unroll
      for (int m = 0; m < kDB; ++m) {
        const int u = u0 + m * 32;
        if (u >= n_routed) break;
        const int ts0 = u / ngf, g = u - ts0 * ngf, t = tk[m], ts = ts0 + t;  // t * k + s + t = t * S + s
        const uint32_t w[8] = {qa[m].x, qa[m].y, qa[m].z, qa[m].w, qb[m].x, qb[m].y, qb[m].z, qb[m].w};
        const float dot = fmaf(16.f * sc[m], group_fdot(w, hs + ((size_t)ts * f + g * 64), g),
                               (bi[m] - 16.f * sc[m]) * hsum[ts * ngf + g]);
        const float v = s_w[ts] * dot;
#pragma unroll
        for (int tt = 0; tt < TB; ++tt)
          if (tt == t) acc[tt] += v;
      }
    }
    if (p.shared)
      for (int g = lane; g < ngf; g += 32) {
        const uint4* q = reinterpret_cast<const uint4*>(p.w.sh_down.q + (size_t)j * (f / 8) + g * 8);
        const uint4 a = q[0], b = q[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const size_t si = (size_t)j * ngf + g;
        const float sc1 = bf16f(p.w.sh_down.scale[si]), bi1 = bf16f(p.w.sh_down.bias[si]);
#pragma unroll
        for (int t = 0; t < TB; ++t)
          if (t < T) {
            const int ts = t * S + k;
            const float dot = fmaf(16.f * sc1, group_fdot(w, hs + ((size_t)ts * f + g * 64), g),
                                   (bi1 - 16.f * sc1) * hsum[ts * ngf + g]);
            acc[t] = fmaf(s_w[ts], dot, acc[t]);
          }
      }
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      if (t >= T) break;
      float v = acc[t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
      if (lane == 0) p.out[(size_t)t * d + j] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
  }
}

int sm_count_b() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

template <typename K>
cudaError_t launch_pdl(K kern, int grid, size_t smem, cudaStream_t s, const BatchParams& p) {
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kBThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

size_t batch_smem_router(int T, int d) { return (size_t)T * d * 2 + (size_t)kBWarps * kBatchMaxT * 8 * 4; }
size_t batch_smem_gateup(int T, int d, int E, int k) {
  const size_t head = (size_t)T * d * 2 + (size_t)T * (d / 64) * 4 + (size_t)T * k * 4;
  const size_t ring = d % 512 == 0 ? 15 + (size_t)kBWarps * kRD * (d + d / 8) : 0;
  return head + std::max((size_t)T * E * 4, ring);
}
size_t batch_smem_down(int T, int k, int f) {
  const int S = k + 1;
  return (size_t)T * S * f * 2 + (size_t)T * S * (f / 64) * 4 + (size_t)T * S * 4 + (size_t)T * k * 4;
}

bool batch_shape_supported(int T, int d, int E, int k, int f) {
  constexpr size_t kLimit = 200 * 1024;
  return T >= 1 && T <= kBatchMaxT && k <= 32 && E <= 1024 && d % 64 == 0 && f % 64 == 0 &&
         batch_smem_router(T, d) <= kLimit && batch_smem_gateup(T, d, E, k) <= kLimit &&
         batch_smem_down(T, k, f) <= kLimit;
}

template <int TB>
cudaError_t launch_tb(const BatchParams& p, cudaStream_t s) {
  cudaError_t err = launch_pdl(batch_router_kernel<TB>, (p.E / 8 + (p.shared ? 1 : 0)) * kBatchKS,
                               batch_smem_router(p.T, p.d), s, p);
  if (err != cudaSuccess) return err;
  const int G = 2 * sm_count_b();  // two blocks per SM
  const bool sd = p.d == 2048 && p.f == 512 && p.k == 8;  // the standard layer shape
  if ((err = sd ? launch_pdl(batch_gateup_kernel<TB, 1>, G, batch_smem_gateup(p.T, p.d, p.E, p.k), s, p)
                : launch_pdl(batch_gateup_kernel<TB, 0>, G, batch_smem_gateup(p.T, p.d, p.E, p.k), s, p)) !=
      cudaSuccess)
    return err;
  return sd ? launch_pdl(batch_down_kernel<TB, 1>, G, batch_smem_down(p.T, p.k, p.f), s, p)
            : launch_pdl(batch_down_kernel<TB, 0>, G, batch_smem_down(p.T, p.k, p.f), s, p);
}

cudaError_t decode_batch_launch(const BatchParams& p, cudaStream_t s) {
  if (p.T <= 2) return launch_tb<2>(p, s);
  if (p.T <= 4) return launch_tb<4>(p, s);
  return launch_tb<8>(p, s);
}

}  // namespace moe
