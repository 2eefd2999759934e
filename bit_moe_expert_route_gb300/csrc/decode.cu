// Batch-1 decode: one token through the MoE layer with matrix-vector kernels
// that stream only the router, the shared expert and the top-k selected
// experts' packed 4-bit weights. ("Perplexity's Lily Beats MLX-LM by 1.35x
// Running Qwen3.6 on Apple Silicon", section "Why prefill and decode get
// different treatment": batch-1 decode is bound by reading the weights, and
// uses matrix-vector kernels on the vector ALUs.)
//
// Three launches chained with programmatic dependent launch (PDL). Each
// kernel first issues the loads that do not depend on the previous kernel
// (weights, and x), then waits (griddepcontrol.wait), so its weight traffic
// overlaps the previous kernel's tail:
//   1. decode_router_shared_kernel  router logits (8 complete logits per
//        block), the shared gate logit, and the shared expert's gate/up rows
//        (h of the shared slot).
//   2. decode_gateup_kernel   every block selects the top k from the logits
//        (warp argmax, ties to the lower id; block 0 also stores ids, weights
//        and the gate), then the routed experts' gate/up rows, h = silu(g)*u.
//   3. decode_down_kernel     selects the top k the same way before its wait
//        (kernel 1 has completed by then) and issues its down-row loads, then
//        waits for h; one warp per output column sums every slot's down row,
//        weighted, in slot order, rounded once to bf16.
// The selection is recomputed per block instead of being published by a
// last-block-done step: it costs one L2 read of E logits per block and
// removes a fence, an atomic and a dependent round trip from the path.
//
// Dot products per 16-byte chunk (32 codes, half a group): a code q becomes the
// float f = 1 + q/16 exactly (bit pattern 0x3F800000 | q << 19), so
// sum_k (s*q_k + b) v_k = 16 s * sum_k f_k v_k + (b - 16 s) * sum_k v_k,
// with the activation chunk sums taken once per chunk. f stays in [1, 2), so
// the fp32 sums cancel no more than a factor of a few.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
// XC = chunks of a d_model-long row per lane = d_model / 1024 (d_model <= 4096).

MOE_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEVINL void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// f = 1 + q/16 for code n (0..7) of a packed word.
MOE_DEVINL float code_f(uint32_t w, int n) {
  const int sh = 19 - 4 * n;
  const uint32_t v = sh >= 0 ? (w << sh) : (w >> (-sh));
  return __uint_as_float((v & 0x00780000u) | 0x3F800000u);
}

// sum over the 32 codes of a chunk of f_k * v_k, v in registers.
MOE_DEVINL float chunk_fdot(const uint4 q, const float (&v)[32]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int n = 0; n < 8; n += 2) {
      a0 = fmaf(code_f(w[i], n), v[8 * i + n], a0);
      a1 = fmaf(code_f(w[i], n + 1), v[8 * i + n + 1], a1);
    }
  }
  return a0 + a1;
}

// Same with v in swizzled shared memory (float4 j of chunk c at c*8 + (j ^ (c & 7))).
MOE_DEVINL int chunk_slot(int c, int j) { return c * 8 + (j ^ (c & 7)); }
MOE_DEVINL float chunk_fdot_smem(const uint4 q, const float4* __restrict__ v, int c) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v0 = v[chunk_slot(c, 2 * i)];
    const float4 v1 = v[chunk_slot(c, 2 * i + 1)];
    a0 = fmaf(code_f(w[i], 0), v0.x, a0);
    a1 = fmaf(code_f(w[i], 1), v0.y, a1);
    a0 = fmaf(code_f(w[i], 2), v0.z, a0);
    a1 = fmaf(code_f(w[i], 3), v0.w, a1);
    a0 = fmaf(code_f(w[i], 4), v1.x, a0);
    a1 = fmaf(code_f(w[i], 5), v1.y, a1);
    a0 = fmaf(code_f(w[i], 6), v1.z, a0);
    a1 = fmaf(code_f(w[i], 7), v1.w, a1);
  }
  return a0 + a1;
}

// 16 s and (b - 16 s) of a group, from bf16 scale/bias bits.
MOE_DEVINL float2 affine_f(uint16_t sbits, uint16_t bbits) {
  const float s16 = 16.f * bf16_bits_to_f32(sbits);
  return make_float2(s16, bf16_bits_to_f32(bbits) - s16);
}

// x chunks of this lane (c = lane + 32 i) as fp32 registers, and their sums.
template <int XC>
struct XChunks {
  float v[XC][32];
  float sum[XC];
};

template <int XC>
MOE_DEVINL void load_x_chunks(const uint16_t* __restrict__ x, int nch, XChunks<XC>& xc) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < XC; ++i) {
    const int c = lane + 32 * i;
    float s = 0.f;
    if (c < nch) {
      const uint4* src = reinterpret_cast<const uint4*>(x + 32 * c);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 b = src[j];
        const uint32_t u[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          xc.v[i][8 * j + 2 * t] = __uint_as_float(u[t] << 16);
          xc.v[i][8 * j + 2 * t + 1] = __uint_as_float(u[t] & 0xFFFF0000u);
          s += xc.v[i][8 * j + 2 * t] + xc.v[i][8 * j + 2 * t + 1];
        }
      }
    }
    xc.sum[i] = s;
  }
}

// One gate row and one up row (K = d codes, group 64): this lane's chunks.
template <int XC>
struct RowPairLoads {
  uint4 g[XC], u[XC];
  uint16_t gs[XC], gb[XC], us[XC], ub[XC];
};

template <int XC>
MOE_DEVINL void load_rowpair(const moe_w4_t& G, const moe_w4_t& U, int64_t r, int d,
                             RowPairLoads<XC>& L) {
  const int lane = threadIdx.x & 31, nch = d / 32;
  const uint4* gq = reinterpret_cast<const uint4*>(G.q + r * (d / 8));
  const uint4* uq = reinterpret_cast<const uint4*>(U.q + r * (d / 8));
  const int64_t gr = r * (d / 64);
#pragma unroll
  for (int i = 0; i < XC; ++i) {
    const int c = lane + 32 * i;
    if (c < nch) {
      L.g[i] = __ldcs(gq + c);
      L.u[i] = __ldcs(uq + c);
      L.gs[i] = __ldcs(G.scale + gr + (c >> 1));
      L.gb[i] = __ldcs(G.bias + gr + (c >> 1));
      L.us[i] = __ldcs(U.scale + gr + (c >> 1));
      L.ub[i] = __ldcs(U.bias + gr + (c >> 1));
    }
  }
}

// h = silu(x . g_row) * (x . u_row), warp-reduced, valid on every lane.
template <int XC>
MOE_DEVINL float rowpair_h(const RowPairLoads<XC>& L, const XChunks<XC>& xc, int d) {
  const int lane = threadIdx.x & 31, nch = d / 32;
  float ag = 0.f, au = 0.f;
#pragma unroll
  for (int i = 0; i < XC; ++i) {
    if (lane + 32 * i < nch) {
      const float2 fg = affine_f(L.gs[i], L.gb[i]);
      const float2 fu = affine_f(L.us[i], L.ub[i]);
      ag = fmaf(fg.x, chunk_fdot(L.g[i], xc.v[i]), fmaf(fg.y, xc.sum[i], ag));
      au = fmaf(fu.x, chunk_fdot(L.u[i], xc.v[i]), fmaf(fu.y, xc.sum[i], au));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ag += __shfl_xor_sync(kFull, ag, off);
    au += __shfl_xor_sync(kFull, au, off);
  }
  return ag / (1.f + expf(-ag)) * au;
}

// Top-k of the E logits (+ router bias) by warp 0 of the block, read from
// global memory (L2): ids, softmax-over-selected weights and the shared gate
// go to shared memory. Descending, ties to the lower id.
template <int NPL>
MOE_DEVINL void block_topk(const DecodeParams& p, int* s_ids, float* s_w) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float z[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = i * 32 + lane;
      z[i] = 0.f;
      if (e < p.E) {
        z[i] = __ldcg(p.logits + e);
        if (p.w.router_bias) z[i] = z[i] + p.w.router_bias[e];
      }
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
        if (e < p.E && !((taken >> i) & 1u) && (be == INT_MAX || z[i] > bv)) {
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
      s_ids[lane] = my_e;
      s_w[lane] = ex / sum;
    }
    if (lane == 0) s_w[p.k] = p.shared ? 1.f / (1.f + expf(-__ldcg(p.gate_logit))) : 0.f;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- kernel 1
// blocks [0, E/8): router logits 8b..8b+7 (thread t takes rows t + 256 j);
// blocks [E/8, E/8 + f/8): shared expert gate/up, one row pair per warp.
template <int XC>
__global__ void __launch_bounds__(256) decode_router_shared_kernel(DecodeParams p) {
  constexpr int kPre = 8;  // router rows per thread loaded before the wait
  __shared__ float s_red[8][8];
  const int E = p.E, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_router = E / 8;
  const bool is_router = (int)blockIdx.x < n_router;
  float4 wa[kPre], wb[kPre];
  RowPairLoads<XC> L;
  int64_t sh_row = -1;
  if (is_router) {
    const int e0 = blockIdx.x * 8;
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      const int k = threadIdx.x + 256 * j;
      if (k < p.d) {
        const float4* w = reinterpret_cast<const float4*>(p.w.router + (size_t)k * E + e0);
        wa[j] = __ldcs(w);
        wb[j] = __ldcs(w + 1);
      }
    }
  } else {
    sh_row = (int64_t)(blockIdx.x - n_router) * 8 + warp;
    if (sh_row < p.f) load_rowpair<XC>(p.w.sh_gate, p.w.sh_up, sh_row, p.d, L);
  }
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x < 4) p.status[threadIdx.x] = 0;
  pdl_launch_dependents();
  if (is_router) {
    const int e0 = blockIdx.x * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      const int k = threadIdx.x + 256 * j;
      if (k < p.d) {
        const float xv = bf16_bits_to_f32(p.x[k]);
        acc[0] = fmaf(xv, wa[j].x, acc[0]); acc[1] = fmaf(xv, wa[j].y, acc[1]);
        acc[2] = fmaf(xv, wa[j].z, acc[2]); acc[3] = fmaf(xv, wa[j].w, acc[3]);
        acc[4] = fmaf(xv, wb[j].x, acc[4]); acc[5] = fmaf(xv, wb[j].y, acc[5]);
        acc[6] = fmaf(xv, wb[j].z, acc[6]); acc[7] = fmaf(xv, wb[j].w, acc[7]);
      }
    }
    for (int k = threadIdx.x + 256 * kPre; k < p.d; k += 256) {
      const float xv = bf16_bits_to_f32(p.x[k]);
      const float4* w = reinterpret_cast<const float4*>(p.w.router + (size_t)k * E + e0);
      const float4 a = __ldcs(w), b = __ldcs(w + 1);
      acc[0] = fmaf(xv, a.x, acc[0]); acc[1] = fmaf(xv, a.y, acc[1]);
      acc[2] = fmaf(xv, a.z, acc[2]); acc[3] = fmaf(xv, a.w, acc[3]);
      acc[4] = fmaf(xv, b.x, acc[4]); acc[5] = fmaf(xv, b.y, acc[5]);
      acc[6] = fmaf(xv, b.z, acc[6]); acc[7] = fmaf(xv, b.w, acc[7]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[i] += __shfl_xor_sync(kFull, acc[i], off);
    if (lane == 0)
#pragma unroll
      for (int i = 0; i < 8; ++i) s_red[warp][i] = acc[i];
    __syncthreads();
    if (threadIdx.x < 8) {
      float v = 0.f;
      for (int w = 0; w < 8; ++w) v += s_red[w][threadIdx.x];
      p.logits[e0 + threadIdx.x] = v;
    }
  } else {
    if (sh_row < p.f) {
      XChunks<XC> xc;
      load_x_chunks<XC>(p.x, p.d / 32, xc);
      const float h = rowpair_h<XC>(L, xc, p.d);
      if (lane == 0) p.h[(size_t)p.k * p.f + sh_row] = h;
    }
    if (blockIdx.x == (unsigned)n_router && threadIdx.x < 32) {  // shared gate logit x . w_sg
      float a = 0.f;
      for (int k = lane; k < p.d; k += 32) a = fmaf(bf16_bits_to_f32(p.x[k]), p.w.shared_gate[k], a);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(kFull, a, off);
      if (lane == 0) p.gate_logit[0] = a;
    }
  }
}

// ---------------------------------------------------------------- kernel 2
// Routed gate/up rows: row pair rp = slot * f + row, two per warp at a time.
template <int NPL, int XC>
__global__ void __launch_bounds__(256, XC <= 2 ? 2 : 1) decode_gateup_kernel(DecodeParams p) {
  __shared__ int s_ids[32];
  __shared__ float s_w[33];
  XChunks<XC> xc;
  load_x_chunks<XC>(p.x, p.d / 32, xc);  // x does not depend on the router
  pdl_wait();
  pdl_launch_dependents();
  block_topk<NPL>(p, s_ids, s_w);
  if (blockIdx.x == 0 && threadIdx.x <= p.k) {
    if (threadIdx.x < p.k) p.ids[threadIdx.x] = s_ids[threadIdx.x];
    p.wts[threadIdx.x] = s_w[threadIdx.x];
  }
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * 8;
  const int total = p.k * p.f;
  for (int rp0 = blockIdx.x * 8 + (threadIdx.x >> 5); rp0 < total; rp0 += 2 * nwarps) {
    const int rp1 = rp0 + nwarps;
    RowPairLoads<XC> L0, L1;
    int e0 = s_ids[rp0 / p.f], e1 = 0;
    const bool ok0 = e0 >= 0 && e0 < p.E;
    if (ok0) load_rowpair<XC>(p.w.gate, p.w.up, (int64_t)e0 * p.f + rp0 % p.f, p.d, L0);
    bool ok1 = false;
    if (rp1 < total) {
      e1 = s_ids[rp1 / p.f];
      ok1 = e1 >= 0 && e1 < p.E;
      if (ok1) load_rowpair<XC>(p.w.gate, p.w.up, (int64_t)e1 * p.f + rp1 % p.f, p.d, L1);
    }
    if (!ok0 || (rp1 < total && !ok1)) report(p.status, MOE_DEV_BAD_EXPERT, 21, ok0 ? e1 : e0);
    if (ok0) {
      const float h = rowpair_h<XC>(L0, xc, p.d);
      if (lane == 0) p.h[rp0] = h;
    }
    if (ok1) {
      const float h = rowpair_h<XC>(L1, xc, p.d);
      if (lane == 0) p.h[rp1] = h;
    }
  }
}

// ---------------------------------------------------------------- kernel 3
// One warp per output column j: chunk idx = slot * (f/32) + c of the down rows
// (slot < k: routed expert ids[slot], slot k: shared), weighted by wts[slot].
template <int NPL, int NI>
__global__ void __launch_bounds__(256) decode_down_kernel(DecodeParams p) {
  extern __shared__ float4 smem4[];
  __shared__ int s_ids[32];
  __shared__ float s_w[33];
  const int nslots = p.k + (p.shared ? 1 : 0);
  const int fch = p.f / 32;
  const int total = nslots * fch;
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t qrow = p.f / 8, grow = p.f / 64;
  // 1. the selection (from kernel 1's logits: kernel 1 has completed, since
  //    every block of kernel 2 waited for it before letting this grid start)
  //    and this warp's down-row chunks
  block_topk<NPL>(p, s_ids, s_w);
  uint4 w[NI];
  uint16_t sc[NI], bi[NI];
  float coef[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int idx = lane + 32 * i;
    coef[i] = 0.f;
    if (idx < total && j < p.d) {
      const int slot = idx / fch, c = idx % fch;
      int64_t e = 0;
      const moe_w4_t* D = &p.w.sh_down;
      if (slot < p.k) {
        e = s_ids[slot];
        D = &p.w.down;
      }
      if (e >= 0 && e < p.E) {
        const int64_t r = e * p.d + j;
        w[i] = __ldcs(reinterpret_cast<const uint4*>(D->q + r * qrow) + c);
        sc[i] = __ldcs(D->scale + r * grow + (c >> 1));
        bi[i] = __ldcs(D->bias + r * grow + (c >> 1));
        coef[i] = 1.f;
      } else {
        report(p.status, MOE_DEV_BAD_EXPERT, 22, (int)e);
      }
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  // 2. h of every slot, staged as swizzled fp32 chunks, with chunk sums
  float4* hv = smem4;
  float* hsum = reinterpret_cast<float*>(smem4 + total * 8);
  for (int i = threadIdx.x; i < total * 8; i += blockDim.x)
    hv[chunk_slot(i >> 3, i & 7)] = __ldcg(reinterpret_cast<const float4*>(p.h) + i);
  __syncthreads();
  for (int c = threadIdx.x; c < total; c += blockDim.x) {
    float s = 0.f;
    for (int t = 0; t < 8; ++t) {
      const float4 f = hv[chunk_slot(c, t)];
      s += (f.x + f.y) + (f.z + f.w);
    }
    hsum[c] = s;
  }
  __syncthreads();
  if (j >= p.d) return;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int idx = lane + 32 * i;
    if (idx < total && coef[i] != 0.f) {
      const float2 a = affine_f(sc[i], bi[i]);
      const float part = fmaf(a.x, chunk_fdot_smem(w[i], hv, idx), a.y * hsum[idx]);
      acc = fmaf(s_w[idx / fch], part, acc);
    }
  }
  // chunks beyond NI * 32 (large k * d_ff): loaded after the wait
  for (int idx = lane + 32 * NI; idx < total; idx += 32) {
    const int slot = idx / fch, c = idx % fch;
    int64_t e = 0;
    const moe_w4_t* D = &p.w.sh_down;
    if (slot < p.k) {
      e = s_ids[slot];
      D = &p.w.down;
    }
    if (e < 0 || e >= p.E) continue;
    const int64_t r = e * p.d + j;
    const uint4 wq = __ldcs(reinterpret_cast<const uint4*>(D->q + r * qrow) + c);
    const float2 a = affine_f(__ldcs(D->scale + r * grow + (c >> 1)), __ldcs(D->bias + r * grow + (c >> 1)));
    const float part = fmaf(a.x, chunk_fdot_smem(wq, hv, idx), a.y * hsum[idx]);
    acc = fmaf(s_w[slot], part, acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
  if (lane == 0) {
    const __nv_bfloat16 o = __float2bfloat16_rn(acc);
    p.out[j] = *reinterpret_cast<const uint16_t*>(&o);
  }
}

// ---------------------------------------------------------------- launch
template <class K, class... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int NPL, int XC>
cudaError_t launch_xc(const DecodeParams& p, cudaStream_t s) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int n1 = p.E / 8 + (p.shared ? (p.f + 7) / 8 : 0);
  cudaError_t err = launch_pdl(decode_router_shared_kernel<XC>, dim3(n1), 0, s, p);
  if (err != cudaSuccess) return err;
  const int rowpairs = p.k * p.f;
  const int n2 = std::max(1, std::min((rowpairs + 15) / 16, 2 * sms));
  err = launch_pdl(decode_gateup_kernel<NPL, XC>, dim3(n2), 0, s, p);
  if (err != cudaSuccess) return err;
  const int nslots = p.k + (p.shared ? 1 : 0);
  const int total = nslots * (p.f / 32);
  const size_t smem = (size_t)total * 8 * 16 + (size_t)total * 4;
  const dim3 g3((p.d + 7) / 8);
  auto k3 = total <= 32 * 2 ? decode_down_kernel<NPL, 2>
            : total <= 32 * 4 ? decode_down_kernel<NPL, 4>
            : total <= 32 * 6 ? decode_down_kernel<NPL, 6> : decode_down_kernel<NPL, 8>;
  if (smem > 48 * 1024) {
    err = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  return launch_pdl(k3, g3, smem, s, p);
}

template <int NPL>
cudaError_t launch_npl(const DecodeParams& p, cudaStream_t s) {
  switch (p.d / 1024) {
    case 0:
    case 1: return launch_xc<NPL, 1>(p, s);
    case 2: return launch_xc<NPL, 2>(p, s);
    case 3: return launch_xc<NPL, 3>(p, s);
    default: return launch_xc<NPL, 4>(p, s);
  }
}

}  // namespace

cudaError_t decode_launch(const DecodeParams& p, cudaStream_t s) {
  const int npl = (p.E + 31) / 32;
  if (npl <= 2) return launch_npl<2>(p, s);
  if (npl <= 8) return launch_npl<8>(p, s);
  return launch_npl<32>(p, s);
}

}  // namespace moe
