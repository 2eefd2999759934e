// Gated DeltaNet scan: the gated delta rule recurrence with the state held in
// registers for the whole sequence.
//
// "Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple Silicon",
// section "Prefill optimizations", third bullet: each SIMD group owns one
// column of the recurrent state and carries it through the entire scan in
// registers, so the state is never spilled to memory between tokens. The
// recurrence (the page gives none; this is the published gated delta rule,
// Yang, Kautz and Hatamizadeh 2024), per value head with S in R^{dv x dk}:
//   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,
//   o_t = S_t q_t.
// Row i of S evolves on its own given k_t, q_t, v_t[i], alpha_t and beta_t:
//   p = s_i . k_t;  s_i = alpha_t s_i + beta_t (v_t[i] - alpha_t p) k_t;
//   o_t[i] = s_i . q_t,
// so one warp owns one row (dk / 32 entries per lane, fp32 in registers) and
// runs the whole sequence: per token two warp sums (butterfly shuffles), no
// shared memory and no barriers. A block holds 8 rows of one value head, which
// read the same k_t and q_t (L1 hits after the first warp). The next token's
// inputs are loaded before the current token's reductions, so their latency
// overlaps the shuffles.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kGdnRowsPerBlock = 8;

template <int DKL>  // state entries per lane: dk / 32
struct Vec;
template <>
struct Vec<2> {
  static MOE_DEVINL void load_bf16(const uint16_t* p, float (&f)[2]) {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(p));
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xFFFF0000u);
  }
  static MOE_DEVINL void load_f32(const float* p, float (&f)[2]) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    f[0] = v.x;
    f[1] = v.y;
  }
  static MOE_DEVINL void store_f32(float* p, const float (&f)[2]) {
    *reinterpret_cast<float2*>(p) = make_float2(f[0], f[1]);
  }
};
template <>
struct Vec<4> {
  static MOE_DEVINL void load_bf16(const uint16_t* p, float (&f)[4]) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  }
  static MOE_DEVINL void load_f32(const float* p, float (&f)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x;
    f[1] = v.y;
    f[2] = v.z;
    f[3] = v.w;
  }
  static MOE_DEVINL void store_f32(float* p, const float (&f)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};

MOE_DEVINL float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

struct TokenIn {
  float k[4], q[4];
  float v, a, b;
};

template <int DKL>
MOE_DEVINL void load_token(const GdnParams& p, int t, int h, int hk, int row, int lane, TokenIn& in) {
  const int64_t kq = ((int64_t)t * p.Hk + hk) * p.dk + lane * DKL;
  float k[DKL], q[DKL];
  Vec<DKL>::load_bf16(p.k + kq, k);
  Vec<DKL>::load_bf16(p.q + kq, q);
#pragma unroll
  for (int j = 0; j < DKL; ++j) {
    in.k[j] = k[j];
    in.q[j] = q[j];
  }
  const uint16_t vb = __ldg(p.v + ((int64_t)t * p.Hv + h) * p.dv + row);
  in.v = __uint_as_float((uint32_t)vb << 16);
  in.a = __ldg(p.alpha + (int64_t)t * p.Hv + h);
  in.b = __ldg(p.beta + (int64_t)t * p.Hv + h);
}

template <int DKL>
__global__ void __launch_bounds__(32 * kGdnRowsPerBlock) gdn_scan_kernel(const GdnParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_head = p.dv / kGdnRowsPerBlock;
  const int h = blockIdx.x / rows_per_head;
  const int row = (blockIdx.x % rows_per_head) * kGdnRowsPerBlock + warp;
  const int hk = h / (p.Hv / p.Hk);
  float* srow = p.state + ((int64_t)h * p.dv + row) * p.dk + lane * DKL;
  float s[DKL];
  Vec<DKL>::load_f32(srow, s);
  TokenIn cur{}, nxt{};
  if (p.T > 0) load_token<DKL>(p, 0, h, hk, row, lane, cur);
#pragma unroll 1
  for (int t = 0; t < p.T; ++t) {
    if (t + 1 < p.T) load_token<DKL>(p, t + 1, h, hk, row, lane, nxt);
    float pk = 0.f;
#pragma unroll
    for (int j = 0; j < DKL; ++j) pk = fmaf(s[j], cur.k[j], pk);
    pk = warp_sum(pk);                                   // s_i . k_t
    const float u = cur.b * (cur.v - cur.a * pk);        // beta (v - alpha s.k)
    float po = 0.f;
#pragma unroll
    for (int j = 0; j < DKL; ++j) {
      s[j] = fmaf(cur.a, s[j], u * cur.k[j]);            // alpha s + u k
      po = fmaf(s[j], cur.q[j], po);
    }
    po = warp_sum(po);                                   // o_t[i] = s_i . q_t
    if (lane == 0) p.out[((int64_t)t * p.Hv + h) * p.dv + row] = po;
    cur = nxt;
  }
  Vec<DKL>::store_f32(srow, s);
}

}  // namespace

bool gdn_shape_supported(int dk, int dv, int Hk, int Hv) {
  return (dk == 64 || dk == 128) && dv >= kGdnRowsPerBlock && dv % kGdnRowsPerBlock == 0 &&
         Hk >= 1 && Hv >= Hk && Hv % Hk == 0;
}

cudaError_t gdn_scan_launch(const GdnParams& p, cudaStream_t s) {
  if (!gdn_shape_supported(p.dk, p.dv, p.Hk, p.Hv)) return cudaErrorInvalidValue;
  const int64_t blocks = (int64_t)p.Hv * (p.dv / kGdnRowsPerBlock);
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  if (p.dk == 128)
    gdn_scan_kernel<4><<<(int)blocks, 32 * kGdnRowsPerBlock, 0, s>>>(p);
  else
    gdn_scan_kernel<2><<<(int)blocks, 32 * kGdnRowsPerBlock, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
