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
// barriers inside a token. A block holds 8 rows of one value head, which read
// the same k_t and q_t: the block stages 32 tokens of k, q, v, alpha and beta
// at a time in shared memory (cp.async, double-buffered, the next chunk in
// flight while the current one is scanned), so a token's inputs come from
// shared memory instead of an L2 round trip each.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kGdnRowsPerBlock = 8;

template <int DKL>  // state entries per lane: dk / 32 (fp32 state row in and out)
struct Vec;
template <>
struct Vec<2> {
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

constexpr int kGdnChunk = 32;  // tokens staged in shared memory per step

MOE_DEVINL void cp_async_4(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}

// Shared-memory staging of one chunk of tokens for the block's value head:
// k and q of its key head, v of its 8 rows, alpha and beta.
template <int DKL>
struct Chunk {
  uint16_t k[kGdnChunk][32 * DKL];
  uint16_t q[kGdnChunk][32 * DKL];
  uint16_t v[kGdnChunk][kGdnRowsPerBlock];
  float a[kGdnChunk];
  float b[kGdnChunk];
};

// The whole block copies tokens t0 .. t0 + n - 1 into `c` (16-byte pieces of
// k, q and v; 4-byte alpha and beta) as one cp.async group.
template <int DKL>
MOE_DEVINL void stage_chunk(const GdnParams& p, int t0, int n, int h, int hk, int row0,
                            Chunk<DKL>& c) {
  constexpr int kPieces = 32 * DKL / 8;  // 16-byte pieces per token of k (and of q)
  const int tid = threadIdx.x;
  for (int i = tid; i < n * kPieces; i += 32 * kGdnRowsPerBlock) {
    const int j = i / kPieces, part = i % kPieces;
    const int64_t src = ((int64_t)(t0 + j) * p.Hk + hk) * p.dk + part * 8;
    cp_async_16(smem_u32(&c.k[j][part * 8]), p.k + src, 16u);
    cp_async_16(smem_u32(&c.q[j][part * 8]), p.q + src, 16u);
  }
  if (tid < n) {
    cp_async_16(smem_u32(&c.v[tid][0]), p.v + ((int64_t)(t0 + tid) * p.Hv + h) * p.dv + row0, 16u);
  } else if (tid >= 64 && tid < 64 + n) {
    cp_async_4(smem_u32(&c.a[tid - 64]), p.alpha + (int64_t)(t0 + tid - 64) * p.Hv + h);
  } else if (tid >= 128 && tid < 128 + n) {
    cp_async_4(smem_u32(&c.b[tid - 128]), p.beta + (int64_t)(t0 + tid - 128) * p.Hv + h);
  }
  cp_async_commit();
}

template <int DKL>
MOE_DEVINL void load_bf16_smem(const uint16_t* p, float (&f)[DKL]) {
  if constexpr (DKL == 4) {
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

template <int DKL>
__global__ void __launch_bounds__(32 * kGdnRowsPerBlock) gdn_scan_kernel(const GdnParams p) {
  __shared__ __align__(16) Chunk<DKL> buf[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_head = p.dv / kGdnRowsPerBlock;
  const int h = blockIdx.x / rows_per_head;
  const int row0 = (blockIdx.x % rows_per_head) * kGdnRowsPerBlock;
  const int row = row0 + warp;
  const int hk = h / (p.Hv / p.Hk);
  float* srow = p.state + ((int64_t)h * p.dv + row) * p.dk + lane * DKL;
  float s[DKL];
  Vec<DKL>::load_f32(srow, s);
  const int n_chunks = (p.T + kGdnChunk - 1) / kGdnChunk;
  if (n_chunks > 0) stage_chunk<DKL>(p, 0, min(kGdnChunk, p.T), h, hk, row0, buf[0]);
#pragma unroll 1
  for (int c = 0; c < n_chunks; ++c) {
    const int t0 = c * kGdnChunk, n = min(kGdnChunk, p.T - t0);
    if (c + 1 < n_chunks) {  // the next chunk streams in while this one is scanned
      const int t1 = t0 + kGdnChunk;
      stage_chunk<DKL>(p, t1, min(kGdnChunk, p.T - t1), h, hk, row0, buf[(c + 1) & 1]);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const Chunk<DKL>& ch = buf[c & 1];
#pragma unroll 1
    for (int j = 0; j < n; ++j) {
      float k[DKL], q[DKL];
      load_bf16_smem<DKL>(&ch.k[j][lane * DKL], k);
      load_bf16_smem<DKL>(&ch.q[j][lane * DKL], q);
      const float v = __uint_as_float((uint32_t)ch.v[j][warp] << 16);
      const float a = ch.a[j], b = ch.b[j];
      float pk = 0.f;
#pragma unroll
      for (int i = 0; i < DKL; ++i) pk = fmaf(s[i], k[i], pk);
      pk = warp_sum(pk);                                 // s_i . k_t
      const float u = b * (v - a * pk);                  // beta (v - alpha s.k)
      float po = 0.f;
#pragma unroll
      for (int i = 0; i < DKL; ++i) {
        s[i] = fmaf(a, s[i], u * k[i]);                  // alpha s + u k
        po = fmaf(s[i], q[i], po);
      }
      po = warp_sum(po);                                 // o_t[i] = s_i . q_t
      if (lane == 0) p.out[((int64_t)(t0 + j) * p.Hv + h) * p.dv + row] = po;
    }
    __syncthreads();  // every warp is done with this buffer before it is refilled
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
