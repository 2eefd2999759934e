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
// so a row lives in the registers of L lanes of one warp (R = 32 / L rows per
// warp, dk / L fp32 entries per lane) for the whole sequence; no barriers
// inside a token. s_i . k_{t+1} is known as soon as s_i is updated, so it is
// summed in the same butterfly as s_i . q_t: one butterfly of log2(L) rounds
// per token on the row's dependency chain. A block holds 8 R rows of one
// value head, which read the same k_t and q_t: the block stages 32 tokens of
// k, q, v, alpha and beta at a time in shared memory (cp.async,
// double-buffered, the next chunk in flight while the current one is
// scanned) and widens k and q to fp32 once per chunk, so a token's inputs
// come from shared memory instead of an L2 round trip each.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kGdnWarps = 8;

// Butterfly sum of v over each aligned group of L lanes (L a power of two).
template <int L>
MOE_DEVINL float group_sum(float v) {
#pragma unroll
  for (int off = L / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
// Two independent sums in one butterfly (their shuffles interleave).
template <int L>
MOE_DEVINL void group_sum2(float& a, float& b) {
#pragma unroll
  for (int off = L / 2; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    b += __shfl_xor_sync(0xffffffffu, b, off);
  }
}

constexpr int kGdnChunk = 32;  // tokens staged in shared memory per step

MOE_DEVINL void cp_async_4(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}

// Shared-memory staging of one chunk of tokens for the block's value head:
// k of its key head (one token more than the chunk, so that the next token's
// k is at hand at the chunk's last token), q, v of the block's RB rows,
// alpha and beta.
template <int DK, int RB>
struct Chunk {
  uint16_t k[kGdnChunk + 1][DK];
  uint16_t q[kGdnChunk][DK];
  uint16_t v[kGdnChunk][RB];
  float a[kGdnChunk];
  float b[kGdnChunk];
};

// The whole block copies tokens t0 .. t0 + n - 1 (k also t0 + n when it
// exists) into `c` (16-byte pieces of k, q and v; 4-byte alpha and beta) as
// one cp.async group.
template <int DK, int RB>
MOE_DEVINL void stage_chunk(const GdnParams& p, int t0, int n, int h, int hk, int row0, Chunk<DK, RB>& c) {
  constexpr int kPieces = DK / 8;   // 16-byte pieces per token of k (and of q)
  constexpr int kVPieces = RB / 8;  // of v
  const int tid = threadIdx.x, nk = n + (t0 + n < p.T ? 1 : 0);
  for (int i = tid; i < nk * kPieces; i += 32 * kGdnWarps) {
    const int j = i / kPieces, part = i % kPieces;
    const int64_t src = ((int64_t)(t0 + j) * p.Hk + hk) * p.dk + part * 8;
    cp_async_16(smem_u32(&c.k[j][part * 8]), p.k + src, 16u);
    if (j < n) cp_async_16(smem_u32(&c.q[j][part * 8]), p.q + src, 16u);
  }
  for (int i = tid; i < n * kVPieces; i += 32 * kGdnWarps) {
    const int j = i / kVPieces, part = i % kVPieces;
    cp_async_16(smem_u32(&c.v[j][part * 8]), p.v + ((int64_t)(t0 + j) * p.Hv + h) * p.dv + row0 + part * 8,
                16u);
  }
  if (tid < n)
    cp_async_4(smem_u32(&c.a[tid]), p.alpha + (int64_t)(t0 + tid) * p.Hv + h);
  else if (tid >= 64 && tid < 64 + n)
    cp_async_4(smem_u32(&c.b[tid - 64]), p.beta + (int64_t)(t0 + tid - 64) * p.Hv + h);
  cp_async_commit();
}

// The current chunk's k and q as fp32, converted once by the whole block
// (every warp reads every token's k and q).
template <int DK>
struct ChunkF {
  float k[kGdnChunk + 1][DK];
  float q[kGdnChunk][DK];
};

template <int DK, int RB>
MOE_DEVINL void widen_chunk(const Chunk<DK, RB>& c, int nk, int n, ChunkF<DK>& f) {
  for (int i = threadIdx.x; i < (nk + n) * DK / 2; i += 32 * kGdnWarps) {
    const int e = 2 * i, j = e / DK, x = e % DK;  // token j of k (then of q), elements x, x + 1
    const uint32_t w = j < nk ? *reinterpret_cast<const uint32_t*>(&c.k[j][x])
                              : *reinterpret_cast<const uint32_t*>(&c.q[j - nk][x]);
    float* dst = j < nk ? &f.k[j][x] : &f.q[j - nk][x];
    *reinterpret_cast<float2*>(dst) = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
}

// Which entries of a row a lane holds. A piece is PS = dk / 32 consecutive
// elements (what a lane holds with one row per warp); a row's L = 32 / R
// lanes take its 32 pieces round robin (lane sl: pieces sl, sl + L, ...),
// so the lanes of a row read consecutive pieces (no shared-memory bank
// conflicts). Entry i of lane sl is element PS (sl + L (i / PS)) + i % PS.
template <int PS, int L>
MOE_DEVINL int lane_elem(int sl, int i) {
  return PS * (sl + L * (i / PS)) + i % PS;
}

// A lane's entries of an fp32 row in shared memory (16- or 8-byte pieces).
template <int PS, int R>
MOE_DEVINL void load_row_f32(const float* row, int sl, float (&f)[PS * R]) {
  constexpr int L = 32 / R;
#pragma unroll
  for (int m = 0; m < R; ++m) {
    const float* src = row + PS * (sl + L * m);
    if constexpr (PS == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      f[4 * m] = v.x;
      f[4 * m + 1] = v.y;
      f[4 * m + 2] = v.z;
      f[4 * m + 3] = v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      f[2 * m] = v.x;
      f[2 * m + 1] = v.y;
    }
  }
}

// Adds a lane's R piece sums in the order of the first log2(R) steps of the
// 32-lane butterfly (pieces m and m + R/2 are lanes p and p ^ 16 there, ...),
// so that with the butterfly over the row's L lanes after it every R gives
// the bits of the one-row-per-warp sum.
template <int R>
MOE_DEVINL float fold_pieces(float (&P)[R]) {
#pragma unroll
  for (int off = R / 2; off >= 1; off >>= 1)
#pragma unroll
    for (int m = 0; m < off; ++m) P[m] += P[m + off];
  return P[0];
}

// The lane's part of s . x, piece by piece (even and odd elements in two
// chains, as with one row per warp), folded.
template <int PS, int R>
MOE_DEVINL float lane_dot(const float (&s)[PS * R], const float (&x)[PS * R]) {
  float P[R];
#pragma unroll
  for (int m = 0; m < R; ++m) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int c = 0; c < PS; c += 2) {
      a0 = fmaf(s[PS * m + c], x[PS * m + c], a0);
      a1 = fmaf(s[PS * m + c + 1], x[PS * m + c + 1], a1);
    }
    P[m] = a0 + a1;
  }
  return fold_pieces<R>(P);
}

// R rows of the state per warp, each on L = 32 / R lanes holding DKL = DK / L
// entries. Per token the row needs s . k_t before its update and s . q_t
// after it; s . k_{t+1} is known right after the update too, so it is summed
// in the same butterfly as s . q_t: one butterfly of log2(L) rounds per token
// on the row's dependency chain.
template <int DK, int R>
__global__ void __launch_bounds__(32 * kGdnWarps) gdn_scan_kernel(const GdnParams p) {
  constexpr int L = 32 / R, PS = DK / 32, DKL = PS * R, RB = kGdnWarps * R;
  // staging buffers (two, or one when the sequence is one chunk), then the fp32 copy
  extern __shared__ __align__(16) uint8_t gdn_smem[];
  Chunk<DK, RB>* buf = reinterpret_cast<Chunk<DK, RB>*>(gdn_smem);
  ChunkF<DK>& cf =
      *reinterpret_cast<ChunkF<DK>*>(gdn_smem + (p.T > kGdnChunk ? 2 : 1) * sizeof(Chunk<DK, RB>));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane / L, sl = lane % L;
  const int rows_per_head = p.dv / RB;
  const int h = blockIdx.x / rows_per_head;
  const int row0 = (blockIdx.x % rows_per_head) * RB;
  const int rr = warp * R + sub, row = row0 + rr;  // this lane's row
  const int hk = h / (p.Hv / p.Hk);
  float* srow = p.state + ((int64_t)h * p.dv + row) * p.dk;
  float s[DKL];
  auto load_state = [&]() {
#pragma unroll
    for (int i = 0; i < DKL; i += 2) {  // 8-byte pieces: the state need only be 8-byte aligned
      const float2 v = *reinterpret_cast<const float2*>(srow + lane_elem<PS, L>(sl, i));
      s[i] = v.x;
      s[i + 1] = v.y;
    }
  };
  // launched as a programmatic dependent: wait for the previous kernel's
  // memory before the first global access (the state may come first when the
  // caller states that the previous launch does not write it), then let the
  // next one launch
  if (p.state_early) load_state();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" :::);
  if (!p.state_early) load_state();
  const int n_chunks = (p.T + kGdnChunk - 1) / kGdnChunk;
  float kc[DKL], pk = 0.f;
#pragma unroll 1
  for (int c = 0; c < n_chunks; ++c) {
    const int t0 = c * kGdnChunk, n = min(kGdnChunk, p.T - t0);
    if (c == 0) stage_chunk<DK, RB>(p, 0, n, h, hk, row0, buf[0]);
    if (c + 1 < n_chunks) {  // the next chunk streams in while this one is scanned
      const int t1 = t0 + kGdnChunk;
      stage_chunk<DK, RB>(p, t1, min(kGdnChunk, p.T - t1), h, hk, row0, buf[(c + 1) & 1]);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const Chunk<DK, RB>& ch = buf[c & 1];
    widen_chunk<DK, RB>(ch, n + (t0 + n < p.T ? 1 : 0), n, cf);
    __syncthreads();
    if (c == 0) {  // the first token's s . k
      load_row_f32<PS, R>(cf.k[0], sl, kc);
      pk = group_sum<L>(lane_dot<PS, R>(s, kc));
    }
    // one token: k_t in kcur, k_{t+1} loaded into knext (the two arrays swap
    // roles from token to token, so no copy between them)
    auto token = [&](int j, const float (&kcur)[DKL], float (&knext)[DKL]) {
      const int t = t0 + j;
      float q[DKL];
      load_row_f32<PS, R>(cf.q[j], sl, q);
      if (t + 1 < p.T) {
        load_row_f32<PS, R>(cf.k[j + 1], sl, knext);
      } else {
#pragma unroll
        for (int i = 0; i < DKL; ++i) knext[i] = 0.f;
      }
      const float v = __uint_as_float((uint32_t)ch.v[j][rr] << 16);
      const float a = ch.a[j], b = ch.b[j];
      const float u = b * (v - a * pk);  // beta (v - alpha s.k)
#pragma unroll
      for (int i = 0; i < DKL; ++i) s[i] = fmaf(a, s[i], u * kcur[i]);  // alpha s + u k
      float po = lane_dot<PS, R>(s, q), pn = lane_dot<PS, R>(s, knext);
      group_sum2<L>(po, pn);  // o_t[row] = s . q_t and the next token's s . k
      if (sl == 0) p.out[((int64_t)t * p.Hv + h) * p.dv + row] = po;
      pk = pn;
    };
    float kn[DKL];
#pragma unroll 1
    for (int j = 0; j < n; j += 2) {
      token(j, kc, kn);
      if (j + 1 < n) {
        token(j + 1, kn, kc);
      } else {  // an odd last token: the next k goes back to kc
#pragma unroll
        for (int i = 0; i < DKL; ++i) kc[i] = kn[i];
      }
    }
    __syncthreads();  // every warp is done with this buffer before it is refilled
  }
#pragma unroll
  for (int i = 0; i < DKL; i += 2)
    *reinterpret_cast<float2*>(srow + lane_elem<PS, L>(sl, i)) = make_float2(s[i], s[i + 1]);
}

template <int DK, int R>
cudaError_t gdn_launch_r(const GdnParams& p, int blocks, cudaStream_t s) {
  constexpr size_t kMax = 2 * sizeof(Chunk<DK, kGdnWarps * R>) + sizeof(ChunkF<DK>);
  static const cudaError_t attr =
      cudaFuncSetAttribute(gdn_scan_kernel<DK, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMax);
  if (attr != cudaSuccess) return attr;
  // a one-chunk sequence (decode) needs one staging buffer: more blocks per SM
  const size_t smem = (p.T > kGdnChunk ? 2 : 1) * sizeof(Chunk<DK, kGdnWarps * R>) + sizeof(ChunkF<DK>);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(32 * kGdnWarps);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr1[1];
  attr1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr1[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr1;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gdn_scan_kernel<DK, R>, p);
}

// Rows per warp: 4 where the value rows split into blocks of 32, else 2, else
// 1, at any length (a single decode token measured 2.80 us per layer with 4
// rows per warp against 2.88 with 1 or 2 and 30 layers in one graph).
int gdn_rows_per_warp(int dv) {
  return dv % (kGdnWarps * 4) == 0 ? 4 : dv % (kGdnWarps * 2) == 0 ? 2 : 1;
}

template <int DK>
cudaError_t gdn_launch_dk(const GdnParams& p, cudaStream_t s) {
  const int R = gdn_rows_per_warp(p.dv);
  const int64_t blocks = (int64_t)p.Hv * (p.dv / (kGdnWarps * R));
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  if (R == 4) return gdn_launch_r<DK, 4>(p, (int)blocks, s);
  if (R == 2) return gdn_launch_r<DK, 2>(p, (int)blocks, s);
  return gdn_launch_r<DK, 1>(p, (int)blocks, s);
}

}  // namespace

bool gdn_shape_supported(int dk, int dv, int Hk, int Hv) {
  return (dk == 64 || dk == 128) && dv >= kGdnWarps && dv % kGdnWarps == 0 && Hk >= 1 && Hv >= Hk &&
         Hv % Hk == 0;
}

cudaError_t gdn_scan_launch(const GdnParams& p, cudaStream_t s) {
  if (!gdn_shape_supported(p.dk, p.dv, p.Hk, p.Hv)) return cudaErrorInvalidValue;
  return p.dk == 128 ? gdn_launch_dk<128>(p, s) : gdn_launch_dk<64>(p, s);
}

}  // namespace moe
