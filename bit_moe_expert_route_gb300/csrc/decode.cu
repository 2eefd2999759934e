// Batch-1 decode: one token through the MoE layer with matrix-vector work
// that streams only the router, the shared expert and the top-k selected
// experts' packed 4-bit weights. ("Perplexity's Lily Beats MLX-LM by 1.35x
// Running Qwen3.6 on Apple Silicon", section "Why prefill and decode get
// different treatment": batch-1 decode is bound by reading the weights, and
// uses matrix-vector work on the vector ALUs.)
//
// One persistent launch per layer: G blocks (one per SM), 256 threads each.
//   before the dependency wait (griddepcontrol.wait; nothing here depends on
//     the previous kernel): TMA bulk copies of this block's shared-expert
//     gate/up rows and shared-expert down rows into shared memory, register
//     loads of its slice of the router; every copy barrier is armed with its
//     byte count (the counts do not depend on the routing).
//   phase A  x into shared memory (one round trip); router partial logits
//     over this block's (8 experts x d/KS rows) slice and the matching
//     partial of the shared gate logit x . w_sg, published at once; then h of
//     the block's shared-expert rows, while the partials travel.
//   phase B  thread e polls the KS partials of expert e's logit (summed in a
//     fixed order); each warp ranks its 32 logits by register shuffles, the
//     warps' top-k candidates are ranked among themselves (descending, ties
//     to the lower id), and the last warp issues the block's bulk copies of
//     the selected experts' rows: its routed gate/up row pairs in two groups
//     with a barrier each (rows land, and are computed, group by group), then
//     its share of every slot's down rows. The other warps compute h of each
//     routed row-pair group as it lands; the issuing warp computes the
//     routing weights.
//   phase C  every block polls h of every slot into shared memory and
//     computes its outputs: every slot's down row, weighted, in slot order,
//     rounded once to bf16.
// Cross-block values are published as 64-bit {value, call epoch} words, so a
// reader's poll is both the synchronisation and the load: one L2 round trip
// per dependency. Block 0 stores the epoch
// for the next call at its end; no counter needs resetting, so consecutive
// calls on one workspace stay one chain of programmatic dependent launches,
// and the next layer's blocks (two blocks fit per SM) fetch their weights
// while this layer runs.
//
// Every block runs each phase once per launch, so the kernel's instruction
// footprint, fetched cold from L2 on every SM, matters as much as its
// arithmetic: each computation has one copy of its code (two rows, or two
// output columns, per pass; an odd one out runs as a duplicate). The kernel,
// the routed rows and the down columns also have instantiations for the
// standard layer shape (d_model 2048, 256 experts, top-8, d_ff 512) with
// those sizes as constants: loop trip counts are known and index splits are
// shifts; a launch runs one instantiation, so only its code is fetched.
//
// Dot products per packed word (8 codes; 4 words = 32 codes = half a group):
// a code q becomes the 16-bit float f = 1 + q/16 exactly (bf16 bits
// 0x3F80 | q << 3, f16 bits 0x3C00 | q << 6), two codes per shift-and-mask,
// and is multiplied with the activation by a mixed-precision FMA (16-bit
// inputs, fp32 accumulate; the product is exact). With the activation chunk
// sums taken once,
//   sum_k (s*q_k + b) v_k = 16 s * sum_k f_k v_k + (b - 16 s) * sum_k v_k.
// f stays in [1, 2), so the fp32 sums cancel no more than a factor of a few.
// x enters as its own bf16 values; h (the SwiGLU output) enters the down
// projection rounded to f16, as in the prefill path.
#include <algorithm>
#include <climits>
#include <mutex>

#include "common.cuh"
#include "gemv_dot.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kIssueWarp = kDecWarps - 1;  // issues the routed copies, then the routing weights
constexpr int kRouterPre = 2;  // router rows per thread loaded before the dependency wait
constexpr int kYGroups = 2;    // routed row-pair groups, each with its own copy barrier
static_assert(kDecodeMaxExperts == kDecThreads, "one expert per thread in the top-k");

MOE_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEVINL void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// 1-D TMA bulk copy global -> this CTA's shared memory, completing on `bar`.
MOE_DEVINL void bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bounded wait on a shared-memory barrier phase (every thread).
MOE_DEVINL void bar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns, int32_t* status, int where) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) {
      report(status, MOE_DEV_TIMEOUT, where, (int)threadIdx.x);
      return;
    }
  }
}

// ---------------------------------------------------------------- dot products
// 16 s and (b - 16 s) of a group, from bf16 scale/bias bits.
MOE_DEVINL float2 affine_f(uint16_t sbits, uint16_t bbits) {
  const float s16 = 16.f * bf16_bits_to_f32(sbits);
  return make_float2(s16, bf16_bits_to_f32(bbits) - s16);
}

// ---------------------------------------------------------------- publishing
// Values other blocks read are published as 64-bit words {payload, call
// epoch}: a reader polls a word until its epoch is this call's, so one L2
// round trip both synchronises and delivers the value. The epoch is one more
// than the last call's (kept in the workspace by block 0).
MOE_DEVINL void publish(unsigned long long* w, float v, uint32_t epoch) {
  const unsigned long long x = ((unsigned long long)epoch << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(w), "l"(x) : "memory");
}
MOE_DEVINL unsigned long long ld_word(const unsigned long long* w) {
  unsigned long long x;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(x) : "l"(w) : "memory");
  return x;
}
MOE_DEVINL void ld_word2(const unsigned long long* w, unsigned long long& a, unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(w) : "memory");
}
MOE_DEVINL bool word_ready(unsigned long long x, uint32_t epoch) { return (uint32_t)(x >> 32) == epoch; }
MOE_DEVINL float word_value(unsigned long long x) { return __uint_as_float((uint32_t)x); }

// Bounded poll helper: true while the caller should keep polling.
struct Poll {
  uint64_t t0 = 0;
  uint32_t i = 0;
  MOE_DEVINL bool again(uint64_t limit_ns, int32_t* status, int where) {
    if (++i == 32) t0 = globaltimer_ns();
    if (i > 32) {
      __nanosleep(32);
      if ((i & 63) == 0 && globaltimer_ns() - t0 > limit_ns) {
        report(status, MOE_DEV_TIMEOUT, where, (int)blockIdx.x);
        return false;
      }
    }
    return true;
  }
};

// ---------------------------------------------------------------- layout
// Shared memory of one block (byte offsets from a 128-byte aligned base):
//   Y   row pairs: gate codes [capY][d/2], up codes [capY][d/2], gate scale,
//       gate bias, up scale, up bias [capY][d/64] each (bf16). Phase C reuses
//       it for h as f16 pairs (see pair_slot), then the h chunk sums (fp32).
//   X   down rows per slot s (S = k routed + shared): codes [capX][f/2],
//       scale, bias [capX][f/64] each.
//   Z   the shared expert's row pairs, laid out as in Y with capS rows.
//   U   x as bf16 pairs (see pair_slot) [d/32 chunks][4 words], then the x
//       chunk sums (fp32 [d/32]).
//   then the selection scratch and the bulk-copy barriers. The router's
//   reduction scratch and the top-k candidates live at the start of Y,
//   which receives no copy before the selection is complete (two blocks per
//   SM need every byte).
struct DecSmem {
  uint8_t* Y;
  uint8_t* X;
  uint8_t* Z;
  uint4* xp;        // [d/32 * 4]
  float* xsum;      // [d/32]
  float* cand_key;  // [8 * kc]
  int* cand_id;     // [8 * kc]
  int* s_ids;       // [32]
  float* s_z;       // [32]
  float* s_w;       // [34]: routing weights, then the shared gate
  float* red;       // [8][9]
  float* s_gp;      // [kDecodeMaxSplits] gate-logit partials
  uint32_t* s_epoch;
  uint64_t* barY;   // [kYGroups]
  uint64_t* barX;
  uint64_t* barZ;
};

MOE_DEVINL int cand_per_warp(const DecodeParams& p) { return min(p.k, 32); }

MOE_DEVINL DecSmem carve_dec_smem(uint8_t* base, const DecodeParams& p) {
  DecSmem m;
  m.Y = base;
  m.X = base + p.y_bytes;
  m.Z = m.X + p.x_bytes;
  m.red = reinterpret_cast<float*>(base);  // aliases in Y (see above)
  m.cand_key = m.red + 8 * 9;
  m.cand_id = reinterpret_cast<int*>(m.cand_key + kDecWarps * cand_per_warp(p));
  uint8_t* u = m.Z + p.z_bytes;
  m.xp = reinterpret_cast<uint4*>(u);
  m.xsum = reinterpret_cast<float*>(u + (size_t)p.d * 2);
  float* f = reinterpret_cast<float*>(u + p.u_bytes);
  m.s_ids = reinterpret_cast<int*>(f);
  f += 32;
  m.s_z = f;
  f += 32;
  m.s_w = f;
  f += 34;
  m.s_gp = f;
  f += kDecodeMaxSplits;
  m.s_epoch = reinterpret_cast<uint32_t*>(f);
  f += 2;
  m.barY = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(f) + 7) & ~uintptr_t(7));
  m.barX = m.barY + kYGroups;
  m.barZ = m.barX + 1;
  return m;
}

// Activations (x, and h in phase C) are held as 16-byte words of four pairs
// (v_i, v_{i+4}), one word per 8 values, 4 words per 32-value chunk. Word j
// of chunk c is slot c*4 + (j ^ ((c >> 1) & 3)): the 8 lanes of a wavefront
// reading word j of chunks c..c+7 then hit 8 different bank groups.
MOE_DEVINL int pair_slot(int c, int j) { return c * 4 + (j ^ ((c >> 1) & 3)); }
// 16-bit element index of value i inside that layout.
MOE_DEVINL int pair_elem(int i) { return pair_slot(i >> 5, (i >> 3) & 3) * 8 + (i & 3) * 2 + ((i >> 2) & 1); }

// Row-pair views inside Y (or Z).
struct RowPairSmem {
  const uint4* gq;
  const uint4* uq;
  const uint16_t *gs, *gb, *us, *ub;
};

MOE_DEVINL RowPairSmem rowpair_smem(const uint8_t* Y, int capY, int i, int d) {
  RowPairSmem r;
  const size_t half_row = (size_t)d / 2, groups = (size_t)d / 64;
  r.gq = reinterpret_cast<const uint4*>(Y + i * half_row);
  r.uq = reinterpret_cast<const uint4*>(Y + ((size_t)capY + i) * half_row);
  const uint16_t* s0 = reinterpret_cast<const uint16_t*>(Y + (size_t)capY * d);
  r.gs = s0 + i * groups;
  r.gb = s0 + (capY + i) * groups;
  r.us = s0 + (2 * capY + i) * groups;
  r.ub = s0 + (3 * capY + i) * groups;
  return r;
}

MOE_DEVINL uint32_t word_of(const uint4& q, int j) { return j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w; }

// v * 1/(1 + e^-v) with a correctly rounded reciprocal (no division slow path)
MOE_DEVINL float silu(float v) { return v * __frcp_rn(1.f + expf(-v)); }

// h of rows [i0, i1) of a row-pair region (region row i = flattened row
// pair r0 + i), by warps [w0, w0 + nw): two consecutive rows per warp per
// pass (a row past i1 runs as a duplicate): h = silu(x . g) * (x . u),
// stored plainly for the workspace view and published. Lanes take the
// 32-code chunks c = lane, lane + 32, ...; 8 independent FMA chains each.
constexpr int kRowsPerPass = 2;
template <int NCH>  // 32-code chunks per row as a compile-time constant, or 0: d / 32 at run time
__device__ __noinline__ void rows_h(const DecodeParams& p, const uint8_t* Y, int cap, const uint4* xp,
                                    const float* xsum, int i0, int i1, int r0, int w0, int nw,
                                    uint32_t epoch) {
  const int lane = threadIdx.x & 31, wr = (int)(threadIdx.x >> 5) - w0, d = NCH ? NCH * 32 : p.d,
            nch = NCH ? NCH : d / 32;
#pragma unroll 1
  for (int i = i0 + kRowsPerPass * wr; i < i1; i += kRowsPerPass * nw) {
    RowPairSmem r[kRowsPerPass];
#pragma unroll
    for (int t = 0; t < kRowsPerPass; ++t) r[t] = rowpair_smem(Y, cap, i + t < i1 ? i + t : i, d);
    float acc[2 * kRowsPerPass];  // gate, up of each row
#pragma unroll
    for (int m = 0; m < 2 * kRowsPerPass; ++m) acc[m] = 0.f;
#pragma unroll(NCH ? NCH / 32 : 1)
    for (int c = lane; c < nch; c += 32) {
      uint4 q[2 * kRowsPerPass];
#pragma unroll
      for (int t = 0; t < kRowsPerPass; ++t) {
        q[2 * t] = r[t].gq[c];
        q[2 * t + 1] = r[t].uq[c];
      }
      float lo[2 * kRowsPerPass], hi[2 * kRowsPerPass];
#pragma unroll
      for (int m = 0; m < 2 * kRowsPerPass; ++m) lo[m] = hi[m] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 vp = xp[pair_slot(c, j)];
#pragma unroll
        for (int m = 0; m < 2 * kRowsPerPass; ++m) word_fdot<true>(word_of(q[m], j), vp, lo[m], hi[m]);
      }
      const int g = c >> 1;
      const float xs = xsum[c];
#pragma unroll
      for (int t = 0; t < kRowsPerPass; ++t) {
        const float2 ag = affine_f(r[t].gs[g], r[t].gb[g]), au = affine_f(r[t].us[g], r[t].ub[g]);
        acc[2 * t] = fmaf(ag.x, lo[2 * t] + hi[2 * t], fmaf(ag.y, xs, acc[2 * t]));
        acc[2 * t + 1] = fmaf(au.x, lo[2 * t + 1] + hi[2 * t + 1], fmaf(au.y, xs, acc[2 * t + 1]));
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int m = 0; m < 2 * kRowsPerPass; ++m) acc[m] += __shfl_xor_sync(kFull, acc[m], off);
    float g = acc[0], u = acc[1];
#pragma unroll
    for (int t = 1; t < kRowsPerPass; ++t)
      if (lane == t) {
        g = acc[2 * t];
        u = acc[2 * t + 1];
      }
    if (lane < kRowsPerPass && i + lane < i1) {
      const float v = silu(g) * u;
      const int row = r0 + i + lane;
      p.h[row] = v;
      publish(p.pub_h + row, v, epoch);
    }
  }
}

// Output columns [j0, j0 + nj) from the down rows in X and h (f16 pairs in
// hp, chunk sums in hsum), two columns per warp per pass (the same h words
// serve both): over the flattened (slot, chunk) index idx = lane + 32 i,
// each slot's part weighted by its routing weight; rounded once to bf16.
// FCH: 32-code chunks per down row as a compile-time constant (the chunk
// index splits into slot and chunk with a shift instead of a division by a
// run-time value in every step), or 0: f / 32 at run time.
template <int FCH>
__device__ __noinline__ void down_cols(const DecodeParams& p, const uint8_t* X, const uint4* hp,
                                       const float* hsum, const float* s_w, int total, int j0, int nj) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, f = FCH ? FCH * 32 : p.f,
            fch = FCH ? FCH : f / 32;
  const size_t half_row = f / 2, groups = f / 64;
  const size_t slot_bytes = (size_t)p.capX * (half_row + 4 * groups);
#pragma unroll 1
  for (int j = warp; j < nj; j += 2 * kDecWarps) {
    const int j1 = j + kDecWarps < nj ? j + kDecWarps : j;
    float acc0 = 0.f, acc1 = 0.f;
    // two chunks per step (idx and idx + 32; the second masked past total)
#pragma unroll 1
    for (int idx0 = lane; idx0 < total; idx0 += 64) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int idx = idx0 + 32 * u;
        if (u == 1 && idx >= total) break;
        const int s = idx / fch, c = idx % fch;
        const uint8_t* base = X + s * slot_bytes;
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(base + (size_t)p.capX * half_row);
        const uint16_t* bi = sc + (size_t)p.capX * groups;
        const uint4 q0 = reinterpret_cast<const uint4*>(base + j * half_row)[c];
        const uint4 q1 = reinterpret_cast<const uint4*>(base + j1 * half_row)[c];
        const float2 a0 = affine_f(sc[j * groups + (c >> 1)], bi[j * groups + (c >> 1)]);
        const float2 a1 = affine_f(sc[j1 * groups + (c >> 1)], bi[j1 * groups + (c >> 1)]);
        float lo0 = 0.f, hi0 = 0.f, lo1 = 0.f, hi1 = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint4 vp = hp[pair_slot(idx, w)];
          word_fdot<false>(word_of(q0, w), vp, lo0, hi0);
          word_fdot<false>(word_of(q1, w), vp, lo1, hi1);
        }
        const float ws = s_w[s], hs = hsum[idx];
        acc0 = fmaf(ws, fmaf(a0.x, lo0 + hi0, a0.y * hs), acc0);
        acc1 = fmaf(ws, fmaf(a1.x, lo1 + hi1, a1.y * hs), acc1);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      acc0 += __shfl_xor_sync(kFull, acc0, off);
      acc1 += __shfl_xor_sync(kFull, acc1, off);
    }
    if (lane < 2 && (lane == 0 || j1 != j)) {
      const __nv_bfloat16 o = __float2bfloat16_rn(lane == 0 ? acc0 : acc1);
      p.out[j0 + (lane == 0 ? j : j1)] = *reinterpret_cast<const uint16_t*>(&o);
    }
  }
}

// Bulk copies of row pairs [r0, r0 + n) of one expert's gate/up into Y slots
// [i0, i0 + n): codes of gate and up, then gate scale, gate bias, up scale,
// up bias. `lane_of`/`lanes`: the calling lane's share of the six copies.
__device__ __noinline__ void issue_rowpairs(uint8_t* Y, int capY, int i0, const moe_w4_t& G,
                                            const moe_w4_t& U, int64_t r0, int n, int d, uint64_t* bar) {
  const uint32_t half_row = d / 2, sbytes = d / 32;  // codes and scale bytes per row
  const uint32_t qb = n * half_row, sb = n * sbytes;
  const int64_t qoff = r0 * half_row, soff = r0 * sbytes;
  uint8_t* s0 = Y + (size_t)capY * d + (size_t)i0 * sbytes;
  const size_t sstride = (size_t)capY * sbytes;
  bulk_load(Y + (size_t)i0 * half_row, reinterpret_cast<const uint8_t*>(G.q) + qoff, qb, bar);
  bulk_load(Y + ((size_t)capY + i0) * half_row, reinterpret_cast<const uint8_t*>(U.q) + qoff, qb, bar);
  bulk_load(s0, reinterpret_cast<const uint8_t*>(G.scale) + soff, sb, bar);
  bulk_load(s0 + sstride, reinterpret_cast<const uint8_t*>(G.bias) + soff, sb, bar);
  bulk_load(s0 + 2 * sstride, reinterpret_cast<const uint8_t*>(U.scale) + soff, sb, bar);
  bulk_load(s0 + 3 * sstride, reinterpret_cast<const uint8_t*>(U.bias) + soff, sb, bar);
}

// Bulk copies of down rows [j0, j0 + n) of expert e (matrix D) into slot s of X.
__device__ __noinline__ void issue_down(uint8_t* X, int capX, int s, const moe_w4_t& D, int64_t e,
                                        int j0, int n, int d, int f, uint64_t* bar) {
  const uint32_t half_row = f / 2, sbytes = f / 32;
  uint8_t* base = X + (size_t)s * capX * (half_row + 2 * sbytes);
  const int64_t r0 = e * d + j0;
  bulk_load(base, reinterpret_cast<const uint8_t*>(D.q) + r0 * half_row, n * half_row, bar);
  bulk_load(base + (size_t)capX * half_row, reinterpret_cast<const uint8_t*>(D.scale) + r0 * sbytes,
            n * sbytes, bar);
  bulk_load(base + (size_t)capX * (half_row + sbytes),
            reinterpret_cast<const uint8_t*>(D.bias) + r0 * sbytes, n * sbytes, bar);
}

// The block's routed region rows (flattened (slot, row) index y0 + i = slot
// * f + row; group g holds region rows [gb[g], gb[g + 1])) cut at group and
// slot boundaries, issued by lane 0 in order, group 0 first, so that the
// groups land in that order; then the down rows [j0, j0 + nj) of every
// routed slot (three copies, one lane per slot). Called by a whole warp.
__device__ __noinline__ void issue_routed(const DecodeParams& p, uint8_t* Y, uint8_t* X, const int* ids,
                                          int y0, const int* gb, int ng, int j0, int nj, uint64_t* barY,
                                          uint64_t* barX) {
  const int lane = threadIdx.x & 31, f = p.f;
  if (lane == 0)
    for (int g = 0; g < ng; ++g) {
      for (int a = gb[g]; a < gb[g + 1];) {
        const int r = y0 + a, slot = r / f, row = r % f;
        const int len = min(gb[g + 1] - a, f - row);
        issue_rowpairs(Y, p.capY, a, p.w.gate, p.w.up, (int64_t)ids[slot] * f + row, len, p.d, barY + g);
        a += len;
      }
    }
  __syncwarp();
  if (nj > 0)
    for (int s = lane; s < p.k; s += 32) issue_down(X, p.capX, s, p.w.down, ids[s], j0, nj, p.d, f, barX);
}

// [lo, hi) of `units` work units for block b of G, scaled by `gran`.
MOE_DEVINL int2 block_range(int units, int b, int G, int gran) {
  const int lo = (int)((int64_t)units * b / G), hi = (int)((int64_t)units * (b + 1) / G);
  return make_int2(lo * gran, hi * gran);
}

// The groups of region rows [0, n) (n a multiple of q, the rows a bulk copy
// moves at least: a row's scales are d/32 bytes, a copy a multiple of 16):
// kYGroups nearly equal parts, each a multiple of q rows.
MOE_DEVINL void y_groups(int n, int q, int* gb) {
  const int units = n / q, ng = units >= kYGroups ? kYGroups : 1;
  for (int g = 0; g <= kYGroups; ++g) gb[g] = g >= ng ? n : (units * g / ng) * q;
}

// ---------------------------------------------------------------- kernel
// SD: the standard layer shape (d_model 2048, 256 experts, top-8, d_ff 512)
// as compile-time constants, so that loops over experts, candidates and
// chunks have known trip counts; otherwise 0 (the sizes come from p).
template <int SD>
__global__ void __launch_bounds__(kDecThreads, 2) decode_layer_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t dsmem[];
  const DecSmem sm = carve_dec_smem(dsmem, p);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int d = SD ? 2048 : p.d, E = SD ? 256 : p.E, k = SD ? 8 : p.k, f = SD ? 512 : p.f;
  const int S = k + (p.shared ? 1 : 0);
  const int ncg = E / 8, n_items = ncg * p.KS, rs = (d + p.KS - 1) / p.KS;
  const uint32_t rp_bytes = d + d / 8;          // one row pair in Y
  const uint32_t dn_bytes = f / 2 + f / 16;     // one down row (codes, scale, bias) in X
  const int2 rr = block_range(k * f / p.qrow, b, G, p.qrow);                       // routed row pairs
  const int2 sr = p.shared ? block_range(f / p.qrow, b, G, p.qrow) : make_int2(0, 0);  // shared row pairs
  const int2 orng = block_range(d / p.qout, b, G, p.qout);                          // outputs
  const int nj0 = min(orng.y - orng.x, p.capX);
  const int nr0 = min(rr.y - rr.x, p.capY);
  const int kc = SD ? 8 : cand_per_warp(p);
  int gb[kYGroups + 1];
  y_groups(nr0, p.qrow, gb);

  if (tid == 0) {
    for (int g = 0; g < kYGroups; ++g) mbar_init(sm.barY + g, 1);
    mbar_init(sm.barZ, 1);
    mbar_init(sm.barX, 1);
    fence_mbar_init();
  }
  for (int i = tid; i < kDecWarps * kc; i += kDecThreads) {
    sm.cand_key[i] = -INFINITY;
    sm.cand_id[i] = INT_MAX;
  }
  if (tid < 32) sm.s_ids[tid] = tid < k ? tid : 0;  // overwritten by the selection
  __syncthreads();

  // ---- before the dependency wait: weights only (nothing the previous
  // kernel writes); every barrier armed with the bytes it will receive
  if (warp == 0) {
    const int ns0 = min(sr.y - sr.x, p.capS), njs = p.shared ? nj0 : 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(sm.barZ, ns0 * rp_bytes);
      mbar_arrive_expect_tx(sm.barX, (njs + k * nj0) * dn_bytes);
      for (int g = 0; g < kYGroups; ++g) mbar_arrive_expect_tx(sm.barY + g, (gb[g + 1] - gb[g]) * rp_bytes);
    }
    __syncwarp();
    if (lane == 0 && ns0 > 0) issue_rowpairs(sm.Z, p.capS, 0, p.w.sh_gate, p.w.sh_up, sr.x, ns0, d, sm.barZ);
    if (lane == 1 && njs > 0) issue_down(sm.X, p.capX, k, p.w.sh_down, 0, orng.x, njs, d, f, sm.barX);
  }
  // this block's first router item (8 experts x d/KS rows): kRouterPre rows per thread
  float4 wa[kRouterPre], wb[kRouterPre];
  float wg[kRouterPre];
  {
    const int cg = b % ncg, ks = b / ncg, row1 = min(d, (ks + 1) * rs);
#pragma unroll
    for (int j = 0; j < kRouterPre; ++j) {
      const int row = ks * rs + tid + kDecThreads * j;
      wa[j] = wb[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      wg[j] = 0.f;
      if (b < n_items && row < row1) {
        const float4* w = reinterpret_cast<const float4*>(p.w.router + (size_t)row * E + cg * 8);
        wa[j] = __ldcs(w);
        wb[j] = __ldcs(w + 1);
        if (cg == 0 && p.shared) wg[j] = __ldcs(p.w.shared_gate + row);
      }
    }
  }

  // One thread waits for the previous kernel (its completion and memory are
  // then visible to the whole grid); the others wait at the block barrier.
  if (tid == 0) pdl_wait();
  __syncthreads();
  pdl_launch_dependents();

  // ---- x (one round trip): paired words and chunk sums; this call's epoch
  if (b == 0 && tid < 4) p.status[tid] = 0;
  if (tid == 0) {
    const uint32_t e = *reinterpret_cast<volatile uint32_t*>(p.sync) + 1;
    *sm.s_epoch = e == 0 ? 1 : e;
  }
  for (int i = tid; i < d / 8; i += kDecThreads) {  // word j = i % 4 of chunk c = i / 4
    const uint4 v = reinterpret_cast<const uint4*>(p.x)[i];
    sm.xp[pair_slot(i >> 2, i & 3)] = pair_up(v);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    float s = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) s += __uint_as_float(u[t] << 16) + __uint_as_float(u[t] & 0xFFFF0000u);
    // the 4 words of a chunk are 4 adjacent lanes, active together (d / 8 is a
    // multiple of 16)
    s += __shfl_xor_sync(__activemask(), s, 1);
    s += __shfl_xor_sync(__activemask(), s, 2);
    if ((i & 3) == 0) sm.xsum[i >> 2] = s;
  }
  __syncthreads();
  const uint32_t epoch = *sm.s_epoch;
  const uint16_t* xh = reinterpret_cast<const uint16_t*>(sm.xp);

  // ---- phase A: router partials (and the shared gate-logit partial)
#pragma unroll 1
  for (int it = b; it < n_items; it += G) {
    const int cg = it % ncg, ks = it / ncg, row1 = min(d, (ks + 1) * rs);
    float acc[9] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int row = ks * rs + tid;
    if (it == b) {  // the rows loaded before the wait
#pragma unroll
      for (int j = 0; j < kRouterPre; ++j, row += kDecThreads) {
        if (row >= row1) continue;
        const float xv = bf16_bits_to_f32(xh[pair_elem(row)]);
        acc[0] = fmaf(xv, wa[j].x, acc[0]); acc[1] = fmaf(xv, wa[j].y, acc[1]);
        acc[2] = fmaf(xv, wa[j].z, acc[2]); acc[3] = fmaf(xv, wa[j].w, acc[3]);
        acc[4] = fmaf(xv, wb[j].x, acc[4]); acc[5] = fmaf(xv, wb[j].y, acc[5]);
        acc[6] = fmaf(xv, wb[j].z, acc[6]); acc[7] = fmaf(xv, wb[j].w, acc[7]);
        acc[8] = fmaf(xv, wg[j], acc[8]);
      }
    }
#pragma unroll 1
    for (; row < row1; row += kDecThreads) {
      const float4* w = reinterpret_cast<const float4*>(p.w.router + (size_t)row * E + cg * 8);
      const float4 a = __ldcs(w), c = __ldcs(w + 1);
      const float g = (cg == 0 && p.shared) ? __ldcs(p.w.shared_gate + row) : 0.f;
      const float xv = bf16_bits_to_f32(xh[pair_elem(row)]);
      acc[0] = fmaf(xv, a.x, acc[0]); acc[1] = fmaf(xv, a.y, acc[1]);
      acc[2] = fmaf(xv, a.z, acc[2]); acc[3] = fmaf(xv, a.w, acc[3]);
      acc[4] = fmaf(xv, c.x, acc[4]); acc[5] = fmaf(xv, c.y, acc[5]);
      acc[6] = fmaf(xv, c.z, acc[6]); acc[7] = fmaf(xv, c.w, acc[7]);
      acc[8] = fmaf(xv, g, acc[8]);
    }
#pragma unroll
    for (int i = 0; i < 9; ++i)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[i] += __shfl_xor_sync(kFull, acc[i], off);
    if (lane == 0)
#pragma unroll
      for (int i = 0; i < 9; ++i) sm.red[warp * 9 + i] = acc[i];
    __syncthreads();
    if (tid < 9 && b != p.silent_block) {
      float v = 0.f;
      for (int w = 0; w < kDecWarps; ++w) v += sm.red[w * 9 + tid];
      if (tid < 8) publish(p.pub + (size_t)ks * E + cg * 8 + tid, v, epoch);
      else if (cg == 0) publish(p.pub + (size_t)kDecodeMaxSplits * E + ks, v, epoch);
    }
    __syncthreads();
  }

  // ---- phase B: logits (polled from the published partials), top k
  float key = -INFINITY;
  if (tid < E) {
    unsigned long long w[kDecodeMaxSplits];
    bool ready = false;
    Poll poll;
    do {
      ready = true;
#pragma unroll
      for (int s = 0; s < kDecodeMaxSplits; ++s)
        if (s < p.KS) {
          w[s] = ld_word(p.pub + (size_t)s * E + tid);
          ready = ready && word_ready(w[s], epoch);
        }
    } while (!ready && poll.again(p.wait_ns, p.status, 41));
    float z = 0.f;
#pragma unroll
    for (int s = 0; s < kDecodeMaxSplits; ++s)
      if (s < p.KS) z += word_value(w[s]);
    if (b == 0) p.logits[tid] = z;
    key = p.w.router_bias ? z + p.w.router_bias[tid] : z;
  }
  if (tid < p.KS) {  // gate-logit partials
    unsigned long long w;
    Poll poll;
    do w = ld_word(p.pub + (size_t)kDecodeMaxSplits * E + tid);
    while (!word_ready(w, epoch) && poll.again(p.wait_ns, p.status, 42));
    sm.s_gp[tid] = word_value(w);
  }
  // rank of each key among its warp's 32 (register shuffles; descending,
  // ties to the lower expert id); the best kc of each warp are candidates
  {
    int rank = 0;
#pragma unroll
    for (int o = 1; o < 32; ++o) {
      const int src = (lane + o) & 31;
      const float kj = __shfl_sync(kFull, key, src);
      rank += (int)(kj > key) | ((int)(kj == key) & (int)(src < lane));
    }
    if (tid < E && rank < kc) {
      sm.cand_key[warp * kc + rank] = key;
      sm.cand_id[warp * kc + rank] = tid;
    }
  }
  __syncthreads();
  // a candidate's rank among all candidates is its overall rank (everything
  // that outranks a top-k expert is a candidate too)
#pragma unroll 1
  for (int t = tid; t < kDecWarps * kc; t += kDecThreads) {
    const float kt = sm.cand_key[t];
    const int et = sm.cand_id[t];
    if (et == INT_MAX) continue;
    int rank = 0;
#pragma unroll 8
    for (int j = 0; j < kDecWarps * kc; ++j) {
      const float kj = sm.cand_key[j];
      rank += (int)(kj > kt) | ((int)(kj == kt) & (int)(sm.cand_id[j] < et));
    }
    if (rank < k) {
      sm.s_ids[rank] = et;
      sm.s_z[rank] = kt;
    }
  }
  fence_proxy_async_smem();  // the aliases in Y are done with before copies land there
  __syncthreads();

  // ---- the routed rows: the issuing warp sends the copies (gate/up row
  // pairs group by group, then the down rows) and computes the routing
  // weights; the other warps compute each row-pair group as it lands
  uint32_t y_phase = 0;
#pragma unroll 1
  for (int c0 = rr.x; c0 < rr.y; c0 += p.capY) {
    const int n = min(p.capY, rr.y - c0);
    y_groups(n, p.qrow, gb);
    if (c0 != rr.x) __syncthreads();  // the previous chunk's rows are consumed
    if (warp == kIssueWarp) {
      if (c0 != rr.x) {
        if (lane == 0) {
          fence_proxy_async_smem();
          for (int g = 0; g < kYGroups; ++g) mbar_arrive_expect_tx(sm.barY + g, (gb[g + 1] - gb[g]) * rp_bytes);
        }
        __syncwarp();
      }
      issue_routed(p, sm.Y, sm.X, sm.s_ids, c0, gb, kYGroups, orng.x, c0 == rr.x ? nj0 : 0, sm.barY, sm.barX);
      if (c0 == rr.x) {  // the routing weights: softmax over the selected biased logits; the shared gate
        const float zmax = sm.s_z[0];
        const float ex = lane < k ? expf(sm.s_z[lane] - zmax) : 0.f;
        float sum = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
        const float wt = ex * __frcp_rn(sum);
        if (lane < k) sm.s_w[lane] = wt;
        float gl = 0.f;
        for (int s = 0; s < p.KS; ++s) gl += sm.s_gp[s];
        const float gate = p.shared ? __frcp_rn(1.f + expf(-gl)) : 0.f;
        if (lane == 0) sm.s_w[k] = gate;
        if (b == 0) {
          if (lane < k) {
            p.ids[lane] = sm.s_ids[lane];
            p.wts[lane] = wt;
          }
          if (lane == 0) {
            p.gate_logit[0] = gl;
            p.wts[k] = gate;
          }
        }
      }
    } else {
      if (c0 == rr.x && warp >= kIssueWarp - 2) {
        // the shared expert's rows (prefetched before the dependency wait) on
        // two warps, while the routed rows are in flight
        uint32_t z_phase = 0;
#pragma unroll 1
        for (int s0 = sr.x; s0 < sr.y; s0 += p.capS) {
          const int n = min(p.capS, sr.y - s0);
          if (s0 != sr.x) {
            named_bar_sync(2, 64);  // both warps are done with the previous chunk
            if (warp == kIssueWarp - 2 && lane == 0) {
              fence_proxy_async_smem();
              mbar_arrive_expect_tx(sm.barZ, n * rp_bytes);
              issue_rowpairs(sm.Z, p.capS, 0, p.w.sh_gate, p.w.sh_up, s0, n, d, sm.barZ);
            }
          }
          bar_wait(sm.barZ, z_phase & 1, p.wait_ns, p.status, 40);
          ++z_phase;
          if (d == 2048)
            rows_h<64>(p, sm.Z, p.capS, sm.xp, sm.xsum, 0, n, k * f + s0, kIssueWarp - 2, 2, epoch);
          else
            rows_h<0>(p, sm.Z, p.capS, sm.xp, sm.xsum, 0, n, k * f + s0, kIssueWarp - 2, 2, epoch);
        }
      }
#pragma unroll 1
      for (int g = 0; g < kYGroups; ++g) {
        if (gb[g + 1] == gb[g]) continue;
        bar_wait(sm.barY + g, y_phase & 1, p.wait_ns, p.status, 43);
        if (d == 2048)
          rows_h<64>(p, sm.Y, p.capY, sm.xp, sm.xsum, gb[g], gb[g + 1], c0, 0, kIssueWarp, epoch);
        else
          rows_h<0>(p, sm.Y, p.capY, sm.xp, sm.xsum, gb[g], gb[g + 1], c0, 0, kIssueWarp, epoch);
      }
    }
    ++y_phase;
  }
  __syncthreads();  // Y is consumed: it holds h from here on; s_w is complete

  // ---- phase C: h of every slot (polled; as f16 pairs), then the block's outputs
  const int total = S * (f / 32);
  uint4* hp = reinterpret_cast<uint4*>(sm.Y);
  float* hsum = reinterpret_cast<float*>(hp + (size_t)total * 4);
  uint16_t* hph = reinterpret_cast<uint16_t*>(hp);
  constexpr int kHB = 12;  // 16-byte words per thread per polling batch (one batch: (k+1) f <= 6144)
  const int n_pairs = total * 16;
#pragma unroll 1
  for (int base = 0; base < n_pairs; base += kHB * kDecThreads) {
    unsigned long long w0[kHB], w1[kHB];
    uint32_t pending = 0;
#pragma unroll
    for (int m = 0; m < kHB; ++m)
      if (base + m * kDecThreads + tid < n_pairs) pending |= 1u << m;
    Poll poll;
    do {
#pragma unroll
      for (int m = 0; m < kHB; ++m)
        if (pending & (1u << m)) ld_word2(p.pub_h + 2 * (base + m * kDecThreads + tid), w0[m], w1[m]);
#pragma unroll
      for (int m = 0; m < kHB; ++m)
        if ((pending & (1u << m)) && word_ready(w0[m], epoch) && word_ready(w1[m], epoch)) {
          const int i = 2 * (base + m * kDecThreads + tid);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const float v = word_value(t == 0 ? w0[m] : w1[m]);
            const __half hv = __float2half_rn(fminf(fmaxf(v, -65504.f), 65504.f));
            hph[pair_elem(i + t)] = *reinterpret_cast<const uint16_t*>(&hv);
          }
          pending &= ~(1u << m);
        }
    } while (pending && poll.again(p.wait_ns, p.status, 44));
  }
  __syncthreads();
#pragma unroll 1
  for (int c = tid; c < total; c += kDecThreads) {  // chunk sums of the f16 values used
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = hp[pair_slot(c, j)];
      const float2 h0 = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
      const float2 h1 = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
      const float2 h2 = __half22float2(*reinterpret_cast<const __half2*>(&v.z));
      const float2 h3 = __half22float2(*reinterpret_cast<const __half2*>(&v.w));
      s += ((h0.x + h0.y) + (h1.x + h1.y)) + ((h2.x + h2.y) + (h3.x + h3.y));
    }
    hsum[c] = s;
  }
  __syncthreads();
  uint32_t x_phase = 0;
#pragma unroll 1
  for (int j0 = orng.x; j0 < orng.y; j0 += p.capX) {
    const int nj = min(p.capX, orng.y - j0);
    if (j0 != orng.x) {
      __syncthreads();
      if (tid == 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(sm.barX, S * nj * dn_bytes);
        for (int s = 0; s < k; ++s) issue_down(sm.X, p.capX, s, p.w.down, sm.s_ids[s], j0, nj, d, f, sm.barX);
        if (p.shared) issue_down(sm.X, p.capX, k, p.w.sh_down, 0, j0, nj, d, f, sm.barX);
      }
    }
    bar_wait(sm.barX, x_phase & 1, p.wait_ns, p.status, 45);
    ++x_phase;
    if (f == 512)
      down_cols<16>(p, sm.X, hp, hsum, sm.s_w, total, j0, nj);
    else
      down_cols<0>(p, sm.X, hp, hsum, sm.s_w, total, j0, nj);
  }

  // ---- block 0 records this call's epoch for the next call (every block
  // read the old value before it published the h block 0 has waited for)
  if (b == 0 && tid == 0) *reinterpret_cast<volatile uint32_t*>(p.sync) = epoch;
}

// ---------------------------------------------------------------- launch
// Two blocks per SM (this layer's and the next layer's, which prefetches):
// 227 KB of shared memory usable by the blocks of one SM, less 1 KB
// reserved per block, halved.
constexpr size_t kDecSmemLimit = (227 * 1024 - 2 * 1024) / 2;

int gcd_int(int a, int b) { return b == 0 ? a : gcd_int(b, a % b); }
int ceil_div(int a, int b) { return (a + b - 1) / b; }
size_t round_up(size_t v, size_t m) { return (v + m - 1) / m * m; }

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

uint32_t u_bytes(const DecodeParams& p) {  // x pairs, x chunk sums
  return (uint32_t)round_up((size_t)p.d * 2 + (size_t)((p.d / 32 + 3) & ~3) * 4, 16);
}

size_t scratch_bytes(const DecodeParams& p) {
  return u_bytes(p) + (size_t)(32 + 32 + 34 + kDecodeMaxSplits + 2) * 4 + 8 + 8 * (kYGroups + 2);
}

// What the aliases at the start of Y need.
size_t y_alias_bytes(const DecodeParams& p) {
  return (size_t)(72 + 2 * kDecWarps * std::min(p.k, 32)) * 4;
}

void size_buffers(DecodeParams& p) {
  const int S = p.k + (p.shared ? 1 : 0);
  const size_t rp = (size_t)p.d + p.d / 8, dn = (size_t)p.f / 2 + p.f / 16;
  const size_t h_bytes = (size_t)S * p.f * 2 + (size_t)S * (p.f / 32) * 4;  // f16 h, chunk sums
  p.y_bytes = (uint32_t)round_up(std::max({(size_t)p.capY * rp, h_bytes, y_alias_bytes(p)}), 128);
  p.x_bytes = (uint32_t)round_up((size_t)p.capX * S * dn, 16);
  p.z_bytes = (uint32_t)round_up((size_t)p.capS * rp, 16);
  p.u_bytes = u_bytes(p);
}

template <class K, class... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int SD>
cudaError_t launch_decode_t(const DecodeParams& p, int G, size_t smem, cudaStream_t s) {
  static std::mutex mu;
  static bool attr_set = false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set) {
      cudaError_t err = cudaFuncSetAttribute(decode_layer_kernel<SD>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecSmemLimit);
      if (err != cudaSuccess) return err;
      // all of the SM's configurable memory as shared memory (two blocks' worth)
      err = cudaFuncSetAttribute(decode_layer_kernel<SD>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (err != cudaSuccess) return err;
      attr_set = true;
    }
  }
  // The blocks wait on one another, so all G must be resident at once (one
  // per SM here), and the next layer's blocks should fit beside them: the
  // occupancy query must allow two blocks per SM, else the launch is refused.
  int per_sm = 0;
  const cudaError_t err =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_layer_kernel<SD>, kDecThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 2 || G > per_sm * sm_count()) return cudaErrorInvalidConfiguration;
  return launch_pdl(decode_layer_kernel<SD>, dim3(G), smem, s, p);
}

cudaError_t launch_decode(const DecodeParams& p, int G, size_t smem, cudaStream_t s) {
  const bool sd = p.d == 2048 && p.E == 256 && p.k == 8 && p.f == 512;  // the standard layer shape
  return sd ? launch_decode_t<1>(p, G, smem, s) : launch_decode_t<0>(p, G, smem, s);
}

// Row granularity of the block ranges: bulk copies move whole 16-byte units
// (d/32 scale bytes per gate/up row, f/32 per down row).
int qrow_of(int d) { return 16 / gcd_int(16, d / 32); }
int qout_of(int f) { return 16 / gcd_int(16, f / 32); }

}  // namespace

size_t decode_pub_words(int E) { return (size_t)kDecodeMaxSplits * E + kDecodeMaxSplits; }

bool decode_shape_supported(int d, int E, int k, int f, bool shared) {
  if (d > 4096 || E % 8 || E > kDecodeMaxExperts || k > 32) return false;
  DecodeParams p = {};
  p.d = d;
  p.E = E;
  p.k = k;
  p.f = f;
  p.shared = shared;
  p.capY = qrow_of(d);  // smallest chunks the kernel can loop over
  p.capX = qout_of(f);
  p.capS = shared ? p.capY : 0;
  size_buffers(p);
  return (size_t)p.y_bytes + p.x_bytes + p.z_bytes + scratch_bytes(p) <= kDecSmemLimit;
}

cudaError_t decode_launch(const DecodeParams& p0, cudaStream_t s) {
  DecodeParams p = p0;
  p.qrow = qrow_of(p.d);
  p.qout = qout_of(p.f);
  // One block per SM, but no more blocks than routed row-pair units: every
  // block then publishes some h, which block 0 waits for before it moves the
  // epoch on (so no block can read the epoch after it changed).
  const int G = std::min(sm_count(), p.k * p.f / p.qrow);
  if (G <= 0) return cudaErrorInvalidDevice;
  const int ncg = p.E / 8;
  p.KS = std::max(1, std::min(kDecodeMaxSplits, G / ncg));
  p.capY = ceil_div(p.k * p.f / p.qrow, G) * p.qrow;
  p.capX = ceil_div(p.d / p.qout, G) * p.qout;
  p.capS = p.shared ? ceil_div(p.f / p.qrow, G) * p.qrow : 0;
  size_buffers(p);
  // too large for two blocks per SM: smaller chunks (the kernel loops over them)
  while ((size_t)p.y_bytes + p.x_bytes + p.z_bytes + scratch_bytes(p) > kDecSmemLimit &&
         (p.capY > p.qrow || p.capX > p.qout || p.capS > p.qrow)) {
    if (p.capS > p.qrow && p.capS >= p.capY)
      p.capS = std::max(p.qrow, (p.capS / 2) / p.qrow * p.qrow);
    else if (p.capY > p.qrow && (p.y_bytes >= p.x_bytes || p.capX <= p.qout))
      p.capY = std::max(p.qrow, (p.capY / 2) / p.qrow * p.qrow);
    else
      p.capX = std::max(p.qout, (p.capX / 2) / p.qout * p.qout);
    size_buffers(p);
  }
  const size_t smem = (size_t)p.y_bytes + p.x_bytes + p.z_bytes + scratch_bytes(p);
  if (smem > kDecSmemLimit) return cudaErrorInvalidValue;
  return launch_decode(p, G, smem, s);
}

}  // namespace moe
