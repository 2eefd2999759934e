// The expert chain fused per row tile: gate/up grouped GEMM + SwiGLU, then
// the down GEMM + weighted combine, with h kept in shared memory.
//
// "Fused dequantization inside the grouped GEMM" and the routing/combine
// around it ("Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on
// Apple Silicon", section "Prefill optimizations"): the 4-bit tiles are
// unpacked on chip just before the multiply. Here the activations between
// the two projections are not written to memory either: a CTA takes one
// tile of up to 64 rows of one expert (or of the shared expert) and runs
//   G slices  f/128 slices of 128 gate rows and the matching 128 up rows,
//             K = d: tcgen05 MMAs into two tensor-memory accumulators, then
//             h = silu(g) * u (f16) written straight into a shared-memory
//             buffer laid out as the down GEMM's B operand (K-major, 128-byte
//             swizzle, one 64-feature block per 8 KB);
//   D slices  d/128 slices of 128 down rows, K = f, B = that h buffer, then
//             row_scale * y added into each row's fp32 output row at L2
//             (one bulk reduce per token row, as the two-kernel path).
// Roles (one persistent CTA per SM, 512 threads), as in the grouped GEMM:
// warp 0 TMA of packed codes (gate+up, or down), warp 1 the MMAs, warps 2-3
// gather the token rows for the G slices (16-byte cp.async, zero past the
// tile), warps 4-11 dequantise into tensor memory (the MMA's A operand),
// warps 12-15 the epilogues (SwiGLU into the h buffer; the combine). Two
// accumulator buffers let one slice's epilogue overlap the next slice's
// MMAs; the h buffer is single: a tile's D MMAs wait until its last G slice
// is written (h_full), and the next tile's SwiGLU waits until those MMAs
// have read it (h_empty). Every wait is bounded (2 s, MOE_DEV_TIMEOUT).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kTileM = 128;                    // weight rows per slice (MMA M)
constexpr int kKB = 64;                        // codes per k-block (= quantisation group)
constexpr int kBN = kFusedBlockN;              // token rows per tile (MMA N)
constexpr int kQK = 4;                         // k-blocks per packed-code stage
constexpr int kSQ = 2;                         // packed-code stages
constexpr int kQStage = kTileM * kKB / 2 * kQK;  // 16 KB per matrix per stage
constexpr int kSA = 4;                         // A stages in tensor memory
constexpr int kAColsStage = 2 * (kKB / 2);     // two matrices' 64 K in 32-bit columns
constexpr int kACol = 2 * 2 * kBN;             // A stages after two buffers of two accumulators
constexpr int kBBytes = kBN * kKB * 2;         // token tile of one k-block: 8 KB
constexpr int kSB = 6;                         // token-tile stages
constexpr int kCH = 32;                        // combine chunk: token rows per pass
constexpr int kHBlocks = kFusedMaxDff / kKB;   // h buffer: 64-feature blocks

constexpr int kOffQ = 0;
constexpr int kOffB = kOffQ + kSQ * 2 * kQStage;
constexpr int kOffH = kOffB + kSB * kBBytes;
constexpr int kOffEpi = kOffH + kHBlocks * kBBytes;
constexpr int kOffRow = kOffEpi + 2 * kCH * kTileM * 4;
constexpr int kOffBar = kOffRow + 2 * kBN * 4;
constexpr int kNumBars = 2 * kSQ + 2 * kSA + 2 * kSB + 4 + 3;
constexpr int kSmem = kOffBar + 8 * kNumBars + 16 + 1024;  // + alignment slack
static_assert(kSmem <= 232448, "shared memory per CTA exceeded");
static_assert(kACol + kSA * kAColsStage <= 512, "tensor memory exceeded");

struct KParams {
  CUtensorMap tm[6];  // codes: gate, up, shared gate, shared up, down, shared down
  FusedParams g;
};

struct Tile {
  int group, row0, rows;
  bool ok, ext;
};

MOE_DEVINL Tile load_tile(const FusedParams& g, int u) {
  const int4 m = reinterpret_cast<const int4*>(g.block_map)[u];
  Tile t;
  t.group = m.x;
  t.row0 = m.y;
  t.rows = m.z;
  t.ext = m.x == g.n_groups;
  t.ok = m.x >= 0 && (m.x < g.n_groups || (g.X[0].q != nullptr && t.ext)) && m.y >= 0 && m.z >= 1 &&
         m.z <= kBN && (int64_t)m.y + m.z <= g.n_rows;
  return t;
}

MOE_DEVINL int num_units(const FusedParams& g) {
  int nt = *g.num_tiles;
  if (nt < 0) nt = 0;
  if (nt > g.max_tiles) nt = g.max_tiles;
  return nt;
}

// 8 codes of a packed word -> 8 f16 RNE(scale * q + bias), as 4 words in K order
// (1024 + q is exact in f16; minus 1024, then one fused f16x2 fma).
MOE_DEVINL uint4 dequant_word_f16(uint32_t w, __half2 s2, __half2 b2) {
  const __half2 m1024 = __floats2half2_rn(-1024.f, -1024.f);
  const __half2 one = __floats2half2_rn(1.f, 1.f);
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;
    __half2 q2 = __hfma2(*reinterpret_cast<const __half2*>(&v), one, m1024);
    __half2 r = __hfma2(s2, q2, b2);
    p[i] = *reinterpret_cast<uint32_t*>(&r);
  }
  uint4 o;
  o.x = __byte_perm(p[0], p[1], 0x5410);
  o.y = __byte_perm(p[2], p[3], 0x5410);
  o.z = __byte_perm(p[0], p[1], 0x7632);
  o.w = __byte_perm(p[2], p[3], 0x7632);
  return o;
}

// bf16 bits -> f16 pair {v, v}
MOE_DEVINL uint32_t splat_f16(uint16_t bf16_bits) {
  const __half h = __float2half_rn(__uint_as_float((uint32_t)bf16_bits << 16));
  return (uint32_t)(*reinterpret_cast<const uint16_t*>(&h)) * 0x10001u;
}

MOE_DEVINL uint16_t to_f16_sat(float v) {
  const __half h = __float2half_rn(fminf(fmaxf(v, -65504.f), 65504.f));
  return *reinterpret_cast<const uint16_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 1) gemm_fused_kernel(const __grid_constant__ KParams kp) {
  const FusedParams& g = kp.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + kSQ;
  uint64_t* a_full = q_empty + kSQ;
  uint64_t* a_empty = a_full + kSA;
  uint64_t* b_full = a_empty + kSA;
  uint64_t* b_empty = b_full + kSB;
  uint64_t* acc_full = b_empty + kSB;  // [2]
  uint64_t* acc_empty = acc_full + 2;  // [2]
  uint64_t* h_full = acc_empty + 2;
  uint64_t* h_empty = h_full + 1;
  uint64_t* drain = h_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = g.d, f = g.f;
  const int MTG = f / kTileM, KBG = d / kKB;  // G slices and their k-blocks
  const int MTD = d / kTileM, KBD = f / kKB;  // D slices and their k-blocks

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 8);  // dequant warps
    }
    for (int i = 0; i < kSA; ++i) {
      mbar_init(&a_full[i], 8);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < kSB; ++i) {
      mbar_init(&b_full[i], 2);  // gather warps
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);  // epilogue warps
    }
    mbar_init(h_full, 4);
    mbar_init(h_empty, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < 6; ++i) tma_prefetch_desc(&kp.tm[i]);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int units = num_units(g);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_last();
      uint32_t qit = 0;
      bool alive = true;
      for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
        const Tile t = load_tile(g, u);
        if (!t.ok) {
          report(g.status, MOE_DEV_BAD_TILE, 61, u);
          continue;
        }
        // G slices: gate and up codes; D slices: down codes
        for (int ph = 0; ph < 2 && alive; ++ph) {
          const int MT = ph == 0 ? MTG : MTD, KB = ph == 0 ? KBG : KBD, nmat = ph == 0 ? 2 : 1;
          for (int mt = 0; mt < MT && alive; ++mt) {
            const int row = (t.ext ? 0 : t.group * (ph == 0 ? f : d)) + mt * kTileM;
            for (int kb = 0; kb < KB; kb += kQK, ++qit) {
              const int s = qit % kSQ;
              if (!mbar_wait(&q_empty[s], ((qit / kSQ) & 1) ^ 1, abort_flag, g.status, 62)) {
                alive = false;
                break;
              }
              mbar_arrive_expect_tx(&q_full[s], nmat * kQStage);
              for (int j = 0; j < nmat; ++j) {
                const int map = ph == 0 ? (t.ext ? 2 : 0) + j : (t.ext ? 5 : 4);
                tma_load_2d(smem + kOffQ + (s * 2 + j) * kQStage, &kp.tm[map], kb * (kKB / 8), row,
                            &q_full[s], policy);
              }
            }
          }
        }
      }
      for (uint32_t j = qit > (uint32_t)kSQ ? qit - kSQ : 0; j < qit; ++j)
        mbar_wait(&q_full[j % kSQ], (j / kSQ) & 1, abort_flag, g.status, 63);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kTileM, kBN);
      uint32_t it = 0, bit = 0, acc_it = 0, ul = 0;  // ul: this CTA's valid tiles so far
      bool alive = true;
      for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
        const Tile t = load_tile(g, u);
        if (!t.ok) continue;
        for (int ph = 0; ph < 2 && alive; ++ph) {
          const int MT = ph == 0 ? MTG : MTD, KB = ph == 0 ? KBG : KBD;
          if (ph == 1) {  // the tile's h is complete in shared memory
            if (!mbar_wait(h_full, ul & 1, abort_flag, g.status, 64)) {
              alive = false;
              break;
            }
            tc_fence_after();
          }
          for (int mt = 0; mt < MT && alive; ++mt, ++acc_it) {
            const uint32_t buf = acc_it & 1;
            if (!mbar_wait(&acc_empty[buf], ((acc_it >> 1) & 1) ^ 1, abort_flag, g.status, 65)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + buf * (2 * kBN);
            for (int kb = 0; kb < KB; ++kb, ++it) {
              const int s = it % kSA;
              if (!mbar_wait(&a_full[s], (it / kSA) & 1, abort_flag, g.status, 66)) {
                alive = false;
                break;
              }
              const uint32_t a0 = tmem_base + kACol + s * kAColsStage;
              if (ph == 0) {
                const int sb = bit % kSB;
                if (!mbar_wait(&b_full[sb], (bit / kSB) & 1, abort_flag, g.status, 67)) {
                  alive = false;
                  break;
                }
                tc_fence_after();
                const uint32_t b_addr = smem_u32(smem + kOffB + sb * kBBytes);
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                  for (int kk = 0; kk < kKB / 16; ++kk)
                    tc_mma_ts(d_tmem + j * kBN, a0 + j * (kKB / 2) + kk * 8, smem_desc_sw128(b_addr + kk * 32),
                              idesc, (kb | kk) != 0);
                tc_commit(&b_empty[sb]);
                ++bit;
              } else {
                tc_fence_after();
                const uint32_t h_addr = smem_u32(smem + kOffH + kb * kBBytes);
#pragma unroll
                for (int kk = 0; kk < kKB / 16; ++kk)
                  tc_mma_ts(d_tmem, a0 + kk * 8, smem_desc_sw128(h_addr + kk * 32), idesc, (kb | kk) != 0);
              }
              tc_commit(&a_empty[s]);
            }
            if (!alive) break;
            tc_commit(&acc_full[buf]);
          }
          if (ph == 1 && alive) tc_commit(h_empty);  // the tile's D MMAs have read h
        }
        ++ul;
      }
      tc_commit(drain);
      mbar_wait(drain, 0, abort_flag, g.status, 68);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ dequantise
    const int dt = threadIdx.x - 128;
    const int m = dt & (kTileM - 1);  // weight row inside the slice
    const int half = dt >> 7;         // codes half*32 .. half*32+31 of each k-block
    uint32_t it = 0, qit = 0;
    bool alive = true;
    for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
      const Tile t = load_tile(g, u);
      if (!t.ok) continue;
      for (int ph = 0; ph < 2 && alive; ++ph) {
        const int MT = ph == 0 ? MTG : MTD, KB = ph == 0 ? KBG : KBD, nmat = ph == 0 ? 2 : 1;
        for (int mt = 0; mt < MT && alive; ++mt) {
          const int64_t row = (t.ext ? 0 : (int64_t)t.group * (ph == 0 ? f : d)) + mt * kTileM + m;
          const uint16_t* sc[2];
          const uint16_t* bi[2];
          for (int j = 0; j < 2; ++j) {
            const GemmW4& w = t.ext ? g.X[ph == 0 ? j : 2] : g.W[ph == 0 ? j : 2];
            sc[j] = w.scale + row * KB;
            bi[j] = w.bias + row * KB;
          }
          for (int kb0 = 0; kb0 < KB && alive; kb0 += 8) {
            // 8 k-blocks' scales and biases per 16-byte load (KB is a multiple of 8)
            uint4 sv[2], bv[2];
            for (int j = 0; j < nmat; ++j) {
              sv[j] = __ldg(reinterpret_cast<const uint4*>(sc[j]) + (kb0 >> 3));
              bv[j] = __ldg(reinterpret_cast<const uint4*>(bi[j]) + (kb0 >> 3));
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int kb = kb0 + i;
              const int sq = qit % kSQ;
              if (kb % kQK == 0 && !mbar_wait(&q_full[sq], (qit / kSQ) & 1, abort_flag, g.status, 69)) {
                alive = false;
                break;
              }
              const int qoff = m * 128 + ((((kb % kQK) * 2 + half) ^ (m & 7)) << 4);
              uint4 qw[2];
              for (int j = 0; j < nmat; ++j)
                qw[j] = *reinterpret_cast<const uint4*>(smem + kOffQ + (sq * 2 + j) * kQStage + qoff);
              const int sa = it % kSA;
              if (!mbar_wait(&a_empty[sa], ((it / kSA) & 1) ^ 1, abort_flag, g.status, 70)) {
                alive = false;
                break;
              }
              for (int j = 0; j < nmat; ++j) {
                const uint32_t sw = i < 2 ? sv[j].x : i < 4 ? sv[j].y : i < 6 ? sv[j].z : sv[j].w;
                const uint32_t bw = i < 2 ? bv[j].x : i < 4 ? bv[j].y : i < 6 ? bv[j].z : bv[j].w;
                const uint32_t s2 = splat_f16((uint16_t)(sw >> ((i & 1) * 16)));
                const uint32_t b2 = splat_f16((uint16_t)(bw >> ((i & 1) * 16)));
                const uint32_t words[4] = {qw[j].x, qw[j].y, qw[j].z, qw[j].w};
                uint32_t r[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  const uint4 o = dequant_word_f16(words[c], *reinterpret_cast<const __half2*>(&s2),
                                                   *reinterpret_cast<const __half2*>(&b2));
                  r[4 * c] = o.x;
                  r[4 * c + 1] = o.y;
                  r[4 * c + 2] = o.z;
                  r[4 * c + 3] = o.w;
                }
                tmem_st_32x32b_x16(tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + kACol + sa * kAColsStage +
                                       j * (kKB / 2) + half * 16,
                                   r);
              }
              tc_wait_st();
              tc_fence_before();
              mbar_arrive_warp(&a_full[sa]);
              if (kb % kQK == kQK - 1) {
                mbar_arrive_warp(&q_empty[sq]);
                ++qit;
              }
              ++it;
            }
          }
        }
      }
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ gather the token rows (G slices)
    constexpr int kD = kSB - 2;
    constexpr int kRowsPerThread = kBN * 8 / 64;  // 16-byte chunks per thread per k-block
    const int gt = threadIdx.x - 64;
    const int c = gt & 7;
    const int n_first = gt >> 3;
    uint32_t it = 0, arrived = 0;
    bool alive = true;
    for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
      const Tile t = load_tile(g, u);
      if (!t.ok) continue;
      int64_t src_row[kRowsPerThread];
      bool valid[kRowsPerThread];
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int n = n_first + 8 * i;
        valid[i] = n < t.rows;
        src_row[i] = 0;
        if (valid[i]) {
          const int64_t r = t.row0 + n;
          const int64_t a = (int64_t)g.row_index[r];
          if (a < 0 || a >= g.A_rows) {
            report(g.status, MOE_DEV_BAD_ROW, 71, (int)r);
            valid[i] = false;
          } else {
            src_row[i] = a;
          }
        }
      }
      for (int mt = 0; mt < MTG && alive; ++mt) {
        for (int kb = 0; kb < KBG; ++kb, ++it) {
          const int sb = it % kSB;
          if (!mbar_wait(&b_empty[sb], ((it / kSB) & 1) ^ 1, abort_flag, g.status, 72)) {
            alive = false;
            break;
          }
          const uint32_t b_tile = smem_u32(smem + kOffB + sb * kBBytes);
#pragma unroll
          for (int i = 0; i < kRowsPerThread; ++i) {
            const int n = n_first + 8 * i;
            const uint16_t* src = g.A + src_row[i] * d + kb * kKB + c * 8;
            cp_async_16(b_tile + sw128_offset(n, c), src, valid[i] ? 16u : 0u);
          }
          cp_async_commit();
          if (it + 1 - arrived > (uint32_t)kD) {
            cp_async_wait<kD>();
            fence_proxy_async_smem();
            mbar_arrive_warp(&b_full[arrived % kSB]);
            ++arrived;
          }
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      for (; arrived < it; ++arrived) mbar_arrive_warp(&b_full[arrived % kSB]);
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (; arrived < it; ++arrived) mbar_arrive_warp(&b_full[arrived % kSB]);
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogues
    const int ew = warp & 3;           // TMEM lane quarter = the warp's 32 weight rows
    const int et = threadIdx.x - 384;  // 0..127 inside the epilogue group
    constexpr int kRowsPerWarp = kCH / 4;
    constexpr int kStage = kCH * kTileM;
    float* s_rscale = reinterpret_cast<float*>(smem + kOffRow);
    int* s_orow = reinterpret_cast<int*>(s_rscale + kBN);
    uint8_t* stage = smem + kOffEpi;
    uint32_t acc_it = 0, chunk = 0, ul = 0;  // ul: this CTA's valid tiles so far
    bool alive = true;
    for (int u = blockIdx.x; u < units && alive; u += gridDim.x, ++ul) {
      const Tile t = load_tile(g, u);
      if (!t.ok) {
        --ul;
        continue;
      }
      // the previous tile's D MMAs are done with the h buffer
      if (!mbar_wait(h_empty, (ul & 1) ^ 1, abort_flag, g.status, 73)) break;
      named_bar_sync(1, 128);  // every epilogue warp is done with the previous tile's rows
      for (int n = et; n < t.rows; n += 128) {
        const int64_t r = (int64_t)t.row0 + n;
        int orow = __ldg(g.row_index + r);
        if (orow < 0 || orow >= g.C_rows) {
          report(g.status, MOE_DEV_BAD_ROW, 74, (int)r);
          orow = -1;
        }
        s_orow[n] = orow;
        s_rscale[n] = __ldg(g.row_scale + r);
      }
      named_bar_sync(1, 128);
      for (int ph = 0; ph < 2 && alive; ++ph) {
        const int MT = ph == 0 ? MTG : MTD;
        for (int mt = 0; mt < MT; ++mt, ++acc_it) {
          const uint32_t buf = acc_it & 1;
          if (!mbar_wait(&acc_full[buf], (acc_it >> 1) & 1, abort_flag, g.status, 75)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + ((uint32_t)(ew * 32) << 16) + buf * (2 * kBN);
          if (ph == 0) {
            // SwiGLU of the warp's 32 features for every token row, into the
            // h buffer: feature fe of row n at block fe / 64, element fe % 64
            const int fe = mt * kTileM + ew * 32 + lane;
            uint8_t* hb = smem + kOffH + (fe >> 6) * kBBytes + ((fe & 7) << 1);
            const int hc = (fe & 63) >> 3;
#pragma unroll 1
            for (int c0 = 0; c0 < kBN; c0 += 32) {
              uint32_t gv[32], uv[32];
              tmem_ld_32x32b_x32(taddr + c0, gv);
              tmem_ld_32x32b_x32(taddr + kBN + c0, uv);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int n = c0 + i;
                const float a = __uint_as_float(gv[i]);
                const float v = __fdividef(a, 1.f + __expf(-a)) * __uint_as_float(uv[i]);
                *reinterpret_cast<uint16_t*>(hb + sw128_offset(n, hc)) = to_f16_sat(v);
              }
            }
            if (mt == MT - 1) {  // h of the tile is complete: the D MMAs may read it
              fence_proxy_async_smem();
              mbar_arrive_warp(h_full);
            }
          } else {
            const int64_t tcol0 = (int64_t)mt * kTileM;
#pragma unroll 1
            for (int c0 = 0; c0 < kBN; c0 += kCH, ++chunk) {
              uint32_t v0[32];
              tmem_ld_32x32b_x32(taddr + c0, v0);
              tc_wait_ld();
              const int sb = chunk & 1;
              if (lane < kRowsPerWarp) bulk_wait_read<1>();
              named_bar_sync(2, 128);
              {
                float* S = reinterpret_cast<float*>(stage) + sb * kStage + ew * 32;
#pragma unroll
                for (int i = 0; i < kCH; ++i) S[i * kTileM + lane] = __uint_as_float(v0[i]) * s_rscale[c0 + i];
              }
              fence_proxy_async_smem();
              named_bar_sync(2, 128);
              if (lane < kRowsPerWarp) {
                const int i = ew * kRowsPerWarp + lane, n = c0 + i;
                if (n < t.rows) {
                  const int orow = s_orow[n];
                  const float* src = reinterpret_cast<const float*>(stage) + sb * kStage + i * kTileM;
                  if (orow >= 0)
                    bulk_reduce_add_f32(g.C + (int64_t)orow * d + tcol0, src, kTileM * 4);
                }
                bulk_commit();
              }
            }
          }
          tc_fence_before();
          mbar_arrive_warp(&acc_empty[buf]);
        }
      }
    }
    if (lane < kRowsPerWarp) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// Packed codes viewed as a 2-D uint32 tensor [rows][K/8]; box 32 words x 128
// rows (4 k-blocks), 128-byte swizzle.
bool make_map(CUtensorMap* tm, const uint32_t* q, int64_t rows, int K) {
  auto fn = tensor_map_encoder();
  if (!fn || !q) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 8) * 4};
  const cuuint32_t box[2] = {(cuuint32_t)(kKB / 8 * kQK), kTileM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool fused_shape_supported(int d, int f) {
  // slices of 128 rows of both projections; K of both a multiple of 8 k-blocks
  // (scale loads) and of the 4-k-block code stages; h fits its buffer
  return d % 512 == 0 && f % 512 == 0 && f <= kFusedMaxDff && d >= 512;
}

cudaError_t gemm_fused_launch(const FusedParams& p, cudaStream_t s) {
  if (!fused_shape_supported(p.d, p.f)) return cudaErrorInvalidValue;
  KParams kp;
  memset(&kp, 0, sizeof kp);
  kp.g = p;
  const int64_t E = p.n_groups;
  if (!make_map(&kp.tm[0], p.W[0].q, E * p.f, p.d) || !make_map(&kp.tm[1], p.W[1].q, E * p.f, p.d) ||
      !make_map(&kp.tm[4], p.W[2].q, E * p.d, p.f))
    return cudaErrorInvalidValue;
  if (p.X[0].q) {
    if (!make_map(&kp.tm[2], p.X[0].q, p.f, p.d) || !make_map(&kp.tm[3], p.X[1].q, p.f, p.d) ||
        !make_map(&kp.tm[5], p.X[2].q, p.d, p.f))
      return cudaErrorInvalidValue;
  } else {  // never read: no tile has the extra group
    kp.tm[2] = kp.tm[0];
    kp.tm[3] = kp.tm[1];
    kp.tm[5] = kp.tm[4];
  }
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::max(1, std::min(sms, p.max_tiles));
  gemm_fused_kernel<<<grid, kThreads, kSmem, s>>>(kp);
  return cudaGetLastError();
}

}  // namespace moe
