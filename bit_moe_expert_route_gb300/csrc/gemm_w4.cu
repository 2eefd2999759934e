// Grouped GEMM with groupwise affine 4-bit weights dequantised on chip.
//
// "Fused dequantization inside the grouped GEMM": the packed weights are
// unpacked one tile at a time into on-chip memory just before the multiply,
// and the expanded weights are never written back to memory
// ("Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple
// Silicon", section "Prefill optimizations", first bullet).
//
// GB300 design (one persistent CTA per SM, warp-specialised):
//   * Swap-AB: the MMA's M side (128) is a tile of weight rows (output
//     features), the N side is a tile of up to block_n token rows; D lives in
//     tensor memory (TMEM), fp32. A tile of work is (block-map entry, 128-row
//     slice of N); the block map is read on the device, so the grid never
//     depends on the routing result.
//   * warp 0       TMA producer: packed-code tiles (128 rows x 64 codes =
//                  4 KB per projection) into a ring of shared-memory stages.
//   * warp 1       allocates TMEM and issues tcgen05.mma (one thread), with
//                  one commit per k-block to a ring of completion barriers
//                  that frees both that k-block's A stage and its token tile.
//   * warps 4-11   dequantise: two threads per weight row, 32 codes each;
//                  RNE(scale*q + bias) (f16 or bf16) goes into the A operand:
//                  in tensor memory (tcgen05.st: row = TMEM lane, two K
//                  elements per column) where it fits beside the
//                  accumulators, else the 128-byte-swizzled K-major tile in
//                  shared memory; then the packed-code stage is freed (only
//                  after its codes are consumed).
//   * warps 2-3    gather: token rows (through row_index) are copied with
//                  16-byte cp.async into the swizzled K-major B operand;
//                  rows past the tile's end are zero-filled. Without a
//                  row_index the rows are contiguous and warp 0 loads each
//                  B tile with one 128-byte-swizzled TMA copy instead.
//   * warps 12-15  epilogue: tcgen05.ld of the accumulators, then
//                  NONE (fp32 store), SWIGLU (silu(g)*u in the operand type,
//                  stored straight from registers) or COMBINE (row_scale * y
//                  staged in shared memory and added into each token's output
//                  row by one TMA bulk fp32 reduce per row, done at L2).
//   Accumulators are double buffered so the epilogue of one tile overlaps the
//   MMAs of the next (256-row gate/up tiles fill TMEM with one buffer). At
//   tiles of up to 64 rows the token tile's producer arrives on the A stage's
//   barrier, so the MMA tests one barrier per k-block. Every wait is bounded;
//   a CTA that gives up records MOE_DEV_TIMEOUT, drains what it issued, frees
//   TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kTileM = 128;      // weight rows per tile (MMA M)
constexpr int kKB = 64;          // codes per k-block (= quantisation group)
constexpr int kQBytes = kTileM * kKB / 2;   // packed codes of one k-block: 4 KB
constexpr int kABytes = kTileM * kKB * 2;   // dequantised tile: 16 KB
constexpr int kSmemBudget = 220 * 1024;

// QK = k-blocks of packed codes per TMA box (and per ring stage). 4: one box
// of 128 rows x 128 bytes (128-byte swizzle) per matrix; 1: 128 rows x 32
// bytes. The wide box moves the same bytes with a quarter of the row
// requests, which is what bounds a stream of narrow strided boxes.
template <int BN, int NMAT, int EPI, int QK>
struct Cfg {
  static constexpr int kSQ = QK == 1 ? 4 : 2;      // packed-code stages
  static constexpr int kQStage = kQBytes * QK;     // bytes per matrix per stage
  static constexpr int kCH = BN < 32 ? BN : 32;  // epilogue chunk: token columns per pass
  // Epilogue staging (COMBINE only): two buffers of kCH token rows x 128
  // fp32 outputs, plus per-row scale and output row.
  static constexpr int kEpiBytes = EPI == MOE_EPI_COMBINE ? 2 * kCH * kTileM * 4 : 0;
  static constexpr int kRowInfoBytes = EPI == MOE_EPI_COMBINE ? 2 * BN * 4 : 0;
  // Rings: packed codes (TMA), dequantised A tiles (dequant warps), token
  // tiles B (gather warps or TMA). B tiles are small, so B runs deepest: it
  // has the longest latency to cover (row gathers from L2/HBM).
  // The dequantised A operand goes to tensor memory instead of shared
  // memory where it fits next to two buffers of accumulators (NMAT x BN
  // columns each; TMEM has 512): the MMA then reads only B from shared memory
  // (the shared-memory traffic per k-block roughly halves). The gate/up GEMM
  // at block_n 128 fills TMEM with its accumulators and keeps A in shared
  // memory: a single accumulator buffer would hold every tile's MMAs behind
  // the previous tile's epilogue, which costs more than the traffic saved.
  static constexpr int kAColsStage = NMAT * (kKB / 2);
  static constexpr int kSA = 2 * NMAT * BN + 4 * kAColsStage <= 512 ? 4 : 2;
  static constexpr bool kATmem = 2 * NMAT * BN + kSA * kAColsStage <= 512;
  static constexpr int kAStage = kATmem ? 0 : NMAT * kABytes;
  static constexpr int kBBytes = BN * kKB * 2;
  static constexpr int kQRing = kSQ * NMAT * kQStage;
  // Two accumulator buffers where they fit (the epilogue of one tile then
  // overlaps the MMAs of the next); 256-row tiles of gate and up fill TMEM
  // with one.
  static constexpr int kAccBufs = 2 * NMAT * BN <= 512 ? 2 : 1;
  static constexpr int kACol = kAccBufs * NMAT * BN;  // first TMEM column of the A stages
  static constexpr int kSB0a =
      (kSmemBudget - kQRing - kEpiBytes - kRowInfoBytes - kSA * kAStage) / kBBytes;
  // a tile too wide for three token stages within the budget takes what is
  // left of the CTA's shared memory (barriers and alignment slack reserved)
  static constexpr int kSB0 =
      kSB0a >= 3 ? kSB0a
                 : (232448 - 1024 - 8 * (2 * kSQ + 2 * kSA + 2 * 8 + 5) - 16 - kQRing - kEpiBytes -
                    kRowInfoBytes - kSA * kAStage) /
                       kBBytes;
  // Tiles of up to 64 rows with A in TMEM: the token ring takes the A ring's
  // depth and its producer arrives on the A stage's barrier, so the MMA tests
  // one barrier per k-block instead of two (a test costs about 100 cycles of
  // the MMA thread, the busiest role at these sizes; taller tiles keep the
  // deeper token ring).
  static constexpr bool kMerge = kATmem && kSA >= 3 && BN <= 64;
  static constexpr int kSB = kMerge ? kSA : (kSB0 > 8 ? 8 : kSB0);
  static constexpr int kSD = kSA > kSB ? kSA : kSB;  // k-block completion barriers
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kSA * kAStage;
  static constexpr int kOffQ = kOffB + kSB * kBBytes;
  static constexpr int kOffEpi = kOffQ + kQRing;
  static constexpr int kOffRowInfo = kOffEpi + kEpiBytes;
  static constexpr int kOffBar = kOffRowInfo + kRowInfoBytes;
  static constexpr int kBarBytes = 8 * (2 * kSQ + 2 * kSA + 2 * kSB + 5) + 16;
  static constexpr int kSmem = kOffBar + kBarBytes + 1024;  // + alignment slack
  static constexpr int kTmemCols0 = kAccBufs * NMAT * BN + (kATmem ? kSA * kAColsStage : 0);
  static constexpr int kTmemCols = kTmemCols0 <= 32 ? 32 : kTmemCols0 <= 64 ? 64
                                   : kTmemCols0 <= 128 ? 128 : kTmemCols0 <= 256 ? 256 : 512;
  static_assert(kSB >= 3, "not enough shared memory for three token-tile stages");
  static_assert(kTmemCols0 <= 512, "accumulators and A stages exceed TMEM");
  static_assert(!kATmem || kACol + kSA * kAColsStage <= 512, "A stages past the end of TMEM");
  static_assert(kSmem <= 232448, "shared memory per CTA exceeded");
};

struct KParams {
  CUtensorMap tm[5];  // packed codes W[0], W[1], X[0], X[1]; [4] activations A (row_index == null)
  GemmParams g;
};

struct TileInfo {
  int group, row0, rows, mt;
  bool ok;
};

MOE_DEVINL TileInfo load_tile(const GemmParams& g, int unit, int MT) {
  TileInfo t;
  const int4 m = reinterpret_cast<const int4*>(g.block_map)[unit / MT];
  t.group = m.x;
  t.row0 = m.y;
  t.rows = m.z;
  t.mt = unit % MT;
  const bool extra = g.X[0].q != nullptr;
  t.ok = m.x >= 0 && (m.x < g.n_groups || (extra && m.x == g.n_groups)) && m.y >= 0 &&
         m.z >= 1 && m.z <= g.block_n && (int64_t)m.y + m.z <= g.n_rows;
  return t;
}

MOE_DEVINL int num_units(const GemmParams& g, int MT) {
  int nt = *g.num_tiles;
  if (nt < 0) nt = 0;
  if (nt > g.max_tiles) nt = g.max_tiles;
  return nt * MT;
}

// Dequantise one packed word (8 codes, low nibble first) into 8 bf16 values
// RNE(scale * q + bias), returned as 4 bf16x2 words in K order.
// The codes become exact bf16 integers through the bit pattern of 128 + q
// (0x4300 | q), minus 128; scale * q + bias is then one fused bf16x2 fma
// (single rounding). Codes are paired (i, i+4) by mask-and-shift and
// regrouped into (2i, 2i+1) order with byte permutes.
MOE_DEVINL uint4 dequant_word(uint32_t w, __nv_bfloat162 s2, __nv_bfloat162 b2) {
  const __nv_bfloat162 m128 = __floats2bfloat162_rn(-128.f, -128.f);
  const __nv_bfloat162 one = __floats2bfloat162_rn(1.f, 1.f);
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;  // {128+q_i, 128+q_{i+4}}
    __nv_bfloat162 q2 = __hfma2(*reinterpret_cast<const __nv_bfloat162*>(&v), one, m128);
    __nv_bfloat162 r = __hfma2(s2, q2, b2);
    p[i] = *reinterpret_cast<uint32_t*>(&r);
  }
  // p[i] = {w_i, w_{i+4}}; want {w0,w1},{w2,w3},{w4,w5},{w6,w7}
  uint4 o;
  o.x = __byte_perm(p[0], p[1], 0x5410);
  o.y = __byte_perm(p[2], p[3], 0x5410);
  o.z = __byte_perm(p[0], p[1], 0x7632);
  o.w = __byte_perm(p[2], p[3], 0x7632);
  return o;
}

// Same, into f16: 0x6400 | q is 1024 + q exactly; minus 1024 gives q; then
// RNE_f16(scale * q + bias) with one fused f16x2 fma.
MOE_DEVINL uint4 dequant_word_f16(uint32_t w, __half2 s2, __half2 b2) {
  const __half2 m1024 = __floats2half2_rn(-1024.f, -1024.f);
  const __half2 one = __floats2half2_rn(1.f, 1.f);
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;  // {1024+q_i, 1024+q_{i+4}}
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

// bf16 bit pattern -> operand-format pair {v, v}
template <bool F16>
MOE_DEVINL uint32_t splat_operand(uint16_t bf16_bits) {
  if constexpr (F16) {
    const __half h = __float2half_rn(__uint_as_float((uint32_t)bf16_bits << 16));
    const uint16_t hb = *reinterpret_cast<const uint16_t*>(&h);
    return (uint32_t)hb * 0x10001u;
  } else {
    return (uint32_t)bf16_bits * 0x10001u;
  }
}

// fp32 -> operand-format bits (RNE); f16 saturates to the largest finite value.
template <bool F16>
MOE_DEVINL uint16_t to_operand(float v) {
  if constexpr (F16) {
    const __half h = __float2half_rn(fminf(fmaxf(v, -65504.f), 65504.f));
    return *reinterpret_cast<const uint16_t*>(&h);
  } else {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<const uint16_t*>(&b);
  }
}

template <int BN, int NMAT, int EPI, bool F16, int QK>
__global__ void __launch_bounds__(kThreads, 1) gemm_w4_kernel(const __grid_constant__ KParams kp) {
  using C = Cfg<BN, NMAT, EPI, QK>;
  constexpr int kSQ = C::kSQ;
  const GemmParams& g = kp.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + kSQ;
  uint64_t* a_full = q_empty + kSQ;
  uint64_t* b_full = a_full + C::kSA;
  // done[i % kSD] completes when the MMAs of k-block i have read their A and
  // B stages: one commit per k-block frees both (the A producer at k-block i
  // waits for k-block i - kSA, the B producer for i - kSB; the MMA cannot run
  // kSD k-blocks past either, so no barrier is two phases ahead of a waiter)
  uint64_t* done = b_full + C::kSB;
  uint64_t* b_ready = C::kMerge ? a_full : b_full;  // where token tiles are signalled
  uint64_t* acc_full = done + C::kSD;      // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* drain = acc_empty + 2;         // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int MT = g.N / kTileM;
  const int KB = g.K / kKB;
  const bool b_by_tma = g.row_index == nullptr;  // contiguous rows: one TMA tile per k-block

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 8);    // dequant warps
    }
    for (int i = 0; i < C::kSA; ++i)  // dequant warps (+ the token tile's producer when merged)
      mbar_init(&a_full[i], 8 + (C::kMerge ? (b_by_tma ? 1 : 2) : 0));
    for (int i = 0; i < C::kSB; ++i) {
      mbar_init(&b_full[i], b_by_tma ? 1 : 2);  // TMA, or the gather warps
    }
    for (int i = 0; i < C::kSD; ++i) mbar_init(&done[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);  // epilogue warps
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&kp.tm[0]);
    if (NMAT == 2) tma_prefetch_desc(&kp.tm[1]);
    if (g.X[0].q) {
      tma_prefetch_desc(&kp.tm[2]);
      if (NMAT == 2) tma_prefetch_desc(&kp.tm[3]);
    }
    if (b_by_tma) tma_prefetch_desc(&kp.tm[4]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int units = num_units(g, MT);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_last();
      uint32_t it = 0, qit = 0;
      bool alive = true;
      for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
        const TileInfo t = load_tile(g, u, MT);
        if (!t.ok) {
          report(g.status, MOE_DEV_BAD_TILE, 31, u / MT);
          continue;
        }
        const bool ext = t.group == g.n_groups;
        const int row = (ext ? 0 : t.group * g.N) + t.mt * kTileM;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          if (kb % QK == 0) {
            const int s = qit % kSQ;
            if (!mbar_wait(&q_empty[s], ((qit / kSQ) & 1) ^ 1, abort_flag, g.status, 1)) {
              alive = false;
              break;
            }
            mbar_arrive_expect_tx(&q_full[s], NMAT * C::kQStage);
#pragma unroll
            for (int j = 0; j < NMAT; ++j)
              tma_load_2d(smem + C::kOffQ + (s * NMAT + j) * C::kQStage, &kp.tm[(ext ? 2 : 0) + j],
                          kb * (kKB / 8), row, &q_full[s], policy);
            ++qit;
          }
          if (b_by_tma) {
            const int sb = it % C::kSB;
            if (it >= (uint32_t)C::kSB &&
                !mbar_wait(&done[(it - C::kSB) % C::kSD], ((it - C::kSB) / C::kSD) & 1, abort_flag, g.status, 10)) {
              alive = false;
              ++it;
              break;
            }
            mbar_arrive_expect_tx(&b_ready[sb], C::kBBytes);
            tma_load_2d(smem + C::kOffB + sb * C::kBBytes, &kp.tm[4], kb * kKB, t.row0, &b_ready[sb],
                        policy);
          }
        }
      }
      // drain: every issued load must land before the CTA exits
      for (uint32_t j = qit > (uint32_t)kSQ ? qit - kSQ : 0; j < qit; ++j)
        mbar_wait(&q_full[j % kSQ], (j / kSQ) & 1, abort_flag, g.status, 2);
      const uint32_t n_issued = it;
      if (b_by_tma)
        for (uint32_t j = n_issued > (uint32_t)C::kSB ? n_issued - C::kSB : 0; j < n_issued; ++j)
          mbar_wait(&b_ready[j % C::kSB], (j / C::kSB) & 1, abort_flag, g.status, 2);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = F16 ? idesc_f16_f32(kTileM, BN) : idesc_bf16_f32(kTileM, BN);
      uint32_t it = 0, acc_it = 0;
      bool alive = true;
      for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
        const TileInfo t = load_tile(g, u, MT);
        if (!t.ok) continue;
        const uint32_t buf = acc_it % C::kAccBufs;
        if (!mbar_wait(&acc_empty[buf], ((acc_it / C::kAccBufs) & 1) ^ 1, abort_flag, g.status, 3))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * (NMAT * BN);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % C::kSA, sb = it % C::kSB;
          if (!mbar_wait(&a_full[s], (it / C::kSA) & 1, abort_flag, g.status, 4) ||
              (!C::kMerge && !mbar_wait(&b_full[sb], (it / C::kSB) & 1, abort_flag, g.status, 4))) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t b_addr = smem_u32(smem + C::kOffB + sb * C::kBBytes);
          if constexpr (C::kATmem) {
#pragma unroll
            for (int j = 0; j < NMAT; ++j) {
              const uint32_t a_tmem = tmem_base + C::kACol + s * C::kAColsStage + j * (kKB / 2);
#pragma unroll
              for (int kk = 0; kk < kKB / 16; ++kk)
                tc_mma_ts(d_tmem + j * BN, a_tmem + kk * 8, smem_desc_sw128(b_addr + kk * 32), idesc,
                          (kb | kk) != 0);
            }
          } else {
#pragma unroll
            for (int j = 0; j < NMAT; ++j) {
              const uint32_t a_addr = smem_u32(smem + C::kOffA + (s * NMAT + j) * kABytes);
#pragma unroll
              for (int kk = 0; kk < kKB / 16; ++kk)
                tc_mma_bf16(d_tmem + j * BN, smem_desc_sw128(a_addr + kk * 32),
                            smem_desc_sw128(b_addr + kk * 32), idesc, (kb | kk) != 0);
            }
          }
          tc_commit(&done[it % C::kSD]);
        }
        if (!alive) break;
        tc_commit(&acc_full[buf]);
        ++acc_it;
      }
      // drain: all issued MMAs complete before TMEM is freed
      tc_commit(drain);
      mbar_wait(drain, 0, abort_flag, g.status, 5);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ dequantise
    const int dt = threadIdx.x - 128;
    const int m = dt & (kTileM - 1);  // weight row inside the tile
    const int half = dt >> 7;         // codes half*32 .. half*32+31 of each k-block
    uint32_t it = 0, qit = 0;
    bool alive = true;
    // One k-block: wait for its packed codes and a free A stage, write the
    // operand tile, signal the MMA; release the code stage after its last
    // k-block (only once its codes are consumed: releasing right after the
    // shared-memory loads let the next TMA refill land before those loads
    // had returned their data).
    auto step = [&](int kb, const uint32_t (&s2)[NMAT], const uint32_t (&b2)[NMAT]) -> bool {
      const int sq = qit % kSQ;
      if (kb % QK == 0 && !mbar_wait(&q_full[sq], (qit / kSQ) & 1, abort_flag, g.status, 6))
        return false;
      // this thread's 16 bytes of codes: row m, k-block kb % QK, half `half`
      // (QK = 4: 128-byte rows, 16-byte chunk index XOR (m % 8) as TMA wrote them)
      const int qoff = QK == 1 ? m * 32 + half * 16
                               : m * 128 + ((((kb % QK) * 2 + half) ^ (m & 7)) << 4);
      uint4 qw[NMAT];
#pragma unroll
      for (int j = 0; j < NMAT; ++j)
        qw[j] = *reinterpret_cast<const uint4*>(smem + C::kOffQ + (sq * NMAT + j) * C::kQStage + qoff);
      const int sa = it % C::kSA;
      if (it >= (uint32_t)C::kSA &&
          !mbar_wait(&done[(it - C::kSA) % C::kSD], ((it - C::kSA) / C::kSD) & 1, abort_flag, g.status, 7))
        return false;
#pragma unroll
      for (int j = 0; j < NMAT; ++j) {
        const uint32_t words[4] = {qw[j].x, qw[j].y, qw[j].z, qw[j].w};
        uint32_t r[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 o;
          if constexpr (F16)
            o = dequant_word_f16(words[c], *reinterpret_cast<const __half2*>(&s2[j]),
                                 *reinterpret_cast<const __half2*>(&b2[j]));
          else
            o = dequant_word(words[c], *reinterpret_cast<const __nv_bfloat162*>(&s2[j]),
                             *reinterpret_cast<const __nv_bfloat162*>(&b2[j]));
          if constexpr (C::kATmem) {
            r[4 * c] = o.x;
            r[4 * c + 1] = o.y;
            r[4 * c + 2] = o.z;
            r[4 * c + 3] = o.w;
          } else {
            uint8_t* a_tile = smem + C::kOffA + (sa * NMAT + j) * kABytes;
            *reinterpret_cast<uint4*>(a_tile + sw128_offset(m, half * 4 + c)) = o;
          }
        }
        if constexpr (C::kATmem)  // row m = lane (quarter warp % 4), columns half*16 .. +15 of the stage
          tmem_st_32x32b_x16(tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + C::kACol +
                                 sa * C::kAColsStage + j * (kKB / 2) + half * 16, r);
      }
      if constexpr (C::kATmem) {
        tc_wait_st();
        tc_fence_before();
      } else {
        fence_proxy_async_smem();
      }
      mbar_arrive_warp(&a_full[sa]);
      if (kb % QK == QK - 1) {
        mbar_arrive_warp(&q_empty[sq]);
        ++qit;
      }
      ++it;
      return true;
    };
    const bool vec = (KB & 7) == 0;  // scale/bias rows load 8 groups (16 bytes) at a time
    for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
      const TileInfo t = load_tile(g, u, MT);
      if (!t.ok) continue;
      const bool ext = t.group == g.n_groups;
      const int64_t row = (ext ? 0 : (int64_t)t.group * g.N) + t.mt * kTileM + m;
      const uint16_t* sc[NMAT];
      const uint16_t* bi[NMAT];
#pragma unroll
      for (int j = 0; j < NMAT; ++j) {
        const GemmW4& w = ext ? g.X[j] : g.W[j];
        sc[j] = w.scale + row * KB;
        bi[j] = w.bias + row * KB;
      }
      if (vec) {
        // 8 k-blocks per scale/bias load, unrolled so every word index is
        // static (a runtime index would put the words in local memory); the
        // next batch is loaded one batch ahead of use
        uint4 s_nxt[NMAT], b_nxt[NMAT];
#pragma unroll
        for (int j = 0; j < NMAT; ++j) {
          s_nxt[j] = __ldg(reinterpret_cast<const uint4*>(sc[j]));
          b_nxt[j] = __ldg(reinterpret_cast<const uint4*>(bi[j]));
        }
        for (int kb0 = 0; kb0 < KB && alive; kb0 += 8) {
          uint4 s_cur[NMAT], b_cur[NMAT];
#pragma unroll
          for (int j = 0; j < NMAT; ++j) {
            s_cur[j] = s_nxt[j];
            b_cur[j] = b_nxt[j];
            if (kb0 + 8 < KB) {
              s_nxt[j] = __ldg(reinterpret_cast<const uint4*>(sc[j]) + (kb0 >> 3) + 1);
              b_nxt[j] = __ldg(reinterpret_cast<const uint4*>(bi[j]) + (kb0 >> 3) + 1);
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t s2[NMAT], b2[NMAT];
#pragma unroll
            for (int j = 0; j < NMAT; ++j) {
              const uint32_t sw = i < 2 ? s_cur[j].x : i < 4 ? s_cur[j].y : i < 6 ? s_cur[j].z : s_cur[j].w;
              const uint32_t bw = i < 2 ? b_cur[j].x : i < 4 ? b_cur[j].y : i < 6 ? b_cur[j].z : b_cur[j].w;
              s2[j] = splat_operand<F16>((uint16_t)(sw >> ((i & 1) * 16)));
              b2[j] = splat_operand<F16>((uint16_t)(bw >> ((i & 1) * 16)));
            }
            if (!step(kb0 + i, s2, b2)) {
              alive = false;
              break;
            }
          }
        }
      } else {
        for (int kb = 0; kb < KB; ++kb) {
          uint32_t s2[NMAT], b2[NMAT];
#pragma unroll
          for (int j = 0; j < NMAT; ++j) {
            s2[j] = splat_operand<F16>(__ldg(sc[j] + kb));
            b2[j] = splat_operand<F16>(__ldg(bi[j] + kb));
          }
          if (!step(kb, s2, b2)) {
            alive = false;
            break;
          }
        }
      }
    }
  } else if ((warp == 2 || warp == 3) && !b_by_tma) {
    // ------------------------------------------------------------ gather B
    // 16-byte cp.async per (row, chunk) into the swizzled tile. A thread
    // signals a step only once its copies have landed (wait_group, then the
    // proxy fence, then the arrive), deferred by kD steps so that kD + 1
    // steps of gathers are in flight at once. The arrival of step i comes
    // after the issue of step i + kD, which waits for the MMA of step
    // i + kD - kSB to release its stage: with kD = kSB - 2 that is the MMA of
    // step i - 2, so the MMA of step i - 1 still runs while step i is being
    // signalled (kD = kSB - 1 would make every MMA wait for the previous
    // one to finish and the copies to be signalled: MMAs one at a time).
    constexpr int kD = C::kSB - 2;
    constexpr int kRowsPerThread = (BN * 8 + 63) / 64;  // 16-byte chunks per thread
    const int gt = threadIdx.x - 64;
    const int c = gt & 7;           // chunk of the 128-byte row slice
    const int n_first = gt >> 3;    // first row handled; rows n_first + 8*i
    uint32_t it = 0, arrived = 0;
    bool alive = true;
    for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
      const TileInfo t = load_tile(g, u, MT);
      if (!t.ok) continue;
      int64_t src_row[kRowsPerThread];
      bool valid[kRowsPerThread];
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int n = n_first + 8 * i;
        valid[i] = n < BN && n < t.rows;
        src_row[i] = 0;
        if (valid[i]) {
          const int64_t r = t.row0 + n;
          const int64_t a = (int64_t)g.row_index[r];
          if (a < 0 || a >= g.A_rows) {
            report(g.status, MOE_DEV_BAD_ROW, 32, (int)r);
            valid[i] = false;
          } else {
            src_row[i] = a;
          }
        }
      }
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int sb = it % C::kSB;
        if (it >= (uint32_t)C::kSB &&
            !mbar_wait(&done[(it - C::kSB) % C::kSD], ((it - C::kSB) / C::kSD) & 1, abort_flag, g.status, 8)) {
          alive = false;
          break;
        }
        const uint32_t b_tile = smem_u32(smem + C::kOffB + sb * C::kBBytes);
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) {
          const int n = n_first + 8 * i;
          if (n < BN) {
            const uint16_t* src = g.A + src_row[i] * g.K + kb * kKB + c * 8;
            cp_async_16(b_tile + sw128_offset(n, c), src, valid[i] ? 16u : 0u);
          }
        }
        cp_async_commit();
        if (it + 1 - arrived > (uint32_t)kD) {  // step `arrived` is kD steps old: complete it
          cp_async_wait<kD>();
          fence_proxy_async_smem();
          mbar_arrive_warp(&b_ready[arrived % C::kSB]);
          ++arrived;
        }
      }
      // End of the tile: signal its last steps as soon as they land. Deferring
      // them behind the next tile's first issues would hold the MMA until the
      // next tile's block-map entry and row indices have come back from memory
      // (several thousand cycles per tile, seen in per-role timestamps).
      cp_async_wait<0>();
      fence_proxy_async_smem();
      for (; arrived < it; ++arrived) mbar_arrive_warp(&b_ready[arrived % C::kSB]);
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (; arrived < it; ++arrived) mbar_arrive_warp(&b_ready[arrived % C::kSB]);
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogue
    // TMEM -> registers -> (NONE) direct fp32 stores; (SWIGLU) silu(g)*u in
    // the operand type, stored directly (64 contiguous bytes per warp and
    // token row); (COMBINE) a staging tile of CH token rows x the tile's 128
    // outputs shared by the 4 epilogue warps (each fills its 32 outputs),
    // double buffered, each row added into the token's fp32 output row at L2
    // by one TMA bulk reduce (the weighted combine of the routed experts and
    // the shared one). Whole rows keep the number of bulk reductions at one
    // per token row (each has a fixed cost in the copy engine and at L2).
    const int ew = warp & 3;             // TMEM lane quarter = the warp's 32 outputs
    const int et = threadIdx.x - 384;    // 0..127 inside the epilogue group
    constexpr int CH = C::kCH;
    constexpr int kRowsPerWarp = CH / 4;  // token rows each warp writes back per chunk
    constexpr int kStage = CH * kTileM;   // elements per staging buffer
    float* s_rscale = reinterpret_cast<float*>(smem + C::kOffRowInfo);
    int* s_orow = reinterpret_cast<int*>(s_rscale + BN);
    uint8_t* stage = smem + C::kOffEpi;
    uint32_t acc_it = 0, chunk = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const TileInfo t = load_tile(g, u, MT);
      if (!t.ok) continue;
      const uint32_t buf = acc_it % C::kAccBufs;
      if (!mbar_wait(&acc_full[buf], (acc_it / C::kAccBufs) & 1, abort_flag, g.status, 9)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(ew * 32) << 16) + buf * (NMAT * BN);
      const int64_t tcol0 = (int64_t)t.mt * kTileM;  // the tile's first output
      if constexpr (EPI == MOE_EPI_COMBINE) {
        named_bar_sync(1, 128);  // every epilogue warp is done with the previous tile's rows
        for (int n = et; n < t.rows; n += 128) {
          const int64_t r = (int64_t)t.row0 + n;
          int orow = __ldg(g.out_row + r);
          if (orow < 0 || orow >= g.C_rows) {
            report(g.status, MOE_DEV_BAD_ROW, 33, (int)r);
            orow = -1;
          }
          s_orow[n] = orow;
          s_rscale[n] = __ldg(g.row_scale + r);
        }
        named_bar_sync(1, 128);
      }
      const int64_t col0 = tcol0 + ew * 32;  // this warp's first output
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += CH, ++chunk) {
        uint32_t v0[32], v1[32];
        if constexpr (CH == 32) {
          tmem_ld_32x32b_x32(taddr + c0, v0);
          if (NMAT == 2) tmem_ld_32x32b_x32(taddr + BN + c0, v1);
        } else {
          uint32_t h0[16], h1[16];
          tmem_ld_32x32b_x16(taddr + c0, h0);
          if (NMAT == 2) tmem_ld_32x32b_x16(taddr + BN + c0, h1);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            v0[i] = h0[i];
            v1[i] = NMAT == 2 ? h1[i] : 0u;
          }
        }
        tc_wait_ld();
        if constexpr (EPI == MOE_EPI_NONE) {
#pragma unroll
          for (int i = 0; i < CH; ++i) {
            const int n = c0 + i;
            if (n >= t.rows) break;
            static_cast<float*>(g.C)[((int64_t)t.row0 + n) * g.ldc + col0 + lane] =
                __uint_as_float(v0[i]);
          }
        } else if constexpr (EPI == MOE_EPI_SWIGLU) {
          // straight from registers: per token row, the warp's 32 outputs are
          // 64 contiguous bytes of h (no staging, barriers or bulk copies).
          // Every column is computed first (columns past the tile's rows are
          // never stored, whatever they hold), so the chunk's exp/reciprocal
          // chains overlap instead of running one token row at a time behind
          // a row-count branch.
          uint16_t* hrow = static_cast<uint16_t*>(g.C) + (int64_t)t.row0 * g.ldc + col0 + lane;
#pragma unroll
          for (int i = 0; i < CH; ++i) {
            const float a = __uint_as_float(v0[i]);
            v0[i] = to_operand<F16>(__fdividef(a, 1.f + __expf(-a)) * __uint_as_float(v1[i]));
          }
          const int nv = t.rows - c0;  // token rows of this chunk inside the tile
#pragma unroll
          for (int i = 0; i < CH; ++i)
            if (i < nv) hrow[(int64_t)(c0 + i) * g.ldc] = (uint16_t)v0[i];
        } else {
          const int sb = chunk & 1;
          // the copies issued from this buffer two chunks ago have read it
          if (lane < kRowsPerWarp) bulk_wait_read<1>();
          named_bar_sync(2, 128);
          {
            float* S = reinterpret_cast<float*>(stage) + sb * kStage + ew * 32;
#pragma unroll
            for (int i = 0; i < CH; ++i) S[i * kTileM + lane] = __uint_as_float(v0[i]) * s_rscale[c0 + i];
          }
          fence_proxy_async_smem();
          named_bar_sync(2, 128);  // the chunk's rows are complete
          if (lane < kRowsPerWarp) {
            const int i = ew * kRowsPerWarp + lane, n = c0 + i;
            if (n < t.rows) {
              const int orow = s_orow[n];
              const float* src = reinterpret_cast<const float*>(stage) + sb * kStage + i * kTileM;
              if (orow >= 0)
                bulk_reduce_add_f32(static_cast<float*>(g.C) + (int64_t)orow * g.ldc + tcol0, src,
                                    kTileM * 4);
            }
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      mbar_arrive_warp(&acc_empty[buf]);
      ++acc_it;
    }
    if (lane < kRowsPerWarp) bulk_wait_all();  // every bulk copy has landed before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() { return tensor_map_encoder(); }

// Packed codes viewed as a 2-D uint32 tensor [rows][K/8]; box 8 words x 128 rows.
bool make_q_map(CUtensorMap* tm, const uint32_t* q, int64_t rows, int K, int qk) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 8) * 4};
  const cuuint32_t box[2] = {(cuuint32_t)(kKB / 8 * qk), kTileM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            qk == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activations viewed as a 2-D 16-bit tensor [rows][K]; box 64 x box_rows,
// 128-byte swizzle: exactly the K-major B operand tile the MMA reads.
bool make_act_map(CUtensorMap* tm, const uint16_t* A, int64_t rows, int K, int box_rows) {
  auto fn = get_encode_fn();
  if (!fn || rows < 1) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {kKB, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(A), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int NMAT, int EPI, bool F16, int QK>
cudaError_t launch_t(const KParams& kp, cudaStream_t s) {
  using C = Cfg<BN, NMAT, EPI, QK>;
  auto kern = gemm_w4_kernel<BN, NMAT, EPI, F16, QK>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t max_units = (int64_t)kp.g.max_tiles * (kp.g.N / kTileM);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, max_units));
  kern<<<grid, kThreads, C::kSmem, s>>>(kp);
  return cudaGetLastError();
}

template <int NMAT, int EPI, bool F16, int QK>
cudaError_t launch_bn(const KParams& kp, cudaStream_t s) {
  switch (kp.g.block_n) {
    case 16: return launch_t<16, NMAT, EPI, F16, QK>(kp, s);
    case 32: return launch_t<32, NMAT, EPI, F16, QK>(kp, s);
    case 64: return launch_t<64, NMAT, EPI, F16, QK>(kp, s);
    case 128: return launch_t<128, NMAT, EPI, F16, QK>(kp, s);
    case 256: return launch_t<256, NMAT, EPI, F16, QK>(kp, s);
    default: return cudaErrorInvalidValue;
  }
}

int q_kblocks_per_stage(int K) { return (K / kKB) % 4 == 0 ? 4 : 1; }

template <bool F16, int QK>
cudaError_t launch_epi(const KParams& kp, cudaStream_t s) {
  switch (kp.g.epilogue) {
    case MOE_EPI_NONE: return launch_bn<1, MOE_EPI_NONE, F16, QK>(kp, s);
    case MOE_EPI_SWIGLU: return launch_bn<2, MOE_EPI_SWIGLU, F16, QK>(kp, s);
    case MOE_EPI_COMBINE: return launch_bn<1, MOE_EPI_COMBINE, F16, QK>(kp, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

cudaError_t gemm_w4_launch(const GemmParams& p, cudaStream_t s) {
  KParams kp;
  memset(&kp, 0, sizeof kp);
  kp.g = p;
  const int nmat = p.epilogue == MOE_EPI_SWIGLU ? 2 : 1;
  const int qk = q_kblocks_per_stage(p.K);
  for (int j = 0; j < nmat; ++j) {
    if (!make_q_map(&kp.tm[j], p.W[j].q, (int64_t)p.n_groups * p.N, p.K, qk))
      return cudaErrorInvalidValue;
    if (p.X[0].q && !make_q_map(&kp.tm[2 + j], p.X[j].q, p.N, p.K, qk)) return cudaErrorInvalidValue;
  }
  if (!p.row_index && !make_act_map(&kp.tm[4], p.A, p.A_rows, p.K, p.block_n))
    return cudaErrorInvalidValue;
  if (qk == 4) return p.operand_f16 ? launch_epi<true, 4>(kp, s) : launch_epi<false, 4>(kp, s);
  return p.operand_f16 ? launch_epi<true, 1>(kp, s) : launch_epi<false, 1>(kp, s);
}

}  // namespace moe
