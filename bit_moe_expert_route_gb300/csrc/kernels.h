// Internal launch interfaces of the CUDA kernels (host side, C++).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------- routing
constexpr int kRouteTPB = 128;  // tokens per block of the top-k and scatter kernels

struct RouteParams {
  const float* logits;     // [T][E]
  const float* bias;       // [E] or null
  int T, E, k, block_n, with_shared;
  // outputs
  int32_t* ids;            // [T][k]
  float* w;                // [T][k]
  int32_t* counts;         // [E]
  int32_t* offsets;        // [E+1]
  int32_t* perm;           // [T*k]
  int32_t* inv_perm;       // [T*k]
  int32_t* row_token;      // [T*k (+T)]
  float* row_weight;       // [T*k (+T)] or null
  int32_t* block_map;      // [max_tiles][4]
  int32_t* num_tiles;      // [1]
  int max_tiles;
  // optional second block map of the same rows in tiles of block_n2 rows;
  // window2 > 0 (a multiple of kRouteTPB) orders it by token window: the
  // tiles of tokens [0, window2) of every expert, then their shared rows,
  // then the next window's (each expert's rows in a window are contiguous,
  // since the scatter keeps every expert's rows in token order)
  int32_t* block_map2;     // [max_tiles2][4] or null
  int32_t* num_tiles2;     // [1]
  int max_tiles2, block_n2, window2;
  // scratch
  int32_t* blk;            // [nblk][E]
  int32_t* status;
};

inline int route_nblk(int T) { return (T + kRouteTPB - 1) / kRouteTPB; }
// Tiles of a block map of T tokens' rows cut per token window of W tokens
// (W = 0: one window): every (window, expert) and (window, shared) piece
// ends in at most one partial tile.
inline int windowed_max_tiles(int T, int E, int k, int bn, int W, bool with_shared) {
  const int64_t nW = W > 0 ? ((int64_t)T + W - 1) / W : 1;
  const int64_t n = ((int64_t)T * k + bn - 1) / bn + nW * E +
                    (with_shared ? ((int64_t)T + bn - 1) / bn + nW - 1 : 0);
  return n > 0x3FFFFFFF ? 0x3FFFFFFF : (int)n;
}
cudaError_t route_launch(const RouteParams& p, cudaStream_t s);

// ---------------------------------------------------------------- router GEMM
// logits[t][e] = sum_k x[t][k] * Wr[k][e] and gate_logit[t] = x_t . wsg, fp32
// accumulation of exact products (the fp32 weights are split into three bf16
// planes, wsplit, rebuilt on every call). Optionally also writes
// x16 = f16(x) (saturated), the tensor-core operand copy.
struct RouterParams {
  const uint16_t* x;        // [T][d] bf16
  int T, d, E, k;
  const float* Wr;          // [d][E]
  const float* wsg;         // [d] or null (no shared expert)
  uint16_t* wsplit;         // scratch [3][router_split_rows(E, wsg != null)][d] bf16
  float* logits;            // [T][E]
  float* gate_logit;        // [T] (with wsg)
  float* row_weight;        // [T*k + T] or null: row T*k + t gets sigmoid(gate_logit[t])
  uint16_t* x16;            // [T][d] or null
  int32_t* status;
};
inline int router_split_rows(int E, bool gate) { return E + (gate ? 16 : 0); }
cudaError_t router_launch(const RouterParams& p, cudaStream_t s);

// cuTensorMapEncodeTiled from the driver (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// ---------------------------------------------------------------- small-batch decode
constexpr int kBatchMaxT = 8;  // tokens per small-batch decode call
constexpr int kBatchKS = 4;    // router K slices
struct BatchParams {
  const uint16_t* x;        // [T][d] bf16
  moe_weights_t w;
  int T, d, E, k, f, shared;
  float* part;              // [kBatchKS][T][E + 1] router partials (column E: the gate)
  float* logits;            // [T][E]
  float* gate_logit;        // [T]
  int32_t* ids;             // [T][k]
  float* wts;               // [T][k + 1]: routing weights, then the shared gate
  float* h;                 // [T][k + 1][f] fp32
  uint16_t* out;            // [T][d] bf16
  int32_t* status;
};
bool batch_shape_supported(int T, int d, int E, int k, int f);
cudaError_t decode_batch_launch(const BatchParams& p, cudaStream_t s);

// ---------------------------------------------------------------- grouped GEMM
struct GemmW4 {
  const uint32_t* q;
  const uint16_t* scale;
  const uint16_t* bias;
};

struct GemmParams {
  const uint16_t* A;        // [A_rows][K] bf16
  int64_t A_rows;
  int K;
  const int32_t* row_index; // [n_rows] or null
  int64_t n_rows;
  GemmW4 W[2];              // routed stack (W[1] = up for SwiGLU)
  GemmW4 X[2];              // extra group (index n_groups), q == null if absent
  int n_groups;
  int N;
  const int32_t* block_map;
  const int32_t* num_tiles;
  int max_tiles;
  int block_n;
  int epilogue;
  int operand_f16;          // 1: A and dequantised weights are f16; 0: bf16
  const float* row_scale;
  const int32_t* out_row;
  void* C;
  int64_t C_rows;
  int64_t ldc;
  int32_t* status;
};

cudaError_t gemm_w4_launch(const GemmParams& p, cudaStream_t s);

// Fused gate/up -> SwiGLU -> down -> weighted combine over tiles of
// kFusedBlockN rows (gemm_fused.cu): h of a tile stays in shared memory.
// f16 operands; W[0..2] = gate, up, down of the routed stack (n_groups
// experts), X[0..2] the shared expert (group n_groups; q == null if absent).
constexpr int kFusedBlockN = 64;
constexpr int kFusedMaxDff = 512;
struct FusedParams {
  const uint16_t* A;        // x16 [A_rows][d] f16
  int64_t A_rows;
  int d, f;
  const int32_t* row_index; // [n_rows]: token of row r
  int64_t n_rows;
  GemmW4 W[3];
  GemmW4 X[3];
  int n_groups;
  const int32_t* block_map; // tiles of at most kFusedBlockN rows
  const int32_t* num_tiles;
  int max_tiles;
  const float* row_scale;   // [n_rows] combine weights
  float* C;                 // [C_rows][d] fp32, added into
  int64_t C_rows;
  int32_t* status;
};
bool fused_shape_supported(int d, int f);
cudaError_t gemm_fused_launch(const FusedParams& p, cudaStream_t s);

// ---------------------------------------------------------------- elementwise
cudaError_t f32_to_bf16_launch(const float* in, uint16_t* out, int64_t n, cudaStream_t s);

// Gated DeltaNet scan (gdn.cu): bf16 q, k [T][Hk][dk], v [T][Hv][dv]; fp32
// alpha, beta [T][Hv]; fp32 state [Hv][dv][dk] in/out; fp32 out [T][Hv][dv].
struct GdnParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const float* alpha;
  const float* beta;
  int T, Hk, Hv, dk, dv;
  float* state;
  float* out;
  int state_early;  // the state may be read before waiting for the previous launch
};
bool gdn_shape_supported(int dk, int dv, int Hk, int Hv);
cudaError_t gdn_scan_launch(const GdnParams& p, cudaStream_t s);

// Batch-1 decode attention with grouped KV heads (attn.cu): bf16 q [Hq][d],
// K, V [L][Hkv][d]; fp32 partials (m, l [Hq][P], o [Hq][P][d], P = splits x 8
// warps) in a workspace; fp32 out [Hq][d].
struct AttnParams {
  const uint16_t* q;
  const uint16_t* K;
  const uint16_t* V;
  int L, Hq, Hkv, d;
  float scale;
  float* ws;      // attn_workspace_floats(...) floats; the launch carves the partials
  float* part_m;  // set by attn_decode_launch
  float* part_l;
  float* part_o;
  float* out;
};
bool attn_shape_supported(int L, int Hq, int Hkv, int d);
int attn_splits(int L, int Hkv, int slots);  // slots: blocks resident at once
size_t attn_workspace_floats(int L, int Hq, int Hkv, int d, int slots);
cudaError_t attn_decode_launch(const AttnParams& p, int sms, cudaStream_t s);

// Deterministic combine: acc[t] = sum, in slot order (routed slots, then the
// shared row when `shared`), of row_weight[row] * y[row], fp32 fused
// multiply-adds; out = bf16 RNE of acc. y [T*k (+T)][d] fp32, d % 4 == 0.
cudaError_t combine_rows_launch(const float* y, const int32_t* inv_perm, const float* row_weight,
                                int T, int k, int d, bool shared, float* acc, uint16_t* out,
                                int32_t* status, cudaStream_t s);

// ---------------------------------------------------------------- decode
struct DecodeParams {
  const uint16_t* x;        // [d]
  moe_weights_t w;
  int d, E, k, f;
  bool shared;
  uint16_t* out;            // [d]
  // workspace
  float* logits;            // [E]
  float* gate_logit;        // [1]
  int32_t* ids;             // [k]
  float* wts;               // [k]
  float* h;                 // [k+1][f]
  int32_t* status;
  // published {value, epoch} words: [kDecodeMaxSplits][E] router partials,
  // then [kDecodeMaxSplits] gate-logit partials; and h [k+1][f]
  unsigned long long* pub;
  unsigned long long* pub_h;
  uint32_t* sync;           // [0]: epoch of the last call (zero before the first call)
  // bounded waits give up after wait_ns; silent_block >= 0 (tests of the
  // timeout path only): that block publishes no router partial sums
  uint64_t wait_ns;
  int silent_block;
  // set by decode_launch
  int KS, qrow, qout, capY, capX, capS;
  uint32_t y_bytes, x_bytes, z_bytes, u_bytes;
};
constexpr int kDecodeMaxSplits = 8;  // router K splits
constexpr int kDecodeMaxExperts = 256;  // one expert per thread in the top-k
size_t decode_pub_words(int E);
// Sizes the decode kernel can run: d <= 4096 and h of every slot fits in shared memory.
bool decode_shape_supported(int d, int E, int k, int f, bool shared);
cudaError_t decode_launch(const DecodeParams& p, cudaStream_t s);
// moe_decode_gemv_w4's argument checks other than the workspace (moe_api.cu).
int decode_args_status(const uint16_t* x, const moe_weights_t* w, const moe_shape_t* shape,
                       const uint16_t* out);

}  // namespace moe
