// C ABI of libmoe_gb300: argument validation, workspace layouts and the
// launch sequences of the routing, grouped-GEMM, whole-layer and decode
// entry points declared in include/moe.h.
#include <atomic>
#include <algorithm>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "gdn.h"
#include "attn.h"

namespace {

using moe::kStatusWords;

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  return (major == 10 && minor == 3) ? MOE_OK : MOE_ERR_ARCH;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  (void)cudaGetLastError();  // clear a non-sticky launch error
  return MOE_ERR_CUDA;
}

bool valid_block_n(int bn) {
  return bn == 16 || bn == 32 || bn == 64 || bn == 128 || bn == 256;
}

// Sequential workspace carve-out.
struct Carve {
  uint8_t* base;
  size_t off = 0;
  explicit Carve(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <class T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += align_up(count * sizeof(T));
    return p;
  }
};

struct RouteWs {
  int32_t* status;
  int32_t* blk;
  size_t bytes;
};

RouteWs route_ws(void* ws, int T, int E) {
  Carve c(ws);
  RouteWs r;
  r.status = c.take<int32_t>(kStatusWords);
  r.blk = c.take<int32_t>((size_t)moe::route_nblk(T) * E);
  r.bytes = c.off;
  return r;
}

// Token window of the down projection's block map under MOE_FWD_DOWN_WINDOWS
// (a multiple of the routing kernels' 128-token blocks): 8192 tokens' fp32
// output rows are 64 MB, about half of L2.
constexpr int kDownWindow = 8192;

// moe_debug_decode_fault's settings (process-wide; tests of the timeout path)
std::atomic<uint64_t> g_decode_wait_ns{0};
std::atomic<int> g_decode_silent_block{-1};

bool shape_ok(const moe_shape_t* s, bool need_tokens) {
  if (!s) return false;
  if (s->T < 0 || (need_tokens && s->T < 1)) return false;
  if (s->group != 64) return false;
  if (s->d_model < 128 || s->d_model % 128) return false;
  if (s->d_ff < 128 || s->d_ff % 128) return false;
  if (s->n_experts < 1 || s->n_experts > 1024 || s->n_experts % 8) return false;
  if (s->top_k < 1 || s->top_k > 32 || s->top_k > s->n_experts) return false;
  if ((int64_t)s->T * (s->top_k + 1) >= (int64_t)1 << 30) return false;
  return true;
}

struct FwdWs {
  moe_forward_views_t v;
  int32_t* blk;  // routing scratch [route_nblk(T)][E]
  uint16_t* wsplit;  // router weights as three bf16 planes [3][Ep][d]
  size_t bytes;
};

FwdWs forward_ws(void* ws, const moe_shape_t* s, int bn, int flags) {
  const int T = s->T, E = s->n_experts, k = s->top_k;
  const int64_t rows = (int64_t)T * k + T;
  Carve c(ws);
  FwdWs r;
  memset(&r.v, 0, sizeof r.v);
  r.v.max_tiles = moe_max_tiles(T, E, k, bn, 1);
  r.v.block_n = bn;
  r.v.status = c.take<int32_t>(kStatusWords);
  r.v.logits = c.take<float>((size_t)T * E);
  r.v.gate_logit = c.take<float>(T);
  r.v.topk_ids = c.take<int32_t>((size_t)T * k);
  r.v.topk_w = c.take<float>((size_t)T * k);
  r.v.counts = c.take<int32_t>(E);
  r.v.offsets = c.take<int32_t>(E + 1);
  r.v.perm = c.take<int32_t>((size_t)T * k);
  r.v.inv_perm = c.take<int32_t>((size_t)T * k);
  r.v.row_token = c.take<int32_t>(rows);
  r.v.row_weight = c.take<float>(rows);
  r.v.block_map = c.take<int32_t>((size_t)r.v.max_tiles * 4);
  r.v.num_tiles = c.take<int32_t>(1);
  r.blk = c.take<int32_t>((size_t)moe::route_nblk(T) * E);
  r.wsplit = c.take<uint16_t>((size_t)3 * moe::router_split_rows(E, true) * s->d_model);
  // 256-row tiles pay off once the experts average 256 rows or more: each
  // tile's weights are dequantised once for twice the rows (below that they
  // are mostly padding, and the combine epilogue's per-row copies dominate);
  // gate/up joins at 512 rows per expert (see moe_forward)
  r.v.down_block_n = bn == 128 && (int64_t)T * k >= (int64_t)256 * E ? 256 : bn;
  // MOE_FWD_DOWN_WINDOWS, above kDownWindow tokens: the down map ordered by
  // token window (see RouteParams::window2)
  r.v.down_window =
      (flags & MOE_FWD_DOWN_WINDOWS) && r.v.down_block_n != bn && T > kDownWindow ? kDownWindow : 0;
  if (r.v.down_block_n != bn) {
    r.v.down_max_tiles = moe::windowed_max_tiles(T, E, k, r.v.down_block_n, r.v.down_window, true);
    r.v.down_block_map = c.take<int32_t>((size_t)r.v.down_max_tiles * 4);
    r.v.down_num_tiles = c.take<int32_t>(1);
  } else {  // one map serves both projections
    r.v.down_max_tiles = r.v.max_tiles;
    r.v.down_block_map = r.v.block_map;
    r.v.down_num_tiles = r.v.num_tiles;
  }
  r.v.x16 = c.take<uint16_t>((size_t)T * s->d_model);
  r.v.h = c.take<uint16_t>((size_t)rows * s->d_ff);
  r.v.out_acc = c.take<float>((size_t)T * s->d_model);
  // deterministic mode: the down projection's unweighted output rows
  r.v.y = (flags & MOE_FWD_DETERMINISTIC) ? c.take<float>((size_t)rows * s->d_model) : nullptr;
  r.bytes = c.off;
  return r;
}

bool flags_ok(int flags) {
  if (flags & ~(MOE_FWD_DETERMINISTIC | MOE_FWD_DOWN_WINDOWS | MOE_FWD_FUSED)) return false;
  return !((flags & MOE_FWD_FUSED) && (flags & (MOE_FWD_DETERMINISTIC | MOE_FWD_DOWN_WINDOWS)));
}

// The row-tile height moe_forward_ex uses: the caller's, else the fused
// chain's own, else the one moe_pick_block_n picks; 0 if unsupported.
int forward_block_n(const moe_shape_t* s, int block_n, int flags) {
  if (flags & MOE_FWD_FUSED) {
    if (block_n == 0) block_n = moe::kFusedBlockN;
    return block_n == moe::kFusedBlockN && moe::fused_shape_supported(s->d_model, s->d_ff) ? block_n : 0;
  }
  if (block_n == 0) block_n = moe_pick_block_n(s->T, s->n_experts, s->top_k);
  return valid_block_n(block_n) && block_n != 256 ? block_n : 0;  // gate/up: 128 rows at most
}

struct DecWs {
  moe_decode_views_t v;
  uint32_t* sync;                // the decode kernel's call epoch (zero before the first call)
  unsigned long long* pub;       // published router and gate-logit partial sums
  unsigned long long* pub_h;     // published h
  size_t bytes;
};

DecWs decode_ws(void* ws, const moe_shape_t* s) {
  const int E = s->n_experts, k = s->top_k;
  Carve c(ws);
  DecWs r;
  memset(&r.v, 0, sizeof r.v);
  r.v.status = c.take<int32_t>(kStatusWords);
  r.sync = c.take<uint32_t>(4);
  r.v.logits = c.take<float>(E);
  r.v.gate_logit = c.take<float>(1);
  r.v.topk_ids = c.take<int32_t>(k);
  r.v.topk_w = c.take<float>(k + 1);
  r.v.h = c.take<float>((size_t)(k + 1) * s->d_ff);
  r.pub = c.take<unsigned long long>(moe::decode_pub_words(E));
  r.pub_h = c.take<unsigned long long>((size_t)(k + 1) * s->d_ff);
  r.bytes = c.off;
  return r;
}

struct BatchWs {
  moe_decode_views_t v;
  float* wts;   // [T][k + 1]
  float* part;  // router partials [kBatchKS][T][E + 1]
  size_t bytes;
};

BatchWs batch_ws(void* ws, const moe_shape_t* s) {
  const int T = s->T, E = s->n_experts, k = s->top_k;
  Carve c(ws);
  BatchWs r;
  memset(&r.v, 0, sizeof r.v);
  r.v.status = c.take<int32_t>(kStatusWords);
  r.v.logits = c.take<float>((size_t)T * E);
  r.v.gate_logit = c.take<float>(T);
  r.v.topk_ids = c.take<int32_t>((size_t)T * k);
  r.wts = c.take<float>((size_t)T * (k + 1));
  r.v.topk_w = r.wts;
  r.v.h = c.take<float>((size_t)T * (k + 1) * s->d_ff);
  r.part = c.take<float>((size_t)moe::kBatchKS * T * (E + 1));
  r.bytes = c.off;
  return r;
}

bool batch_shape_ok(const moe_shape_t* s) {
  return shape_ok(s, true) && moe::batch_shape_supported(s->T, s->d_model, s->n_experts, s->top_k,
                                                          s->d_ff);
}


bool w4_ok(const moe_w4_t& w) {
  return w.q && w.scale && w.bias && aligned(w.q, 16) && aligned(w.scale, 16) &&
         aligned(w.bias, 16);
}

int check_weights(const moe_weights_t* w, const moe_shape_t* s) {
  if (!w || !w->router) return MOE_ERR_NULL;
  const moe_w4_t* all[6] = {&w->gate, &w->up, &w->down, &w->sh_gate, &w->sh_up, &w->sh_down};
  const int n = w->shared_gate ? 6 : 3;
  for (int i = 0; i < n; ++i) {
    if (!all[i]->q || !all[i]->scale || !all[i]->bias) return MOE_ERR_NULL;
    if (!w4_ok(*all[i])) return MOE_ERR_ALIGN;
  }
  if (!aligned(w->router, 16) || (w->router_bias && !aligned(w->router_bias, 4)) ||
      (w->shared_gate && !aligned(w->shared_gate, 16)))
    return MOE_ERR_ALIGN;
  if (w->shared_gate && s->d_ff_shared != s->d_ff) return MOE_ERR_SHAPE;
  return MOE_OK;
}

}  // namespace

// Checks of moe_decode_gemv_w4's arguments other than the workspace.
int moe::decode_args_status(const uint16_t* x, const moe_weights_t* w, const moe_shape_t* shape,
                            const uint16_t* out) {
  if (!shape_ok(shape, true) || shape->T != 1) return MOE_ERR_SHAPE;
  if (!moe::decode_shape_supported(shape->d_model, shape->n_experts, shape->top_k, shape->d_ff,
                                   w && w->shared_gate))
    return MOE_ERR_SHAPE;
  int rc = check_weights(w, shape);
  if (rc != MOE_OK) return rc;
  if (!x || !out) return MOE_ERR_NULL;
  if (!aligned(x, 16) || !aligned(out, 4)) return MOE_ERR_ALIGN;
  return MOE_OK;
}

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer is NULL";
    case MOE_ERR_ALIGN: return "a pointer is not aligned as required";
    case MOE_ERR_SHAPE: return "unsupported or inconsistent sizes";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case MOE_ERR_DEVICE: return "a kernel recorded a fault in the device status word";
    case MOE_ERR_ARCH: return "the current device is not a compute capability 10.3 GPU";
    case 100 + MOE_DEV_OK: return "device: ok";
    case 100 + MOE_DEV_BAD_TILE: return "device: block-map entry out of range";
    case 100 + MOE_DEV_BAD_ROW: return "device: row index out of range";
    case 100 + MOE_DEV_TIMEOUT: return "device: bounded wait ran out";
    case 100 + MOE_DEV_BAD_EXPERT: return "device: expert id out of range";
    default: return "unknown status";
  }
}

int moe_version(void) { return 100; }

// Measured on GB300 (d_model 2048, 256 experts, top-8, layer times with L2
// flushed): 64-row tiles beat 16- and 32-row tiles from about 8 rows per
// expert on (T = 512: 0.453 -> 0.338 ms; T = 1024: 0.461 -> 0.364 ms), since
// a tile's fixed costs (block-map entry, gathers, accumulator hand-offs)
// outweigh its padding; 128-row tiles win once experts average more than 64.
int moe_pick_block_n(int T, int n_experts, int top_k) {
  if (T <= 0 || n_experts <= 0) return 16;
  const double per_expert = (double)T * top_k / n_experts;
  if (per_expert <= 4) return 16;
  if (per_expert <= 64) return 64;
  return 128;
}

int moe_max_tiles(int T, int n_experts, int top_k, int block_n, int with_shared) {
  if (T < 0 || block_n <= 0) return 0;
  return (int)(cdiv((int64_t)T * top_k, block_n) + n_experts +
               (with_shared ? cdiv(T, block_n) : 0));
}

size_t moe_route_workspace_bytes(int T, int n_experts) {
  if (T < 0 || n_experts < 1) return 0;
  return route_ws(nullptr, T, n_experts).bytes;
}

int moe_route(const float* logits, const float* logit_bias, int T, int n_experts, int top_k,
              int block_n, int with_shared, int32_t* topk_ids, float* topk_w, int32_t* counts,
              int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* row_token,
              float* row_weight, int32_t* block_map, int32_t* num_tiles, int max_tiles, void* ws,
              size_t ws_bytes, void* stream) {
  if (T < 0 || n_experts < 1 || n_experts > 1024 || top_k < 1 || top_k > 32 ||
      top_k > n_experts || !valid_block_n(block_n) || (int64_t)T * (top_k + 1) >= (1 << 30))
    return MOE_ERR_SHAPE;
  if (!counts || !offsets || !num_tiles) return MOE_ERR_NULL;
  if (T > 0 && (!logits || !topk_ids || !topk_w || !perm || !inv_perm || !row_token || !block_map))
    return MOE_ERR_NULL;
  if (max_tiles < moe_max_tiles(T, n_experts, top_k, block_n, with_shared)) return MOE_ERR_SHAPE;
  if (!aligned(block_map, 16) || !aligned(logits, 4)) return MOE_ERR_ALIGN;
  const RouteWs rw = route_ws(ws, T, n_experts);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < rw.bytes) return MOE_ERR_WORKSPACE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = cuda_status(cudaMemsetAsync(rw.status, 0, kStatusWords * 4, s))) != MOE_OK) return rc;
  if (T == 0) {  // nothing routed: empty histogram, zero offsets, no tiles
    if ((rc = cuda_status(cudaMemsetAsync(counts, 0, n_experts * 4, s))) != MOE_OK) return rc;
    if ((rc = cuda_status(cudaMemsetAsync(offsets, 0, (n_experts + 1) * 4, s))) != MOE_OK) return rc;
    return cuda_status(cudaMemsetAsync(num_tiles, 0, 4, s));
  }
  moe::RouteParams p;
  memset(&p, 0, sizeof p);
  p.logits = logits;
  p.bias = logit_bias;
  p.T = T;
  p.E = n_experts;
  p.k = top_k;
  p.block_n = block_n;
  p.with_shared = with_shared ? 1 : 0;
  p.ids = topk_ids;
  p.w = topk_w;
  p.counts = counts;
  p.offsets = offsets;
  p.perm = perm;
  p.inv_perm = inv_perm;
  p.row_token = row_token;
  p.row_weight = row_weight;
  p.block_map = block_map;
  p.num_tiles = num_tiles;
  p.max_tiles = max_tiles;
  p.blk = rw.blk;
  p.status = rw.status;
  return cuda_status(moe::route_launch(p, s));
}

size_t moe_gemm_workspace_bytes(void) { return kStatusWords * 4; }

int moe_grouped_gemm_w4a16(const uint16_t* A, int64_t A_rows, int K, const int32_t* row_index,
                           int64_t n_rows, const moe_w4_t* W, int n_groups, int N,
                           const moe_w4_t* W_extra, const int32_t* block_map,
                           const int32_t* num_tiles, int max_tiles, int block_n, int epilogue,
                           int operand_format, const float* row_scale, const int32_t* out_row, void* C,
                           int64_t C_rows, int64_t ldc, void* ws, size_t ws_bytes, void* stream) {
  if (epilogue != MOE_EPI_NONE && epilogue != MOE_EPI_SWIGLU && epilogue != MOE_EPI_COMBINE)
    return MOE_ERR_SHAPE;
  if (operand_format != MOE_OPERAND_BF16 && operand_format != MOE_OPERAND_F16) return MOE_ERR_SHAPE;
  if (K < 64 || K % 64 || N < 128 || N % 128 || n_groups < 1 || A_rows < 0 || n_rows < 0 ||
      max_tiles < 0 || ldc < N || C_rows < 0)
    return MOE_ERR_SHAPE;
  if (!valid_block_n(block_n)) return MOE_ERR_SHAPE;
  if (epilogue != MOE_EPI_COMBINE && C_rows < n_rows) return MOE_ERR_SHAPE;
  // SWIGLU and COMBINE write 16-byte token-row segments (bulk copies)
  if (epilogue == MOE_EPI_SWIGLU && ldc % 8) return MOE_ERR_SHAPE;
  if (epilogue == MOE_EPI_COMBINE && ldc % 4) return MOE_ERR_SHAPE;
  if (!A || !W || !block_map || !num_tiles || !C) return MOE_ERR_NULL;
  if (epilogue == MOE_EPI_COMBINE && (!row_scale || !out_row)) return MOE_ERR_NULL;
  const int nmat = epilogue == MOE_EPI_SWIGLU ? 2 : 1;
  for (int j = 0; j < nmat; ++j) {
    if (!W[j].q || !W[j].scale || !W[j].bias) return MOE_ERR_NULL;
    if (!w4_ok(W[j])) return MOE_ERR_ALIGN;
    if (W_extra) {
      if (!W_extra[j].q || !W_extra[j].scale || !W_extra[j].bias) return MOE_ERR_NULL;
      if (!w4_ok(W_extra[j])) return MOE_ERR_ALIGN;
    }
  }
  if (!aligned(A, 16) || !aligned(block_map, 16) || !aligned(C, 16)) return MOE_ERR_ALIGN;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < moe_gemm_workspace_bytes()) return MOE_ERR_WORKSPACE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* status = static_cast<int32_t*>(ws);
  if ((rc = cuda_status(cudaMemsetAsync(status, 0, kStatusWords * 4, s))) != MOE_OK) return rc;
  if (max_tiles == 0 || n_rows == 0) return MOE_OK;
  moe::GemmParams p;
  memset(&p, 0, sizeof p);
  p.A = A;
  p.A_rows = A_rows;
  p.K = K;
  p.row_index = row_index;
  p.n_rows = n_rows;
  for (int j = 0; j < nmat; ++j) {
    p.W[j] = {W[j].q, W[j].scale, W[j].bias};
    if (W_extra) p.X[j] = {W_extra[j].q, W_extra[j].scale, W_extra[j].bias};
  }
  p.n_groups = n_groups;
  p.N = N;
  p.block_map = block_map;
  p.num_tiles = num_tiles;
  p.max_tiles = max_tiles;
  p.block_n = block_n;
  p.epilogue = epilogue;
  p.operand_f16 = operand_format == MOE_OPERAND_F16 ? 1 : 0;
  p.row_scale = row_scale;
  p.out_row = out_row;
  p.C = C;
  p.C_rows = C_rows;
  p.ldc = ldc;
  p.status = status;
  return cuda_status(moe::gemm_w4_launch(p, s));
}

size_t moe_workspace_bytes_ex(const moe_shape_t* shape, int block_n, int flags) {
  if (!shape_ok(shape, false) || !flags_ok(flags)) return 0;
  if ((block_n = forward_block_n(shape, block_n, flags)) == 0) return 0;
  return forward_ws(nullptr, shape, block_n, flags).bytes;
}

size_t moe_workspace_bytes(const moe_shape_t* shape, int block_n) {
  return moe_workspace_bytes_ex(shape, block_n, 0);
}

int moe_forward_views_ex(void* ws, size_t ws_bytes, const moe_shape_t* shape, int block_n,
                         int flags, moe_forward_views_t* views) {
  if (!shape_ok(shape, false) || !flags_ok(flags)) return MOE_ERR_SHAPE;
  if ((block_n = forward_block_n(shape, block_n, flags)) == 0) return MOE_ERR_SHAPE;
  if (!views) return MOE_ERR_NULL;
  const FwdWs fw = forward_ws(ws, shape, block_n, flags);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < fw.bytes) return MOE_ERR_WORKSPACE;
  *views = fw.v;
  return MOE_OK;
}

int moe_forward_views(void* ws, size_t ws_bytes, const moe_shape_t* shape, int block_n,
                      moe_forward_views_t* views) {
  return moe_forward_views_ex(ws, ws_bytes, shape, block_n, 0, views);
}

int moe_forward(const uint16_t* x, const moe_weights_t* w, const moe_shape_t* shape, int block_n,
                uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  return moe_forward_ex(x, w, shape, block_n, 0, out, ws, ws_bytes, stream);
}

int moe_forward_ex(const uint16_t* x, const moe_weights_t* w, const moe_shape_t* shape,
                   int block_n, int flags, uint16_t* out, void* ws, size_t ws_bytes,
                   void* stream) {
  if (!shape_ok(shape, false) || !flags_ok(flags)) return MOE_ERR_SHAPE;
  if ((block_n = forward_block_n(shape, block_n, flags)) == 0) return MOE_ERR_SHAPE;
  const int T = shape->T, E = shape->n_experts, k = shape->top_k, d = shape->d_model,
            f = shape->d_ff;
  int rc = check_weights(w, shape);
  if (rc != MOE_OK) return rc;
  if (T > 0 && (!x || !out)) return MOE_ERR_NULL;
  if (!aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_ALIGN;
  const FwdWs fw = forward_ws(ws, shape, block_n, flags);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < fw.bytes) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const moe_forward_views_t& v = fw.v;
  if ((rc = cuda_status(cudaMemsetAsync(v.status, 0, kStatusWords * 4, s))) != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  const bool shared = w->shared_gate != nullptr;
  const int64_t rows = (int64_t)T * k + (shared ? T : 0);

  // 1. router logits, shared-expert gate logit and the f16 copy of x
  moe::RouterParams rt;
  memset(&rt, 0, sizeof rt);
  rt.x = x;
  rt.T = T;
  rt.d = d;
  rt.E = E;
  rt.k = k;
  rt.Wr = w->router;
  rt.wsg = w->shared_gate;
  rt.wsplit = fw.wsplit;
  rt.logits = v.logits;
  rt.gate_logit = v.gate_logit;
  rt.row_weight = v.row_weight;
  rt.x16 = v.x16;
  rt.status = v.status;
  if ((rc = cuda_status(moe::router_launch(rt, s))) != MOE_OK) return rc;
  // 2. top-k, shared gate, histogram, scan, scatter, block map
  moe::RouteParams rp;
  memset(&rp, 0, sizeof rp);
  rp.logits = v.logits;
  rp.bias = w->router_bias;
  rp.T = T;
  rp.E = E;
  rp.k = k;
  rp.block_n = block_n;
  rp.with_shared = shared ? 1 : 0;
  rp.ids = v.topk_ids;
  rp.w = v.topk_w;
  rp.counts = v.counts;
  rp.offsets = v.offsets;
  rp.perm = v.perm;
  rp.inv_perm = v.inv_perm;
  rp.row_token = v.row_token;
  rp.row_weight = v.row_weight;
  rp.block_map = v.block_map;
  rp.num_tiles = v.num_tiles;
  rp.max_tiles = v.max_tiles;
  rp.blk = fw.blk;
  rp.status = v.status;
  if (v.down_block_map != v.block_map) {  // a second map for the down projection
    rp.block_map2 = v.down_block_map;
    rp.num_tiles2 = v.down_num_tiles;
    rp.max_tiles2 = v.down_max_tiles;
    rp.block_n2 = v.down_block_n;
    rp.window2 = v.down_window;
  }
  if ((rc = cuda_status(moe::route_launch(rp, s))) != MOE_OK) return rc;
  if (flags & MOE_FWD_FUSED) {
    // 3-4. the fused chain: per 64-row tile, gate/up + SwiGLU into shared
    // memory, then down + weighted combine into the fp32 accumulator
    if ((rc = cuda_status(cudaMemsetAsync(v.out_acc, 0, (size_t)T * d * 4, s))) != MOE_OK) return rc;
    moe::FusedParams fp;
    memset(&fp, 0, sizeof fp);
    fp.A = v.x16;
    fp.A_rows = T;
    fp.d = d;
    fp.f = f;
    fp.row_index = v.row_token;
    fp.n_rows = rows;
    fp.W[0] = {w->gate.q, w->gate.scale, w->gate.bias};
    fp.W[1] = {w->up.q, w->up.scale, w->up.bias};
    fp.W[2] = {w->down.q, w->down.scale, w->down.bias};
    if (shared) {
      fp.X[0] = {w->sh_gate.q, w->sh_gate.scale, w->sh_gate.bias};
      fp.X[1] = {w->sh_up.q, w->sh_up.scale, w->sh_up.bias};
      fp.X[2] = {w->sh_down.q, w->sh_down.scale, w->sh_down.bias};
    }
    fp.n_groups = E;
    fp.block_map = v.block_map;
    fp.num_tiles = v.num_tiles;
    fp.max_tiles = v.max_tiles;
    fp.row_scale = v.row_weight;
    fp.C = v.out_acc;
    fp.C_rows = T;
    fp.status = v.status;
    if ((rc = cuda_status(moe::gemm_fused_launch(fp, s))) != MOE_OK) return rc;
    return cuda_status(moe::f32_to_bf16_launch(v.out_acc, out, (int64_t)T * d, s));
  }
  // 3. gate/up grouped GEMM with SwiGLU -> h (rows in expert order, shared rows last)
  moe::GemmParams g;
  memset(&g, 0, sizeof g);
  g.A = v.x16;
  g.A_rows = T;
  g.K = d;
  g.row_index = v.row_token;
  g.n_rows = rows;
  g.W[0] = {w->gate.q, w->gate.scale, w->gate.bias};
  g.W[1] = {w->up.q, w->up.scale, w->up.bias};
  if (shared) {
    g.X[0] = {w->sh_gate.q, w->sh_gate.scale, w->sh_gate.bias};
    g.X[1] = {w->sh_up.q, w->sh_up.scale, w->sh_up.bias};
  }
  g.n_groups = E;
  g.N = f;
  // From 512 rows per expert on average, gate/up also runs on the down
  // projection's 256-row map (one accumulator buffer then fills TMEM); at
  // 256-511 rows per expert the 128-row tiles measured faster.
  const bool tall = v.down_block_n == 256 && v.down_window == 0 && (int64_t)T * k >= (int64_t)512 * E;
  g.block_map = tall ? v.down_block_map : v.block_map;
  g.num_tiles = tall ? v.down_num_tiles : v.num_tiles;
  g.max_tiles = tall ? v.down_max_tiles : v.max_tiles;
  g.block_n = tall ? 256 : block_n;
  g.epilogue = MOE_EPI_SWIGLU;
  g.operand_f16 = 1;
  g.C = v.h;
  g.C_rows = rows;
  g.ldc = f;
  g.status = v.status;
  if ((rc = cuda_status(moe::gemm_w4_launch(g, s))) != MOE_OK) return rc;
  // 4. down grouped GEMM, weighted combine into the fp32 accumulator (or, in
  // deterministic mode, every row's output stored for a fixed-order sum)
  const bool det = v.y != nullptr;
  if (!det && (rc = cuda_status(cudaMemsetAsync(v.out_acc, 0, (size_t)T * d * 4, s))) != MOE_OK)
    return rc;
  moe::GemmParams g2 = g;
  g2.A = v.h;
  g2.A_rows = rows;
  g2.K = f;
  g2.row_index = nullptr;
  g2.W[0] = {w->down.q, w->down.scale, w->down.bias};
  g2.W[1] = {};
  g2.X[0] = shared ? moe::GemmW4{w->sh_down.q, w->sh_down.scale, w->sh_down.bias} : moe::GemmW4{};
  g2.X[1] = {};
  g2.N = d;
  g2.block_map = v.down_block_map;
  g2.num_tiles = v.down_num_tiles;
  g2.max_tiles = v.down_max_tiles;
  g2.block_n = v.down_block_n;
  g2.epilogue = MOE_EPI_COMBINE;
  g2.row_scale = v.row_weight;
  g2.out_row = v.row_token;
  g2.C = v.out_acc;
  g2.C_rows = T;
  g2.ldc = d;
  if (det) {
    g2.epilogue = MOE_EPI_NONE;
    g2.row_scale = nullptr;
    g2.out_row = nullptr;
    g2.C = v.y;
    g2.C_rows = rows;
  }
  if ((rc = cuda_status(moe::gemm_w4_launch(g2, s))) != MOE_OK) return rc;
  // 5. bf16 output
  if (det)
    return cuda_status(moe::combine_rows_launch(v.y, v.inv_perm, v.row_weight, T, k, d, shared,
                                                v.out_acc, out, v.status, s));
  return cuda_status(moe::f32_to_bf16_launch(v.out_acc, out, (int64_t)T * d, s));
}

size_t moe_decode_workspace_bytes(const moe_shape_t* shape) {
  if (!shape_ok(shape, false)) return 0;
  return decode_ws(nullptr, shape).bytes;
}

int moe_decode_views(void* ws, size_t ws_bytes, const moe_shape_t* shape,
                     moe_decode_views_t* views) {
  if (!shape_ok(shape, false)) return MOE_ERR_SHAPE;
  if (!views) return MOE_ERR_NULL;
  const DecWs dw = decode_ws(ws, shape);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < dw.bytes) return MOE_ERR_WORKSPACE;
  *views = dw.v;
  return MOE_OK;
}

int moe_decode_gemv_w4(const uint16_t* x, const moe_weights_t* w, const moe_shape_t* shape,
                       uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  int rc = moe::decode_args_status(x, w, shape, out);
  if (rc != MOE_OK) return rc;
  const DecWs dw = decode_ws(ws, shape);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < dw.bytes) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the decode kernel clears the status word itself (after its dependency
  // wait) and keeps its epoch in the workspace, so consecutive calls stay one
  // chain of PDL launches with no memset between them
  moe::DecodeParams p;
  memset(&p, 0, sizeof p);
  p.x = x;
  p.w = *w;
  p.d = shape->d_model;
  p.E = shape->n_experts;
  p.k = shape->top_k;
  p.f = shape->d_ff;
  p.shared = w->shared_gate != nullptr;
  p.out = out;
  p.logits = dw.v.logits;
  p.gate_logit = dw.v.gate_logit;
  p.ids = dw.v.topk_ids;
  p.wts = dw.v.topk_w;
  p.h = dw.v.h;
  p.status = dw.v.status;
  p.pub = dw.pub;
  p.pub_h = dw.pub_h;
  p.sync = dw.sync;
  const uint64_t limit = g_decode_wait_ns.load(std::memory_order_relaxed);
  p.wait_ns = limit ? limit : moe::kWaitLimitNs;
  p.silent_block = g_decode_silent_block.load(std::memory_order_relaxed);
  return cuda_status(moe::decode_launch(p, s));
}

size_t moe_decode_batch_workspace_bytes(const moe_shape_t* shape) {
  if (!batch_shape_ok(shape)) return 0;
  return batch_ws(nullptr, shape).bytes;
}

int moe_decode_batch_views(void* ws, size_t ws_bytes, const moe_shape_t* shape,
                           moe_decode_views_t* views) {
  if (!batch_shape_ok(shape)) return MOE_ERR_SHAPE;
  if (!views) return MOE_ERR_NULL;
  const BatchWs bw = batch_ws(ws, shape);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < bw.bytes) return MOE_ERR_WORKSPACE;
  *views = bw.v;
  return MOE_OK;
}

int moe_decode_batch_w4(const uint16_t* x, const moe_weights_t* w, const moe_shape_t* shape,
                        uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  if (!batch_shape_ok(shape)) return MOE_ERR_SHAPE;
  int rc = check_weights(w, shape);
  if (rc != MOE_OK) return rc;
  if (!x || !out) return MOE_ERR_NULL;
  if (!aligned(x, 16) || !aligned(out, 2)) return MOE_ERR_ALIGN;
  const BatchWs bw = batch_ws(ws, shape);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < bw.bytes) return MOE_ERR_WORKSPACE;
  if ((rc = check_device()) != MOE_OK) return rc;
  moe::BatchParams p;
  memset(&p, 0, sizeof p);
  p.x = x;
  p.w = *w;
  p.T = shape->T;
  p.d = shape->d_model;
  p.E = shape->n_experts;
  p.k = shape->top_k;
  p.f = shape->d_ff;
  p.shared = w->shared_gate != nullptr;
  p.part = bw.part;
  p.logits = bw.v.logits;
  p.gate_logit = bw.v.gate_logit;
  p.ids = bw.v.topk_ids;
  p.wts = bw.wts;
  p.h = bw.v.h;
  p.out = out;
  p.status = bw.v.status;
  return cuda_status(moe::decode_batch_launch(p, static_cast<cudaStream_t>(stream)));
}

int moe_debug_decode_fault(uint64_t wait_limit_ns, int silent_block) {
  g_decode_wait_ns.store(wait_limit_ns, std::memory_order_relaxed);
  g_decode_silent_block.store(silent_block < 0 ? -1 : silent_block, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_get_device_status(const void* ws, void* stream, int32_t* device_status) {
  if (!ws || !device_status) return MOE_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  int rc = cuda_status(cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s));
  if (rc != MOE_OK) return rc;
  if ((rc = cuda_status(cudaStreamSynchronize(s))) != MOE_OK) return rc;
  *device_status = v;
  return v == MOE_DEV_OK ? MOE_OK : MOE_ERR_DEVICE;
}

}  // extern "C"

int moe_gdn_scan(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                 const float* beta, int T, int n_k_heads, int n_v_heads, int d_k, int d_v,
                 float* state, float* out, void* stream) {
  return moe_gdn_scan_ex(q, k, v, alpha, beta, T, n_k_heads, n_v_heads, d_k, d_v, state, out, 0,
                         stream);
}

int moe_gdn_scan_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                    const float* beta, int T, int n_k_heads, int n_v_heads, int d_k, int d_v,
                    float* state, float* out, int flags, void* stream) {
  if ((flags & ~MOE_GDN_STATE_EARLY) != 0) return MOE_ERR_SHAPE;
  if (T < 0 || !moe::gdn_shape_supported(d_k, d_v, n_k_heads, n_v_heads)) return MOE_ERR_SHAPE;
  if ((int64_t)T * n_v_heads * d_v >= (int64_t)1 << 40) return MOE_ERR_SHAPE;
  if (!state) return MOE_ERR_NULL;
  if (T > 0 && (!q || !k || !v || !alpha || !beta || !out)) return MOE_ERR_NULL;
  const size_t state_align = d_k == 128 ? 16 : 8;  // q, k, v are staged in 16-byte pieces
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(alpha, 4) ||
      !aligned(beta, 4) || !aligned(state, state_align))
    return MOE_ERR_ALIGN;
  if (T == 0) return MOE_OK;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  moe::GdnParams p;
  memset(&p, 0, sizeof p);
  p.q = q;
  p.k = k;
  p.v = v;
  p.alpha = alpha;
  p.beta = beta;
  p.T = T;
  p.Hk = n_k_heads;
  p.Hv = n_v_heads;
  p.dk = d_k;
  p.dv = d_v;
  p.state = state;
  p.out = out;
  p.state_early = (flags & MOE_GDN_STATE_EARLY) != 0;
  return cuda_status(moe::gdn_scan_launch(p, static_cast<cudaStream_t>(stream)));
}

size_t moe_decode_attention_workspace_bytes(int L, int n_q_heads, int n_kv_heads, int d) {
  if (!moe::attn_shape_supported(L, n_q_heads, n_kv_heads, d)) return 0;
  // the split count never exceeds one per 64 positions, whatever the SM count
  return moe::attn_workspace_floats(L, n_q_heads, n_kv_heads, d, 1 << 20) * sizeof(float);
}

int moe_decode_attention(const uint16_t* q, const uint16_t* K, const uint16_t* V, int L,
                         int n_q_heads, int n_kv_heads, int d, float scale, float* out, void* ws,
                         size_t ws_bytes, void* stream) {
  if (!moe::attn_shape_supported(L, n_q_heads, n_kv_heads, d)) return MOE_ERR_SHAPE;
  if ((int64_t)L * n_kv_heads * d >= (int64_t)1 << 40) return MOE_ERR_SHAPE;
  if (!q || !K || !V || !out) return MOE_ERR_NULL;
  if (!aligned(q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(out, 4))
    return MOE_ERR_ALIGN;
  if (!ws || !aligned(ws, 4) ||
      ws_bytes < moe_decode_attention_workspace_bytes(L, n_q_heads, n_kv_heads, d))
    return MOE_ERR_WORKSPACE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  moe::AttnParams p;
  memset(&p, 0, sizeof p);
  p.q = q;
  p.K = K;
  p.V = V;
  p.L = L;
  p.Hq = n_q_heads;
  p.Hkv = n_kv_heads;
  p.d = d;
  p.scale = scale > 0.f ? scale : 1.f / sqrtf((float)d);
  p.ws = static_cast<float*>(ws);
  p.out = out;
  return cuda_status(moe::attn_decode_launch(p, sms, static_cast<cudaStream_t>(stream)));
}
