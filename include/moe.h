/*
 * moe.h: C ABI of libmoe_gb300, a GB300 (sm_103a) implementation of the
 * sparse mixture-of-experts layer of a Qwen3.6-35B-A3B-style model.
 *
 * The layer (as the pages describe it):
 *   - a router picks 8 of 256 experts per token, plus one shared expert that
 *     every token uses ("Perplexity's Lily Beats MLX-LM by 1.35x Running
 *     Qwen3.6 on Apple Silicon", section "What Lily actually does");
 *   - expert weights are groupwise affine 4-bit, unpacked tile by tile on
 *     chip just before the multiply, never expanded in memory (same page,
 *     "Prefill optimizations", first bullet; "Perplexity Open Sources Lily:
 *     Rust & Metal Engine for Qwen3.6", body);
 *   - the routing metadata (histogram, prefix scan, scatter, block map) is
 *     built and consumed on the GPU with no host round trip ("Prefill
 *     optimizations", second bullet);
 *   - batch-1 decode is a matrix-vector product over only the selected
 *     experts' weights ("Why prefill and decode get different treatment").
 * The same library also exports the model's Gated DeltaNet scan (gdn.h) and
 * batch-1 decode attention with grouped KV heads (attn.h), under the
 * conventions below.
 *
 * Conventions shared by every call
 *   - bf16 values are passed as uint16_t bit patterns.
 *   - All device pointers are caller-owned. The library allocates nothing,
 *     keeps no state between calls and creates no streams. Every call only
 *     enqueues work on `stream` (a cudaStream_t passed as void*, NULL = the
 *     legacy default stream) and returns without synchronising; no call
 *     copies data to the host except moe_get_device_status.
 *   - 4-bit weights, one projection of a stack of G experts (moe_w4_t):
 *       q     uint32 [G][N][K/8]  code k of row n is nibble (k % 8) of word
 *                                 k/8, lowest nibble first
 *       scale bf16   [G][N][K/group]
 *       bias  bf16   [G][N][K/group]
 *     element value w[g][n][k] = scale * q + bias (one scale/bias per group
 *     of `group` consecutive codes along K). q, scale and bias must be
 *     16-byte aligned.
 *   - Supported sizes: group == 64; d_model and d_ff multiples of 128;
 *     1 <= top_k <= 32, top_k <= n_experts <= 1024; d_ff_shared == d_ff
 *     when a shared expert is present.
 *   - Return value: MOE_OK or a negative moe_status code. Host-side argument
 *     checks run before anything is enqueued. Faults that kernels detect
 *     (an out-of-range block-map entry or row index, a bounded wait that ran
 *     out) are recorded in the device status word in the workspace; each
 *     call clears that word when it starts, moe_get_device_status reads it.
 *   - No function aborts, exits or throws.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_NULL = -1,      /* a required pointer is NULL */
  MOE_ERR_ALIGN = -2,     /* a pointer is not aligned as documented */
  MOE_ERR_SHAPE = -3,     /* unsupported or inconsistent sizes */
  MOE_ERR_WORKSPACE = -4, /* workspace NULL, misaligned (256 B) or too small */
  MOE_ERR_CUDA = -5,      /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_DEVICE = -6,    /* a kernel recorded a fault in the device status word */
  MOE_ERR_ARCH = -7       /* the current device is not a compute capability 10.3 GPU */
};

/* Device status word values (read with moe_get_device_status). */
enum moe_device_status {
  MOE_DEV_OK = 0,
  MOE_DEV_BAD_TILE = 1,    /* a block-map entry points outside the rows or groups */
  MOE_DEV_BAD_ROW = 2,     /* a row index or output row is out of range */
  MOE_DEV_TIMEOUT = 3,     /* a bounded wait inside a kernel ran out */
  MOE_DEV_BAD_EXPERT = 4   /* a top-k id outside [0, n_experts) */
};

enum moe_epilogue {
  MOE_EPI_NONE = 0,    /* C fp32 [rows][N] = A_row . W^T                          */
  MOE_EPI_SWIGLU = 1,  /* C bf16 [rows][N] = silu(A_row . Wg^T) * (A_row . Wu^T)  */
  MOE_EPI_COMBINE = 2  /* C fp32 [out rows][N] += row_scale[row] * (A_row . W^T)  */
};

/* Tensor-core operand type of the grouped GEMM: activations A and the
 * dequantised weights are both of this type (fp32 accumulation). */
enum moe_operand_format {
  MOE_OPERAND_BF16 = 0, /* A bf16; weights RNE_bf16(scale*q + bias) */
  MOE_OPERAND_F16 = 1   /* A f16; weights RNE_f16(scale*q + bias); values must lie within
                           the f16 range (|v| < 65504), larger ones saturate */
};

typedef struct {
  int32_t T;           /* tokens */
  int32_t d_model;     /* hidden size (K of gate/up, N of down) */
  int32_t n_experts;   /* routed experts E */
  int32_t top_k;       /* experts per token */
  int32_t d_ff;        /* routed expert intermediate size */
  int32_t d_ff_shared; /* shared expert intermediate size */
  int32_t group;       /* quantisation group along K (64) */
} moe_shape_t;

typedef struct {
  const uint32_t* q;
  const uint16_t* scale;
  const uint16_t* bias;
} moe_w4_t;

typedef struct {
  moe_w4_t gate, up, down;          /* routed experts: [E][d_ff][d_model/8], [E][d_model][d_ff/8] */
  moe_w4_t sh_gate, sh_up, sh_down; /* shared expert (one group); ignored when shared_gate is NULL */
  const float* router;              /* fp32 [d_model][n_experts], row-major */
  const float* router_bias;         /* fp32 [n_experts] added to the logits, or NULL */
  const float* shared_gate;         /* fp32 [d_model]: shared expert scaled by sigmoid(x . w); NULL = none */
} moe_weights_t;

/* Text for a moe_status or (offset by 100) a moe_device_status value. */
const char* moe_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int moe_version(void);

/* Row-tile height used by moe_forward when block_n == 0: 16 up to 4 rows per
 * expert on average (T * top_k / n_experts), 64 up to 64, else 128. */
int moe_pick_block_n(int T, int n_experts, int top_k);

/* Upper bound on block-map entries: ceil(T*k/bn) + E + (with_shared ? ceil(T/bn) : 0). */
int moe_max_tiles(int T, int n_experts, int top_k, int block_n, int with_shared);

/*
 * moe_route: GPU-resident routing from fp32 router logits.
 * ("Prefill optimizations", second bullet: histogram, prefix scan, scatter
 * and block-map build stay on the GPU.)
 *
 *   logits      fp32 [T][E] device; logit_bias fp32 [E] or NULL.
 *               z = fp32(logits + bias). ids = the top_k largest z
 *               (descending, ties to the lower expert id);
 *               w_j = exp(z_j - z_max) / sum over the selected of exp(.).
 *   topk_ids    int32 [T][top_k] out;  topk_w fp32 [T][top_k] out.
 *   counts      int32 [E] out: assignments per expert.
 *   offsets     int32 [E+1] out: exclusive prefix sum, offsets[E] = T*top_k.
 *   perm        int32 [T*top_k] out: assignment a = t*top_k + j listed by
 *               expert, then by a (a stable counting sort).
 *   inv_perm    int32 [T*top_k] out: inv_perm[perm[p]] = p.
 *   row_token   int32 [T*top_k (+T)] out: token of each row (perm[p]/top_k);
 *               with_shared appends rows T*top_k + t -> t.
 *   row_weight  fp32 [T*top_k] out or NULL: topk_w of each row's assignment.
 *   block_map   int32 [max_tiles][4] out: {group, first row, rows, 0} per
 *               tile of block_n rows: expert 0's rows, expert 1's, ...;
 *               then (with_shared) the T shared rows as group E.
 *               max_tiles must be >= moe_max_tiles(T, E, top_k, block_n, with_shared).
 *   num_tiles   int32 [1] out: entries written.
 *   ws          device workspace of moe_route_workspace_bytes(T, E) bytes,
 *               256-byte aligned; holds the status word.
 * Every output is bit-exact given the same logits except topk_w (expf).
 * block_n in {16, 32, 64, 128, 256}.
 */
size_t moe_route_workspace_bytes(int T, int n_experts);
int moe_route(const float* logits, const float* logit_bias, int T, int n_experts, int top_k,
              int block_n, int with_shared, int32_t* topk_ids, float* topk_w, int32_t* counts,
              int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* row_token,
              float* row_weight, int32_t* block_map, int32_t* num_tiles, int max_tiles,
              void* ws, size_t ws_bytes, void* stream);

/*
 * moe_grouped_gemm_w4a16: grouped GEMM over row tiles with 4-bit weights
 * dequantised on chip ("Prefill optimizations", first bullet). Tensor-core
 * (tcgen05) kernel: packed tiles arrive by TMA and are unpacked to the
 * operand type (f16 or bf16, as operand_format says) into the MMA's A
 * operand, in tensor memory where it fits beside two accumulator buffers
 * (always for a single weight matrix, e.g. the down projection) and in
 * shared memory otherwise; products accumulate in fp32 in tensor memory.
 *
 *   A           [A_rows][K] device, row-major (K contiguous), bf16 or f16 as
 *               operand_format says (moe_operand_format).
 *   row_index   int32 [n_rows]: A row of GEMM row r; NULL = r itself.
 *   W           MOE_EPI_SWIGLU: W[0] = gate, W[1] = up; otherwise W[0].
 *               Each a stack of n_groups experts: q [n_groups][N][K/8].
 *   W_extra     optional: weights of group index n_groups (one expert, same
 *               layout, W_extra[0..1] like W), e.g. the shared expert; NULL = none.
 *   block_map   int32 [max_tiles][4] {group, first row, rows, 0} device;
 *   num_tiles   int32 [1] device: entries to process (read on the device).
 *               Rows r of a tile are first..first+rows-1 < n_rows, rows <= block_n.
 *   epilogue    moe_epilogue.
 *   row_scale   COMBINE: fp32 [n_rows] factor of each GEMM row.
 *   out_row     COMBINE: int32 [n_rows] destination row of each GEMM row.
 *   C           NONE: fp32 [n_rows][ldc]; SWIGLU: [n_rows][ldc] of the operand type;
 *               COMBINE: fp32 [C_rows][ldc], accumulated with atomic adds
 *               (order of the adds is not fixed). ldc >= N, in elements;
 *               SWIGLU needs ldc % 8 == 0, COMBINE ldc % 4 == 0.
 *   N           output columns (multiple of 128); K multiple of 64.
 *   ws          256-byte aligned, >= moe_gemm_workspace_bytes() bytes.
 * block_n in {16, 32, 64, 128, 256}. At 256 with SWIGLU the two 256-column
 * accumulators fill tensor memory, so a tile's epilogue no longer overlaps
 * the next tile's products.
 */
size_t moe_gemm_workspace_bytes(void);
int moe_grouped_gemm_w4a16(const uint16_t* A, int64_t A_rows, int K, const int32_t* row_index,
                           int64_t n_rows, const moe_w4_t* W, int n_groups, int N,
                           const moe_w4_t* W_extra, const int32_t* block_map,
                           const int32_t* num_tiles, int max_tiles, int block_n, int epilogue,
                           int operand_format, const float* row_scale, const int32_t* out_row, void* C,
                           int64_t C_rows, int64_t ldc, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward: the whole layer for T tokens.
 *   out[t] = sum_j w[t][j] * Expert_{ids[t][j]}(x_t) + sigmoid(x_t . w_sg) * Shared(x_t)
 * with Expert(x) = (silu(x Wg^T) * (x Wu^T)) Wd^T.
 *   x    bf16 [T][d_model] device;  out bf16 [T][d_model] device.
 *   block_n  row-tile height (16/32/64/128) or 0 for moe_pick_block_n.
 *   ws   256-byte aligned, >= moe_workspace_bytes(shape, block_n) bytes.
 * Pipeline: router and shared-gate logits on the tensor cores (the fp32
 * router weights split exactly into three bf16 planes in the workspace on
 * every call; fp32 accumulation; also writing an f16 copy of x) -> top-k ->
 * histogram -> scan -> scatter + block map -> grouped GEMM (gate/up + SwiGLU)
 * -> grouped GEMM (down + weighted combine) -> bf16 output.
 * The grouped GEMMs use f16 tensor-core operands (MOE_OPERAND_F16): x, the
 * dequantised weights and the intermediate h are f16 (11-bit significand),
 * accumulation is fp32. x, the weights and h must lie within the f16 range.
 */
size_t moe_workspace_bytes(const moe_shape_t* shape, int block_n);
int moe_forward(const uint16_t* x, const moe_weights_t* w, const moe_shape_t* shape, int block_n,
                uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward_ex: moe_forward with option flags; flags 0 is moe_forward.
 * MOE_FWD_DETERMINISTIC makes the output reproducible bit for bit from run
 * to run: the down grouped GEMM stores every row's (unweighted) output, fp32
 * [T*top_k + T][d_model] in the workspace, instead of adding it into the
 * token's accumulator at L2 (whose order of fp32 additions varies between
 * runs), and one more kernel sums each token's rows in slot order (routed
 * slots 0..top_k-1 by descending logit, then the shared expert), one fp32
 * fused multiply-add per row, and rounds the sum to bf16. It costs the y
 * rows' bytes in the workspace (2.4 GB at T = 32768, d_model 2048) and one
 * write and one read of them per call.
 * MOE_FWD_DOWN_WINDOWS orders the down projection's tiles by token window
 * (8192 tokens) when it runs on its own 256-row map (T * top_k >= 256 *
 * n_experts with 128-row gate/up tiles) and T > 8192: every expert's rows of
 * one window, then the next window's, so the fp32 rows the combine adds into
 * stay in L2 while their contributions arrive. Each (window, expert) piece
 * may end in a partial tile.
 * MOE_FWD_FUSED runs the two projections as one kernel over 64-row tiles
 * (block_n 0 or 64): per tile, the gate/up products and SwiGLU go into
 * shared memory (h is not written to the workspace; its view stays
 * unwritten), then the down products of that h are weighted and added into
 * the fp32 accumulator. Needs d_model and d_ff multiples of 512, d_ff <= 512;
 * not combinable with the other flags. Other flag bits, or those cases,
 * return MOE_ERR_SHAPE.
 * moe_workspace_bytes_ex / moe_forward_views_ex take the same flags (the
 * views' y is set only with MOE_FWD_DETERMINISTIC).
 */
#define MOE_FWD_DETERMINISTIC 1
#define MOE_FWD_DOWN_WINDOWS 2
#define MOE_FWD_FUSED 4
size_t moe_workspace_bytes_ex(const moe_shape_t* shape, int block_n, int flags);
int moe_forward_ex(const uint16_t* x, const moe_weights_t* w, const moe_shape_t* shape,
                   int block_n, int flags, uint16_t* out, void* ws, size_t ws_bytes,
                   void* stream);

/* Device pointers of moe_forward's intermediates inside its workspace. */
typedef struct {
  float* logits;       /* [T][E] router logits (without router_bias) */
  float* gate_logit;   /* [T] x . w_sg */
  int32_t* topk_ids;   /* [T][k] */
  float* topk_w;       /* [T][k] */
  int32_t* counts;     /* [E] */
  int32_t* offsets;    /* [E+1] */
  int32_t* perm;       /* [T*k] */
  int32_t* inv_perm;   /* [T*k] */
  int32_t* row_token;  /* [T*k + T] */
  float* row_weight;   /* [T*k + T] routing weight, then sigmoid gate */
  int32_t* block_map;  /* [max_tiles][4] */
  int32_t* num_tiles;  /* [1] */
  uint16_t* x16;       /* f16 [T][d_model]: x as the tensor-core operand */
  uint16_t* h;         /* f16 [T*k + T][d_ff] */
  float* out_acc;      /* fp32 [T][d_model] */
  int32_t* status;     /* device status word */
  int32_t max_tiles;
  int32_t block_n;     /* gate/up row-tile height */
  /* The down projection's block map. Equal to block_map/num_tiles/max_tiles
     unless block_n is 128 and T*top_k >= 256*n_experts: the down projection
     then runs on 256-row tiles of a second map, and from T*top_k >=
     512*n_experts (without MOE_FWD_DOWN_WINDOWS) so does gate/up. */
  int32_t* down_block_map;
  int32_t* down_num_tiles;
  int32_t down_max_tiles;
  int32_t down_block_n;
  /* MOE_FWD_DETERMINISTIC only (else NULL): fp32 [T*k + T][d_model], row r =
     h row r . W_down^T of its expert, unweighted; out_acc then holds the
     fixed-order weighted sum. */
  float* y;
  /* Tokens per window of the down projection's block map (0: one window).
     With a window W, down_block_map lists, for tokens [0, W), every expert's
     tiles in expert order and then the shared rows' tiles, then the same for
     [W, 2W), and so on. */
  int32_t down_window;
} moe_forward_views_t;
int moe_forward_views(void* ws, size_t ws_bytes, const moe_shape_t* shape, int block_n,
                      moe_forward_views_t* views);
int moe_forward_views_ex(void* ws, size_t ws_bytes, const moe_shape_t* shape, int block_n,
                         int flags, moe_forward_views_t* views);

/*
 * moe_decode_gemv_w4: one token (shape->T == 1) through the layer with
 * matrix-vector work that reads only the router, the shared expert and the
 * top_k selected experts' packed weights ("Why prefill and decode get
 * different treatment"). One kernel launch per call, one block per SM; the
 * blocks synchronise through counters in the workspace, so the call needs
 * the whole GPU to itself while it runs (other work on the GPU only delays
 * it; a wait that exceeds 2 s records MOE_DEV_TIMEOUT).
 *   x bf16 [d_model] device; out bf16 [d_model] device; d_model <= 4096,
 *   n_experts <= 256, top_k <= 32 and (top_k + 1) * d_ff <= about 24000 (h
 *   of every slot is staged on chip); other sizes return MOE_ERR_SHAPE.
 *   ws 256-byte aligned, >= moe_decode_workspace_bytes(shape) bytes, and
 *   zero-filled before its first use (cudaMemset); every call leaves its
 *   counters at zero for the next one. Zero it again after a call whose
 *   device status reports MOE_DEV_TIMEOUT. Calls on one workspace must not
 *   overlap on the GPU.
 */
size_t moe_decode_workspace_bytes(const moe_shape_t* shape);
int moe_decode_gemv_w4(const uint16_t* x, const moe_weights_t* w, const moe_shape_t* shape,
                       uint16_t* out, void* ws, size_t ws_bytes, void* stream);

typedef struct {
  float* logits;      /* [E] */
  float* gate_logit;  /* [1] */
  int32_t* topk_ids;  /* [k] */
  float* topk_w;      /* [k] */
  float* h;           /* fp32 [k + 1][d_ff]: SwiGLU activations, shared expert last */
  int32_t* status;
} moe_decode_views_t;
int moe_decode_views(void* ws, size_t ws_bytes, const moe_shape_t* shape,
                     moe_decode_views_t* views);

/*
 * moe_decode_gemv_w4_noalloc: moe_decode_gemv_w4 without a caller workspace.
 * The pages have no counterpart to this call; it exists for callers that may
 * not allocate device memory, such as plug-ins running inside a framework
 * whose memory pool owns the GPU, or serving loops that cannot afford an
 * allocation's synchronisation. Its scratch is a 256 KB array compiled into
 * the library (each GPU that loads the library holds one until the process
 * exits); the call itself allocates nothing.
 *   x, w, shape, out, stream: as for moe_decode_gemv_w4 (shape->T == 1), with
 *   the same argument checks and return codes; then MOE_ERR_WORKSPACE when
 *   moe_decode_workspace_bytes(shape) exceeds 256 KB (the top-8-of-256 layer
 *   with d_ff 512 needs 74,240 bytes), and MOE_ERR_CUDA if the scratch's
 *   device address cannot be obtained.
 * The first call on each device looks the scratch up (cudaGetSymbolAddress,
 * which may load the library's device code onto that device); make that
 * first call before any stream capture. All calls share the one array, which
 * keeps the previous call's contents (a static device array starts at zero,
 * and every call leaves the kernel's counters as the next call needs them).
 * Calls that overlap on the GPU, e.g. on two streams, race on the array.
 * The array's device status word is read with
 * moe_decode_noalloc_device_status; after a call that recorded
 * MOE_DEV_TIMEOUT, moe_decode_noalloc_reset zeroes the array (the decode
 * contract's "zero the workspace again"), and later calls are correct again.
 */
int moe_decode_gemv_w4_noalloc(const uint16_t* x, const moe_weights_t* w,
                               const moe_shape_t* shape, uint16_t* out, void* stream);
/* The built-in scratch's device status word (synchronises `stream`; returns
 * MOE_ERR_DEVICE when the word holds a fault), as moe_get_device_status. */
int moe_decode_noalloc_device_status(void* stream, int32_t* device_status);
/* Zeroes the built-in scratch on `stream` (cudaMemsetAsync; allocates nothing). */
int moe_decode_noalloc_reset(void* stream);

/*
 * moe_decode_batch_w4: a small batch of tokens (1 <= shape->T <= 8, e.g. a
 * speculative-decoding verification batch whose tokens select different
 * experts) through the layer with matrix-vector work, as in
 * moe_decode_gemv_w4 ("Why prefill and decode get different treatment"):
 * the router, the shared expert and each selected expert's rows are read
 * once per call and applied to every token that uses them. Three kernel
 * launches chained by programmatic dependent launch; no waits between
 * blocks, so the call shares the GPU with other work.
 *   x bf16 [T][d_model] device (16-byte aligned); out bf16 [T][d_model].
 *   Routing as in moe_forward: top_k by logit (plus router_bias), ties to the
 *   lower id, softmax over the selected; the shared expert (if any) scaled by
 *   sigmoid(x . shared_gate).
 *   Shapes: d_model, d_ff multiples of 128, n_experts <= 1024, top_k <= 32,
 *   and the per-block staging (about T*d_model*2 and T*(top_k+1)*d_ff*2
 *   bytes) within 200 KB; otherwise MOE_ERR_SHAPE.
 *   ws 256-byte aligned, >= moe_decode_batch_workspace_bytes(shape) bytes (no
 *   initialisation needed). Calls on one workspace must not overlap on the GPU.
 */
size_t moe_decode_batch_workspace_bytes(const moe_shape_t* shape);
int moe_decode_batch_w4(const uint16_t* x, const moe_weights_t* w, const moe_shape_t* shape,
                        uint16_t* out, void* ws, size_t ws_bytes, void* stream);
/* Views of a batch-decode workspace, every array with a leading [T]: logits
 * [T][E], gate_logit [T], topk_ids [T][k], topk_w [T][k + 1] (the shared
 * gate last), h fp32 [T][k + 1][d_ff]. */
int moe_decode_batch_views(void* ws, size_t ws_bytes, const moe_shape_t* shape,
                           moe_decode_views_t* views);

/*
 * moe_debug_decode_fault: a test hook for the decode path's failure
 * detection (no counterpart on the pages). Later moe_decode_gemv_w4 calls
 * (and moe_decode_gemv_w4_noalloc) give up a cross-block wait after
 * wait_limit_ns instead of 2 s (0 restores 2 s), and, when silent_block >= 0,
 * that block of each call publishes no router partial sums, so every other
 * block's wait for them runs out: the call then records MOE_DEV_TIMEOUT in
 * the workspace's status word and runs to its end with a wrong output. The
 * settings are process-wide and apply to calls enqueued after this one
 * (CUDA graphs keep the settings they were captured with). Returns MOE_OK.
 */
int moe_debug_decode_fault(uint64_t wait_limit_ns, int silent_block);

/*
 * Reads the device status word of a workspace (synchronises `stream`).
 * *device_status receives a moe_device_status value.
 */
int moe_get_device_status(const void* ws, void* stream, int32_t* device_status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
