// ORACLE: plain, slow CPU reference of the 4-bit sparse MoE layer.
//
// This file is TEST INFRASTRUCTURE. Only the test suite, the package smoke
// check and the benchmark's CPU-baseline leg load it. The CUDA library never
// links, includes or calls it, and it shares no code with the CUDA path.
//
// What it computes, and the passage each step follows:
//   * Router: a linear router picks 8 of 256 experts per token, plus one
//     shared expert that every token uses.
//     ("Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple
//     Silicon", section "What Lily actually does"; also "Perplexity Open
//     Sources Lily Inference Engine for Apple Silicon", third paragraph.)
//   * Groupwise affine 4-bit weights: each group of `G` consecutive codes
//     along K shares one scale and one bias, w = scale * q + bias.
//     ("Perplexity Open Sources Lily: Rust & Metal Engine for Qwen3.6", body;
//     "Perplexity's Lily Beats MLX-LM ...", section "Prefill optimizations".)
//     Dequantising a tile before the multiply leaves the product unchanged,
//     so here the weight is dequantised element by element, exactly, in
//     double precision.
//   * Routing metadata: per-expert histogram, prefix scan, scatter of the
//     (token, slot) assignments into expert order, and a block map of
//     fixed-size row tiles ("Prefill optimizations", second bullet). Here it
//     is built by brute force: a stable selection per expert.
//   * Batch-1 decode is the same arithmetic at T = 1
//     ("Why prefill and decode get different treatment").
//
// Readings adopted where the pages are silent:
//   nibble k%8 of word k/8 holds code k, low nibble first; SwiGLU experts
//   h = silu(x Wg^T) * (x Wu^T), y = h Wd^T; softmax over the selected
//   logits (softmax over all, renormalised over the top k); top-k ties go to
//   the lower expert id; an optional per-expert router bias is added to the
//   fp32 logits before selection and weighting; the shared expert's output
//   is scaled by sigmoid(x . w_sg).
//
// Precision: inputs are exact (bf16 / fp32 / 4-bit codes); every sum is
// accumulated in double in index order; results are rounded to fp32 once.
// The one decision taken in fp32 is top-k selection, on z = fp32(l + b),
// which is the precision the fp32 logits carry.
//
// ORACLE_MUTANT (compile-time, default 0) plants one known mistake so the
// test suite can show that its pins catch it. A normal build never sets it.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif
#define MUT(n) (ORACLE_MUTANT == (n))

namespace {

double bf16_value(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// One projection of a stack of experts: codes q[g][n][K/8], scale and bias
// s[g][n][K/G], b[g][n][K/G] (bf16 bit patterns).
struct W4 {
  const uint32_t* q;
  const uint16_t* s;
  const uint16_t* b;
  int N, K, G;
};

// The 4-bit code of element k of row (g, n).
int code_at(const W4& w, int64_t g, int n, int k) {
  const uint32_t word = w.q[(g * w.N + n) * (int64_t)(w.K / 8) + k / 8];
  const int nib = MUT(1) ? (7 - (k % 8)) : (k % 8);
  return static_cast<int>((word >> (4 * nib)) & 0xFu);
}

// w = scale * q + bias for element k of row (g, n), exact in double.
double dequant_at(const W4& w, int64_t g, int n, int k) {
  const int64_t gi = MUT(7) ? g * w.N * (int64_t)(w.K / w.G) + (int64_t)(k / w.G) * w.N + n
                            : (g * w.N + n) * (int64_t)(w.K / w.G) + k / w.G;
  const double scale = bf16_value(w.s[gi]);
  const double bias = MUT(2) ? 0.0 : bf16_value(w.b[gi]);
  return scale * code_at(w, g, n, k) + bias;
}

// Sum_k W[g][n][k] * v[k]
double row_dot(const W4& w, int64_t g, int n, const double* v) {
  double acc = 0.0;
  for (int k = 0; k < w.K; ++k) acc += dequant_at(w, g, n, k) * v[k];
  return acc;
}

double silu(double z) { return z / (1.0 + std::exp(-z)); }

// Router logit of expert e: Sum_k x[k] * Wr[k][e], Wr row-major [d][E].
double router_logit(const double* x, const float* Wr, int d, int E, int e) {
  double acc = 0.0;
  for (int k = 0; k < d; ++k)
    acc += x[k] * (MUT(8) ? Wr[(int64_t)e * d + k] : Wr[(int64_t)k * E + e]);
  return acc;
}

// One SwiGLU expert g applied to one token: y = (silu(x Wg^T) * x Wu^T) Wd^T.
void expert_forward(const W4& gate, const W4& up, const W4& down, int64_t g, const double* x,
                    double* y) {
  const int f = gate.N, d = down.N;
  std::vector<double> h(f);
  for (int i = 0; i < f; ++i) {
    const double gi = row_dot(gate, g, i, x);
    const double ui = row_dot(up, g, i, x);
    h[i] = MUT(3) ? silu(ui) * gi : silu(gi) * ui;
  }
  for (int j = 0; j < d; ++j) y[j] = row_dot(down, g, j, h.data());
}

// Top-k of one token's biased logits z (descending, ties to the lower id),
// and the routing weights: softmax of the selected z.
void topk_one(const float* logits, const float* bias, int E, int k, int32_t* ids, double* w) {
  std::vector<float> z(E);
  for (int e = 0; e < E; ++e) z[e] = bias ? logits[e] + bias[e] : logits[e];  // fp32 add
  std::vector<char> taken(E, 0);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      const bool better = best < 0 || z[e] > z[best] || (MUT(5) && z[e] == z[best]);
      if (better) best = e;
    }
    taken[best] = 1;
    ids[j] = best;
  }
  const double zmax = z[ids[0]];
  double denom = 0.0;
  if (MUT(4)) {  // softmax over all experts, not renormalised over the top k
    for (int e = 0; e < E; ++e) denom += std::exp(z[e] - zmax);
  } else {
    for (int j = 0; j < k; ++j) denom += std::exp(z[ids[j]] - zmax);
  }
  for (int j = 0; j < k; ++j) w[j] = std::exp(z[ids[j]] - zmax) / denom;
}

}  // namespace

extern "C" {

// Dequantise rows [0, rows) of one stacked projection (group index g folded
// into rows): W[r][k] = scale * q + bias, exact, written as fp64.
int oracle_dequant(const uint32_t* q, const uint16_t* s, const uint16_t* b, int rows, int K,
                   int G, double* W) {
  if (K % 8 || K % G) return -1;
  const W4 w{q, s, b, rows, K, G};
  for (int r = 0; r < rows; ++r)
    for (int k = 0; k < K; ++k) W[(int64_t)r * K + k] = dequant_at(w, 0, r, k);
  return 0;
}

// logits[t][e] = fp32( Sum_k x[t][k] * Wr[k][e] ), Wr row-major [d][E].
// gate_logit[t] = fp32( Sum_k x[t][k] * wsg[k] ) when wsg != NULL.
int oracle_router(const uint16_t* x, const float* Wr, const float* wsg, int T, int d, int E,
                  float* logits, float* gate_logit) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < T; ++t) {
    std::vector<double> xt(d);
    for (int k = 0; k < d; ++k) xt[k] = bf16_value(x[(int64_t)t * d + k]);
    for (int e = 0; e < E; ++e)
      logits[(int64_t)t * E + e] = static_cast<float>(router_logit(xt.data(), Wr, d, E, e));
    if (wsg && gate_logit) {
      double acc = 0.0;
      for (int k = 0; k < d; ++k) acc += xt[k] * wsg[k];
      gate_logit[t] = static_cast<float>(acc);
    }
  }
  return 0;
}

// Top-k selection and routing weights for T tokens.
int oracle_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* ids,
                float* w) {
  if (k < 1 || k > E) return -1;
  std::vector<double> wd(k);
  for (int t = 0; t < T; ++t) {
    topk_one(logits + (int64_t)t * E, bias, E, k, ids + (int64_t)t * k, wd.data());
    for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = static_cast<float>(wd[j]);
  }
  return 0;
}

// Routing metadata from the top-k ids (assignment a = t*k + j):
//   counts[e]      = #{a : ids[a] == e}
//   offsets[0..E]  = exclusive prefix sum of counts, offsets[E] = T*k
//   perm[pos]      = a, listing assignments by expert, then by a (stable)
//   inv_perm[a]    = pos
//   row_token[pos] = a / k; when with_shared, row_token[T*k + t] = t
//   block_map[i]   = {group, first row, rows, 0}: expert e's rows cut into
//                    tiles of block_n, experts in order; then, when
//                    with_shared, the T shared-expert rows as group E.
//   num_tiles      = number of block_map entries.
int oracle_route_meta(const int32_t* ids, int T, int k, int E, int block_n, int with_shared,
                      int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                      int32_t* row_token, int32_t* block_map, int32_t* num_tiles,
                      int max_tiles) {
  const int64_t A = (int64_t)T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t a = 0; a < A; ++a) counts[ids[a]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int64_t pos = 0;
  for (int e = 0; e < E; ++e) {
    if (MUT(9)) {
      for (int64_t a = A - 1; a >= 0; --a)
        if (ids[a] == e) { perm[pos] = (int32_t)a; inv_perm[a] = (int32_t)pos; row_token[pos] = (int32_t)(a / k); ++pos; }
    } else {
      for (int64_t a = 0; a < A; ++a)
        if (ids[a] == e) { perm[pos] = (int32_t)a; inv_perm[a] = (int32_t)pos; row_token[pos] = (int32_t)(a / k); ++pos; }
    }
  }
  if (with_shared)
    for (int t = 0; t < T; ++t) row_token[A + t] = t;
  int n = 0;
  auto emit = [&](int g, int64_t first, int rows) -> bool {
    for (int r0 = 0; r0 < rows; r0 += block_n) {
      if (n >= max_tiles) return false;
      const int r = MUT(10) ? block_n : (rows - r0 < block_n ? rows - r0 : block_n);
      int32_t* m = block_map + 4 * (int64_t)n;
      m[0] = g; m[1] = (int32_t)(first + r0); m[2] = r; m[3] = 0;
      ++n;
    }
    return true;
  };
  for (int e = 0; e < E; ++e)
    if (!emit(e, offsets[e], counts[e])) return -2;
  if (with_shared && !emit(E, A, T)) return -2;
  *num_tiles = n;
  return 0;
}

// One SwiGLU expert (group g of the stacks) applied to T tokens:
// y[t] = (silu(x Wg^T) * (x Wu^T)) Wd^T, fp64 output.
int oracle_expert(const uint16_t* x, int T, int d, int f, int G, int g, const uint32_t* gq,
                  const uint16_t* gs, const uint16_t* gb, const uint32_t* uq, const uint16_t* us,
                  const uint16_t* ub, const uint32_t* dq, const uint16_t* ds, const uint16_t* db,
                  double* y) {
  const W4 gate{gq, gs, gb, f, d, G}, up{uq, us, ub, f, d, G}, down{dq, ds, db, d, f, G};
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < T; ++t) {
    std::vector<double> xt(d);
    for (int kk = 0; kk < d; ++kk) xt[kk] = bf16_value(x[(int64_t)t * d + kk]);
    expert_forward(gate, up, down, g, xt.data(), y + (int64_t)t * d);
  }
  return 0;
}

// The whole layer for T tokens:
//   out[t] = Sum_j w[t][j] * Expert_{ids[t][j]}(x_t) + sigmoid(x_t . w_sg) * Shared(x_t)
// logits_in (optional) replaces the router's own logits (fp32 [T][E]); the
// optional outputs receive the logits, ids, fp32 weights and shared gate.
int oracle_moe_forward(int T, int d, int E, int k, int f, int f_sh, int G, const uint16_t* x,
                       const float* Wr, const float* router_bias, const float* wsg,
                       const uint32_t* gq, const uint16_t* gs, const uint16_t* gb,
                       const uint32_t* uq, const uint16_t* us, const uint16_t* ub,
                       const uint32_t* dq, const uint16_t* ds, const uint16_t* db,
                       const uint32_t* sgq, const uint16_t* sgs, const uint16_t* sgb,
                       const uint32_t* suq, const uint16_t* sus, const uint16_t* sub,
                       const uint32_t* sdq, const uint16_t* sds, const uint16_t* sdb,
                       const float* logits_in, float* out, float* logits_out, int32_t* ids_out,
                       float* w_out, float* gate_out) {
  if (d % 8 || f % 8 || d % G || f % G || k < 1 || k > E) return -1;
  const bool shared = wsg != nullptr;
  if (shared && (f_sh % 8 || f_sh % G)) return -1;
  const W4 gate{gq, gs, gb, f, d, G}, up{uq, us, ub, f, d, G}, down{dq, ds, db, d, f, G};
  const W4 sgate{sgq, sgs, sgb, f_sh, d, G}, sup{suq, sus, sub, f_sh, d, G},
      sdown{sdq, sds, sdb, d, f_sh, G};
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < T; ++t) {
    std::vector<double> xt(d), y(d), acc(d, 0.0), w(k);
    std::vector<float> lg(E);
    std::vector<int32_t> ids(k);
    for (int kk = 0; kk < d; ++kk) xt[kk] = bf16_value(x[(int64_t)t * d + kk]);
    if (logits_in) {
      for (int e = 0; e < E; ++e) lg[e] = logits_in[(int64_t)t * E + e];
    } else {
      for (int e = 0; e < E; ++e) lg[e] = static_cast<float>(router_logit(xt.data(), Wr, d, E, e));
    }
    topk_one(lg.data(), router_bias, E, k, ids.data(), w.data());
    for (int j = 0; j < k; ++j) {
      expert_forward(gate, up, down, ids[j], xt.data(), y.data());
      for (int i = 0; i < d; ++i) acc[i] += (MUT(11) ? 1.0 : w[j]) * y[i];
    }
    double gval = 0.0;
    if (shared) {
      double a = 0.0;
      for (int kk = 0; kk < d; ++kk) a += xt[kk] * wsg[kk];
      const float s = static_cast<float>(a);
      gval = MUT(6) ? (double)s : 1.0 / (1.0 + std::exp(-(double)s));
      expert_forward(sgate, sup, sdown, 0, xt.data(), y.data());
      for (int i = 0; i < d; ++i) acc[i] += gval * y[i];
    }
    for (int i = 0; i < d; ++i) out[(int64_t)t * d + i] = static_cast<float>(acc[i]);
    if (logits_out)
      for (int e = 0; e < E; ++e) logits_out[(int64_t)t * E + e] = lg[e];
    if (ids_out)
      for (int j = 0; j < k; ++j) ids_out[(int64_t)t * k + j] = ids[j];
    if (w_out)
      for (int j = 0; j < k; ++j) w_out[(int64_t)t * k + j] = static_cast<float>(w[j]);
    if (gate_out) gate_out[t] = static_cast<float>(gval);
  }
  return 0;
}

}  // extern "C"
