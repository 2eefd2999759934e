/*
 * Seeded synthetic inputs for the 4-bit MoE layer (inputs only: no routing,
 * dequantisation or expert arithmetic lives here).
 *
 * Every value is a pure function of (key, element index), so any slice of a
 * tensor (one expert, one token) can be regenerated without producing the
 * rest, and results do not depend on the number of OpenMP threads.
 *
 * Generator: the i-th output of a splitmix64 stream seeded with `key`
 * (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014): z = key + (i+1)*0x9E3779B97F4A7C15 followed by the
 * splitmix64 finaliser.  Normals use the Box-Muller transform (cosine
 * branch, one normal per pair of uniforms) in double precision.
 *
 * bf16 values are produced by round-to-nearest-even of the fp32 value.
 */
#include <math.h>
#include <stdint.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_at(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * GOLDEN);
}

/* uniform in [0, 1) with 53 random bits */
static inline double unif01(uint64_t h) { return (double)(h >> 11) * 0x1.0p-53; }

static inline double normal_at(uint64_t key, uint64_t i) {
  double u1 = ((double)(stream_at(key, 2 * i) >> 11) + 1.0) * 0x1.0p-53; /* (0,1] */
  double u2 = unif01(stream_at(key, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t lsb = (v.u >> 16) & 1u;
  v.u += 0x7FFFu + lsb;
  return (uint16_t)(v.u >> 16);
}

static inline float bf16_to_f32(uint16_t b) {
  union { float f; uint32_t u; } v;
  v.u = ((uint32_t)b) << 16;
  return v.f;
}

uint64_t synth_key(uint64_t seed, uint64_t layer, uint64_t tensor) {
  uint64_t k = mix64(seed + GOLDEN);
  k = mix64(k ^ (layer + 2 * GOLDEN));
  return mix64(k ^ (tensor + 3 * GOLDEN));
}

/* out[j] = float(sigma * N(0,1)) for element off+j */
void synth_normal_f32(uint64_t key, int64_t off, int64_t n, double sigma, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) out[j] = (float)(sigma * normal_at(key, (uint64_t)(off + j)));
}

/* out[j] = bf16(float(sigma * N(0,1))) */
void synth_normal_bf16(uint64_t key, int64_t off, int64_t n, double sigma, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j)
    out[j] = f32_to_bf16_rne((float)(sigma * normal_at(key, (uint64_t)(off + j))));
}

/* packed words of eight uniform 4-bit codes: the high 32 bits of each draw */
void synth_q4(uint64_t key, int64_t off, int64_t nwords, uint32_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nwords; ++j)
    out[j] = (uint32_t)(stream_at(key, (uint64_t)(off + j)) >> 32);
}

/*
 * Per-group scale ~ U[lo, hi] rounded to bf16, and
 * bias = bf16(float(-8 * scale_bf16 + noise * N(0,1))), the affine offset
 * that centres the codes 0..15 near zero.
 */
void synth_scale_bias(uint64_t key_s, uint64_t key_b, int64_t off, int64_t n, double lo,
                      double hi, double noise, uint16_t* scale, uint16_t* bias) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) {
    uint64_t i = (uint64_t)(off + j);
    uint16_t s = f32_to_bf16_rne((float)(lo + (hi - lo) * unif01(stream_at(key_s, i))));
    double b = -8.0 * (double)bf16_to_f32(s) + noise * normal_at(key_b, i);
    scale[j] = s;
    bias[j] = f32_to_bf16_rne((float)b);
  }
}

/* uniform integers in [0, n_range) (used for random tie and permutation tests) */
void synth_uniform_int(uint64_t key, int64_t off, int64_t n, uint32_t n_range, int32_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j)
    out[j] = (int32_t)((stream_at(key, (uint64_t)(off + j)) >> 32) % n_range);
}
