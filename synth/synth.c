/*
 * Seeded synthetic inputs for the pruned gated-MLP workloads.
 *
 * This file draws random numbers and rounds them to bf16. It holds none of
 * the FFN arithmetic: both the CPU oracle and the GPU tests take their inputs
 * from here, so that the two sides see the same bytes.
 *
 * Generator (counter based, so any element can be drawn on its own and the
 * result does not depend on the thread count):
 *   key       = mix(mix(seed + G) ^ (tensor_id * 0xD1B54A32D192ED03))
 *   bits(e)   = mix(key + (e + 1) * G)                   G = 0x9E3779B97F4A7C15
 *   u1        = ((bits >> 32) + 1) / 2^32                in (0, 1]
 *   u2        = (bits & 0xffffffff) / 2^32               in [0, 1)
 *   normal(e) = sqrt(-2 ln u1) * cos(2 pi u2)            (Box-Muller, one output per draw)
 * where mix() is the SplitMix64 finaliser (Steele, Lea, Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014).
 *
 * Rounding: double -> float (round to nearest even) -> bf16 (round to nearest
 * even on the top 16 bits). Build with -ffp-contract=off so that no fused
 * multiply-add changes a result between machines.
 */
#include <math.h>
#include <stdint.h>

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
  return mix64(mix64(seed + SYNTH_GOLDEN) ^ (tensor_id * 0xD1B54A32D192ED03ULL));
}

static inline double normal_at(uint64_t key, uint64_t e) {
  uint64_t bits = mix64(key + (e + 1ULL) * SYNTH_GOLDEN);
  double u1 = ((double)(bits >> 32) + 1.0) * (1.0 / 4294967296.0);
  double u2 = (double)(bits & 0xffffffffULL) * (1.0 / 4294967296.0);
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

static inline uint16_t to_bf16(double v) {
  float f = (float)v;
  union { float f; uint32_t u; } c;
  c.f = f;
  uint32_t u = c.u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* out[e] = normal(offset + e) as double, e in [0, n). */
void synth_normal_f64(uint64_t seed, uint64_t tensor_id, uint64_t offset, int64_t n, double* out) {
  uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < n; ++e) out[e] = normal_at(key, offset + (uint64_t)e);
}

/* out[e] = bf16(mean + std * normal(offset + e)). */
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t offset, int64_t n, double mean,
                       double std, uint16_t* out) {
  uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < n; ++e) out[e] = to_bf16(mean + std * normal_at(key, offset + (uint64_t)e));
}

/* Rows of width `cols` with a per-column scale:
 * out[r*cols + c] = bf16(normal(offset + r*cols + c) * scale[c]). */
void synth_scaled_rows_bf16(uint64_t seed, uint64_t tensor_id, uint64_t offset, int64_t rows, int64_t cols,
                            const double* scale, uint16_t* out) {
  uint64_t key = stream_key(seed, tensor_id);
  int64_t n = rows * cols;
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < n; ++e) out[e] = to_bf16(normal_at(key, offset + (uint64_t)e) * scale[e % cols]);
}

/* Rounds doubles to bf16 with the same rule as above. */
void synth_round_bf16(int64_t n, const double* in, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < n; ++e) out[e] = to_bf16(in[e]);
}
