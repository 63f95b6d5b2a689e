/*
 * Seeded, counter-based synthetic inputs for the selective-scan workloads.
 *
 * This file draws random numbers and encodes them; it contains none of the
 * scan's arithmetic.  Both the fp64 oracle and the CUDA path read arrays
 * produced here, so the two sides always see bit-identical inputs.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014).  Element i of stream s under seed k is
 *     w(k, s, i) = mix64(key(k, s) + (i + 1) * GAMMA),
 *     key(k, s)  = mix64(k * GAMMA ^ (s << 40) ^ 0x5DEECE66D),
 * i.e. the (i+1)-th output of a SplitMix64 sequence whose state starts at
 * key(k, s).  Any slice of any tensor can be regenerated on its own.
 *
 * Uniforms use the top 53 bits: U = (w >> 11) * 2^-53 + 2^-54, in (0, 1).
 * Normals use the Box-Muller transform (Box & Muller, 1958) on the two
 * uniforms drawn from words 2i and 2i+1: z = sqrt(-2 ln U1) cos(2 pi U2).
 * Values are formed in double, rounded to float (round to nearest even),
 * and, for bfloat16 tensors, rounded again to bfloat16 (round to nearest
 * even on the float bit pattern; NaN never occurs for these draws).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * GAMMA ^ (stream << 40) ^ 0x5DEECE66DULL);
}

static inline double uniform01(uint64_t key, uint64_t i) {
  uint64_t w = mix64(key + (i + 1) * GAMMA);
  return (double)(w >> 11) * 0x1.0p-53 + 0x1.0p-54;
}

static inline double normal01(uint64_t key, uint64_t i) {
  double u1 = uniform01(key, 2 * i), u2 = uniform01(key, 2 * i + 1);
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  union { float f; uint32_t u; } v = {f};
  uint32_t lsb = (v.u >> 16) & 1u;
  return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

/* kind: 0 = normal(p0 = mean, p1 = std); 1 = uniform(p0 = lo, p1 = hi);
 *       2 = log-uniform(p0 = lo, p1 = hi), i.e. exp(U(ln lo, ln hi)). */
static inline double draw(int kind, uint64_t key, uint64_t i, double p0, double p1) {
  if (kind == 0) return p0 + p1 * normal01(key, i);
  double u = uniform01(key, i);
  if (kind == 1) return p0 + (p1 - p0) * u;
  return exp(log(p0) + (log(p1) - log(p0)) * u);
}

/* Fill out[0..n) with elements offset..offset+n of (seed, stream), as float. */
void synth_fill_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                    int kind, double p0, double p1, float* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) out[j] = (float)draw(kind, key, offset + (uint64_t)j, p0, p1);
}

/* Same draws, stored as bfloat16 bit patterns. */
void synth_fill_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                     int kind, double p0, double p1, uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j)
    out[j] = f32_to_bf16_rne((float)draw(kind, key, offset + (uint64_t)j, p0, p1));
}

/* Same draws, kept in double (used where a recipe transforms a draw). */
void synth_fill_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                    int kind, double p0, double p1, double* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) out[j] = draw(kind, key, offset + (uint64_t)j, p0, p1);
}

/* Raw 64-bit words, for tests of the generator itself. */
void synth_words(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint64_t* out) {
  uint64_t key = stream_key(seed, stream);
  for (int64_t j = 0; j < n; ++j) out[j] = mix64(key + (offset + (uint64_t)j + 1) * GAMMA);
}

/* float -> bfloat16 bits (round to nearest even); exposed for the encoder test. */
void synth_f32_to_bf16(const float* in, int64_t n, uint16_t* out) {
  for (int64_t j = 0; j < n; ++j) out[j] = f32_to_bf16_rne(in[j]);
}
