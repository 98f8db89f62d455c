/*
 * Seeded synthetic inputs for the KDA recurrence, shared by the fp64 oracle's
 * tests and by the GPU tests / benchmark.  This file holds no arithmetic of the
 * recurrence itself: it only draws numbers and rounds them to storage types.
 *
 * Generator (counter based, so any slice can be regenerated on its own):
 *   - SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom
 *     number generators", OOPSLA 2014; constants of S. Vigna's splitmix64.c):
 *     the n-th output of a stream with key K is mix64(K + (n + 1) * 0x9E3779B97F4A7C15).
 *   - Box-Muller (G. Box, M. Muller, 1958): element i of a stream uses the outputs
 *     2i and 2i+1, u1 = (a >> 11 + 1) * 2^-53 in (0, 1], u2 = (b >> 11) * 2^-53 in [0, 1),
 *     x = sqrt(-2 ln u1) * cos(2 pi u2).
 * Storage rounding: fp64 -> fp32 round-to-nearest, then fp32 -> bf16 round-to-nearest-even.
 *
 * Everything is plain C99 with OpenMP; compile with -ffp-contract=off so that
 * x86-64 and aarch64 hosts give the same bits.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_F32 0
#define SYNTH_BF16 1
#define SYNTH_F64 2

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t sm64_at(uint64_t key, uint64_t n) {
  return mix64(key + (n + 1ULL) * 0x9E3779B97F4A7C15ULL);
}

/* Key of stream `stream` under `seed`: two SplitMix64 draws, so nearby seeds
 * and streams give unrelated keys. */
uint64_t synth_stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed * 0x9E3779B97F4A7C15ULL + 0x632BE59BD9B4E019ULL) ^ (stream * 0xD1B54A32D192ED03ULL + 1ULL));
}

static inline double normal_at(uint64_t key, uint64_t i) {
  const uint64_t a = sm64_at(key, 2ULL * i);
  const uint64_t b = sm64_at(key, 2ULL * i + 1ULL);
  const double u1 = (double)((a >> 11) + 1ULL) * 0x1.0p-53;
  const double u2 = (double)(b >> 11) * 0x1.0p-53;
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) {            /* inf or nan */
    return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  }
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline void store_as(void* out, int dtype, int64_t i, double x) {
  if (dtype == SYNTH_F64) {
    ((double*)out)[i] = x;
  } else if (dtype == SYNTH_F32) {
    ((float*)out)[i] = (float)x;
  } else {
    ((uint16_t*)out)[i] = f32_to_bf16_rne((float)x);
  }
}

/* Raw standard normals, counter indices [offset, offset + n), as fp64. */
void synth_normal_f64(uint64_t seed, uint64_t stream, int64_t offset, int64_t n, double* out) {
  const uint64_t key = synth_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = normal_at(key, (uint64_t)(offset + i));
}

/*
 * Rows of `d` values.  Row r of the output is logical row
 * first_row + r * row_stride of the stream (logical row R covers counter
 * indices [R*d, R*d + d)).  Each value is scale * N(0,1); with unit_norm != 0
 * the row is first divided by its fp64 Euclidean norm (an all-zero row is kept
 * as zeros).  Results are rounded to `dtype`.  Returns 0 on success.
 */
int synth_rows(uint64_t seed, uint64_t stream, int64_t first_row, int64_t row_stride, int64_t nrows,
               int32_t d, double scale, int32_t unit_norm, int32_t dtype, void* out) {
  if (d <= 0 || d > 4096 || nrows < 0) return 1;
  if (dtype != SYNTH_F32 && dtype != SYNTH_BF16 && dtype != SYNTH_F64) return 1;
  const uint64_t key = synth_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r) {
    double buf[4096];
    const uint64_t row = (uint64_t)(first_row + r * row_stride);
    double ss = 0.0;
    for (int32_t j = 0; j < d; ++j) {
      buf[j] = scale * normal_at(key, row * (uint64_t)d + (uint64_t)j);
      ss += buf[j] * buf[j];
    }
    double inv = 1.0;
    if (unit_norm && ss > 0.0) inv = 1.0 / sqrt(ss);
    for (int32_t j = 0; j < d; ++j) store_as(out, dtype, r * (int64_t)d + j, buf[j] * inv);
  }
  return 0;
}

/* Per-element sigmoid(N(0,1)) in fp32 (the write strengths), counter indices
 * first + r * stride for r in [0, n). */
int synth_sigmoid_normal_f32(uint64_t seed, uint64_t stream, int64_t first, int64_t stride, int64_t n,
                             float* out) {
  if (n < 0) return 1;
  const uint64_t key = synth_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    const double x = normal_at(key, (uint64_t)(first + r * stride));
    out[r] = (float)(1.0 / (1.0 + exp(-x)));
  }
  return 0;
}

/* fp32 -> bf16 (round to nearest even), the rounding every bf16 value of this
 * module goes through. */
void synth_f32_to_bf16(const float* in, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

/* Uniforms in [0, 1): (x >> 11) * 2^-53 of outputs first + r*stride. */
void synth_uniform_f64(uint64_t seed, uint64_t stream, int64_t first, int64_t n, double* out) {
  const uint64_t key = synth_stream_key(seed, stream);
  for (int64_t r = 0; r < n; ++r) out[r] = (double)(sm64_at(key, (uint64_t)(first + r)) >> 11) * 0x1.0p-53;
}
