/*
 * Seeded synthetic inputs: initial weights and token/label streams.
 *
 * This module is shared by the CUDA path's harness and by the oracle. It holds
 * none of the training step's arithmetic: it only turns (seed, stream, index)
 * into numbers, so that both sides see the same bytes.
 *
 * Generator definition (counter-based, so any element can be produced alone
 * and the fill parallelises without changing a single bit):
 *   mix(z)        = SplitMix64 finaliser (Steele, Lea, Flood 2014):
 *                   z ^= z >> 30; z *= 0xbf58476d1ce4e5b9;
 *                   z ^= z >> 27; z *= 0x94d049bb133111eb; z ^= z >> 31
 *   key(seed, s)  = mix(seed ^ mix(s + 1))
 *   word(key, n)  = mix(key + (n + 1) * 0x9e3779b97f4a7c15)   (n-th SplitMix64 output)
 * Normal values (Box-Muller, computed in double):
 *   element pair p uses w1 = word(key, 2p), w2 = word(key, 2p + 1)
 *   u1 = ((w1 >> 11) + 1) * 2^-53  in (0, 1]
 *   u2 =  (w2 >> 11)      * 2^-53  in [0, 1)
 *   rad = sqrt(-2 ln u1);  z[2p] = rad cos(2 pi u2),  z[2p+1] = rad sin(2 pi u2)
 *   value = (float)(z * std), then rounded to bfloat16 to nearest-even.
 * Integers in [0, range) (Lemire's multiply-shift reduction of the top 32 bits):
 *   out[i] = ((word(key, i) >> 32) * range) >> 32
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9e3779b97f4a7c15ULL

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xbf58476d1ce4e5b9ULL;
  z ^= z >> 27;
  z *= 0x94d049bb133111ebULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed ^ mix64(stream + 1));
}

static inline uint64_t word(uint64_t key, uint64_t n) { return mix64(key + (n + 1) * GOLDEN); }

/* float -> bfloat16 bits, round to nearest even (NaN kept quiet). */
static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline void normal_pair(uint64_t key, uint64_t p, double* z0, double* z1) {
  const double two_m53 = 1.0 / 9007199254740992.0;
  uint64_t w1 = word(key, 2 * p), w2 = word(key, 2 * p + 1);
  double u1 = (double)((w1 >> 11) + 1) * two_m53;
  double u2 = (double)(w2 >> 11) * two_m53;
  double rad = sqrt(-2.0 * log(u1));
  double ang = 6.283185307179586476925286766559 * u2;
  *z0 = rad * cos(ang);
  *z1 = rad * sin(ang);
}

/* Fill out[0..n) with bfloat16 N(0, std^2) values of stream `stream`. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, double std_dev, uint16_t* out, int64_t n) {
  const uint64_t key = stream_key(seed, stream);
  const int64_t npairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < npairs; ++p) {
    double z0, z1;
    normal_pair(key, (uint64_t)p, &z0, &z1);
    out[2 * p] = f32_to_bf16_rne((float)(z0 * std_dev));
    if (2 * p + 1 < n) out[2 * p + 1] = f32_to_bf16_rne((float)(z1 * std_dev));
  }
}

/* Fill out[0..n) with the bfloat16 constant `value`. */
void synth_const_bf16(double value, uint16_t* out, int64_t n) {
  const uint16_t b = f32_to_bf16_rne((float)value);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = b;
}

/* Fill out[0..n) with integers uniform in [0, range). */
void synth_uniform_i32(uint64_t seed, uint64_t stream, uint32_t range, int32_t* out, int64_t n) {
  const uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t hi = word(key, (uint64_t)i) >> 32;
    out[i] = (int32_t)((hi * (uint64_t)range) >> 32);
  }
}

/* Zero a byte range in parallel (first touch spreads pages over the cores). */
void synth_zero(void* dst, int64_t nbytes) {
  const int64_t chunk = 1 << 22;
  const int64_t nchunks = (nbytes + chunk - 1) / chunk;
#pragma omp parallel for schedule(static)
  for (int64_t c = 0; c < nchunks; ++c) {
    int64_t off = c * chunk;
    int64_t len = nbytes - off < chunk ? nbytes - off : chunk;
    memset((char*)dst + off, 0, (size_t)len);
  }
}
