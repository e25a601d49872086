/*
 * Seeded synthetic-input arithmetic shared by the host and device fillers.
 *
 * This header is the whole definition of every synthetic tensor used by the
 * tests and the benchmark. It holds no arithmetic of the decode path itself:
 * only a counter-based random stream and the rounding of its draws to the
 * storage types (bf16, fp32). Both fillers compile this same text, and every
 * step is exact integer arithmetic or a single correctly rounded IEEE
 * operation, so the host and device produce identical bits.
 *
 *  - Random stream: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 *    pseudorandom number generators", OOPSLA 2014; finaliser constants as in
 *    Vigna's public-domain splitmix64.c). Output n of the stream keyed by `key`
 *    is mix(key + (n+1) * 0x9E3779B97F4A7C15), all arithmetic mod 2^64.
 *  - Normal draws: the Irwin–Hall sum of twelve uniforms minus its mean
 *    (mean 0, variance 1 up to 2^-32, tails cut at +-6). Each element takes
 *    stream outputs 3i, 3i+1, 3i+2, split into four 16-bit uniforms each.
 *  - Scaling by sigma and rounding to bf16 / fp32 (round to nearest, ties to
 *    even) from double, done here in integer code so that no compiler or
 *    library rounding mode enters.
 */
#ifndef SYNTH_ARITH_H
#define SYNTH_ARITH_H

#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define SYNTH_FN __host__ __device__ static inline
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ull

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Output n (n >= 0) of the SplitMix64 sequence whose state starts at `key`. */
SYNTH_FN uint64_t synth_stream(uint64_t key, uint64_t n) {
  return synth_mix64(key + (n + 1ull) * SYNTH_GAMMA);
}

/* Key of one synthetic tensor: a function of the global seed and a tensor id. */
SYNTH_FN uint64_t synth_key(uint64_t seed, uint64_t tensor_id) {
  return synth_mix64(synth_mix64(seed + SYNTH_GAMMA) ^ (tensor_id * 0xD1B54A32D192ED03ull + 0x632BE59BD9B4E019ull));
}

/* Approximately standard normal draw for element i: exact multiple of 2^-17. */
SYNTH_FN double synth_normal(uint64_t key, uint64_t i) {
  int64_t s = 0;
  for (int j = 0; j < 3; ++j) {
    uint64_t r = synth_stream(key, 3ull * i + (uint64_t)j);
    s += (int64_t)(r & 0xFFFFu) + (int64_t)((r >> 16) & 0xFFFFu) +
         (int64_t)((r >> 32) & 0xFFFFu) + (int64_t)(r >> 48);
  }
  const int64_t num = 2 * s - 12 * 65535; /* |num| < 2^21: exact in double */
  return (double)num * 0x1p-17;           /* power-of-two scale: exact */
}

SYNTH_FN uint64_t synth_f64_bits(double v) {
  uint64_t b;
  memcpy(&b, &v, sizeof b);
  return b;
}

/*
 * Round a finite double to a binary format with an 8-bit exponent (bias 127)
 * and `mbits` stored mantissa bits, nearest-even. mbits = 7 gives bfloat16,
 * mbits = 23 gives IEEE binary32. Returns the encoded bits.
 */
SYNTH_FN uint32_t synth_round_e8(double v, int mbits) {
  const uint64_t b = synth_f64_bits(v);
  const uint32_t sign = (uint32_t)(b >> 63) << (8 + mbits);
  const int e = (int)((b >> 52) & 0x7FF);
  if (e == 0) return sign; /* zero (double subnormals are far below range) */
  const uint64_t sig = (b & 0xFFFFFFFFFFFFFull) | (1ull << 52);
  int be = e - 1023 + 127;
  int shift = 52 - mbits;
  if (be <= 0) { /* result is subnormal in the target format */
    shift += 1 - be;
    be = 0;
  }
  if (shift > 62) return sign;
  uint64_t q = sig >> shift;
  const uint64_t rem = sig & ((1ull << shift) - 1ull);
  const uint64_t half = 1ull << (shift - 1);
  if (rem > half || (rem == half && (q & 1ull))) q += 1ull;
  if (be == 0) return sign | (uint32_t)q; /* may carry into the exponent: still right */
  if (q >> (mbits + 1)) {
    q >>= 1;
    be += 1;
  }
  if (be >= 255) return sign | (0xFFu << mbits);
  return sign | ((uint32_t)be << mbits) | (uint32_t)(q & ((1ull << mbits) - 1ull));
}

SYNTH_FN uint16_t synth_bf16(uint64_t key, uint64_t i, double sigma) {
  return (uint16_t)synth_round_e8(synth_normal(key, i) * sigma, 7);
}

SYNTH_FN uint32_t synth_f32(uint64_t key, uint64_t i, double sigma) {
  return synth_round_e8(synth_normal(key, i) * sigma, 23);
}

#endif /* SYNTH_ARITH_H */
