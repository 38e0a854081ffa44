/*
 * synth_core.h - counter-based seeded input generator.
 *
 * This header is the single definition of the synthetic inputs used by the
 * tests, the bench and the CPU oracle's callers.  It holds no arithmetic of
 * the decode-MLP method itself: only pseudo-random numbers, the shape of their
 * distribution, and the fp32 -> bf16 storage conversion of activations.
 *
 * It compiles as plain C (host, gcc, built with -ffp-contract=off) and as CUDA
 * device code, and produces bit-identical values on both, because every
 * floating-point step is one IEEE-754 operation with round-to-nearest-even:
 *
 *   draw(seed, c)  = mix64(seed + (c + 1) * 0x9E3779B97F4A7C15)   (mod 2^64)
 *     mix64 is the SplitMix64 output function (Steele, Lea, Flood, "Fast
 *     splittable pseudorandom number generators", OOPSLA 2014), so draw() is
 *     the c-th output of a SplitMix64 stream started at `seed`.
 *   z(i)           = (S_i - 393210) * 2^-16,  S_i = sum of the twelve 16-bit
 *     fields of draw(seed, 4i), draw(seed, 4i+1), draw(seed, 4i+2).
 *     This is the Irwin-Hall "sum of twelve uniforms" approximation of a
 *     standard normal: mean 0, variance (65536^2 - 1)/65536^2, support
 *     [-6, 6].  The integer difference is below 2^19, so z is exact in fp32.
 *   normal(i)      = fl(mean + fl(z(i) * std))   (one rounding per operation;
 *     the add is skipped when mean == 0)
 *   outliers       : if (draw(seed, 4i+3) >> 32) < p32 then value = fl(value *
 *     outlier_scale)   (a Bernoulli(p32 / 2^32) mask)
 *   bf16 storage   : round-to-nearest-even of the fp32 bit pattern.
 *
 * Element i of a row-major [N][K] tensor is element n*K + k, so any row range
 * can be regenerated on its own.
 */
#ifndef MT_SYNTH_CORE_H
#define MT_SYNTH_CORE_H

#include <stdint.h>

#ifdef __CUDACC__
#define SYN_FN static __host__ __device__ __forceinline__
#else
#define SYN_FN static inline
#endif

#define SYN_GOLDEN 0x9E3779B97F4A7C15ULL
#define SYN_IH_MEAN 393210 /* 12 * 65535 / 2 */

SYN_FN uint64_t syn_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

SYN_FN uint64_t syn_draw(uint64_t seed, uint64_t ctr) {
  return syn_mix64(seed + (ctr + 1ULL) * SYN_GOLDEN);
}

SYN_FN int32_t syn_fields16(uint64_t r) {
  return (int32_t)(r & 0xFFFF) + (int32_t)((r >> 16) & 0xFFFF) +
         (int32_t)((r >> 32) & 0xFFFF) + (int32_t)(r >> 48);
}

SYN_FN float syn_mul(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fmul_rn(a, b);
#else
  return a * b;
#endif
}

SYN_FN float syn_add(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fadd_rn(a, b);
#else
  return a + b;
#endif
}

/* Standard-normal approximation for element i (exact in fp32). */
SYN_FN float syn_z(uint64_t seed, uint64_t i) {
  int32_t s = syn_fields16(syn_draw(seed, 4 * i)) +
              syn_fields16(syn_draw(seed, 4 * i + 1)) +
              syn_fields16(syn_draw(seed, 4 * i + 2));
  return (float)(s - SYN_IH_MEAN) * (1.0f / 65536.0f);
}

SYN_FN float syn_value(uint64_t seed, uint64_t i, float mean, float stdv,
                       uint32_t outlier_p32, float outlier_scale) {
  float v = syn_mul(syn_z(seed, i), stdv);
  if (mean != 0.0f) v = syn_add(mean, v);
  if (outlier_p32 != 0u) {
    uint32_t u = (uint32_t)(syn_draw(seed, 4 * i + 3) >> 32);
    if (u < outlier_p32) v = syn_mul(v, outlier_scale);
  }
  return v;
}

SYN_FN uint32_t syn_f32_bits(float f) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(f);
#else
  union { float f; uint32_t u; } c;
  c.f = f;
  return c.u;
#endif
}

/* fp32 -> bf16 storage conversion, round to nearest even; NaN -> quiet NaN. */
SYN_FN uint16_t syn_bf16(float f) {
  uint32_t u = syn_f32_bits(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
    return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

#endif /* MT_SYNTH_CORE_H */
