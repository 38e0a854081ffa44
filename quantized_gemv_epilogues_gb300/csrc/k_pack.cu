// k_pack.cu - affine group quantiser / packer and the matching dequantiser.
//
// meTile docs, "MLX-LM Backend": affine INT8 and 4-bit "affine nibbles,
// scales, and biases", groups of 32, 64 and 128 along K, prepared ahead of
// time.  Per group, in binary64:
//   bias  = bf16(min)   (a zero minimum gives the bias +0)
//   scale = bf16((max - min) / (2^bits - 1))
//   q     = clamp(round_half_even((w - bias) / scale), 0, 2^bits - 1),
//           and q = 0 when scale == 0.
// Stored layout: INT8 one code per byte; INT4 byte j of a row holds code 2j
// in bits 0..3 and code 2j+1 in bits 4..7.
//
// One warp per group.  Every step is an IEEE binary64 operation with explicit
// round-to-nearest intrinsics, so the codes do not depend on the compiler's
// contraction choices.
#include <math.h>

#include "mt_device.cuh"
#include "mt_internal.h"

namespace mt {

// binary64 -> bf16, round to nearest even, by integer operations on the
// binary64 fields: keep the top 8 significant bits (fewer for bf16
// subnormals), round on the discarded bits.
__device__ uint16_t bf16_rne_from_f64(double x) {
  const unsigned long long u = (unsigned long long)__double_as_longlong(x);
  const uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
  const unsigned long long mag = u & 0x7FFFFFFFFFFFFFFFull;
  if (mag > 0x7FF0000000000000ull) return (uint16_t)(sign | 0x7FC0u);
  if (mag == 0x7FF0000000000000ull) return (uint16_t)(sign | 0x7F80u);
  const int E = (int)(mag >> 52);
  if (E == 0) return sign;  // binary64 subnormal or zero: below half a bf16 unit
  const int e = E - 1023;
  const unsigned long long sig = (mag & 0xFFFFFFFFFFFFFull) | (1ull << 52);
  if (e >= -126) {
    unsigned long long keep = sig >> 45;
    const unsigned long long rem = sig & ((1ull << 45) - 1), half = 1ull << 44;
    if (rem > half || (rem == half && (keep & 1ull))) ++keep;
    int be = e + 127;
    if (keep == 256ull) { keep = 128ull; ++be; }
    if (be >= 255) return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (uint16_t)(be << 7) | (uint16_t)(keep & 0x7Fu));
  }
  const int sh = -81 - e;  // bf16 subnormal: value / 2^-133 = sig >> sh
  if (sh > 54) return sign;
  unsigned long long keep = sig >> sh;
  const unsigned long long rem = sig & ((1ull << sh) - 1), half = 1ull << (sh - 1);
  if (rem > half || (rem == half && (keep & 1ull))) ++keep;
  return (uint16_t)(sign | (uint16_t)keep);
}

__device__ __forceinline__ double bf16_to_f64(uint16_t h) {
  return (double)__uint_as_float((uint32_t)h << 16);
}

template <int BITS>
__global__ void __launch_bounds__(256) pack_affine_kernel(const float* __restrict__ W, int N, int K,
                                                           int group, uint8_t* __restrict__ q,
                                                           uint16_t* __restrict__ s,
                                                           uint16_t* __restrict__ b) {
  pdl_wait();
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int G = K / group;
  if (gw >= (long long)N * G) return;
  const long long n = gw / G;
  const int gi = (int)(gw - n * G);
  const float* src = W + n * K + (long long)gi * group;
  const int npairs = group >> 1;

  float mn = INFINITY, mx = -INFINITY;
  for (int p = lane; p < npairs; p += 32) {
    const float2 v = *reinterpret_cast<const float2*>(src + 2 * p);
    mn = fminf(mn, fminf(v.x, v.y));
    mx = fmaxf(mx, fmaxf(v.x, v.y));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  double dmn = (double)mn;
  if (dmn == 0.0) dmn = 0.0;  // a zero minimum is +0
  const double dmx = (double)mx;
  const double qmax = (double)((1 << BITS) - 1);
  const uint16_t b16 = bf16_rne_from_f64(dmn);
  const uint16_t s16 = bf16_rne_from_f64(__ddiv_rn(__dsub_rn(dmx, dmn), qmax));
  const double bias = bf16_to_f64(b16), scale = bf16_to_f64(s16);
  if (lane == 0) {
    s[n * G + gi] = s16;
    b[n * G + gi] = b16;
  }
  for (int p = lane; p < npairs; p += 32) {
    const float2 v = *reinterpret_cast<const float2*>(src + 2 * p);
    uint32_t c[2];
    const float vv[2] = {v.x, v.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      double t = 0.0;
      if (scale != 0.0) {
        t = rint(__ddiv_rn(__dsub_rn((double)vv[i], bias), scale));
        t = fmin(fmax(t, 0.0), qmax);
      }
      c[i] = (uint32_t)t;
    }
    const long long k = (long long)gi * group + 2 * p;
    if (BITS == 8) {
      *reinterpret_cast<uint16_t*>(q + n * K + k) = (uint16_t)(c[0] | (c[1] << 8));
    } else {
      q[n * (K / 2) + k / 2] = (uint8_t)(c[0] | (c[1] << 4));
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(256) unpack_affine_kernel(const uint8_t* __restrict__ q,
                                                             const uint16_t* __restrict__ s,
                                                             const uint16_t* __restrict__ b, int N,
                                                             int K, int group, float* __restrict__ W) {
  pdl_wait();
  const long long total = (long long)N * K;
  const int G = K / group;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long n = i / K;
    const int k = (int)(i - n * K);
    uint32_t code;
    if (BITS == 8) {
      code = q[i];
    } else {
      const uint8_t byte = q[n * (K / 2) + k / 2];
      code = (k & 1) ? (byte >> 4) : (byte & 0xF);
    }
    const float sc = bf16f(s[n * G + k / group]), bi = bf16f(b[n * G + k / group]);
    W[i] = fmaf(sc, (float)code, bi);
  }
}

mt_status launch_pack_affine(const float* W, int N, int K, int group, int bits, uint8_t* q,
                             uint16_t* s, uint16_t* b, const Launch& l) {
  const long long groups = (long long)N * (K / group);
  if (groups == 0) return MT_OK;
  const long long blocks = (groups + 7) / 8;
  if (blocks > 0x7FFFFFFFll) return MT_ERR_SHAPE;
  if (bits == 8)
    return launch(pack_affine_kernel<8>, dim3((unsigned)blocks), dim3(256), 0, l, W, N, K, group, q, s, b);
  return launch(pack_affine_kernel<4>, dim3((unsigned)blocks), dim3(256), 0, l, W, N, K, group, q, s, b);
}

mt_status launch_unpack_affine(const uint8_t* q, const uint16_t* s, const uint16_t* b, int N,
                               int K, int group, int bits, float* W, const Launch& l) {
  const long long total = (long long)N * K;
  if (total == 0) return MT_OK;
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (bits == 8)
    return launch(unpack_affine_kernel<8>, dim3((unsigned)blocks), dim3(256), 0, l, q, s, b, N, K, group, W);
  return launch(unpack_affine_kernel<4>, dim3((unsigned)blocks), dim3(256), 0, l, q, s, b, N, K, group, W);
}

// ------------------------------------------------------------ MX packer
//
// meTile docs, "MLX-LM Backend", Block-Scaled MLX Primitive: MXFP8 / MXFP4
// weights quantised ahead of time, E4M3 / E2M1 values with E8M0 scales.  The
// encodings and the block of 32 elements along K are those of the OCP
// Microscaling Formats (MX) v1.0 specification named by the format:
//   scale field E = clamp(floor(log2(amax)) - emax + 127, 0, 254), emax the
//                   element format's largest exponent (8 for E4M3, 2 for
//                   E2M1); an all-zero block takes E = 0
//   element       = w / 2^(E - 127) rounded to nearest-even in the element
//                   format, magnitudes above its largest finite value clamped
//                   to it, the sign kept.
// One warp per block, one element per lane; the rounding is done in binary64
// (the division by a power of two is exact there).

// floor(log2(a)) of a positive finite float (subnormals included).
__device__ __forceinline__ int floor_log2_pos(float a) {
  const uint32_t u = __float_as_uint(a);
  const int e = (int)(u >> 23);
  return e ? e - 127 : (31 - __clz((int)u)) - 149;
}

// Nearest E4M3 code (sign, 4 exponent bits with bias 7, 3 fraction bits).
__device__ uint8_t e4m3_rne(double v) {
  const uint8_t sign = signbit(v) ? 0x80 : 0;
  const double a = fabs(v);
  if (!(a < 448.0)) return (uint8_t)(sign | 0x7E);  // the largest finite, 448
  if (a < 0x1p-6) return (uint8_t)(sign | (int)rint(a * 512.0));  // multiples of 2^-9; 8 = 2^-6
  int e = ilogb(a);                        // a in [2^e, 2^(e+1)), -6 <= e <= 8
  int m = (int)rint(ldexp(a, 3 - e));      // 8 .. 16
  if (m == 16) { m = 8; ++e; }
  return (uint8_t)(sign | ((e + 7) << 3) | (m - 8));
}

// Nearest E2M1 code (sign, 2 exponent bits with bias 1, 1 fraction bit).
__device__ uint8_t e2m1_rne(double v) {
  const uint8_t sign = signbit(v) ? 8 : 0;
  const double a = fabs(v);
  if (!(a < 6.0)) return (uint8_t)(sign | 7);  // the largest finite, 6
  if (a < 1.0) return (uint8_t)(sign | (int)rint(a * 2.0));  // 0, 0.5; 2 = 1.0
  int e = ilogb(a);                        // 0 .. 2
  int m = (int)rint(ldexp(a, 1 - e));      // 2 .. 4
  if (m == 4) { m = 2; ++e; }
  return (uint8_t)(sign | ((e + 1) << 1) | (m - 2));
}

template <int BITS>
__global__ void __launch_bounds__(256) pack_mx_kernel(const float* __restrict__ W, int N, int K,
                                                       uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  const int lane = threadIdx.x & 31;
  const long long nb = (long long)N * (K / 32);
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long b = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nb; b += warps) {
    const long long n = b / (K / 32), kb = b - n * (K / 32);
    const float w = W[n * K + kb * 32 + lane];
    float amax = fabsf(w);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    constexpr int EMAX = BITS == 8 ? 8 : 2;
    const int E = amax > 0.f ? max(0, min(254, floor_log2_pos(amax) - EMAX + 127)) : 0;
    const double v = ldexp((double)w, 127 - E);
    const uint32_t c = BITS == 8 ? e4m3_rne(v) : e2m1_rne(v);
    if (BITS == 8) {
      q[n * K + kb * 32 + lane] = (uint8_t)c;
    } else {
      const uint32_t hi = __shfl_down_sync(0xffffffffu, c, 1);
      if ((lane & 1) == 0) q[n * (K / 2) + kb * 16 + (lane >> 1)] = (uint8_t)(c | (hi << 4));
    }
    if (lane == 0) s[b] = (uint8_t)E;
  }
}

mt_status launch_pack_mx(const float* W, int N, int K, int bits, uint8_t* q, uint8_t* s,
                         const Launch& l) {
  const long long nb = (long long)N * (K / 32);
  if (nb == 0) return MT_OK;
  long long blocks = (nb + 7) / 8;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (bits == 8) return launch(pack_mx_kernel<8>, dim3((unsigned)blocks), dim3(256), 0, l, W, N, K, q, s);
  return launch(pack_mx_kernel<4>, dim3((unsigned)blocks), dim3(256), 0, l, W, N, K, q, s);
}

}  // namespace mt
