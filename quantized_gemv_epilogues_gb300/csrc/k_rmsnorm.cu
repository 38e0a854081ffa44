// k_rmsnorm.cu - K1: residual add + RMSNorm as one multi-output kernel.
//
// meTile docs, "Compute-Graph Fusion" (opening example): summed = values +
// residual and normalized = rms_norm(summed, weight, eps) are both graph
// outputs, so the fused kernel writes both.  "MLX-LM Backend", Dispatch
// Policy: RMSNorm over BF16 values with FP32 accumulation.
//
// One CTA per row.  Each thread owns CPT 16-byte chunks (8 bf16) of the row,
// keeps the rounded sum in registers between the two passes, and the sum of
// squares is reduced with warp shuffles and one shared-memory step.
#include "mt_device.cuh"
#include "mt_internal.h"

namespace mt {

template <int CPT, bool NORM_F32>
__global__ void __launch_bounds__(1024) add_rmsnorm_kernel(
    const uint16_t* __restrict__ v, const uint16_t* __restrict__ r,
    const uint16_t* __restrict__ w, float eps, uint16_t* out_sum, void* out_norm, int d) {
  __shared__ float warp_ss[32];
  pdl_trigger();
  const int m = blockIdx.x;
  const int nch = d >> 3;
  const size_t row = (size_t)m * d;

  // The gain is static: read it before waiting for the preceding kernel.
  uint4 wv[CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * blockDim.x;
    wv[j] = c < nch ? ldg_nc(w + (size_t)c * 8) : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();

  uint4 sv[CPT];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * blockDim.x;
    sv[j] = make_uint4(0, 0, 0, 0);
    if (c < nch) {
      // plain (coherent) loads: out_sum may alias residual
      const uint4 a = *reinterpret_cast<const uint4*>(v + row + (size_t)c * 8);
      const uint4 b = *reinterpret_cast<const uint4*>(r + row + (size_t)c * 8);
      const uint32_t* aw = &a.x;
      const uint32_t* bw = &b.x;
      uint32_t* sw = &sv[j].x;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // fp32 sum of two bf16 values, rounded once to bf16
        const uint16_t lo = f2bf(bf16lo(aw[i]) + bf16lo(bw[i]));
        const uint16_t hi = f2bf(bf16hi(aw[i]) + bf16hi(bw[i]));
        const float flo = bf16f(lo), fhi = bf16f(hi);
        ss = fmaf(flo, flo, ss);
        ss = fmaf(fhi, fhi, ss);
        sw[i] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      *reinterpret_cast<uint4*>(out_sum + row + (size_t)c * 8) = sv[j];
    }
  }

#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) warp_ss[warp] = ss;
  __syncthreads();
  const int nwarps = (blockDim.x + 31) >> 5;
  float tot = 0.f;
  for (int i = 0; i < nwarps; ++i) tot += warp_ss[i];
  const float inv = rsqrtf(tot / (float)d + eps);

#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * blockDim.x;
    if (c >= nch) continue;
    const uint32_t* sw = &sv[j].x;
    const uint32_t* ww = &wv[j].x;
    float o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = bf16lo(sw[i]) * inv * bf16lo(ww[i]);
      o[2 * i + 1] = bf16hi(sw[i]) * inv * bf16hi(ww[i]);
    }
    if (NORM_F32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out_norm) + row + (size_t)c * 8);
      dst[0] = make_float4(o[0], o[1], o[2], o[3]);
      dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    } else {
      uint4 pk;
      uint32_t* pw = &pk.x;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        pw[i] = (uint32_t)f2bf(o[2 * i]) | ((uint32_t)f2bf(o[2 * i + 1]) << 16);
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out_norm) + row + (size_t)c * 8) = pk;
    }
  }
}

template <int CPT>
static mt_status go(const uint16_t* v, const uint16_t* r, const uint16_t* w, float eps,
                    uint16_t* out_sum, void* out_norm, int M, int d, bool f32, int threads,
                    const Launch& l) {
  if (f32)
    return launch(add_rmsnorm_kernel<CPT, true>, dim3(M), dim3(threads), 0, l, v, r, w, eps,
                  out_sum, out_norm, d);
  return launch(add_rmsnorm_kernel<CPT, false>, dim3(M), dim3(threads), 0, l, v, r, w, eps,
                out_sum, out_norm, d);
}

mt_status launch_add_rmsnorm(const uint16_t* v, const uint16_t* r, const uint16_t* w, float eps,
                             uint16_t* out_sum, void* out_norm, int M, int d, bool norm_f32,
                             const Launch& l) {
  const int nch = d / 8;
  int cpt = 1;
  while (cpt < 8 && nch > cpt * 1024) cpt *= 2;
  int threads = (nch + cpt - 1) / cpt;
  threads = ((threads + 31) / 32) * 32;
  if (threads > 1024) threads = 1024;
  switch (cpt) {
    case 1: return go<1>(v, r, w, eps, out_sum, out_norm, M, d, norm_f32, threads, l);
    case 2: return go<2>(v, r, w, eps, out_sum, out_norm, M, d, norm_f32, threads, l);
    case 4: return go<4>(v, r, w, eps, out_sum, out_norm, M, d, norm_f32, threads, l);
    default: return go<8>(v, r, w, eps, out_sum, out_norm, M, d, norm_f32, threads, l);
  }
}

}  // namespace mt
