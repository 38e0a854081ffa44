// k_gemv_warp.cuh - one-row (M == 1) GEMV with the SwiGLU or residual
// epilogue as a single kernel: one warp-task phase (k_phase.cuh) between
// programmatic-dependent-launch edges.
//
// meTile docs, "Compute-Graph Fusion", Automatic Gated Epilogues (gate and up
// share the activation, silu(gate) * up before the only store; the down
// projection adds the residual in its epilogue); "MLX-LM Backend", Dispatch
// Policy (affine w = scale * q + bias per group of 32/64/128 along K).
//
// The weights of a CTA's first two tasks and its scales and biases are
// requested before the kernel waits for the preceding kernel on the stream;
// x, the residual and the output follow that wait.  No thread waits on
// another CTA or on a flag: the only waits are cp.async group completions and
// CTA barriers.
#pragma once
#include "k_phase.cuh"

namespace mt {

struct WarpArgs {
  PhaseGeom g;
  PhaseW w;
  const uint16_t* x;    // [MR][K]
  const uint16_t* res;  // [MR][N] residual (res_ld N), bias [N] (res_ld 0), or nullptr
  int res_ld;
  void* out;            // [MR][N]
  int out_f32;
};

// RS: rows per load stream (g.RS; 2 for rows of exactly 64 chunks).  MR:
// activation rows (1, or 2 for affine INT8 with RS == 1): every weight chunk
// is used for both rows, and each row's result is the one-row kernel's.  PL:
// bytes of the fixed-point x (affine; 2 for bf16 outputs, 3 for fp32).
template <int FMT, int KIND, int RS, int MR, int PL>
__global__ void __launch_bounds__(WT_THREADS, 1) gemv_warp_kernel(const WarpArgs a) {
  constexpr bool AFF = FmtTraits<FMT>::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;
  static_assert(MR == 1 || (MR == 2 && FMT == FMT_A8 && RS == 1), "two activation rows: affine INT8");
  const PhaseGeom& g = a.g;

  // shared memory: xraw [MR][K] bf16, xs [MR] staging layouts, the phase
  // tail, then (down / projection) the addends [MR][rows]
  extern __shared__ __align__(128) unsigned char smem[];
  const size_t xs_row = xs_bytes<FMT, PL>(g.K);
  PhaseSmem sm;
  sm.xraw = reinterpret_cast<uint16_t*>(smem);
  sm.xs = reinterpret_cast<uint4*>(smem + (size_t)MR * g.K * 2);
  sm.xs_stride = (int)(xs_row / 16);
  phase_tail_carve<FMT, KIND, MR>(g, smem + (size_t)MR * (g.K * 2 + xs_row), sm);
  uint16_t* res_s = reinterpret_cast<uint16_t*>(smem + (size_t)MR * (g.K * 2 + xs_row) +
                                                phase_tail_bytes<FMT, KIND, MR>(g));
  __shared__ int task_ctr;
  __shared__ float red[WARP_TASK_WARPS];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PhaseCta c = phase_cta<KIND, RS>(g, blockIdx.x);
  const int rows_alloc = g.rows_alloc;

  if (tid == 0) task_ctr = 2 * WARP_TASK_WARPS;  // tasks 0..2W-1 are taken statically
  __syncthreads();
  pdl_trigger();

  const uint64_t pol = l2_evict_first_policy();
  uint4 bufA[WT_NS][WT_CL], bufB[WT_NS][WT_CL];
  const int tA = warp, tB = warp + WARP_TASK_WARPS;
  wt_load<KIND, RS>(g, a.w, c, tA, bufA, pol, lane);
  wt_load<KIND, RS>(g, a.w, c, tB, bufB, pol, lane);
  wt_prefetch<KIND, RS>(g, a.w, c, tA + 2 * WARP_TASK_WARPS, lane);
  wt_prefetch<KIND, RS>(g, a.w, c, tB + 2 * WARP_TASK_WARPS, lane);
  if constexpr (AFF) {
    stage_sb<KIND>(g, a.w, c, sm.sbr, tid, WT_THREADS);
    cp_async_commit();
  }

  pdl_wait();  // x, the residual and the output buffer follow the preceding kernel
  // the addends of the CTA's rows (residual or bias), requested with x so the
  // epilogue does not wait on an L2 round trip; each row's addend is read
  // here and its output written later by the same thread's row loop, so an
  // output that is also the residual stays correct
  if constexpr (KIND == 1)
    if (a.res)
#pragma unroll
      for (int r = 0; r < MR; ++r)
        for (int rl = tid; rl < c.rows; rl += WT_THREADS)
          res_s[r * rows_alloc + rl] = a.res[(size_t)r * a.res_ld + c.r_begin + rl];
  // x into shared memory and (affine) its largest |x|, then one staging pass
  // with the vector's fixed-point scale
  const int nu = g.K / 8;
  float mx[MR];
#pragma unroll
  for (int r = 0; r < MR; ++r) {
    float m = 0.f;
    const uint16_t* xr = a.x + (size_t)r * g.K;
    uint16_t* xw = sm.xraw + (size_t)r * g.K;
    // plain (coherent) loads, all of a thread's units requested before any is
    // used (K <= 16384 in one batch): x was written by the preceding kernel
    constexpr int XU = 4;
    uint4 xv[XU];
#pragma unroll
    for (int k = 0; k < XU; ++k) {
      const int i = tid + k * WT_THREADS;
      xv[k] = i < nu ? *reinterpret_cast<const uint4*>(xr + (size_t)i * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < XU; ++k) {
      const int i = tid + k * WT_THREADS;
      if (i < nu) {
        reinterpret_cast<uint4*>(xw)[i] = xv[k];
        if constexpr (AFF) m = fmaxf(m, unit_absmax(xv[k]));
      }
    }
    for (int i = tid + XU * WT_THREADS; i < nu; i += WT_THREADS) {
      const uint4 v = *reinterpret_cast<const uint4*>(xr + (size_t)i * 8);
      reinterpret_cast<uint4*>(xw)[i] = v;
      if constexpr (AFF) m = fmaxf(m, unit_absmax(v));
    }
    mx[r] = m;
  }
  // each row's largest |x| (one CTA reduction per row), then one staging
  // pass per row with that row's fixed-point scale
#pragma unroll
  for (int r = 0; r < MR; ++r) {
    int ex = 0;
    if constexpr (AFF) ex = fx_exponent<PL>(cta_max(mx[r], red, tid));  // its barrier also publishes xraw
    else __syncthreads();
    const float xscale = exp2i(ex);
    PhaseSmem smr = sm;
    smr.xraw = sm.xraw + (size_t)r * g.K;
    smr.xs = sm.xs + (size_t)r * sm.xs_stride;
    smr.gsum = sm.gsum + (size_t)r * g.G;
    smr.xinv = sm.xinv + (size_t)r * g.P;
    for (int base = warp * 32; base < nu; base += WT_THREADS) {
      const int i = base + lane < nu ? base + lane : -1;
      x_stage_unit<FMT, PL>(g, smr, i, i >= 0 ? reinterpret_cast<const uint4*>(smr.xraw)[i] : make_uint4(0, 0, 0, 0),
                        xscale, false);
    }
    x_set_scale<FMT>(g, smr, ex, tid, WT_THREADS);
    if (MR > 1) __syncthreads();  // red is reused by the next row's reduction
  }
  cp_async_wait_all();  // scales and biases
  __syncthreads();

  wt_run<FMT, KIND, PL, RS, MR, RS == 1>(g, a.w, c, sm, bufA, bufB, tA, tB, &task_ctr, pol, lane);
  __syncthreads();

  // epilogue: one thread per row adds the pieces in a fixed order
  for (int rl = tid; rl < c.rows; rl += WT_THREADS) {
    const int n = c.r_begin + rl;
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      const float v0 = row_total<NW, MR>(g, sm.parts, rl, 0, r);
      float outv;
      if constexpr (KIND == 0) {
        const float v1 = row_total<NW, MR>(g, sm.parts, rl, 1, r);
        outv = v0 / (1.0f + expf(-v0)) * v1;  // silu(gate) * up
      } else {
        outv = a.res ? v0 + bf16f(res_s[r * rows_alloc + rl]) : v0;  // + residual or bias
      }
      const size_t o = (size_t)r * g.N + n;
      if (a.out_f32)
        static_cast<float*>(a.out)[o] = outv;
      else
        static_cast<uint16_t*>(a.out)[o] = f2bf(outv);
    }
  }
}

using WarpKernT = void (*)(WarpArgs);

// The instantiation for MR activation rows and RS rows per load stream.
template <int FMT, int KIND, int PL>
WarpKernT warp_kernel_for(int MR, int RS) {
  constexpr int MR2 = FMT == FMT_A8 ? 2 : 1;  // the two-row instantiation (affine INT8 only)
  return MR == 2 ? gemv_warp_kernel<FMT, KIND, 1, MR2, PL>
                 : (RS == 2 ? gemv_warp_kernel<FMT, KIND, 2, 1, PL> : gemv_warp_kernel<FMT, KIND, 1, 1, PL>);
}

// Host plan and launch of the warp-task kernel for one (format, kind).
// Returns MT_ERR_SHAPE when the problem does not fit its shared-memory
// layout (the caller then uses the team kernel).
template <int FMT, int KIND>
mt_status run_gemv_warp(const GemvProblem& p, const Launch& l) {
  // one activation row, or two over affine INT8 weights
  if (!(p.M == 1 || (p.M == 2 && FMT == FMT_A8))) return MT_ERR_SHAPE;
  static OccCache cache;  // only the attribute flags are used
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  if (!di) return cuda_fail((cudaError_t)derr);

  const int grid = di->sm_count < p.N ? di->sm_count : p.N;
  const int MR = p.M;
  WarpArgs a = {};
  size_t smem_parts = 0;
  if (!plan_phase<FMT, KIND>(p.K, p.N, p.group, grid, &a.g, &smem_parts, 1, MR == 1 ? 2 : 1)) return MT_ERR_SHAPE;
  if (MR == 2) smem_parts = phase_tail_bytes<FMT, KIND, 2>(a.g);
  a.w.W0 = static_cast<const uint8_t*>(p.W0);
  a.w.W1 = static_cast<const uint8_t*>(p.W1);
  a.w.s0 = p.s0; a.w.b0 = p.b0; a.w.s1 = p.s1; a.w.b1 = p.b1;
  a.x = p.x;
  a.res = p.res;
  a.res_ld = p.res_ld;
  a.out = p.out;
  a.out_f32 = p.out_f32 ? 1 : 0;

  // affine weights with bf16 outputs: x in 16-bit fixed point (2 byte planes)
  // unless MT_OPT_ACT_BITS asks for 24; with fp32 outputs in 24-bit (3
  // planes); dense bf16 weights: x as stored
  constexpr bool AFF = FmtTraits<FMT>::AFFINE;
  const bool pl2 = AFF && !p.out_f32 && act_bits() == 16;
  const size_t smem = (size_t)MR * ((size_t)p.K * 2 + (pl2 ? xs_bytes<FMT, 2>(p.K) : xs_bytes<FMT, 3>(p.K))) +
                      smem_parts +
                      (KIND == 1 ? ((size_t)MR * a.g.rows_alloc * 2 + 15) / 16 * 16 : 0);  // res_s
  const size_t budget = (size_t)di->max_smem_optin - 1024;  // static smem and slack
  if (smem > budget) return MT_ERR_SHAPE;

  WarpKernT kern = warp_kernel_for<FMT, KIND, 3>(MR, a.g.RS);
  if constexpr (AFF)
    if (pl2) kern = warp_kernel_for<FMT, KIND, 2>(MR, a.g.RS);
  {
    std::lock_guard<std::mutex> g(cache.mu);
    if (dev < 64 && !cache.attr_set[dev]) {
      for (int mr = 1; mr <= 2; ++mr)
        for (int rs = 1; rs <= 2; ++rs)
          for (int pl = AFF ? 2 : 3; pl <= 3; ++pl) {
            WarpKernT k = warp_kernel_for<FMT, KIND, 3>(mr, rs);
            if constexpr (AFF)
              if (pl == 2) k = warp_kernel_for<FMT, KIND, 2>(mr, rs);
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
            if (e != cudaSuccess) return cuda_fail(e);
          }
      cache.attr_set[dev] = 1;
    }
  }
  return launch(kern, dim3(grid), dim3(WT_THREADS), smem, l, a);
}

}  // namespace mt
