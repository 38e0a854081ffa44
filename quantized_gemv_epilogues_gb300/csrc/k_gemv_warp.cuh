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
  const uint16_t* x;
  const uint16_t* res;
  void* out;
  int out_f32;
};

// RS: rows per load stream (g.RS; 2 for rows of exactly 64 chunks).
template <int FMT, int KIND, int RS>
__global__ void __launch_bounds__(WT_THREADS, 1) gemv_warp_kernel(const WarpArgs a) {
  constexpr bool AFF = FmtTraits<FMT>::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;
  const PhaseGeom& g = a.g;

  extern __shared__ __align__(128) unsigned char smem[];
  PhaseSmem sm;
  sm.xraw = reinterpret_cast<uint16_t*>(smem);
  sm.xs = reinterpret_cast<uint4*>(smem + (size_t)g.K * 2);
  phase_tail_carve<FMT, KIND>(g, smem + (size_t)g.K * 2 + xs_bytes<FMT>(g.K), sm);
  // down / projection: the addend of each of the CTA's rows, after the tail
  uint16_t* res_s = reinterpret_cast<uint16_t*>(smem + (size_t)g.K * 2 + xs_bytes<FMT>(g.K) +
                                                phase_tail_bytes<FMT, KIND>(g));
  __shared__ int task_ctr;
  __shared__ float red[WARP_TASK_WARPS];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PhaseCta c = phase_cta<KIND, RS>(g, blockIdx.x);

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
      for (int rl = tid; rl < c.rows; rl += WT_THREADS) res_s[rl] = a.res[c.r_begin + rl];
  // x into shared memory and (affine) its largest |x|, then one staging pass
  // with the vector's fixed-point scale
  const int nu = g.K / 8;
  float m = 0.f;
  {
    // plain (coherent) loads, all of a thread's units requested before any is
    // used (K <= 16384 in one batch): x was written by the preceding kernel
    constexpr int XU = 4;
    uint4 xv[XU];
#pragma unroll
    for (int k = 0; k < XU; ++k) {
      const int i = tid + k * WT_THREADS;
      xv[k] = i < nu ? *reinterpret_cast<const uint4*>(a.x + (size_t)i * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < XU; ++k) {
      const int i = tid + k * WT_THREADS;
      if (i < nu) {
        reinterpret_cast<uint4*>(sm.xraw)[i] = xv[k];
        if constexpr (AFF) m = fmaxf(m, unit_absmax(xv[k]));
      }
    }
    for (int i = tid + XU * WT_THREADS; i < nu; i += WT_THREADS) {
      const uint4 v = *reinterpret_cast<const uint4*>(a.x + (size_t)i * 8);
      reinterpret_cast<uint4*>(sm.xraw)[i] = v;
      if constexpr (AFF) m = fmaxf(m, unit_absmax(v));
    }
  }
  int ex = 0;
  if constexpr (AFF) ex = fx_exponent(cta_max(m, red, tid));  // its barrier also publishes xraw
  else __syncthreads();
  const float xscale = exp2i(ex);
  for (int base = warp * 32; base < nu; base += WT_THREADS) {
    const int i = base + lane < nu ? base + lane : -1;
    x_stage_unit<FMT>(g, sm, i, i >= 0 ? reinterpret_cast<const uint4*>(sm.xraw)[i] : make_uint4(0, 0, 0, 0),
                      xscale, false);
  }
  x_set_scale<FMT>(g, sm, ex, tid, WT_THREADS);
  cp_async_wait_all();  // scales and biases
  __syncthreads();

  wt_run<FMT, KIND, RS>(g, a.w, c, sm, bufA, bufB, tA, tB, &task_ctr, pol, lane);
  __syncthreads();

  // epilogue: one thread per row adds the pieces in a fixed order
  for (int rl = tid; rl < c.rows; rl += WT_THREADS) {
    const float v0 = row_total<NW>(g, sm.parts, rl, 0);
    const int n = c.r_begin + rl;
    float outv;
    if constexpr (KIND == 0) {
      const float v1 = row_total<NW>(g, sm.parts, rl, 1);
      outv = v0 / (1.0f + expf(-v0)) * v1;  // silu(gate) * up
    } else {
      outv = a.res ? v0 + bf16f(res_s[rl]) : v0;  // + residual or bias (one row)
    }
    if (a.out_f32)
      static_cast<float*>(a.out)[n] = outv;
    else
      static_cast<uint16_t*>(a.out)[n] = f2bf(outv);
  }
}

// Host plan and launch of the warp-task kernel for one (format, kind).
// Returns MT_ERR_SHAPE when the problem does not fit its shared-memory
// layout (the caller then uses the team kernel).
template <int FMT, int KIND>
mt_status run_gemv_warp(const GemvProblem& p, const Launch& l) {
  if (p.M != 1) return MT_ERR_SHAPE;
  static OccCache cache;  // only the attribute flags are used
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  if (!di) return cuda_fail((cudaError_t)derr);

  const int grid = di->sm_count < p.N ? di->sm_count : p.N;
  WarpArgs a = {};
  size_t smem_parts = 0;
  if (!plan_phase<FMT, KIND>(p.K, p.N, p.group, grid, &a.g, &smem_parts)) return MT_ERR_SHAPE;
  a.w.W0 = static_cast<const uint8_t*>(p.W0);
  a.w.W1 = static_cast<const uint8_t*>(p.W1);
  a.w.s0 = p.s0; a.w.b0 = p.b0; a.w.s1 = p.s1; a.w.b1 = p.b1;
  a.x = p.x;
  a.res = p.res;
  a.out = p.out;
  a.out_f32 = p.out_f32 ? 1 : 0;

  const size_t smem = (size_t)p.K * 2 + xs_bytes<FMT>(p.K) + smem_parts +
                      (KIND == 1 ? ((size_t)a.g.rows_alloc * 2 + 15) / 16 * 16 : 0);  // res_s
  const size_t budget = (size_t)di->max_smem_optin - 1024;  // static smem and slack
  if (smem > budget) return MT_ERR_SHAPE;

  auto kern = a.g.RS == 2 ? gemv_warp_kernel<FMT, KIND, 2> : gemv_warp_kernel<FMT, KIND, 1>;
  {
    std::lock_guard<std::mutex> g(cache.mu);
    if (dev < 64 && !cache.attr_set[dev]) {
      for (auto k : {gemv_warp_kernel<FMT, KIND, 1>, gemv_warp_kernel<FMT, KIND, 2>}) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
        if (e != cudaSuccess) return cuda_fail(e);
      }
      cache.attr_set[dev] = 1;
    }
  }
  return launch(kern, dim3(grid), dim3(WT_THREADS), smem, l, a);
}

}  // namespace mt
