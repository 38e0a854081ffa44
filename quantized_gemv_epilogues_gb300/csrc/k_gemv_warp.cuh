// k_gemv_warp.cuh - one-row (M == 1) GEMV with the SwiGLU or residual
// epilogue: warp-task register pipeline.
//
// meTile docs, "Compute-Graph Fusion", Automatic Gated Epilogues (gate and up
// share the activation, silu(gate) * up before the only store; the down
// projection adds the residual in its epilogue); "MLX-LM Backend", Dispatch
// Policy (affine w = scale * q + bias per group of 32/64/128 along K).
//
// GB300 design (each choice measured on this part; see the design notes):
//  * One persistent CTA of 16 warps per SM owns a contiguous range of output
//    rows.  The range is cut into tasks of one row piece (B bytes of each of
//    the NW weight matrices), handed out dynamically through a shared-memory
//    counter, so warps finish within about one task of each other.
//  * A warp holds a small queue of task ids: the lines of the tasks two and
//    three ahead are prefetched into L2 (one prefetch per lane), the next
//    task's weights are loaded into registers with 128-bit evict-first loads
//    while the current one is computed (register double buffer, up to 8 x
//    16 B per lane per task).  HBM sees ~200 KB in flight per SM while the
//    register pipeline only has to cover L2 latency, with no per-copy issue
//    cost (bulk TMA copies cost the issuing thread ~350 cycles each on this
//    part, which capped a TMA-ring design near 3.5 TB/s for 2-4 KB pieces).
//    The first tasks are requested before waiting on the preceding kernel
//    (programmatic dependent launch).
//  * x (fp32, unit-transposed: 16-byte unit k of chunk c at index k*CPR + c,
//    so the lanes of a warp read consecutive words) and the CTA's scales and
//    biases (bf16) are staged once in shared memory with cp.async 16-byte
//    copies issued by every thread.
//  * The affine term is factored as
//      sum_k (s q_k + b) x_k = sum_chunks s * (sum q_k x_k) + sum_groups b * X_g
//    with X_g the sum of x over group g: per weight one byte permute
//    (exponent-bias conversion), half a packed fp32x2 add and half a packed
//    fp32x2 FMA.
//  * A task's partial sums are reduced inside the warp (shuffles) and stored
//    per piece in shared memory; after one barrier, one thread per row adds
//    the pieces in a fixed order (deterministic) and runs the epilogue.
//  * No thread waits on another CTA or on a flag: the only waits are
//    cp.async group completions and CTA barriers.
#pragma once
#include "k_gemv.cuh"

namespace mt {

constexpr int WARP_TASK_WARPS = 16;  // warps per CTA
constexpr int WARP_TASK_UPL = 8;     // 16-byte loads per lane per task (all matrices)

struct WarpArgs {
  const uint16_t* x;
  const uint8_t* W0;
  const uint8_t* W1;
  const uint16_t* s0;
  const uint16_t* b0;
  const uint16_t* s1;
  const uint16_t* b1;
  const uint16_t* res;
  void* out;
  int K, N;
  int group, lg_group, G;  // group size, log2(group), groups per row (affine)
  int CPR;                 // 16-byte chunks per row
  int row_bytes;           // bytes of one weight row
  int rows_base, rows_extra;
  int P;                   // pieces per row
  int B;                   // bytes per piece (multiple of 16)
  int CPP;                 // 16-byte chunks per piece (<= 32 * UPL / NW)
  int GPP;                 // groups per piece (affine)
  int rows_alloc;          // rows of the staged arrays
  int sb_stride;           // elements per staged scale or bias array (multiple of 8)
  int sb_vec;              // 1: scales/biases are staged in 16-byte copies (G % 8 == 0)
  int out_f32;
};

// Float index of element e of x in the unit-transposed staging layout.
template <int EPC>
__device__ __forceinline__ int xt_index(int e, int CPR) {
  const int c = e / EPC;
  const int k = (e % EPC) >> 2;
  return (k * CPR + c) * 4 + (e & 3);
}

// Dot product of one 16-byte weight chunk (chunk c of its row) with its EPC
// activations, as a pair of partial sums (packed fp32x2).
template <int FMT>
__device__ __forceinline__ float2 chunk_dot(const uint4 w, const float4* __restrict__ xt, int c,
                                            int CPR) {
  const float2 neg = make_float2(-8388608.0f, -8388608.0f);
  float2 d0 = make_float2(0.f, 0.f), d1 = make_float2(0.f, 0.f);
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  if constexpr (FMT == FMT_A8) {
    // word wi holds elements 4wi..4wi+3, one byte each
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const float4 xv = xt[wi * CPR + c];
      const float2 qa = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(ww[wi], 0x4B000000u, 0x7540u)),
                                               __uint_as_float(__byte_perm(ww[wi], 0x4B000000u, 0x7541u))), neg);
      const float2 qb = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(ww[wi], 0x4B000000u, 0x7542u)),
                                               __uint_as_float(__byte_perm(ww[wi], 0x4B000000u, 0x7543u))), neg);
      d0 = __ffma2_rn(qa, make_float2(xv.x, xv.y), d0);
      d1 = __ffma2_rn(qb, make_float2(xv.z, xv.w), d1);
    }
  } else if constexpr (FMT == FMT_A4) {
    // word wi holds elements 8wi..8wi+7: byte j = (2j low nibble, 2j+1 high)
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const uint32_t lo = ww[wi] & 0x0F0F0F0Fu, hi = (ww[wi] >> 4) & 0x0F0F0F0Fu;
      const float4 xa = xt[(2 * wi) * CPR + c];      // elements 8wi .. 8wi+3
      const float4 xb = xt[(2 * wi + 1) * CPR + c];  // elements 8wi+4 .. 8wi+7
      const float2 q01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7540u)),
                                                __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7540u))), neg);
      const float2 q23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7541u)),
                                                __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7541u))), neg);
      const float2 q45 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7542u)),
                                                __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7542u))), neg);
      const float2 q67 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7543u)),
                                                __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7543u))), neg);
      d0 = __ffma2_rn(q01, make_float2(xa.x, xa.y), d0);
      d1 = __ffma2_rn(q23, make_float2(xa.z, xa.w), d1);
      d0 = __ffma2_rn(q45, make_float2(xb.x, xb.y), d0);
      d1 = __ffma2_rn(q67, make_float2(xb.z, xb.w), d1);
    }
  } else {
    // dense bf16: word wi holds elements 2wi (low half) and 2wi+1 (high half)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float4 xv = xt[u * CPR + c];
      d0 = __ffma2_rn(make_float2(bf16lo(ww[2 * u]), bf16hi(ww[2 * u])), make_float2(xv.x, xv.y), d0);
      d1 = __ffma2_rn(make_float2(bf16lo(ww[2 * u + 1]), bf16hi(ww[2 * u + 1])), make_float2(xv.z, xv.w), d1);
    }
  }
  return __fadd2_rn(d0, d1);
}

template <int FMT, int KIND>
__global__ void __launch_bounds__(WARP_TASK_WARPS * 32, 1) gemv_warp_kernel(const WarpArgs a) {
  using T = FmtTraits<FMT>;
  constexpr int EPC = T::EPC;
  constexpr bool AFF = T::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;
  constexpr int CL = WARP_TASK_UPL / NW;  // chunks per lane per matrix per task
  constexpr int NT = WARP_TASK_WARPS * 32;

  extern __shared__ __align__(128) unsigned char smem[];
  uint16_t* xraw = reinterpret_cast<uint16_t*>(smem);             // [K] bf16
  float4* xt = reinterpret_cast<float4*>(xraw + a.K);             // [K/4]
  float* gsum = reinterpret_cast<float*>(xt + a.K / 4);           // [G]
  uint16_t* sbr = reinterpret_cast<uint16_t*>(gsum + (AFF ? (a.G + 3) / 4 * 4 : 0));
  // sbr: 2*NW arrays of sb_stride bf16: 2m = scales, 2m+1 = biases of matrix m
  float* parts = reinterpret_cast<float*>(sbr + (AFF ? (size_t)2 * NW * a.sb_stride : 0));  // [rows][P][NW]
  __shared__ int task_ctr;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int r_begin = cta * a.rows_base + min(cta, a.rows_extra);
  const int rows = a.rows_base + (cta < a.rows_extra ? 1 : 0);
  const int T_tasks = rows * a.P;

  if (tid == 0) task_ctr = WARP_TASK_WARPS;  // tasks 0..W-1 are taken statically
  __syncthreads();
  pdl_trigger();

  const uint64_t pol = l2_evict_first_policy();
  auto load_task = [&](int t, uint4 (&buf)[NW][CL]) {
    const bool ok = t < T_tasks;
    const int rl = ok ? t / a.P : 0, p = ok ? t - rl * a.P : 0;
    const size_t base = (size_t)(r_begin + rl) * a.row_bytes + (size_t)p * a.B;
#pragma unroll
    for (int m = 0; m < NW; ++m)
#pragma unroll
      for (int k = 0; k < CL; ++k) {
        const int j = lane + 32 * k;
        buf[m][k] = (ok && j < a.CPP) ? ldg_stream_pol((m ? a.W1 : a.W0) + base + (size_t)j * 16, pol)
                                      : make_uint4(0, 0, 0, 0);
      }
  };
  // one L2 prefetch per lane per 128-byte line of task t
  const int lines_pm = (a.B + 127) >> 7;
  auto prefetch_task = [&](int t) {
    if (t >= T_tasks) return;
    const int rl = t / a.P, p = t - rl * a.P;
    const size_t base = (size_t)(r_begin + rl) * a.row_bytes + (size_t)p * a.B;
    for (int li = lane; li < NW * lines_pm; li += 32) {
      const int m = li / lines_pm;
      prefetch_l2((m ? a.W1 : a.W0) + base + (size_t)(li - m * lines_pm) * 128);
    }
  };
  auto next_task = [&]() -> int {
    int t = 0;
    if (lane == 0) t = atomicAdd(&task_ctr, 1);
    return __shfl_sync(0xffffffffu, t, 0);
  };

  // the first tasks: static weights, requested before the wait
  uint4 bufA[NW][CL], bufB[NW][CL];
  int tc = warp;
  load_task(tc, bufA);
  int tl = next_task(), tp1 = next_task(), tp2 = next_task();
  prefetch_task(tl);
  prefetch_task(tp1);
  prefetch_task(tp2);

  if constexpr (AFF) {
    // the CTA's scales and biases (contiguous [rows][G] blocks)
    if (a.sb_vec) {
      const int n16 = rows * a.G / 8;
      const size_t off = (size_t)r_begin * a.G;
      for (int i = tid; i < n16; i += NT) {
#pragma unroll
        for (int m = 0; m < NW; ++m) {
          cp_async16(sbr + (size_t)(2 * m) * a.sb_stride + i * 8, (m ? a.s1 : a.s0) + off + i * 8);
          cp_async16(sbr + (size_t)(2 * m + 1) * a.sb_stride + i * 8, (m ? a.b1 : a.b0) + off + i * 8);
        }
      }
      cp_async_commit();
    } else {
      const int n_sb = rows * a.G;
      for (int i = tid; i < n_sb; i += NT) {
        const size_t gi = (size_t)r_begin * a.G + i;
#pragma unroll
        for (int m = 0; m < NW; ++m) {
          sbr[(size_t)(2 * m) * a.sb_stride + i] = ldg_u16((m ? a.s1 : a.s0) + gi);
          sbr[(size_t)(2 * m + 1) * a.sb_stride + i] = ldg_u16((m ? a.b1 : a.b0) + gi);
        }
      }
    }
  }

  pdl_wait();  // x, the residual and the output buffer follow the preceding kernel
  for (int i = tid; i < a.K / 8; i += NT) cp_async16(xraw + (size_t)i * 8, a.x + (size_t)i * 8);
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  for (int i = tid; i < a.K / 8; i += NT) {
    const uint4 v = *reinterpret_cast<const uint4*>(xraw + (size_t)i * 8);
    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
    float* xf = reinterpret_cast<float*>(xt);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      xf[xt_index<EPC>(i * 8 + 2 * j, a.CPR)] = bf16lo(vw[j]);
      xf[xt_index<EPC>(i * 8 + 2 * j + 1, a.CPR)] = bf16hi(vw[j]);
    }
  }
  __syncthreads();
  if constexpr (AFF) {
    // X_g = sum of x over group g (one warp per group)
    const float* xf = reinterpret_cast<const float*>(xt);
    for (int g = warp; g < a.G; g += WARP_TASK_WARPS) {
      float sum = 0.f;
      for (int e = lane; e < a.group; e += 32) sum += xf[xt_index<EPC>(g * a.group + e, a.CPR)];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane == 0) gsum[g] = sum;
    }
    __syncthreads();
  }

  // computes task t from the weights in buf and stores its partial sums
  auto compute_task = [&](int t, const uint4 (&buf)[NW][CL]) {
    const int rl = t / a.P, p = t - rl * a.P;
    float2 acc[NW];
#pragma unroll
    for (int m = 0; m < NW; ++m) acc[m] = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < CL; ++k) {
      const int j = lane + 32 * k;
      if (j < a.CPP) {
        const int c = p * a.CPP + j;
#pragma unroll
        for (int m = 0; m < NW; ++m) {
          const float2 d = chunk_dot<FMT>(buf[m][k], xt, c, a.CPR);
          if constexpr (AFF) {
            const int gi = (c * EPC) >> a.lg_group;
            const float sc = bf16f(sbr[(size_t)(2 * m) * a.sb_stride + rl * a.G + gi]);
            acc[m] = __ffma2_rn(make_float2(sc, sc), d, acc[m]);
          } else {
            acc[m] = __fadd2_rn(acc[m], d);
          }
        }
      }
    }
    float vals[NW];
#pragma unroll
    for (int m = 0; m < NW; ++m) vals[m] = acc[m].x + acc[m].y;
    if constexpr (AFF) {
      // bias terms of the groups in this piece: sum_g b_g * X_g
      for (int gl = lane; gl < a.GPP; gl += 32) {
        const int g = p * a.GPP + gl;
        const float xg = gsum[g];
#pragma unroll
        for (int m = 0; m < NW; ++m)
          vals[m] = fmaf(bf16f(sbr[(size_t)(2 * m + 1) * a.sb_stride + rl * a.G + g]), xg, vals[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < NW; ++m)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) vals[m] += __shfl_xor_sync(0xffffffffu, vals[m], off);
    if (lane < NW) {
      float v = vals[0];
#pragma unroll
      for (int m = 1; m < NW; ++m)
        if (lane == m) v = vals[m];
      parts[((size_t)rl * a.P + p) * NW + lane] = v;
    }
  };

  // register ping-pong: the next task's loads are in flight while the
  // current one is computed; two tasks per iteration keep indices static
  while (tc < T_tasks) {
    load_task(tl, bufB);
    compute_task(tc, bufA);
    tc = tl; tl = tp1; tp1 = tp2; tp2 = next_task();
    prefetch_task(tp2);
    if (tc >= T_tasks) break;
    load_task(tl, bufA);
    compute_task(tc, bufB);
    tc = tl; tl = tp1; tp1 = tp2; tp2 = next_task();
    prefetch_task(tp2);
  }
  __syncthreads();

  // epilogue: one thread per row adds the pieces in a fixed order
  for (int rl = tid; rl < rows; rl += NT) {
    float v0 = 0.f, v1 = 0.f;
    for (int q = 0; q < a.P; ++q) {
      v0 += parts[((size_t)rl * a.P + q) * NW];
      if (NW == 2) v1 += parts[((size_t)rl * a.P + q) * NW + 1];
    }
    const int n = r_begin + rl;
    float outv;
    if constexpr (KIND == 0) {
      outv = v0 / (1.0f + expf(-v0)) * v1;  // silu(gate) * up
    } else {
      outv = v0 + bf16f(a.res[n]);  // + residual
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
  using T = FmtTraits<FMT>;
  constexpr int EPC = T::EPC;
  constexpr bool AFF = T::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;
  constexpr int CL = WARP_TASK_UPL / NW;
  if (p.M != 1) return MT_ERR_SHAPE;
  static OccCache cache;  // only the attribute flags are used
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  if (!di) return cuda_fail((cudaError_t)derr);

  WarpArgs a = {};
  a.x = p.x;
  a.W0 = static_cast<const uint8_t*>(p.W0);
  a.W1 = static_cast<const uint8_t*>(p.W1);
  a.s0 = p.s0; a.b0 = p.b0; a.s1 = p.s1; a.b1 = p.b1;
  a.res = p.res;
  a.out = p.out;
  a.K = p.K; a.N = p.N;
  a.group = AFF ? p.group : 1;
  a.lg_group = AFF ? (p.group == 32 ? 5 : (p.group == 64 ? 6 : 7)) : 0;
  a.G = AFF ? p.K / p.group : 0;
  a.row_bytes = FMT == FMT_BF16 ? p.K * 2 : (FMT == FMT_A8 ? p.K : p.K / 2);
  a.out_f32 = p.out_f32 ? 1 : 0;
  a.CPR = p.K / EPC;

  // Pieces per row: the fewest whose chunks fit the lanes' register buffer
  // (32 * CL chunks per matrix), dividing the row's chunks and (affine) its
  // groups, so a piece holds whole groups.
  int P = 0;
  for (int q = 1; q <= a.CPR; ++q) {
    if (a.CPR % q || (AFF && a.G % q)) continue;
    if (a.CPR / q <= 32 * CL) { P = q; break; }
  }
  if (P == 0) return MT_ERR_SHAPE;
  a.P = P;
  a.B = a.row_bytes / P;
  a.CPP = a.CPR / P;
  a.GPP = AFF ? a.G / P : 0;

  const int N = p.N;
  int grid = di->sm_count;
  if (grid > N) grid = N;
  a.rows_base = N / grid;
  a.rows_extra = N % grid;
  const int rows_max = a.rows_base + (a.rows_extra ? 1 : 0);
  a.rows_alloc = rows_max;
  a.sb_stride = AFF ? (a.rows_alloc * a.G + 7) / 8 * 8 : 0;
  a.sb_vec = (AFF && a.G % 8 == 0) ? 1 : 0;

  const size_t smem = (size_t)p.K * 2 + (size_t)p.K * 4 +
                      (AFF ? (size_t)(a.G + 3) / 4 * 16 + (size_t)2 * NW * a.sb_stride * 2 : 0) +
                      (size_t)a.rows_alloc * P * NW * 4;
  const size_t budget = (size_t)di->max_smem_optin - 1024;  // static smem and slack
  if (smem > budget) return MT_ERR_SHAPE;

  auto kern = gemv_warp_kernel<FMT, KIND>;
  {
    std::lock_guard<std::mutex> g(cache.mu);
    if (dev < 64 && !cache.attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)budget);
      if (e != cudaSuccess) return cuda_fail(e);
      cache.attr_set[dev] = 1;
    }
  }
  return launch(kern, dim3(grid), dim3(WARP_TASK_WARPS * 32), smem, l, a);
}

}  // namespace mt
