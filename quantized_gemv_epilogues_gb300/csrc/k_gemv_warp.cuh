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
//    rows.  The range is cut into tasks of two weight streams of B bytes
//    that share their activations: gate and up of one row (gate/up), or two
//    consecutive rows (down).  Tasks are handed out dynamically through a
//    shared-memory counter, so warps finish within about one task of each
//    other.
//  * A warp loads its next task's weights into registers with 128-bit
//    evict-first loads while it computes the current one (register double
//    buffer, up to 8 x 16 B per lane per task), ~64-128 KB in flight per SM
//    with no per-copy issue cost.  (Bulk TMA copies cost the issuing thread
//    ~350 cycles each on this part, which capped a TMA-ring design near
//    3.5 TB/s for 2-4 KB pieces.)  The first task is requested before
//    waiting on the preceding kernel (programmatic dependent launch).
//  * The CTA's scales and biases (bf16) and x are staged once in shared
//    memory with cp.async 16-byte copies issued by every thread.  x is then
//    laid out unit-transposed (the x words of chunk c for word k at index
//    k*CPR + c) so the lanes of a warp read consecutive words.
//  * The affine term is factored as
//      sum_k (s q_k + b) x_k = sum_chunks s * (sum q_k x_k) + sum_groups b * X_g
//    with X_g the sum of x over group g (fp32, from the bf16 values).  The
//    codes are turned into fp16 with the exponent-bias trick (a byte permute
//    or a mask builds 1024 + q, one packed fp16 subtract leaves q exactly),
//    and each product q * x is one mixed-precision FMA (fp16 x fp16, exact
//    product, fp32 accumulation).  x enters that FMA as fp16 after an exact
//    power-of-two scaling chosen per CTA from max|x| (so nothing overflows;
//    only elements below ~2^-24 of the scaled maximum lose bits); the scale is
//    divided out of the partial sums.  Dense bf16 weights use the bf16 form of
//    the same FMA with x unchanged.  About two instructions per weight.
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
  unsigned long long p_mul;  // ceil(2^32 / P): t / P == (t * p_mul) >> 32 for t < 2^32 / P
  int B;                   // bytes per piece (multiple of 16)
  int CPP;                 // 16-byte chunks per piece (<= 32 * UPL / 2)
  int GPP;                 // groups per piece (affine)
  int rows_alloc;          // rows of the staged arrays
  int sb_stride;           // elements per staged scale or bias array (multiple of 8)
  int sb_vec;              // 1: scales/biases are staged in 16-byte copies (G % 8 == 0)
  int out_f32;
};

// Staging layout of x (16-bit elements), read by chunk_dot:
// A8: word wi of chunk c is 4 fp16 (elements 4wi..4wi+3) at unit wi*CPR + c.
// A4: word wi of chunk c is 8 fp16 at unit wi*CPR + c, in the order
//     {0,4,1,5,2,6,3,7} that matches the nibble pairs of one weight word.
// BF16: words 2u, 2u+1 of chunk c read 4 bf16 (elements 4u..4u+3) at unit
//     u*CPR + c.

// acc_lo += lo(a) * lo(b), acc_hi += hi(a) * hi(b): fp16 x fp16 products
// (exact in fp32) accumulated in fp32.
__device__ __forceinline__ void fma2_f16_f32(float& lo, float& hi, uint32_t a, uint32_t b) {
  asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
      "mov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
      "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %1, a1, b1, %1;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "r"(a), "r"(b));
}

// The same with bf16 operands (exact products in fp32).
__device__ __forceinline__ void fma2_bf16_f32(float& lo, float& hi, uint32_t a, uint32_t b) {
  asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
      "mov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
      "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %1, a1, b1, %1;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "r"(a), "r"(b));
}

// Two fp16 codes 1024 + q (built with the exponent-bias trick) -> q, exactly.
__device__ __forceinline__ uint32_t unbias_f16x2(uint32_t h) {
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(h) : "r"(0x64006400u));
  return h;
}

// Dot product of one 16-byte weight chunk (chunk c of its row) with its
// activations from the staging layout: sum of q * x (affine, x scaled) or of
// w * x (bf16).
template <int FMT>
__device__ __forceinline__ float chunk_dot(const uint4 w, const uint16_t* __restrict__ xs, int c,
                                           int CPR) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if constexpr (FMT == FMT_A8) {
    const uint2* xu = reinterpret_cast<const uint2*>(xs);
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const uint2 xv = xu[wi * CPR + c];
      const uint32_t h01 = unbias_f16x2(__byte_perm(ww[wi], 0x64646464u, 0x5140u));
      const uint32_t h23 = unbias_f16x2(__byte_perm(ww[wi], 0x64646464u, 0x7342u));
      fma2_f16_f32(a0, a1, h01, xv.x);
      fma2_f16_f32(a2, a3, h23, xv.y);
    }
  } else if constexpr (FMT == FMT_A4) {
    const uint4* xu = reinterpret_cast<const uint4*>(xs);
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const uint4 xv = xu[wi * CPR + c];
      const uint32_t v = ww[wi];
      const uint32_t p0 = unbias_f16x2((v & 0x000F000Fu) | 0x64006400u);          // q0, q4
      const uint32_t p1 = unbias_f16x2(((v >> 4) & 0x000F000Fu) | 0x64006400u);   // q1, q5
      const uint32_t p2 = unbias_f16x2(((v >> 8) & 0x000F000Fu) | 0x64006400u);   // q2, q6
      const uint32_t p3 = unbias_f16x2(((v >> 12) & 0x000F000Fu) | 0x64006400u);  // q3, q7
      fma2_f16_f32(a0, a1, p0, xv.x);
      fma2_f16_f32(a2, a3, p1, xv.y);
      fma2_f16_f32(a0, a1, p2, xv.z);
      fma2_f16_f32(a2, a3, p3, xv.w);
    }
  } else {
    const uint2* xu = reinterpret_cast<const uint2*>(xs);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint2 xv = xu[u * CPR + c];
      fma2_bf16_f32(a0, a1, ww[2 * u], xv.x);
      fma2_bf16_f32(a2, a3, ww[2 * u + 1], xv.y);
    }
  }
  return (a0 + a1) + (a2 + a3);
}

template <int FMT, int KIND>
__global__ void __launch_bounds__(WARP_TASK_WARPS * 32, 1) gemv_warp_kernel(const WarpArgs a) {
  using T = FmtTraits<FMT>;
  constexpr int EPC = T::EPC;
  constexpr bool AFF = T::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;   // weight matrices
  constexpr int RW = KIND == 0 ? 1 : 2;   // rows per task
  constexpr int NS = 2;                   // weight streams per task: NW * RW
  constexpr int CL = WARP_TASK_UPL / NS;  // chunks per lane per stream per task
  constexpr int NT = WARP_TASK_WARPS * 32;

  extern __shared__ __align__(128) unsigned char smem[];
  uint16_t* xraw = reinterpret_cast<uint16_t*>(smem);             // [K] bf16
  uint16_t* xs = xraw + a.K;                                      // [K] staging layout
  float* gsum = reinterpret_cast<float*>(xs + a.K);               // [G]
  uint16_t* sbr = reinterpret_cast<uint16_t*>(gsum + (AFF ? (a.G + 3) / 4 * 4 : 0));
  // sbr: 2*NW arrays of sb_stride bf16: 2m = scales, 2m+1 = biases of matrix m
  float* parts = reinterpret_cast<float*>(sbr + (AFF ? (size_t)2 * NW * a.sb_stride : 0));  // [rows][P][NW]
  __shared__ int task_ctr;
  __shared__ float red_max[WARP_TASK_WARPS];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int r_begin = cta * a.rows_base + min(cta, a.rows_extra);
  const int rows = a.rows_base + (cta < a.rows_extra ? 1 : 0);
  const int T_tasks = (rows + RW - 1) / RW * a.P;

  if (tid == 0) task_ctr = WARP_TASK_WARPS;  // tasks 0..W-1 are taken statically
  __syncthreads();
  pdl_trigger();

  const uint64_t pol = l2_evict_first_policy();
  // stream v of a task: matrix v of row rl0 (gate/up) or row rl0 + v (down)
  auto load_task = [&](int t, uint4 (&buf)[NS][CL]) {
    const int rg = (int)(((unsigned long long)(unsigned)t * a.p_mul) >> 32);
    const int p = t - rg * a.P;
#pragma unroll
    for (int v = 0; v < NS; ++v) {
      const int rl = rg * RW + (KIND == 0 ? 0 : v);
      const bool ok = t < T_tasks && rl < rows;
      const uint8_t* src = (KIND == 0 && v ? a.W1 : a.W0) +
                           (size_t)(r_begin + (ok ? rl : 0)) * a.row_bytes + (size_t)p * a.B;
#pragma unroll
      for (int k = 0; k < CL; ++k) {
        const int j = lane + 32 * k;
        buf[v][k] = (ok && j < a.CPP) ? ldg_stream_pol(src + (size_t)j * 16, pol) : make_uint4(0, 0, 0, 0);
      }
    }
  };
  auto next_task = [&]() -> int {
    int t = 0;
    if (lane == 0) t = atomicAdd(&task_ctr, 1);
    return __shfl_sync(0xffffffffu, t, 0);
  };

  // the first tasks: static weights, requested before the wait
  uint4 bufA[NS][CL], bufB[NS][CL];
  int tc = warp;
  load_task(tc, bufA);

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
  // x scale (affine): 2^e with max|x| * 2^e in [2^14, 2^15), exact
  float xscale = 1.f, xinv = 1.f;
  if constexpr (AFF) {
    float mx = 0.f;
    for (int i = tid; i < a.K / 8; i += NT) {
      const uint4 v = reinterpret_cast<const uint4*>(xraw)[i];
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16lo(v.x)), fabsf(bf16hi(v.x))),
                           fmaxf(fabsf(bf16lo(v.y)), fabsf(bf16hi(v.y)))));
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16lo(v.z)), fabsf(bf16hi(v.z))),
                           fmaxf(fabsf(bf16lo(v.w)), fabsf(bf16hi(v.w)))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red_max[warp] = mx;
    // X_g = sum of x over group g (fp32, unscaled; one warp per group)
    for (int g = warp; g < a.G; g += WARP_TASK_WARPS) {
      float sum = 0.f;
      for (int e = 4 * lane; e < a.group; e += 128) {
        const uint2 v = *reinterpret_cast<const uint2*>(xraw + g * a.group + e);
        sum += (bf16lo(v.x) + bf16hi(v.x)) + (bf16lo(v.y) + bf16hi(v.y));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane == 0) gsum[g] = sum;
    }
    __syncthreads();
    mx = 0.f;
#pragma unroll
    for (int w = 0; w < WARP_TASK_WARPS; ++w) mx = fmaxf(mx, red_max[w]);
    if (mx > 0.f && mx < 3.0e38f) {
      const int ex = max(-126, min(126, 14 - ilogbf(mx)));
      xscale = ldexpf(1.f, ex);
      xinv = ldexpf(1.f, -ex);
    }
  }
  // staging layout: consecutive threads write consecutive words
  {
    const int CPR = a.CPR;
    if constexpr (FMT == FMT_A4) {
#pragma unroll 1
      for (int k = 0; k < 4; ++k)
        for (int c = tid; c < CPR; c += NT) {
          const uint4 v = *reinterpret_cast<const uint4*>(xraw + c * 32 + 8 * k);  // elements 0..7 of word k
          const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
          float f[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            f[2 * j] = bf16lo(vw[j]) * xscale;
            f[2 * j + 1] = bf16hi(vw[j]) * xscale;
          }
          // order {0,4,1,5,2,6,3,7}
          uint4 o;
          o.x = (uint32_t)__half_as_ushort(__float2half_rn(f[0])) | ((uint32_t)__half_as_ushort(__float2half_rn(f[4])) << 16);
          o.y = (uint32_t)__half_as_ushort(__float2half_rn(f[1])) | ((uint32_t)__half_as_ushort(__float2half_rn(f[5])) << 16);
          o.z = (uint32_t)__half_as_ushort(__float2half_rn(f[2])) | ((uint32_t)__half_as_ushort(__float2half_rn(f[6])) << 16);
          o.w = (uint32_t)__half_as_ushort(__float2half_rn(f[3])) | ((uint32_t)__half_as_ushort(__float2half_rn(f[7])) << 16);
          reinterpret_cast<uint4*>(xs)[k * CPR + c] = o;
        }
    } else {
      constexpr int U = EPC / 4;  // words of 4 elements per chunk
#pragma unroll 1
      for (int k = 0; k < U; ++k)
        for (int c = tid; c < CPR; c += NT) {
          const uint2 v = *reinterpret_cast<const uint2*>(xraw + c * EPC + 4 * k);
          uint2 o;
          if constexpr (AFF) {
            o.x = (uint32_t)__half_as_ushort(__float2half_rn(bf16lo(v.x) * xscale)) |
                  ((uint32_t)__half_as_ushort(__float2half_rn(bf16hi(v.x) * xscale)) << 16);
            o.y = (uint32_t)__half_as_ushort(__float2half_rn(bf16lo(v.y) * xscale)) |
                  ((uint32_t)__half_as_ushort(__float2half_rn(bf16hi(v.y) * xscale)) << 16);
          } else {
            o = v;
          }
          reinterpret_cast<uint2*>(xs)[k * CPR + c] = o;
        }
    }
  }
  __syncthreads();

  // computes task t from the weights in buf and stores its partial sums
  auto compute_task = [&](int t, const uint4 (&buf)[NS][CL]) {
    const int rg = (int)(((unsigned long long)(unsigned)t * a.p_mul) >> 32);
    const int p = t - rg * a.P;
    const int rl0 = rg * RW;
    float acc[NS];
#pragma unroll
    for (int v = 0; v < NS; ++v) acc[v] = 0.f;
#pragma unroll
    for (int k = 0; k < CL; ++k) {
      const int j = lane + 32 * k;
      if (j < a.CPP) {
        const int c = p * a.CPP + j;
#pragma unroll
        for (int v = 0; v < NS; ++v) {
          const float d = chunk_dot<FMT>(buf[v][k], xs, c, a.CPR);
          if constexpr (AFF) {
            const int m = KIND == 0 ? v : 0, rl = min(rl0 + (KIND == 0 ? 0 : v), rows - 1);
            const int gi = (c * EPC) >> a.lg_group;
            acc[v] = fmaf(bf16f(sbr[(size_t)(2 * m) * a.sb_stride + rl * a.G + gi]), d, acc[v]);
          } else {
            acc[v] += d;
          }
        }
      }
    }
    float vals[NS];
#pragma unroll
    for (int v = 0; v < NS; ++v) vals[v] = acc[v] * xinv;
    if constexpr (AFF) {
      // bias terms of the groups in this piece: sum_g b_g * X_g
      for (int gl = lane; gl < a.GPP; gl += 32) {
        const int g = p * a.GPP + gl;
        const float xg = gsum[g];
#pragma unroll
        for (int v = 0; v < NS; ++v) {
          const int m = KIND == 0 ? v : 0, rl = min(rl0 + (KIND == 0 ? 0 : v), rows - 1);
          vals[v] = fmaf(bf16f(sbr[(size_t)(2 * m + 1) * a.sb_stride + rl * a.G + g]), xg, vals[v]);
        }
      }
    }
#pragma unroll
    for (int v = 0; v < NS; ++v)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) vals[v] += __shfl_xor_sync(0xffffffffu, vals[v], off);
    if (lane < NS) {
      float val = vals[0];
#pragma unroll
      for (int v = 1; v < NS; ++v)
        if (lane == v) val = vals[v];
      const int m = KIND == 0 ? lane : 0, rl = rl0 + (KIND == 0 ? 0 : lane);
      if (rl < rows) parts[((size_t)rl * a.P + p) * NW + m] = val;
    }
  };

  // register ping-pong: the next task's loads are in flight while the
  // current one is computed; two tasks per iteration keep indices static
  while (tc < T_tasks) {
    const int tB = next_task();
    load_task(tB, bufB);
    compute_task(tc, bufA);
    if (tB >= T_tasks) break;
    tc = next_task();
    load_task(tc, bufA);
    compute_task(tB, bufB);
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
  constexpr int CL = WARP_TASK_UPL / 2;  // chunks per lane per stream
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
  // (32 * CL chunks per stream), dividing the row's chunks and (affine) its
  // groups, so a piece holds whole groups.
  int P = 0;
  for (int q = 1; q <= a.CPR; ++q) {
    if (a.CPR % q || (AFF && a.G % q)) continue;
    if (a.CPR / q <= 32 * CL) { P = q; break; }
  }
  if (P == 0) return MT_ERR_SHAPE;
  a.P = P;
  a.p_mul = ((1ull << 32) + (unsigned long long)P - 1) / (unsigned long long)P;
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

  const size_t smem = (size_t)p.K * 2 + (size_t)p.K * 2 +
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
