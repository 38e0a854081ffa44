// k_gemv.cuh - K2 (gate/up GEMV + SwiGLU epilogue) and K3 (down GEMV +
// residual epilogue) over dense bf16 or group-wise affine INT8/INT4 weights.
//
// meTile docs, "Compute-Graph Fusion", Automatic Gated Epilogues: the gate and
// up projections share one activation input and silu(gate) * up is applied
// on-chip before the only store; a second epilogue adds the transformer
// residual to the down projection in the same kernel.  "MLX-LM Backend",
// Dispatch Policy: affine weights w = scale * q + bias per group of 32/64/128
// along K; dense BF16 gate/up dot products share each activation load.
//
// GB300 mapping (prior art on the pages is a Metal SIMD-group schedule; this
// is written for sm_103a instead):
//  * Weights stream from HBM with 128-bit non-allocating loads, one 16-byte
//    "chunk" per thread per row and step, so a warp reads 512 contiguous
//    bytes of a row per instruction.
//  * A CTA owns a contiguous range of output rows (the grid is persistent,
//    sized to the SM count times the CTAs that fit per SM), so rows are
//    balanced to within one row per CTA.  Inside a CTA, teams of TS threads
//    split K of each row (split-K) and reduce their partial sums with warp
//    shuffles and one shared-memory step per tile of R rows.
//  * x, its per-chunk sums and the CTA's group scales/biases are staged in
//    shared memory once (16-byte loads / cp.async), so the weight stream is
//    the only HBM traffic of the mainloop.
//  * Dequantisation happens in registers.  For one row (M == 1) the affine
//    term is factored per 16-byte chunk: sum_k (s*q_k + b) x_k =
//    s * sum_k q_k x_k + b * sum_k x_k, with sum_k x_k precomputed per chunk.
//    For M > 1 each weight is dequantised once (one FMA) and reused for the
//    M rows.  Accumulation is fp32 throughout.
//  * The next step's weights are loaded before the current step is computed
//    (register double buffering); the first step's weights and the
//    scales/biases are loaded before waiting on the preceding kernel
//    (programmatic dependent launch), hiding the launch gap.
#pragma once
#include "mt_device.cuh"
#include "mt_internal.h"

namespace mt {

struct GemvArgs {
  const uint16_t* x;
  const uint8_t* W0;
  const uint8_t* W1;
  const uint16_t* s0;
  const uint16_t* b0;
  const uint16_t* s1;
  const uint16_t* b1;
  const uint16_t* res;  // addend (residual or bias) or nullptr
  int res_ld;           // its row stride in elements (0: one bias row for every m)
  void* out;
  int M, K, N;
  int group, G;         // group size along K and groups per row
  int CPR;              // 16-byte chunks per row
  int row_bytes;        // bytes per weight row
  int TS, NT, CPT;      // threads per team, teams per CTA, chunks per thread per row
  int rows_base, rows_extra;  // row partition: CTA i gets rows_base + (i < rows_extra)
  int sb_rows;          // rows of scale/bias staged per CTA (allocation)
  int out_f32;
};

// Weight formats (the values of mt_wfmt).  MX8 / MX4: OCP MX block-scaled
// E4M3 / E2M1 elements with one E8M0 scale per 32 elements along K; only the
// tensor-core kernel (k_gemv_mma.cuh) takes them.
constexpr int FMT_BF16 = 0, FMT_A8 = 1, FMT_A4 = 2, FMT_MX8 = 3, FMT_MX4 = 4;

template <int FMT> struct FmtTraits;
template <> struct FmtTraits<FMT_BF16> { static constexpr int EPC = 8, EPW = 2; static constexpr bool AFFINE = false, MX = false; };
template <> struct FmtTraits<FMT_A8> { static constexpr int EPC = 16, EPW = 4; static constexpr bool AFFINE = true, MX = false; };
template <> struct FmtTraits<FMT_A4> { static constexpr int EPC = 32, EPW = 8; static constexpr bool AFFINE = true, MX = false; };
template <> struct FmtTraits<FMT_MX8> { static constexpr int EPC = 16, EPW = 4; static constexpr bool AFFINE = false, MX = true; };
template <> struct FmtTraits<FMT_MX4> { static constexpr int EPC = 32, EPW = 8; static constexpr bool AFFINE = false, MX = true; };

// Decodes word i of a 16-byte weight chunk into EPW floats: the raw codes q
// (affine) or the bf16 weights.
template <int FMT>
__device__ __forceinline__ void decode_word(uint32_t w, float* q) {
  if constexpr (FMT == FMT_BF16) {
    q[0] = bf16lo(w);
    q[1] = bf16hi(w);
  } else if constexpr (FMT == FMT_A8) {
#pragma unroll
    for (int b = 0; b < 4; ++b) q[b] = u8_to_f32(w, b);
  } else {
    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      q[2 * b] = u8_to_f32(lo, b);
      q[2 * b + 1] = u8_to_f32(hi, b);
    }
  }
}

// Loads EPW bf16 activations (elements [e0, e0+EPW) of row m) from shared memory.
template <int EPW>
__device__ __forceinline__ void load_x_word(const uint16_t* xs_row, int e0, float* xv) {
  if constexpr (EPW == 2) {
    const uint32_t a = *reinterpret_cast<const uint32_t*>(xs_row + e0);
    xv[0] = bf16lo(a); xv[1] = bf16hi(a);
  } else if constexpr (EPW == 4) {
    const uint2 a = *reinterpret_cast<const uint2*>(xs_row + e0);
    xv[0] = bf16lo(a.x); xv[1] = bf16hi(a.x); xv[2] = bf16lo(a.y); xv[3] = bf16hi(a.y);
  } else {
    const uint4 a = *reinterpret_cast<const uint4*>(xs_row + e0);
    xv[0] = bf16lo(a.x); xv[1] = bf16hi(a.x); xv[2] = bf16lo(a.y); xv[3] = bf16hi(a.y);
    xv[4] = bf16lo(a.z); xv[5] = bf16hi(a.z); xv[6] = bf16lo(a.w); xv[7] = bf16hi(a.w);
  }
}

__device__ __forceinline__ void team_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int FMT, int KIND, int MR, int R>
__global__ void __launch_bounds__(256) gemv_kernel(const GemvArgs a) {
  using T = FmtTraits<FMT>;
  constexpr int EPC = T::EPC, EPW = T::EPW;
  constexpr bool AFF = T::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;    // weight matrices per output
  constexpr int V = R * NW * MR;           // partial sums per thread per tile
  constexpr bool FACTOR = AFF && MR == 1;  // s * sum(q x) + b * sum(x) per chunk

  extern __shared__ __align__(128) unsigned char smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                       // [MR][K] bf16
  float* sxs = reinterpret_cast<float*>(smem + (size_t)MR * a.K * 2);     // [CPR] (FACTOR)
  uint32_t* sbs = reinterpret_cast<uint32_t*>(
      reinterpret_cast<unsigned char*>(sxs) + (FACTOR ? (size_t)a.CPR * 4 : 0));  // [sb_rows][NW][G]
  float* red = reinterpret_cast<float*>(
      reinterpret_cast<unsigned char*>(sbs) + (AFF ? (size_t)a.sb_rows * NW * a.G * 4 : 0));

  const int tid = threadIdx.x;
  const int team = tid / a.TS, t = tid - team * a.TS;
  const int cta = blockIdx.x;
  const int r_begin = cta * a.rows_base + min(cta, a.rows_extra);
  const int rows = a.rows_base + (cta < a.rows_extra ? 1 : 0);
  const int tiles = (rows + R - 1) / R;
  const int my_tiles = team < tiles ? (tiles - team + a.NT - 1) / a.NT : 0;
  const int steps = my_tiles * a.CPT;

  // ---- step -> (rows, chunk) and the weight loads of one step
  auto load_step = [&](int s, uint4 (&dst)[R][NW]) {
    const int tile = team + (s / a.CPT) * a.NT;
    const int c = (s % a.CPT) * a.TS + t;
    const int row0 = r_begin + tile * R;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const bool ok = (s < steps) && (c < a.CPR) && (tile * R + r < rows);
      const size_t off = (size_t)(row0 + r) * a.row_bytes + (size_t)c * 16;
      dst[r][0] = ok ? ldg_stream(a.W0 + off) : make_uint4(0, 0, 0, 0);
      if constexpr (NW == 2) dst[r][1] = ok ? ldg_stream(a.W1 + off) : make_uint4(0, 0, 0, 0);
    }
  };

  // ---- prologue: static data first (weights of step 0, scales/biases)
  uint4 wA[R][NW], wB[R][NW];
  load_step(0, wA);
  if constexpr (AFF) {
    const int n_sb = rows * NW * a.G;
    for (int i = tid; i < n_sb; i += blockDim.x) {
      const int rl = i / (NW * a.G);
      const int rem = i - rl * NW * a.G;
      const int mat = rem / a.G, gi = rem - mat * a.G;
      const size_t gidx = (size_t)(r_begin + rl) * a.G + gi;
      const uint16_t sv = ldg_u16((mat ? a.s1 : a.s0) + gidx);
      const uint16_t bv = ldg_u16((mat ? a.b1 : a.b0) + gidx);
      sbs[i] = (uint32_t)sv | ((uint32_t)bv << 16);
    }
  }
  pdl_trigger();
  pdl_wait();  // x (and the residual) come from the preceding kernels

  // ---- stage x [M][K] (rows >= M zero) into shared memory
  {
    const int n16 = a.K / 8;  // 16-byte pieces per row
    for (int i = tid; i < MR * n16; i += blockDim.x) {
      const int m = i / n16, p = i - m * n16;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (m < a.M) v = *reinterpret_cast<const uint4*>(a.x + (size_t)m * a.K + (size_t)p * 8);
      *reinterpret_cast<uint4*>(xs + (size_t)m * a.K + (size_t)p * 8) = v;
    }
  }
  __syncthreads();
  if constexpr (FACTOR) {
    for (int c = tid; c < a.CPR; c += blockDim.x) {
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < EPC; e += 8) {
        float xv[8];
        load_x_word<8>(xs + (size_t)c * EPC, e, xv);
#pragma unroll
        for (int i = 0; i < 8; ++i) sum += xv[i];
      }
      sxs[c] = sum;
    }
    __syncthreads();
  }

  // ---- mainloop
  float acc[R][NW][MR];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int k = 0; k < NW; ++k)
#pragma unroll
      for (int m = 0; m < MR; ++m) acc[r][k][m] = 0.f;

  int rbuf = 0;
  const int nwarp_team = a.TS >> 5;

  // Computes step s from the weights in w, then, at the end of a tile,
  // reduces over the team and runs the epilogue.
  auto compute_step = [&](int s, const uint4 (&w)[R][NW]) {
    const int tile = team + (s / a.CPT) * a.NT;
    const int j = s - (s / a.CPT) * a.CPT;
    const int c = j * a.TS + t;
    if (c < a.CPR) {
      const int e_base = c * EPC;
      const int gi = AFF ? e_base / a.group : 0;
      float sc[R][NW], bi[R][NW];
      if constexpr (AFF) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int k = 0; k < NW; ++k) {
            const uint32_t p = sbs[((tile * R + r) * NW + k) * a.G + gi];
            sc[r][k] = bf16lo(p);
            bi[r][k] = bf16hi(p);
          }
      }
      if constexpr (FACTOR) {
        float dot[R][NW];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int k = 0; k < NW; ++k) dot[r][k] = 0.f;
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          float xv[EPW];
          load_x_word<EPW>(xs, e_base + wi * EPW, xv);
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int k = 0; k < NW; ++k) {
              const uint32_t word = wi == 0 ? w[r][k].x : wi == 1 ? w[r][k].y : wi == 2 ? w[r][k].z : w[r][k].w;
              float q[EPW];
              decode_word<FMT>(word, q);
#pragma unroll
              for (int e = 0; e < EPW; ++e) dot[r][k] = fmaf(q[e], xv[e], dot[r][k]);
            }
        }
        const float sxv = sxs[c];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int k = 0; k < NW; ++k)
            acc[r][k][0] = fmaf(sc[r][k], dot[r][k], fmaf(bi[r][k], sxv, acc[r][k][0]));
      } else {
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          float xv[MR][EPW];
#pragma unroll
          for (int m = 0; m < MR; ++m) load_x_word<EPW>(xs + (size_t)m * a.K, e_base + wi * EPW, xv[m]);
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int k = 0; k < NW; ++k) {
              const uint32_t word = wi == 0 ? w[r][k].x : wi == 1 ? w[r][k].y : wi == 2 ? w[r][k].z : w[r][k].w;
              float q[EPW];
              decode_word<FMT>(word, q);
#pragma unroll
              for (int e = 0; e < EPW; ++e) {
                const float wv = AFF ? fmaf(sc[r][k], q[e], bi[r][k]) : q[e];
#pragma unroll
                for (int m = 0; m < MR; ++m) acc[r][k][m] = fmaf(wv, xv[m][e], acc[r][k][m]);
              }
            }
        }
      }
    }

    if (j == a.CPT - 1) {
      // ---- end of a tile: reduce over the team, epilogue, store
      float vals[V];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int k = 0; k < NW; ++k)
#pragma unroll
          for (int m = 0; m < MR; ++m) {
            vals[(r * NW + k) * MR + m] = acc[r][k][m];
            acc[r][k][m] = 0.f;
          }
#pragma unroll
      for (int v = 0; v < V; ++v)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) vals[v] += __shfl_xor_sync(0xffffffffu, vals[v], off);
      const int warp = t >> 5, lane = t & 31;
      float* rb = red + ((size_t)(rbuf * a.NT + team) * nwarp_team) * V;
      if (lane == 0) {
#pragma unroll
        for (int v = 0; v < V; ++v) rb[warp * V + v] = vals[v];
      }
      team_barrier(1 + team, a.TS);
      for (int o = t; o < R * MR; o += a.TS) {
        const int r = o / MR, m = o - r * MR;
        const int rl = tile * R + r;
        if (m >= a.M || rl >= rows) continue;
        const int n = r_begin + rl;
        float v0 = 0.f, v1 = 0.f;
        for (int w2 = 0; w2 < nwarp_team; ++w2) {
          v0 += rb[w2 * V + (r * NW + 0) * MR + m];
          if constexpr (NW == 2) v1 += rb[w2 * V + (r * NW + 1) * MR + m];
        }
        float outv;
        if constexpr (KIND == 0) {
          outv = v0 / (1.0f + expf(-v0)) * v1;  // silu(gate) * up
        } else {
          if (a.res) outv = v0 + bf16f(a.res[(size_t)m * a.res_ld + n]);  // + residual or bias
          else outv = v0;
        }
        if (a.out_f32)
          static_cast<float*>(a.out)[(size_t)m * a.N + n] = outv;
        else
          static_cast<uint16_t*>(a.out)[(size_t)m * a.N + n] = f2bf(outv);
      }
      rbuf ^= 1;
    }
  };

  // Register ping-pong: the loads of step s+1 are in flight while step s is
  // computed.  Two steps per iteration keep every register index static.
  for (int s = 0; s < steps; s += 2) {
    load_step(s + 1, wB);
    compute_step(s, wA);
    if (s + 1 >= steps) break;
    load_step(s + 2, wA);
    compute_step(s + 1, wB);
  }
}

// Host-side planning and launch of one instantiation.
template <int FMT, int KIND, int MR, int R>
mt_status run_gemv(const GemvProblem& p, const Launch& l);

}  // namespace mt
