// k_phase.cuh - one "phase" of the one-row (M == 1) decode MLP on a
// persistent CTA: a GEMV over group-wise affine (INT8, INT4) or dense bf16
// weights whose rows are split into warp tasks.  Used by the single-call
// GEMV kernel (k_gemv_warp.cuh) and by the whole-stack kernel (k_stack.cu).
//
// meTile docs, "Compute-Graph Fusion", Automatic Gated Epilogues (gate and up
// share the activation; silu(gate) * up and the residual add are epilogues);
// "MLX-LM Backend", Dispatch Policy (affine w = scale * q + bias per group of
// 32/64/128 along K, fp32 accumulation).
//
// GB300 design (each choice measured on this part):
//  * One CTA of 16 warps per SM owns a contiguous range of output rows.  The
//    range is cut into tasks of two weight streams of B bytes that share
//    their activations: gate and up of one row (gate/up), or two consecutive
//    rows (down).  A row of exactly 64 chunks (INT4 K = 2048, INT8 K = 1024,
//    bf16 K = 512) would fill only half of a lane's registers, so there a
//    stream spans two consecutive rows (RS = 2): every task still moves 4 KB,
//    which doubles the bytes in flight for those shapes.  Tasks are handed
//    out through a shared-memory counter, so the warps of a CTA finish within
//    about one task of each other.
//  * A warp holds two tasks' weights in registers (128-bit evict-first
//    loads, up to 8 x 16 B per lane per task): it computes one while the
//    other is in flight, ~128 KB in flight per SM with no per-copy issue
//    cost.  (Bulk TMA copies cost the issuing thread ~350 cycles each on
//    this part, which capped a TMA-ring design near 3.5 TB/s for 2-4 KB
//    pieces.)  The first two tasks of a phase are requested before anything
//    the phase depends on is awaited.
//  * Besides its own two tasks, a warp that takes task t asks L2 for task
//    t + 2W (W warps), which some warp will take about one round later: the
//    HBM requests in flight are no longer limited by the register buffers.
//  * The CTA's scales and biases (bf16) and x are staged once in shared
//    memory with cp.async 16-byte copies issued by every thread.
//  * The affine term is factored as
//      sum_k (s q_k + b) x_k = sum_chunks s * (sum q_k x_k) + sum_groups b * X_g
//    with X_g the sum of x over group g (fp32, from the bf16 values).  x is
//    held as a fixed-point integer X = round(x * 2^e) of PL bytes, one 2^e
//    for the whole vector chosen from its max|x|:
//      PL = 2 (bf16 outputs): |X| <= 2^14; every element within 2^6 of the
//        vector's maximum is exact, smaller ones are rounded to 2^-14 of it,
//        below the outputs' own bf16 rounding (2^-9 relative);
//      PL = 3 (fp32 outputs): |X| <= 2^22; every element within 2^14 of the
//        maximum is exact, smaller ones are rounded to 2^-22 of it.
//    X is split into PL byte planes (the top one signed), and the packed
//    codes are used as they are stored: one dp4a (four u8 x s8/u8 products
//    added to an int32) per weight word and plane, so a 16-byte chunk of INT8
//    codes costs 4 PL dp4a.  The plane sums of a chunk are exact integers;
//    combining them into fp32 rounds once (PL = 2) or at most twice (PL = 3),
//    and the scale 2^-e is divided out of the partial sums.  INT4 words are
//    split into their low and high nibbles (two masks) against even/odd
//    element planes.
//    This replaced an fp16 exponent-bias dequant + mixed-precision FMA chain
//    that was instruction-bound at ~4.6 instructions per weight.  Dense bf16
//    weights use mixed-precision bf16 FMAs (exact products, fp32
//    accumulation) with x unchanged.
//  * A task's partial sums are reduced inside the warp (shuffles) and stored
//    per piece in shared memory; after one barrier the caller's epilogue adds
//    the pieces of a row in a fixed order (deterministic).
#pragma once
#include "k_gemv.cuh"

namespace mt {

constexpr int WARP_TASK_WARPS = 16;  // warps per CTA
constexpr int WARP_TASK_UPL = 8;     // 16-byte loads per lane per task (all matrices)
constexpr int WT_NS = 2;             // weight streams per task
constexpr int WT_CL = WARP_TASK_UPL / WT_NS;  // chunks per lane per stream per task
constexpr int WT_THREADS = WARP_TASK_WARPS * 32;

// Geometry of one phase: the GEMV's K and N, the cut of a row into P pieces
// (tasks) and the partition of the N rows over the grid.
struct PhaseGeom {
  int K, N;
  int group, lg_group, G;    // group size, log2(group), groups per row (affine)
  int CPR;                   // 16-byte chunks per row
  int row_bytes;             // bytes of one weight row
  int row_unit;              // rows are dealt out in units of row_unit consecutive rows
  int rows_base, rows_extra; // CTA i owns row_unit * (rows_base + (i < rows_extra)) rows
  int rows_alloc;            // row_unit * (rows_base + (rows_extra != 0))
  int P;                     // pieces per row
  unsigned long long p_mul;  // ceil(2^32 / P): t / P == (t * p_mul) >> 32 for t < 2^32 / P
  int B;                     // bytes per piece (multiple of 16)
  int CPP;                   // 16-byte chunks per piece (<= 32 * WT_CL)
  int GPP;                   // groups per piece (affine)
  int sb_stride;             // elements per staged scale or bias array (multiple of 8)
  int sb_vec;                // 1: scales/biases are staged in 16-byte copies (G % 8 == 0)
  int RS;                    // rows per stream: 1, or 2 when P == 1 and CPR == 16 * WT_CL
                             // (the kernel instantiated for it is chosen on the host)
};

// Weights of one phase.  Gate/up: W0 = gate, W1 = up.  Down: W0 only.
struct PhaseW {
  const uint8_t* W0;
  const uint8_t* W1;
  const uint16_t* s0;
  const uint16_t* b0;
  const uint16_t* s1;
  const uint16_t* b1;
};

// Shared-memory arrays of one phase.
struct PhaseSmem {
  uint16_t* xraw;  // [K] bf16 activations
  uint4* xs;       // staging layout of x (see below), xs_bytes<FMT, PL>(K) bytes
  int xs_stride;   // 16-byte units between two activation rows' staging (MR = 2)
  float* gsum;     // [G] X_g (affine)
  float* xinv;     // [P] 2^-e, undoing the x scale (the same for every piece; affine)
  uint16_t* sbr;   // 2*NW arrays of sb_stride bf16: 2m = scales, 2m+1 = biases of matrix m
  float* parts;    // [rows][P][NW] partial sums of the pieces
};

// Bytes of a phase's shared arrays other than xraw and xs, in the order gsum,
// xinv, sbr, parts (each a multiple of 16 bytes).  MR: activation rows (the
// one-row kernel also takes two): gsum [MR][G], xinv [MR][P], parts
// [rows][P][NW][MR].
template <int FMT, int KIND, int MR = 1>
__host__ __device__ inline size_t phase_tail_bytes(const PhaseGeom& g) {
  constexpr bool AFF = FmtTraits<FMT>::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;
  size_t n = 0;
  if (AFF) {
    n += (size_t)(MR * g.G + 3) / 4 * 16;
    n += (size_t)(MR * g.P + 3) / 4 * 16;
    n += (size_t)2 * NW * g.sb_stride * 2;
  }
  n += ((size_t)g.rows_alloc * g.P * NW * MR * 4 + 15) / 16 * 16;
  return n;
}

// Points sm's gsum, xinv, sbr and parts into the tail at p (16-byte aligned,
// phase_tail_bytes long).
template <int FMT, int KIND, int MR = 1>
__device__ __forceinline__ void phase_tail_carve(const PhaseGeom& g, unsigned char* p, PhaseSmem& sm) {
  constexpr bool AFF = FmtTraits<FMT>::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;
  sm.gsum = reinterpret_cast<float*>(p);
  if (AFF) p += (size_t)(MR * g.G + 3) / 4 * 16;
  sm.xinv = reinterpret_cast<float*>(p);
  if (AFF) p += (size_t)(MR * g.P + 3) / 4 * 16;
  sm.sbr = reinterpret_cast<uint16_t*>(p);
  if (AFF) p += (size_t)2 * NW * g.sb_stride * 2;
  sm.parts = reinterpret_cast<float*>(p);
}

// The rows a CTA owns in one phase and its task count.
struct PhaseCta {
  int r_begin, rows, T;
};

template <int KIND, int RS = 1>
__device__ __forceinline__ PhaseCta phase_cta(const PhaseGeom& g, int cta) {
  constexpr int RW = (KIND == 0 ? 1 : 2) * RS;  // rows per task (RS == g.RS)
  PhaseCta c;
  c.r_begin = g.row_unit * (cta * g.rows_base + min(cta, g.rows_extra));
  c.rows = g.row_unit * (g.rows_base + (cta < g.rows_extra ? 1 : 0));
  c.T = (c.rows + RW - 1) / RW * g.P;
  return c;
}

// Staging layout of x, read by chunk_dot (16-byte units; CPR chunks per row).
// Affine formats hold x as a fixed-point integer X of PL bytes (PL = 3: 24
// bits, for fp32 outputs; PL = 2: 16 bits, for bf16 outputs), stored as PL
// byte planes; plane 0 is the most significant byte (signed), the others are
// unsigned:
// A8:   unit p*CPR + c holds byte plane p (byte PL-1-p of X) of the 16
//       elements of chunk c, in element order.
// A4:   unit (2p + h)*CPR + c holds byte plane p of the even (h = 0) or odd
//       (h = 1) elements of chunk c's 32: byte b of word wi is element
//       8wi + 2b + h, matching the low / high nibbles of weight word wi.
// BF16: words 2u, 2u+1 of chunk c read 4 bf16 (elements 4u..4u+3) at 8-byte
//       unit u*CPR + c.
template <int FMT, int PL>
__host__ __device__ constexpr size_t xs_bytes(int K) {
  return FMT == FMT_BF16 ? (size_t)K * 2 : (size_t)K * PL;
}

// s += the four byte products of a (unsigned codes) and b (signed or
// unsigned x bytes), exactly, in int32.
__device__ __forceinline__ void dp4a_us(int& s, uint32_t a, uint32_t b) {
  asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(s) : "r"(a), "r"(b));
}
__device__ __forceinline__ void dp4a_uu(uint32_t& s, uint32_t a, uint32_t b) {
  asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(s) : "r"(a), "r"(b));
}

// The plane sums of one chunk, S = 65536 S2 + 256 S1 + S0 = sum q_k X_k, in
// fp32.  The plane sums are exact; S1, S0 <= 255 * 255 * 32, so 256 S1 + S0 <
// 2^31 is exact in int32.  Its conversion to fp32 rounds when it exceeds 2^24
// and the final fma rounds once more, so S carries at most two fp32 roundings.
__device__ __forceinline__ float combine_planes(int s2, uint32_t s1, uint32_t s0) {
  return fmaf((float)s2, 65536.f, (float)(int)(s1 * 256u + s0));
}
// Two planes (16-bit X): S = 256 S1 + S0 with |S1| <= 32 * 255 * 128 and S0 <=
// 32 * 255 * 255, exact in int32; one rounding in the conversion to fp32.
__device__ __forceinline__ float combine_planes(int s1, uint32_t s0) {
  return (float)(s1 * 256 + (int)s0);
}

// acc_lo += lo(a) * lo(b), acc_hi += hi(a) * hi(b) for bf16 pairs: exact
// products in fp32, fp32 accumulation.
__device__ __forceinline__ void fma2_bf16_f32(float& lo, float& hi, uint32_t a, uint32_t b) {
  asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
      "mov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
      "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %1, a1, b1, %1;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "r"(a), "r"(b));
}

// Dot product of one 16-byte weight chunk (chunk c of its row) with its
// activations from the staging layout: sum of q * X (affine, PL byte planes,
// exact but for the final conversion, returned in fp32) or of w * x (bf16,
// fp32 accumulation).
template <int FMT, int PL>
__device__ __forceinline__ float chunk_dot(const uint4 w, const uint4* __restrict__ xs, int c,
                                           int CPR) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  if constexpr (FMT == FMT_A8 && PL == 2) {
    const uint4 p1 = xs[c], p0 = xs[CPR + c];
    const uint32_t x1[4] = {p1.x, p1.y, p1.z, p1.w};
    const uint32_t x0[4] = {p0.x, p0.y, p0.z, p0.w};
    int s1 = 0;
    uint32_t s0 = 0;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      dp4a_us(s1, ww[wi], x1[wi]);
      dp4a_uu(s0, ww[wi], x0[wi]);
    }
    return combine_planes(s1, s0);
  } else if constexpr (FMT == FMT_A4 && PL == 2) {
    const uint4 e1 = xs[c], o1 = xs[CPR + c], e0 = xs[2 * CPR + c], o0 = xs[3 * CPR + c];
    const uint32_t xe1[4] = {e1.x, e1.y, e1.z, e1.w}, xo1[4] = {o1.x, o1.y, o1.z, o1.w};
    const uint32_t xe0[4] = {e0.x, e0.y, e0.z, e0.w}, xo0[4] = {o0.x, o0.y, o0.z, o0.w};
    int s1 = 0;
    uint32_t s0 = 0;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const uint32_t lo = ww[wi] & 0x0F0F0F0Fu;         // codes 8wi + 0, 2, 4, 6
      const uint32_t hi = (ww[wi] >> 4) & 0x0F0F0F0Fu;  // codes 8wi + 1, 3, 5, 7
      dp4a_us(s1, lo, xe1[wi]);
      dp4a_us(s1, hi, xo1[wi]);
      dp4a_uu(s0, lo, xe0[wi]);
      dp4a_uu(s0, hi, xo0[wi]);
    }
    return combine_planes(s1, s0);
  } else if constexpr (FMT == FMT_A8) {
    const uint4 p2 = xs[c], p1 = xs[CPR + c], p0 = xs[2 * CPR + c];
    const uint32_t x2[4] = {p2.x, p2.y, p2.z, p2.w};
    const uint32_t x1[4] = {p1.x, p1.y, p1.z, p1.w};
    const uint32_t x0[4] = {p0.x, p0.y, p0.z, p0.w};
    int s2 = 0;
    uint32_t s1 = 0, s0 = 0;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      dp4a_us(s2, ww[wi], x2[wi]);
      dp4a_uu(s1, ww[wi], x1[wi]);
      dp4a_uu(s0, ww[wi], x0[wi]);
    }
    return combine_planes(s2, s1, s0);
  } else if constexpr (FMT == FMT_A4) {
    const uint4 e2 = xs[c], o2 = xs[CPR + c], e1 = xs[2 * CPR + c], o1 = xs[3 * CPR + c];
    const uint4 e0 = xs[4 * CPR + c], o0 = xs[5 * CPR + c];
    const uint32_t xe2[4] = {e2.x, e2.y, e2.z, e2.w}, xo2[4] = {o2.x, o2.y, o2.z, o2.w};
    const uint32_t xe1[4] = {e1.x, e1.y, e1.z, e1.w}, xo1[4] = {o1.x, o1.y, o1.z, o1.w};
    const uint32_t xe0[4] = {e0.x, e0.y, e0.z, e0.w}, xo0[4] = {o0.x, o0.y, o0.z, o0.w};
    int s2 = 0;
    uint32_t s1 = 0, s0 = 0;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const uint32_t lo = ww[wi] & 0x0F0F0F0Fu;         // codes 8wi + 0, 2, 4, 6
      const uint32_t hi = (ww[wi] >> 4) & 0x0F0F0F0Fu;  // codes 8wi + 1, 3, 5, 7
      dp4a_us(s2, lo, xe2[wi]);
      dp4a_us(s2, hi, xo2[wi]);
      dp4a_uu(s1, lo, xe1[wi]);
      dp4a_uu(s1, hi, xo1[wi]);
      dp4a_uu(s0, lo, xe0[wi]);
      dp4a_uu(s0, hi, xo0[wi]);
    }
    return combine_planes(s2, s1, s0);
  } else {
    const uint2* xu = reinterpret_cast<const uint2*>(xs);
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint2 xv = xu[u * CPR + c];
      fma2_bf16_f32(a0, a1, ww[2 * u], xv.x);
      fma2_bf16_f32(a2, a3, ww[2 * u + 1], xv.y);
    }
    return (a0 + a1) + (a2 + a3);
  }
}

// Asks L2 for the weights of task t (one 128-byte line per lane; no
// registers are written).
template <int KIND, int RS = 1>
__device__ __forceinline__ void wt_prefetch(const PhaseGeom& g, const PhaseW& w, const PhaseCta& c,
                                            int t, int lane) {
  constexpr int RW = KIND == 0 ? 1 : 2;
  if (t >= c.T) return;
  const int rg = (int)(((unsigned long long)(unsigned)t * g.p_mul) >> 32);
  const int p = t - rg * g.P;
  const int v = lane >> 4, line = lane & 15;  // lanes 0-15: stream 0, 16-31: stream 1
  // with RS = 2 the stream is two whole rows (P == 1): lines 0-7 and 8-15
  const int rl = (rg * RW + (KIND == 0 ? 0 : v)) * RS + (RS == 2 ? line * 128 / g.row_bytes : 0);
  if (rl >= c.rows || line * 128 >= g.B * RS) return;
  const uint8_t* src = (KIND == 0 && v ? w.W1 : w.W0) + (size_t)(c.r_begin + rl) * g.row_bytes +
                       (size_t)p * g.B + (size_t)(RS == 2 ? line * 128 % g.row_bytes : line * 128);
  prefetch_l2_normal(src);
}

// Requests chunk slot k of every stream of task t into buf[.][k] (zeros
// for t >= T or rows past the CTA's range).  Stream v of a task: matrix v of
// row rg (gate/up) or row 2*rg + v (down); piece p of the row.  Lane chunk
// slot k is chunk lane + 32 k of the piece (RS = 1), or chunk lane + 32 (k & 1)
// of row k >> 1 of the stream's two rows (RS = 2: whole rows of 64 chunks).
template <int KIND, int RS = 1>
__device__ __forceinline__ void wt_load_chunk(const PhaseGeom& g, const PhaseW& w, const PhaseCta& c,
                                              int t, uint4 (&buf)[WT_NS][WT_CL], int k, uint64_t pol,
                                              int lane) {
  constexpr int RW = KIND == 0 ? 1 : 2;
  const int rg = (int)(((unsigned long long)(unsigned)t * g.p_mul) >> 32);
  const int p = t - rg * g.P;
#pragma unroll
  for (int v = 0; v < WT_NS; ++v) {
    const uint8_t* W = KIND == 0 && v ? w.W1 : w.W0;
    if constexpr (RS == 1) {
      const int rl = rg * RW + (KIND == 0 ? 0 : v);
      const int j = lane + 32 * k;
      const bool ok = t < c.T && rl < c.rows && j < g.CPP;
      buf[v][k] = ok ? ldg_stream_pol(W + (size_t)(c.r_begin + rl) * g.row_bytes + (size_t)p * g.B + (size_t)j * 16, pol)
                     : make_uint4(0, 0, 0, 0);
    } else {
      const int r = (rg * RW + (KIND == 0 ? 0 : v)) * 2 + (k >> 1);
      const bool ok = t < c.T && r < c.rows;
      buf[v][k] = ok ? ldg_stream_pol(W + (size_t)(c.r_begin + r) * g.row_bytes + (size_t)(lane + 32 * (k & 1)) * 16, pol)
                     : make_uint4(0, 0, 0, 0);
    }
  }
}

// Requests the weights of task t into buf (every chunk slot).
template <int KIND, int RS = 1>
__device__ __forceinline__ void wt_load(const PhaseGeom& g, const PhaseW& w, const PhaseCta& c,
                                        int t, uint4 (&buf)[WT_NS][WT_CL], uint64_t pol,
                                        int lane) {
#pragma unroll
  for (int k = 0; k < WT_CL; ++k) wt_load_chunk<KIND, RS>(g, w, c, t, buf, k, pol, lane);
}

// Stages the CTA's scales and biases (contiguous [rows][G] blocks) into
// sbr, spread over threads t = 0 .. nt-1 of the CTA.  16-byte path: cp.async
// copies, committed by the caller.
template <int KIND>
__device__ __forceinline__ void stage_sb(const PhaseGeom& g, const PhaseW& w, const PhaseCta& c,
                                         uint16_t* sbr, int t, int nt) {
  constexpr int NW = KIND == 0 ? 2 : 1;
  if (g.sb_vec) {
    const int n16 = c.rows * g.G / 8;
    const size_t off = (size_t)c.r_begin * g.G;
    for (int i = t; i < n16; i += nt) {
#pragma unroll
      for (int m = 0; m < NW; ++m) {
        cp_async16(sbr + (size_t)(2 * m) * g.sb_stride + i * 8, (m ? w.s1 : w.s0) + off + i * 8);
        cp_async16(sbr + (size_t)(2 * m + 1) * g.sb_stride + i * 8, (m ? w.b1 : w.b0) + off + i * 8);
      }
    }
  } else {
    const int n_sb = c.rows * g.G;
    for (int i = t; i < n_sb; i += nt) {
      const size_t gi = (size_t)c.r_begin * g.G + i;
#pragma unroll
      for (int m = 0; m < NW; ++m) {
        sbr[(size_t)(2 * m) * g.sb_stride + i] = ldg_u16((m ? w.s1 : w.s0) + gi);
        sbr[(size_t)(2 * m + 1) * g.sb_stride + i] = ldg_u16((m ? w.b1 : w.b0) + gi);
      }
    }
  }
}

// Staging of x, in 8-element units (one uint4 of bf16).
//
// The largest |x| of a unit (exact).
__device__ __forceinline__ float unit_absmax(const uint4 v) {
  const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16lo(vw[j])), fabsf(bf16hi(vw[j]))));
  return m;
}

// The exponent e with m * 2^e in [2^(8 PL - 3), 2^(8 PL - 2)) for the
// largest |x| m of the vector (a zero or subnormal m takes the largest
// exponent, 126): then X = round(x * 2^e) has |X| <= 2^(8 PL - 2) for every
// element, within the signed range of PL bytes (24 bits: 2^22; 16 bits: 2^14).
template <int PL>
__device__ __forceinline__ int fx_exponent(float m) {
  const int mb = __float_as_int(m);
  return (mb >> 23) >= 255 ? 0 : max(-126, min(126, (8 * PL - 3) - ((mb >> 23) - 127)));
}

// Byte k of each of a, b, c, d, packed as one word (a in the low byte).
__device__ __forceinline__ uint32_t byte_plane(uint32_t a, uint32_t b, uint32_t c, uint32_t d, int k) {
  const uint32_t sel = (uint32_t)k | ((uint32_t)(k + 4) << 4);
  return __byte_perm(__byte_perm(a, b, sel), __byte_perm(c, d, sel), 0x5410);
}

// Unit i of x (0 <= i < K/8): stored in sm.xraw (when store_raw), in the
// staging layout sm.xs with the scale xscale = 2^e (affine), and its sum
// added into the group sum X_g = sm.gsum[g] (fp32).  Every lane of a warp
// calls it together for units base + lane (base a multiple of 32; i = -1 for
// a lane without a unit), so the group/8 units of a quantisation group sit in
// consecutive lanes and are summed with a fixed shuffle tree.  The caller ends
// the staging with a CTA barrier before sm.xs is read.
template <int FMT, int PL>
__device__ __forceinline__ void x_stage_unit(const PhaseGeom& g, const PhaseSmem& sm, int i, const uint4 v,
                                             float xscale, bool store_raw) {
  static_assert(PL == 2 || PL == 3, "16- or 24-bit fixed point");
  if (store_raw && i >= 0) reinterpret_cast<uint4*>(sm.xraw)[i] = v;
  const int CPR = g.CPR;
  if constexpr (!FmtTraits<FMT>::AFFINE) {
    // bf16: a unit is a chunk; its words 2u, 2u+1 go to 8-byte unit u*CPR + c
    if (i >= 0) {
      reinterpret_cast<uint2*>(sm.xs)[i] = make_uint2(v.x, v.y);
      reinterpret_cast<uint2*>(sm.xs)[CPR + i] = make_uint2(v.z, v.w);
    }
  } else {
    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
    float sum = 0.f;
    uint32_t X[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = bf16lo(vw[j]), hi = bf16hi(vw[j]);
      sum += lo + hi;
      // |x * xscale| <= 2^(8 PL - 2) by the choice of the scale
      X[2 * j] = (uint32_t)round_small_to_int(lo * xscale);
      X[2 * j + 1] = (uint32_t)round_small_to_int(hi * xscale);
    }
    const int upg = g.group >> 3;  // units per group: 4, 8 or 16
    for (int off = 1; off < upg; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (i < 0) return;
    if ((i & (upg - 1)) == 0) sm.gsum[i >> (g.lg_group - 3)] = sum;
    if constexpr (FMT == FMT_A8) {
      // unit i = words 2(i&1), 2(i&1)+1 of chunk i>>1; plane p byte PL-1-p of X
      uint2* xs2 = reinterpret_cast<uint2*>(sm.xs);
      const int c = i >> 1, h = i & 1;
#pragma unroll
      for (int p = 0; p < PL; ++p)
        xs2[(size_t)(p * CPR + c) * 2 + h] = make_uint2(byte_plane(X[0], X[1], X[2], X[3], PL - 1 - p),
                                                        byte_plane(X[4], X[5], X[6], X[7], PL - 1 - p));
    } else {
      // unit i = word i&3 of chunk i>>2: even elements -> half 0, odd -> half 1
      uint32_t* xs4 = reinterpret_cast<uint32_t*>(sm.xs);
      const int c = i >> 2, wi = i & 3;
#pragma unroll
      for (int p = 0; p < PL; ++p) {
        xs4[(size_t)((2 * p) * CPR + c) * 4 + wi] = byte_plane(X[0], X[2], X[4], X[6], PL - 1 - p);
        xs4[(size_t)((2 * p + 1) * CPR + c) * 4 + wi] = byte_plane(X[1], X[3], X[5], X[7], PL - 1 - p);
      }
    }
  }
}

// Records the scale 2^-e for every piece (affine; threads t < P of nt).
template <int FMT>
__device__ __forceinline__ void x_set_scale(const PhaseGeom& g, const PhaseSmem& sm, int ex, int t, int nt) {
  if constexpr (FmtTraits<FMT>::AFFINE)
    for (int p = t; p < g.P; p += nt) sm.xinv[p] = exp2i(-ex);
}

// The largest value over the CTA of one float per thread; every thread gets
// it.  red: WARP_TASK_WARPS floats of shared memory, free on entry and not
// reused before the next CTA barrier.
__device__ __forceinline__ float cta_max(float v, float* red, int tid) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  if ((tid & 31) == 0) red[tid >> 5] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < WARP_TASK_WARPS; ++w) m = fmaxf(m, red[w]);
  return m;
}

// Sums four values over the warp in one butterfly: at step 16 a lane keeps
// a, b (bit 4 clear) or c, d (set) and sends the other pair; at step 8 it
// keeps the first (bit 3 clear) or second of its pair; steps 4, 2, 1 finish.
// Lane l returns the warp sum of value 2 * bit4(l) + bit3(l) of (a, b, c, d),
// added in the same tree as a full butterfly of that value.
__device__ __forceinline__ float reduce4_lanes(float a, float b, float c, float d, int lane) {
  const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
  float x = h16 ? c : a, y = h16 ? d : b;
  x += __shfl_xor_sync(0xffffffffu, h16 ? a : c, 16);
  y += __shfl_xor_sync(0xffffffffu, h16 ? b : d, 16);
  float z = h8 ? y : x;
  z += __shfl_xor_sync(0xffffffffu, h8 ? x : y, 8);
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  return z;
}

// wt_compute for RS = 2 (P == 1, rows of 64 chunks): stream v holds rows
// r_v and r_v + 1, r_v = 2 (t * RW + v) for down and 2t (both matrices) for
// gate/up; a lane's chunks k = 0, 1 (chunk lane + 32 k) are row r_v and
// k = 2, 3 (chunk lane + 32 (k - 2)) row r_v + 1.  Each row's partial sum is
// formed exactly as in wt_compute (the same chunk, group and lane order, the
// same reduction), so it does not depend on whether the row is the first or
// second of its stream, and is stored as its single piece.
template <int FMT, int KIND, int PL, class AfterChunk>
__device__ __forceinline__ void wt_compute_rs2(const PhaseGeom& g, const PhaseCta& c,
                                               const PhaseSmem& sm, int t,
                                               const uint4 (&buf)[WT_NS][WT_CL], int lane,
                                               AfterChunk after) {
  using T = FmtTraits<FMT>;
  constexpr int EPC = T::EPC;
  constexpr bool AFF = T::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;
  constexpr int RW = KIND == 0 ? 1 : 2;
  static_assert(WT_CL == 4, "two rows of two chunks per lane");
  auto row_of = [&](int v, int r) { return (t * RW + (KIND == 0 ? 0 : v)) * 2 + r; };
  // scales of stream v, row r: chunk lane + 32 (k & 1) is in group gi0 +
  // (k & 1) * gstep (exact, as in wt_compute)
  const uint16_t* sc[WT_NS][2];
  int gstep = 0;
  if constexpr (AFF) {
    const int gi0 = (lane * EPC) >> g.lg_group;
    gstep = (32 * EPC) >> g.lg_group;
#pragma unroll
    for (int v = 0; v < WT_NS; ++v)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int m = KIND == 0 ? v : 0, rl = min(row_of(v, r), c.rows - 1);
        sc[v][r] = sm.sbr + (size_t)(2 * m) * g.sb_stride + rl * g.G + gi0;
      }
  }
  float acc[WT_NS][2];
#pragma unroll
  for (int v = 0; v < WT_NS; ++v) acc[v][0] = acc[v][1] = 0.f;
#pragma unroll
  for (int k = 0; k < WT_CL; ++k) {
    const int r = k >> 1, ch = lane + 32 * (k & 1);
#pragma unroll
    for (int v = 0; v < WT_NS; ++v) {
      const float d = chunk_dot<FMT, PL>(buf[v][k], sm.xs, ch, g.CPR);
      if constexpr (AFF) acc[v][r] = fmaf(bf16f(sc[v][r][(k & 1) * gstep]), d, acc[v][r]);
      else acc[v][r] += d;
    }
    after(k);
  }
  float vals[WT_NS][2];
#pragma unroll
  for (int v = 0; v < WT_NS; ++v)
#pragma unroll
    for (int r = 0; r < 2; ++r) vals[v][r] = AFF ? acc[v][r] * sm.xinv[0] : acc[v][r];
  if constexpr (AFF) {
    // bias terms: sum_g b_g * X_g over each row's groups, group g on lane
    // g mod 32 for both rows, as in wt_compute, so a row's sum does not depend
    // on its place in the stream (the partition of rows over CTAs may differ)
    for (int gi = lane; gi < g.G; gi += 32) {
      const float xg = sm.gsum[gi];
#pragma unroll
      for (int v = 0; v < WT_NS; ++v)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int m = KIND == 0 ? v : 0, rl = min(row_of(v, r), c.rows - 1);
          vals[v][r] = fmaf(bf16f(sm.sbr[(size_t)(2 * m + 1) * g.sb_stride + rl * g.G + gi]), xg, vals[v][r]);
        }
    }
  }
  // the four warp sums in one butterfly: lanes keep stream v = bit 4 and row
  // r = bit 3 of their index, sending the others at the first two steps
  const float s = reduce4_lanes(vals[0][0], vals[0][1], vals[1][0], vals[1][1], lane);
  if ((lane & 7) == 0) {
    const int v = (lane >> 4) & 1, r = (lane >> 3) & 1;
    const int m = KIND == 0 ? v : 0, rl = row_of(v, r);
    if (rl < c.rows) sm.parts[(size_t)rl * NW + m] = s;
  }
}

// wt_compute for two activation rows (MR = 2; affine INT8, one row per
// stream): each weight chunk is multiplied with both rows' staged x (row m's
// staging at sm.xs + m * xs_stride, its group sums at sm.gsum + m * G, its
// scale at sm.xinv[m * P + p]).  Each row's sum is formed as in wt_compute;
// parts hold [rows][P][NW][2].
template <int FMT, int KIND, int PL, class AfterChunk>
__device__ __forceinline__ void wt_compute_mr2(const PhaseGeom& g, const PhaseCta& c,
                                               const PhaseSmem& sm, int t,
                                               const uint4 (&buf)[WT_NS][WT_CL], int lane,
                                               AfterChunk after) {
  using T = FmtTraits<FMT>;
  constexpr int EPC = T::EPC;
  constexpr int NW = KIND == 0 ? 2 : 1;
  constexpr int RW = KIND == 0 ? 1 : 2;
  static_assert(FMT == FMT_A8, "two activation rows: affine INT8");
  const int rg = (int)(((unsigned long long)(unsigned)t * g.p_mul) >> 32);
  const int p = t - rg * g.P;
  const int rl0 = rg * RW;
  float acc[WT_NS][2];
#pragma unroll
  for (int v = 0; v < WT_NS; ++v) acc[v][0] = acc[v][1] = 0.f;
  // scales: slot k in group gi0 + k*gstep (exact, as in wt_compute)
  const int gstep = (32 * EPC) >> g.lg_group;
  const uint16_t* sc[WT_NS];
#pragma unroll
  for (int v = 0; v < WT_NS; ++v) {
    const int mt = KIND == 0 ? v : 0, rl = min(rl0 + (KIND == 0 ? 0 : v), c.rows - 1);
    sc[v] = sm.sbr + (size_t)(2 * mt) * g.sb_stride + rl * g.G + (((p * g.CPP + lane) * EPC) >> g.lg_group);
  }
#pragma unroll
  for (int k = 0; k < WT_CL; ++k) {
    const int j = lane + 32 * k;
    if (j < g.CPP) {
      const int ch = p * g.CPP + j;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint4* xs = sm.xs + (size_t)m * sm.xs_stride;
#pragma unroll
        for (int v = 0; v < WT_NS; ++v) {
          const float d = chunk_dot<FMT, PL>(buf[v][k], xs, ch, g.CPR);
          acc[v][m] = fmaf(bf16f(sc[v][k * gstep]), d, acc[v][m]);
        }
      }
    }
    after(k);
  }
  float vals[WT_NS][2];
#pragma unroll
  for (int v = 0; v < WT_NS; ++v)
#pragma unroll
    for (int m = 0; m < 2; ++m) vals[v][m] = acc[v][m] * sm.xinv[m * g.P + p];
  // bias terms of the groups in this piece: sum_g b_g * X_g, per row of x
  for (int gl = lane; gl < g.GPP; gl += 32) {
    const int gi = p * g.GPP + gl;
#pragma unroll
    for (int v = 0; v < WT_NS; ++v) {
      const int mt = KIND == 0 ? v : 0, rl = min(rl0 + (KIND == 0 ? 0 : v), c.rows - 1);
      const float b = bf16f(sm.sbr[(size_t)(2 * mt + 1) * g.sb_stride + rl * g.G + gi]);
#pragma unroll
      for (int m = 0; m < 2; ++m) vals[v][m] = fmaf(b, sm.gsum[m * g.G + gi], vals[v][m]);
    }
  }
  // the four warp sums in one butterfly (stream v = bit 4, activation row m
  // = bit 3 of the lane that ends with the sum)
  const float s = reduce4_lanes(vals[0][0], vals[0][1], vals[1][0], vals[1][1], lane);
  if ((lane & 7) == 0) {
    const int v = (lane >> 4) & 1, m = (lane >> 3) & 1;
    const int mt = KIND == 0 ? v : 0, rl = rl0 + (KIND == 0 ? 0 : v);
    if (rl < c.rows) sm.parts[(((size_t)rl * g.P + p) * NW + mt) * 2 + m] = s;
  }
}

// Computes task t from the weights in buf and stores its partial sums (one
// per stream) in sm.parts.  after(k) runs once chunk slot k of every stream
// has been consumed, so that the slot's registers can be refilled while the
// rest of the task is computed.
template <int FMT, int KIND, int PL, int RS = 1, int MR = 1, class AfterChunk>
__device__ __forceinline__ void wt_compute(const PhaseGeom& g, const PhaseCta& c,
                                           const PhaseSmem& sm, int t,
                                           const uint4 (&buf)[WT_NS][WT_CL], int lane,
                                           AfterChunk after) {
  using T = FmtTraits<FMT>;
  constexpr int EPC = T::EPC;
  constexpr bool AFF = T::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;
  constexpr int RW = KIND == 0 ? 1 : 2;
  if constexpr (RS == 2) {
    wt_compute_rs2<FMT, KIND, PL>(g, c, sm, t, buf, lane, after);
    return;
  }
  if constexpr (MR == 2) {
    wt_compute_mr2<FMT, KIND, PL>(g, c, sm, t, buf, lane, after);
    return;
  }
  const int rg = (int)(((unsigned long long)(unsigned)t * g.p_mul) >> 32);
  const int p = t - rg * g.P;
  const int rl0 = rg * RW;
  // scales: chunk slot k of this lane is chunk p*CPP + lane + 32k of the row,
  // in group gi0 + k*gstep (32 chunks span whole groups, so the step is exact)
  const uint16_t* sc[WT_NS];
  int gstep = 0;
  if constexpr (AFF) {
    const int gi0 = ((p * g.CPP + lane) * EPC) >> g.lg_group;
    gstep = (32 * EPC) >> g.lg_group;
#pragma unroll
    for (int v = 0; v < WT_NS; ++v) {
      const int m = KIND == 0 ? v : 0, rl = min(rl0 + (KIND == 0 ? 0 : v), c.rows - 1);
      sc[v] = sm.sbr + (size_t)(2 * m) * g.sb_stride + rl * g.G + gi0;
    }
  }
  float acc[WT_NS];
#pragma unroll
  for (int v = 0; v < WT_NS; ++v) acc[v] = 0.f;
#pragma unroll
  for (int k = 0; k < WT_CL; ++k) {
    const int j = lane + 32 * k;
    if (j < g.CPP) {
      const int ch = p * g.CPP + j;
#pragma unroll
      for (int v = 0; v < WT_NS; ++v) {
        const float d = chunk_dot<FMT, PL>(buf[v][k], sm.xs, ch, g.CPR);
        if constexpr (AFF) acc[v] = fmaf(bf16f(sc[v][k * gstep]), d, acc[v]);
        else acc[v] += d;
      }
    }
    after(k);
  }
  float vals[WT_NS];
#pragma unroll
  for (int v = 0; v < WT_NS; ++v) vals[v] = AFF ? acc[v] * sm.xinv[p] : acc[v];
  if constexpr (AFF) {
    // bias terms of the groups in this piece: sum_g b_g * X_g
    for (int gl = lane; gl < g.GPP; gl += 32) {
      const int gi = p * g.GPP + gl;
      const float xg = sm.gsum[gi];
#pragma unroll
      for (int v = 0; v < WT_NS; ++v) {
        const int m = KIND == 0 ? v : 0, rl = min(rl0 + (KIND == 0 ? 0 : v), c.rows - 1);
        vals[v] = fmaf(bf16f(sm.sbr[(size_t)(2 * m + 1) * g.sb_stride + rl * g.G + gi]), xg, vals[v]);
      }
    }
  }
  // the two streams' warp sums in one butterfly: at its first step lanes
  // 0-15 keep stream 0 and lanes 16-31 stream 1, each sending the other
  static_assert(WT_NS == 2, "two streams per task");
  const bool hi = (lane & 16) != 0;
  float r = hi ? vals[1] : vals[0];
  r += __shfl_xor_sync(0xffffffffu, hi ? vals[0] : vals[1], 16);
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  if ((lane & 15) == 0) {
    const int v = lane >> 4;
    const int m = KIND == 0 ? v : 0, rl = rl0 + (KIND == 0 ? 0 : v);
    if (rl < c.rows) sm.parts[((size_t)rl * g.P + p) * NW + m] = r;
  }
}

// The task loop of one warp.  On entry bufA holds task tA and bufB task tB
// (tA < tB, both requested) and tasks tA + 2W, tB + 2W have been asked of L2
// (wt_prefetch); task_ctr (shared) hands out the next task numbers.  Register
// ping-pong: one task is in flight while the other is computed; two tasks per
// iteration keep the buffer indices static.  EAGER: the task that replaces
// the one being computed is drawn first, and each of its chunk slots is
// requested as soon as the slot has been consumed, so the warp keeps nearly
// two tasks of weights in flight while it computes; otherwise the whole task
// is requested after the computation (one task in flight meanwhile, but the
// computation's shared-memory reads do not queue behind weight loads).
template <int FMT, int KIND, int PL, int RS = 1, int MR = 1, bool EAGER = false>
__device__ __forceinline__ void wt_run(const PhaseGeom& g, const PhaseW& w, const PhaseCta& c,
                                       const PhaseSmem& sm, uint4 (&bufA)[WT_NS][WT_CL],
                                       uint4 (&bufB)[WT_NS][WT_CL], int tA, int tB, int* task_ctr,
                                       uint64_t pol, int lane) {
  auto next_task = [&]() -> int {
    int t = 0;
    if (lane == 0) t = atomicAdd(task_ctr, 1);
    return __shfl_sync(0xffffffffu, t, 0);
  };
  constexpr int AHEAD = 2 * WARP_TASK_WARPS;  // L2 lookahead in tasks
  auto no_op = [](int) {};
  if constexpr (!EAGER) {
    for (;;) {
      if (tA >= c.T) break;  // tA < tB here
      wt_compute<FMT, KIND, PL, RS, MR>(g, c, sm, tA, bufA, lane, no_op);
      tA = next_task();
      wt_load<KIND, RS>(g, w, c, tA, bufA, pol, lane);
      wt_prefetch<KIND, RS>(g, w, c, tA + AHEAD, lane);
      if (tB >= c.T) break;  // tB < tA here
      wt_compute<FMT, KIND, PL, RS, MR>(g, c, sm, tB, bufB, lane, no_op);
      tB = next_task();
      wt_load<KIND, RS>(g, w, c, tB, bufB, pol, lane);
      wt_prefetch<KIND, RS>(g, w, c, tB + AHEAD, lane);
    }
  } else {
    for (;;) {
      if (tA >= c.T) break;  // tA < tB here
      const int nA = next_task();
      wt_prefetch<KIND, RS>(g, w, c, nA + AHEAD, lane);
      wt_compute<FMT, KIND, PL, RS, MR>(g, c, sm, tA, bufA, lane,
                                    [&](int k) { wt_load_chunk<KIND, RS>(g, w, c, nA, bufA, k, pol, lane); });
      tA = nA;
      if (tB >= c.T) break;  // tB < tA here
      const int nB = next_task();
      wt_prefetch<KIND, RS>(g, w, c, nB + AHEAD, lane);
      wt_compute<FMT, KIND, PL, RS, MR>(g, c, sm, tB, bufB, lane,
                                    [&](int k) { wt_load_chunk<KIND, RS>(g, w, c, nB, bufB, k, pol, lane); });
      tB = nB;
    }
  }
}

// Sum of the pieces of CTA row rl of matrix m (for activation row r of MR),
// in piece order.
template <int NW, int MR = 1>
__device__ __forceinline__ float row_total(const PhaseGeom& g, const float* parts, int rl, int m, int r = 0) {
  float v = 0.f;
  for (int q = 0; q < g.P; ++q) v += parts[(((size_t)rl * g.P + q) * NW + m) * MR + r];
  return v;
}

// ---------------------------------------------------------------- host side

// Plans one phase for a grid of `grid` CTAs: the fewest pieces per row whose
// chunks fit the lanes' register buffer (32 * WT_CL chunks per stream),
// dividing the row's chunks and (affine) its groups, so a piece holds whole
// groups.  The N rows are dealt out to the CTAs in contiguous ranges of whole
// units of row_unit rows (N % row_unit == 0).  Returns false if no such cut
// exists.  *smem_parts receives the bytes of the phase's shared arrays other
// than x (phase_tail_bytes).
template <int FMT, int KIND>
bool plan_phase(int K, int N, int group, int grid, PhaseGeom* out, size_t* smem_parts,
                int row_unit = 1, int max_rs = 2) {
  using T = FmtTraits<FMT>;
  constexpr int EPC = T::EPC;
  constexpr bool AFF = T::AFFINE;
  PhaseGeom g = {};
  g.K = K;
  g.N = N;
  g.group = AFF ? group : 1;
  g.lg_group = AFF ? (group == 32 ? 5 : (group == 64 ? 6 : 7)) : 0;
  g.G = AFF ? K / group : 0;
  g.row_bytes = FMT == FMT_BF16 ? K * 2 : (FMT == FMT_A8 ? K : K / 2);
  g.CPR = K / EPC;
  int P = 0;
  for (int q = 1; q <= g.CPR; ++q) {
    if (g.CPR % q || (AFF && g.G % q)) continue;
    if (g.CPR / q <= 32 * WT_CL) { P = q; break; }
  }
  if (P == 0 || grid < 1 || row_unit < 1 || N % row_unit) return false;
  g.P = P;
  g.RS = (max_rs >= 2 && P == 1 && g.CPR == 16 * WT_CL) ? 2 : 1;
  g.p_mul = ((1ull << 32) + (unsigned long long)P - 1) / (unsigned long long)P;
  g.B = g.row_bytes / P;
  g.CPP = g.CPR / P;
  g.GPP = AFF ? g.G / P : 0;
  g.row_unit = row_unit;
  g.rows_base = N / row_unit / grid;
  g.rows_extra = N / row_unit % grid;
  g.rows_alloc = row_unit * (g.rows_base + (g.rows_extra ? 1 : 0));
  g.sb_stride = AFF ? (g.rows_alloc * g.G + 7) / 8 * 8 : 0;
  g.sb_vec = (AFF && g.G % 8 == 0) ? 1 : 0;
  *out = g;
  *smem_parts = phase_tail_bytes<FMT, KIND>(g);
  return true;
}

}  // namespace mt
