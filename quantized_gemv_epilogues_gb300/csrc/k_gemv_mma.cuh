// k_gemv_mma.cuh - multi-row GEMV (1 <= M <= 8 activation rows) with the
// SwiGLU or residual epilogue, its dot products on the tensor cores.
//
// meTile docs, "Compute-Graph Fusion", Automatic Gated Epilogues (gate and up
// share the activation; silu(gate) * up and the residual add are epilogues
// before the only store); "MLX-LM Backend", Dispatch Policy (affine
// w = scale * q + bias per group of 32/64/128 along K, fp32 accumulation).
//
// GB300 design:
//  * Dot products are mma.sync m16n8k16 with fp32 accumulators: A = 16
//    weight rows x 16 K, B = 16 K x 8 activation rows (B columns >= M repeat
//    row M-1 and their results are dropped).  Each weight is read once for
//    all M rows, and the per-weight work does not grow with M.
//  * Affine codes enter A exactly as fp16 subnormals: the 16-bit pattern
//    0x00qq is the fp16 value q * 2^-24 (exponent field zero, spacing
//    2^-24), so one mask or byte permute per two codes places them, with no
//    arithmetic.  A high INT4 nibble stays in place as 16 q * 2^-24, and the
//    x it meets is staged divided by 16.  Products with x (fp16 up to 2^15)
//    are exact in the fp32 accumulator; the 2^24 goes into the staged group
//    scale.  Each group's fp32 accumulator is then scaled by the row's group
//    scale and the bias enters as b * X_g, both in
//    fp32; X_g, the group sum of x, comes from one more mma per k step with
//    an all-ones A (the tensor pipe is otherwise idle most of the time).
//    Dense bf16 weights are A as stored.
//  * x enters B as fp16 scaled per quantisation group by a power of two 2^e
//    (max|x| 2^e in [2^14, 2^15) over the group): a bf16 value is exact in
//    fp16 unless it lies below 2^-28 of its group's maximum (those are
//    flushed); the scale is divided out at each group's fp32 flush.  Every
//    CTA stages and converts all of x: asynchronous 16-byte copies, then one
//    pass of packed bf16 maxima and an integer re-biasing of the
//    bf16 exponent (bf16x2_to_f16x2).  Dense bf16 weights take x as stored
//    (bf16 mma).
//  * K order: a dot product does not depend on which physical K index meets
//    which mma k slot, as long as A and B agree.  A lane takes WPL
//    consecutive 4-byte words of its row with one 16-, 8- or 4-byte load and
//    uses them in register order; x is staged in shared memory in the same
//    order, so a lane reads its B fragments with 16-byte loads and no
//    shuffles.  The 16 K indices of one k step lie in one quantisation group
//    (the load width is chosen from the group size).
//  * Work split: one CTA of 16 warps per SM.  A contiguous range of output
//    rows (within one row of every other range) belongs to a cluster of two
//    CTAs that take one half of K each (each stages and converts half of x;
//    their totals meet through distributed shared memory), or to one CTA
//    when K does not halve into whole groups; a range is cut into tiles of
//    at most 16 rows.  A unit is one tile x UK of K: 32 words (128 bytes) per lane.  The
//    CTA's units are dealt to its warps in contiguous ranges; a warp
//    accumulates along K in registers and writes one partial per tile it
//    touched, and the epilogue adds a row's partials in warp order
//    (deterministic).  Two units are in flight per warp (register double
//    buffer) and the unit after them is asked of L2.
#pragma once
#include <algorithm>

#include "k_gemv_run.cuh"

namespace mt {

constexpr int MMA_WARPS = 16;
constexpr int MMA_THREADS = 32 * MMA_WARPS;
constexpr int MMA_WORDS = 32;  // 4-byte weight words per lane per unit

struct MmaArgs {
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
  int out_f32;
  int M, K, N;
  int group, lg_group, G;
  int ck;      // CTAs per cluster sharing a row range: 1, or 2 (each takes half of K)
  int Kc, Gc;  // K and groups per CTA (K / ck, G / ck)
  int row_bytes;
  int rows_base, rows_extra;  // row range r owns rows_base + (r < rows_extra) rows
  int KB;                     // units per tile along K: ceil(K / UK)
  int NS;                     // partial slots per warp
  int xstride;                // bytes per staged x row
  int raw_vec;                // 1: raw scales/biases are copied in 16-byte pieces
  // shared-memory byte offsets
  int off_sbf, off_ginv, off_raw, off_parts, off_tstart, off_tot;
};

// Compile-time shape of one (format, kind, load width) instantiation.
template <int FMT, int KIND, int WPL>
struct MmaCfg {
  static constexpr int NW = KIND == 0 ? 2 : 1;                               // weight matrices
  static constexpr int EPW = FmtTraits<FMT>::EPW;                           // codes per word
  static constexpr int CPL = WPL * EPW;  // codes per lane per chunk
  static constexpr int CW = 4 * CPL;     // codes of a row per chunk (4 lanes)
  static constexpr int LB = 2 * CPL;     // bytes of staged x per lane per chunk
  static constexpr int CPU = MMA_WORDS / (NW * 2 * WPL);  // chunks per unit
  static constexpr int UK = CPU * CW;                       // K per unit
  static constexpr int KSC = EPW * WPL / 4;  // k steps per chunk (16 K indices = 4 per lane each)
  static_assert(CPU >= 1 && KSC >= 1, "load width");
};

// Byte offset of code k within a weight row.
template <int FMT>
__host__ __device__ constexpr size_t code_bytes(int k) {
  return FmtTraits<FMT>::EPW == 4 ? (size_t)k : (FmtTraits<FMT>::EPW == 8 ? (size_t)k / 2 : (size_t)k * 2);
}

// Streaming loads of WPL words (no L1 allocation, L2 policy).
template <int WPL>
__device__ __forceinline__ void ldw(uint32_t (&d)[WPL], const uint8_t* p, uint64_t pol) {
  if constexpr (WPL == 4) {
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "l"(p), "l"(pol));
  } else if constexpr (WPL == 2) {
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
                 : "=r"(d[0]), "=r"(d[1])
                 : "l"(p), "l"(pol));
  } else {
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;"
                 : "=r"(d[0])
                 : "l"(p), "l"(pol));
  }
}

// Thread-block cluster helpers (distributed shared memory).
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster: the shared-memory writes before
// it are visible to every CTA after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The float at this CTA's shared address p, read from the same address in
// the shared memory of cluster CTA `rank`.
__device__ __forceinline__ float ld_cluster_f32(const float* p, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// Packed bf16 maxima.  On non-negative finite values the bf16 order is the
// order of the 16-bit patterns, so this is also a packed unsigned 16-bit
// maximum of such patterns.
__device__ __forceinline__ uint32_t hmax2_bf16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// fp16 bit patterns of x * 2^e for the two bf16 values of w, by integer
// arithmetic on the bit fields: an fp16 exponent field is the bf16 one minus
// 112 plus e, and the 7 bf16 fraction bits become the top 7 of the 10.  thr2
// holds (112 - e) << 7 in both halves (0 <= 112 - e < 256): a packed
// maximum clamps magnitudes below 2^-15 after scaling to that threshold, so
// the subtraction never borrows across halves and they come out as zero (or,
// in [2^-15, 2^-14), as some value below 2^-14).  Exact for every |x 2^e| in
// [2^-14, 2^15); the caller's e keeps the group's maximum below 2^15.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, uint32_t thr2) {
  const uint32_t t = hmax2_bf16(w & 0x7FFF7FFFu, thr2) - thr2;
  return (t << 3) | (w & 0x80008000u);
}

// d += A * B for one m16n8k16 tile, fp32 accumulation; A/B fp16 or bf16.
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Exact fp16 values of block-scaled elements (the E8M0 block scale is applied
// at the group flush): lo = codes (c0, c1), hi = (c2, c3) of the word's four
// E4M3 bytes, or of the two E2M1 bytes in its low 16 bits (byte b holds
// c_2b in bits 0..3 and c_2b+1 in bits 4..7).  Every E4M3 and E2M1 value is
// an fp16 value.
__device__ __forceinline__ void e4m3x2_to_f16x2(uint32_t v, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(v));
}
__device__ __forceinline__ void e2m1x2_to_f16x2(uint32_t v, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(v));
}

// The two A registers of k step ks (within its chunk) from one row's words:
// lo holds the codes of mma k slots (2t, 2t+1), hi those of (2t+8, 2t+9).
//   A8:   word ks = codes c0..c3;   lo = (c0, c1), hi = (c2, c3)
//   A4:   word ks/2 = codes c0..c7 (byte b: c_2b low nibble, c_2b+1 high);
//         even ks: lo = (c0, c4), hi = (c1, c5); odd ks: lo = (c2, c6), hi = (c3, c7)
//   BF16: words 2ks, 2ks+1 as stored (elements in order)
//   MX8:  as A8, the E4M3 codes converted to fp16 values
//   MX4:  word ks/2, its low (even ks) or high (odd ks) 16 bits = codes
//         c0..c3 of the step in order: lo = (c0, c1), hi = (c2, c3)
// The staged x of a lane's chunk follows the same order (A8, MX8, MX4 and
// bf16: the elements in order; A4: permuted within each 8), and when a lane's
// block is 64 bytes (A4 or MX4 with 16-byte loads) lanes t = 2, 3 keep its 16-byte
// pieces swapped in pairs (piece q at q ^ 1), so the quarter-warps of a
// 16-byte shared load hit distinct banks.
template <int FMT, int WPL>
__device__ __forceinline__ void a_regs(const uint32_t (&w)[WPL], int ks, uint32_t& lo, uint32_t& hi) {
  if constexpr (FMT == FMT_MX8) {
    e4m3x2_to_f16x2(w[ks], lo, hi);
  } else if constexpr (FMT == FMT_MX4) {
    e2m1x2_to_f16x2((ks & 1) ? (w[ks >> 1] >> 16) : w[ks >> 1], lo, hi);
  } else if constexpr (FMT == FMT_A8) {
    const uint32_t v = w[ks];
    lo = __byte_perm(v, 0u, 0x4140);  // (c0, c1) * 2^-24
    hi = __byte_perm(v, 0u, 0x4342);  // (c2, c3) * 2^-24
  } else if constexpr (FMT == FMT_A4) {
    const uint32_t v = (ks & 1) ? (w[ks >> 1] >> 8) : w[ks >> 1];
    lo = v & 0x000F000Fu;  // (c0, c4) * 2^-24
    hi = v & 0x00F000F0u;  // (c1, c5) * 2^-20: B holds x / 16 in these slots
  } else {
    lo = w[2 * ks];
    hi = w[2 * ks + 1];
  }
}

// Bytes added to a staged x row so that rows gid and gid + 1 start 16, 32 or
// 64 bytes apart modulo 128 (conflict-free 16-byte B-fragment loads).
template <int LB>
__host__ __device__ constexpr int mma_row_pad() {
  return LB == 16 ? 64 : (LB == 32 ? 16 : 32);
}

template <int FMT, int KIND, int WPL>
__global__ void __launch_bounds__(MMA_THREADS, 1) gemv_mma_kernel(const MmaArgs a) {
  using C = MmaCfg<FMT, KIND, WPL>;
  constexpr int NW = C::NW, CPU = C::CPU, UK = C::UK, CW = C::CW, LB = C::LB, KSC = C::KSC;
  constexpr bool AFF = FmtTraits<FMT>::AFFINE;
  constexpr bool MX = FmtTraits<FMT>::MX;
  constexpr bool GRP = AFF || MX;  // per-group flush (x scaled per group)
  constexpr bool BF = FMT == FMT_BF16;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* xs = smem;                                                   // [M][xstride]
  float4* sbf = reinterpret_cast<float4*>(smem + a.off_sbf);                  // [NW][RT][G][8] (affine)
  float2* sbf2 = reinterpret_cast<float2*>(smem + a.off_sbf);                 // [NW][RT][G][8] (MX)
  uint16_t* raw = reinterpret_cast<uint16_t*>(smem + a.off_raw);              // [NW][2][rows*G] (affine)
  uint8_t* raw8 = reinterpret_cast<uint8_t*>(smem + a.off_raw);               // [NW][rows*G] (MX)
  float* parts = reinterpret_cast<float*>(smem + a.off_parts);                // [W][NS][16][M][NW]
  float* ginv = reinterpret_cast<float*>(smem + a.off_ginv);                  // [Gc][8] 2^-e_g
  int* tstart = reinterpret_cast<int*>(smem + a.off_tstart);                  // [RT + 1]
  float* tot = reinterpret_cast<float*>(smem + a.off_tot);                    // [rows][M][NW] (ck 2)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, t = lane & 3;
  // a cluster of ck CTAs owns a row range; CTA `rank` of it takes the K
  // range [rank Kc, (rank + 1) Kc) of every row
  const int rr = blockIdx.x / a.ck;
  const int rank = a.ck == 2 ? (int)cluster_ctarank() : 0;
  const int r_begin = rr * a.rows_base + min(rr, a.rows_extra);
  const int rows = a.rows_base + (rr < a.rows_extra ? 1 : 0);
  const int RT = (rows + 15) >> 4;
  const int KB = a.KB, M = a.M, K = a.K, G = a.G;
  const int Kc = a.Kc, Gc = a.Gc, K_lo = rank * Kc, g_lo = rank * Gc;
  const int U = RT * KB;
  const int u0 = (int)((long)warp * U / MMA_WARPS), u1 = (int)((long)(warp + 1) * U / MMA_WARPS);

  if (tid <= RT) tstart[tid] = tid * rows / RT;
  __syncthreads();
  pdl_trigger();

  const uint64_t pol = l2_evict_first_policy();

  // Unit cursors: tile j, K block kb, units left in the warp's range.
  struct Cur {
    int j, kb, left;
  };
  auto advance = [&](Cur& c) {
    if (++c.kb == KB) { c.kb = 0; ++c.j; }
    --c.left;
  };

  auto load_unit = [&](const Cur& c, uint32_t (&buf)[NW][2][CPU][WPL]) {
    if (c.left <= 0) return;
    const int j = c.j, k0 = c.kb * UK;
    const int tr0 = tstart[j], tr1 = tstart[j + 1];
#pragma unroll
    for (int mat = 0; mat < NW; ++mat)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rl = tr0 + gid + 8 * h;
        const bool okr = rl < tr1;
        const uint8_t* src = (mat ? a.W1 : a.W0) + (size_t)(r_begin + (okr ? rl : tr0)) * a.row_bytes +
                             code_bytes<FMT>(K_lo + k0) + t * WPL * 4;
#pragma unroll
        for (int ch = 0; ch < CPU; ++ch) {
          if (okr && k0 + ch * CW < Kc) {
            ldw<WPL>(buf[mat][h][ch], src + code_bytes<FMT>(ch * CW), pol);
          } else {
#pragma unroll
            for (int i = 0; i < WPL; ++i) buf[mat][h][ch][i] = 0u;
          }
        }
      }
  };
  // one 128-byte line per lane: the unit's 16 rows x UK codes of each matrix
  auto prefetch_unit = [&](const Cur& c) {
    if (c.left <= 0) return;
    const int j = c.j, k0 = c.kb * UK;
    const int tr0 = tstart[j], tr1 = tstart[j + 1];
    constexpr int LPR = (int)(code_bytes<FMT>(UK) / 128);  // lines per row and matrix
    const int mat = NW == 2 ? (lane >> 4) : 0;
    const int idx = NW == 2 ? (lane & 15) : lane;
    const int rl = tr0 + idx / LPR, line = idx % LPR;
    if (rl < tr1 && (size_t)line * 128 < code_bytes<FMT>(Kc) - code_bytes<FMT>(k0))
      prefetch_l2_normal((mat ? a.W1 : a.W0) + (size_t)(r_begin + rl) * a.row_bytes +
                         code_bytes<FMT>(K_lo + k0) + line * 128);
  };

  // cc: the unit computed next; cl: the next unit to load; cp: the next unit
  // asked of L2 (two ahead of cl)
  Cur cc = {u0 / KB, u0 % KB, u1 - u0};
  Cur cl = cc, cp;
  uint32_t bufA[NW][2][CPU][WPL], bufB[NW][2][CPU][WPL];
  load_unit(cl, bufA);
  advance(cl);
  load_unit(cl, bufB);
  advance(cl);
  cp = cl;
  prefetch_unit(cp);
  advance(cp);
  prefetch_unit(cp);
  advance(cp);

  // raw scales and biases of the CTA's rows (static data: before the wait)
  if constexpr (AFF) {
    // [rows][Gc] per array: this CTA's groups of each of its rows
    const int n = rows * Gc;
#pragma unroll
    for (int mat = 0; mat < NW; ++mat) {
      const uint16_t* s = mat ? a.s1 : a.s0;
      const uint16_t* b = mat ? a.b1 : a.b0;
      uint16_t* rs = raw + (size_t)(2 * mat) * n;
      uint16_t* rb = rs + n;
      if (a.raw_vec) {  // Gc % 8 == 0: 16-byte pieces
        const int upr = Gc >> 3;
        for (int i = tid; i < n / 8; i += MMA_THREADS) {
          const int rl = i / upr, c = i - rl * upr;
          const size_t src = (size_t)(r_begin + rl) * G + g_lo + c * 8;
          cp_async16(rs + i * 8, s + src);
          cp_async16(rb + i * 8, b + src);
        }
      } else {
        for (int i = tid; i < n; i += MMA_THREADS) {
          const int rl = i / Gc, c = i - rl * Gc;
          const size_t src = (size_t)(r_begin + rl) * G + g_lo + c;
          rs[i] = ldg_u16(s + src);
          rb[i] = ldg_u16(b + src);
        }
      }
    }
    cp_async_commit();
  }
  if constexpr (MX) {
    // [rows][Gc] E8M0 bytes per matrix
    const int n = rows * Gc;
#pragma unroll
    for (int mat = 0; mat < NW; ++mat) {
      const uint8_t* s = reinterpret_cast<const uint8_t*>(mat ? a.s1 : a.s0);
      uint8_t* rs = raw8 + (size_t)mat * n;
      if (a.raw_vec) {  // Gc % 16 == 0: 16-byte pieces
        const int upr = Gc >> 4;
        for (int i = tid; i < n / 16; i += MMA_THREADS) {
          const int rl = i / upr, c = i - rl * upr;
          cp_async16(rs + i * 16, s + (size_t)(r_begin + rl) * G + g_lo + c * 16);
        }
      } else {
        for (int i = tid; i < n; i += MMA_THREADS) {
          const int rl = i / Gc, c = i - rl * Gc;
          rs[i] = s[(size_t)(r_begin + rl) * G + g_lo + c];
        }
      }
    }
    cp_async_commit();
  }

  pdl_wait();  // x, the residual and the output follow the preceding kernel

  // ---- x: raw bf16 rows into shared memory (16-byte asynchronous copies,
  // all in flight together)
  const int U8 = Kc / 8;  // 8-element units of this CTA's K range
  {
    int m = 0, u = tid;
    while (m < M && u >= U8) { u -= U8; ++m; }
    while (m < M) {
      cp_async16(xs + (size_t)m * a.xstride + (size_t)u * 16, a.x + (size_t)m * K + K_lo + (size_t)u * 8);
      u += MMA_THREADS;
      while (m < M && u >= U8) { u -= U8; ++m; }
    }
    cp_async_commit();
  }
  cp_async_wait_all();  // x (and the raw scales/biases)
  __syncthreads();

  if constexpr (GRP) {
    // ---- x as fp16 in place, scaled per quantisation group by 2^e_g with
    // max|x| 2^e_g in [2^14, 2^15) (a zero or tiny maximum gives 2^112);
    // ginv[g][m] = 2^-e_g.  One 16-byte unit (8 elements) per lane and step,
    // consecutive lanes on consecutive units (conflict-free shared accesses):
    // a group's upg = group / 8 units sit in consecutive lanes and its
    // maximum (packed bf16 maxima of the magnitudes) is combined by shuffles.
    // Element order within a unit as a_regs reads it: in order (A8); (c0, c4),
    // (c1, c5), (c2, c6), (c3, c7) (A4), and with 64-byte lane blocks (A4,
    // 16-byte loads) the units of lanes t = 2, 3 of each chunk swapped in
    // pairs; the swap partner is the neighbouring lane, whose load precedes
    // both stores.
    const int upg = a.group >> 3, lg_upg = a.lg_group - 3;
    // units per lane and task: the most (up to 4) that still give every warp
    // a task
    constexpr int PU = 4;
    int pu = PU;
    while (pu > 1 && M * ((U8 + 32 * pu - 1) / (32 * pu)) < MMA_WARPS) pu >>= 1;
    const int usegs = (U8 + 32 * pu - 1) / (32 * pu);
    for (int task = warp; task < M * usegs; task += MMA_WARPS) {  // warp-uniform
      const int m = task / usegs, sg = task - m * usegs;
      unsigned char* row = xs + (size_t)m * a.xstride;
      uint4 v[PU];
#pragma unroll
      for (int j = 0; j < PU; ++j) {
        const int u = (sg * pu + j) * 32 + lane;
        v[j] = (j < pu && u < U8) ? *reinterpret_cast<const uint4*>(row + (size_t)u * 16)
                                  : make_uint4(0, 0, 0, 0);
      }
      // the PU units' maxima advance in lockstep (independent shuffle chains)
      uint32_t mx[PU];
#pragma unroll
      for (int j = 0; j < PU; ++j) {
        mx[j] = hmax2_bf16(hmax2_bf16(v[j].x & 0x7FFF7FFFu, v[j].y & 0x7FFF7FFFu),
                           hmax2_bf16(v[j].z & 0x7FFF7FFFu, v[j].w & 0x7FFF7FFFu));
        mx[j] = max(mx[j] & 0xFFFFu, mx[j] >> 16);
      }
      for (int off = 1; off < upg; off <<= 1) {
#pragma unroll
        for (int j = 0; j < PU; ++j) mx[j] = max(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], off));
      }
#pragma unroll
      for (int j = 0; j < PU; ++j) {
        const int u = (sg * pu + j) * 32 + lane;
        // mx: bf16 bits of the group's max|x|; e <= 112 keeps the threshold
        // of bf16x2_to_f16x2 non-negative (groups below 2^-98 lose precision)
        const int e = max(-126, min(112, 14 - ((int)(mx[j] >> 7) - 127)));
        const uint32_t thr = (uint32_t)(112 - e) << 7, t2 = thr | (thr << 16);
        uint4 o;
        if constexpr (FMT != FMT_A4) {
          o = make_uint4(bf16x2_to_f16x2(v[j].x, t2), bf16x2_to_f16x2(v[j].y, t2),
                         bf16x2_to_f16x2(v[j].z, t2), bf16x2_to_f16x2(v[j].w, t2));
        } else {
          // (x0,x1) (x2,x3) (x4,x5) (x6,x7) -> (x0,x4) (x1,x5) (x2,x6) (x3,x7);
          // the odd codes of each byte pair sit 16x high in A (see a_regs), so
          // their x is scaled by 2^(e-4)
          const uint32_t to = (uint32_t)(116 - e) << 7, t2o = to | (to << 16);
          o = make_uint4(bf16x2_to_f16x2(__byte_perm(v[j].x, v[j].z, 0x5410), t2),
                         bf16x2_to_f16x2(__byte_perm(v[j].x, v[j].z, 0x7632), t2o),
                         bf16x2_to_f16x2(__byte_perm(v[j].y, v[j].w, 0x5410), t2),
                         bf16x2_to_f16x2(__byte_perm(v[j].y, v[j].w, 0x7632), t2o));
        }
        if (j < pu && u < U8) {
          const int ud = (LB == 64) ? (u ^ ((u >> 3) & 1)) : u;
          *reinterpret_cast<uint4*>(row + (size_t)ud * 16) = o;
          if ((u & (upg - 1)) == 0) ginv[(u >> lg_upg) * 8 + m] = exp2i(-e);
        }
      }
    }
    // scales and biases: entry (mat, tile j, group g, gid) at thread i; the
    // thread's next entry is MMA_THREADS further (gid stays: 8 | MMA_THREADS)
    const int n = rows * Gc, ne = RT * Gc * 8;
    {
      const int gi = tid & 7;
      int g = tid >> 3, j = 0, mat = 0;
      while (g >= Gc) { g -= Gc; ++j; }
      while (j >= RT) { j -= RT; ++mat; }
      for (int i = tid; i < NW * ne; i += MMA_THREADS) {
        const int tr0 = tstart[j], tr1 = tstart[j + 1];
        const int ra = tr0 + gi, rbw = tr0 + gi + 8;
        if constexpr (MX) {
          // E8M0 field E: 2^(E - 127) (E = 0: 2^-127, an fp32 subnormal)
          const uint8_t* rs = raw8 + (size_t)mat * n;
          auto e8m0 = [](uint32_t E) { return E ? __int_as_float((int)(E << 23)) : __int_as_float(0x00400000); };
          float2 e = make_float2(0.f, 0.f);
          if (ra < tr1) e.x = e8m0(rs[ra * Gc + g]);
          if (rbw < tr1) e.y = e8m0(rs[rbw * Gc + g]);
          sbf2[i] = e;
        } else {
          const uint16_t* rs = raw + (size_t)(2 * mat) * n;
          const uint16_t* rb = rs + n;
          float4 e = make_float4(0.f, 0.f, 0.f, 0.f);
          constexpr float TWO24 = 16777216.f;  // the codes enter the mma as q * 2^-24
          if (ra < tr1) { e.x = bf16f(rs[ra * Gc + g]) * TWO24; e.z = bf16f(rb[ra * Gc + g]); }
          if (rbw < tr1) { e.y = bf16f(rs[rbw * Gc + g]) * TWO24; e.w = bf16f(rb[rbw * Gc + g]); }
          sbf[i] = e;
        }
        g += MMA_THREADS / 8;
        while (g >= Gc) { g -= Gc; ++j; }
        while (j >= RT) { j -= RT; ++mat; }
      }
    }
    __syncthreads();
  }

  // ---- mainloop
  float acc[NW][4];
#pragma unroll
  for (int mat = 0; mat < NW; ++mat)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[mat][i] = 0.f;
  const unsigned char* xrow = xs + (size_t)min(gid, M - 1) * a.xstride + t * LB;
  const int ne = RT * Gc * 8;

  const int jfirst = u0 / KB;
  auto compute_unit = [&](const Cur& c, const uint32_t (&buf)[NW][2][CPU][WPL]) {
    const int j = c.j, kb = c.kb, k0 = kb * UK;
    float d[NW][4] = {}, d1[4] = {};  // d1: group sums of B (A = ones)
#pragma unroll
    for (int ch = 0; ch < CPU; ++ch) {
      const int kc = k0 + ch * CW;
      if (kc >= Kc) break;
      if constexpr (GRP) {
        if ((kc & (a.group - 1)) == 0) {
#pragma unroll
          for (int mat = 0; mat < NW; ++mat)
#pragma unroll
            for (int i = 0; i < 4; ++i) d[mat][i] = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) d1[i] = 0.f;
        }
      }
      // 64-byte lane blocks (A4, MX4 with 16-byte loads): lanes t = 2, 3 hold
      // their pieces swapped
      constexpr bool SWP = LB == 64;
      uint32_t xr[LB / 4];
#pragma unroll
      for (int q = 0; q < LB / 16; ++q) {
        const int pos = SWP ? (q ^ ((t >> 1) & 1)) : q;
        const uint4 v = *reinterpret_cast<const uint4*>(xrow + (size_t)kc * 2 + pos * 16);
        xr[4 * q] = v.x; xr[4 * q + 1] = v.y; xr[4 * q + 2] = v.z; xr[4 * q + 3] = v.w;
      }
#pragma unroll
      for (int ks = 0; ks < KSC; ++ks) {
        const uint32_t b0 = xr[2 * ks], b1 = xr[2 * ks + 1];
        if constexpr (AFF) {  // sum of x over the group: A = 1 (16 where B holds x / 16)
          constexpr uint32_t ONE = 0x3C003C00u, HI = FMT == FMT_A4 ? 0x4C004C00u : ONE;
          mma16816<false>(d1, ONE, ONE, HI, HI, b0, b1);
        }
#pragma unroll
        for (int mat = 0; mat < NW; ++mat) {
          uint32_t lo0, hi0, lo1, hi1;
          a_regs<FMT, WPL>(buf[mat][0][ch], ks, lo0, hi0);
          a_regs<FMT, WPL>(buf[mat][1][ch], ks, lo1, hi1);
          if constexpr (GRP)
            mma16816<false>(d[mat], lo0, lo1, hi0, hi1, b0, b1);
          else
            mma16816<BF>(acc[mat], lo0, lo1, hi0, hi1, b0, b1);
        }
      }
      if constexpr (MX) {
        if (((kc + CW) & (a.group - 1)) == 0) {  // the block ends with this chunk
          const int g = kc >> a.lg_group;
          // block scale * sum(w x) in the group's x scale, then undone
          const float2 gi = *reinterpret_cast<const float2*>(ginv + g * 8 + 2 * t);
#pragma unroll
          for (int mat = 0; mat < NW; ++mat) {
            const float2 sb = sbf2[(size_t)mat * ne + (j * Gc + g) * 8 + gid];
            acc[mat][0] = fmaf(sb.x * d[mat][0], gi.x, acc[mat][0]);
            acc[mat][1] = fmaf(sb.x * d[mat][1], gi.y, acc[mat][1]);
            acc[mat][2] = fmaf(sb.y * d[mat][2], gi.x, acc[mat][2]);
            acc[mat][3] = fmaf(sb.y * d[mat][3], gi.y, acc[mat][3]);
          }
        }
      }
      if constexpr (AFF) {
        if (((kc + CW) & (a.group - 1)) == 0) {  // the group ends with this chunk
          const int g = kc >> a.lg_group;
          // s * sum(q x) + b * X_g in the group's x scale, then undone
          const float2 gi = *reinterpret_cast<const float2*>(ginv + g * 8 + 2 * t);
#pragma unroll
          for (int mat = 0; mat < NW; ++mat) {
            const float4 sb = sbf[(size_t)mat * ne + (j * Gc + g) * 8 + gid];
            acc[mat][0] = fmaf(fmaf(sb.x, d[mat][0], sb.z * d1[0]), gi.x, acc[mat][0]);
            acc[mat][1] = fmaf(fmaf(sb.x, d[mat][1], sb.z * d1[1]), gi.y, acc[mat][1]);
            acc[mat][2] = fmaf(fmaf(sb.y, d[mat][2], sb.w * d1[0]), gi.x, acc[mat][2]);
            acc[mat][3] = fmaf(fmaf(sb.y, d[mat][3], sb.w * d1[1]), gi.y, acc[mat][3]);
          }
        }
      }
    }
    if (c.left == 1 || kb + 1 == KB) {  // last unit of this warp in tile j
      const int slot = j - jfirst;
      float* pp = parts + (size_t)(warp * a.NS + slot) * 16 * M * NW;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int m = 2 * t + c;
        if (m < M) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int mat = 0; mat < NW; ++mat)
              pp[((gid + 8 * h) * M + m) * NW + mat] = acc[mat][2 * h + c];
        }
      }
#pragma unroll
      for (int mat = 0; mat < NW; ++mat)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mat][i] = 0.f;
    }
  };

  // register ping-pong: two units per iteration keep the buffer indices static
  while (cc.left > 0) {
    compute_unit(cc, bufA);
    advance(cc);
    load_unit(cl, bufA);
    advance(cl);
    prefetch_unit(cp);
    advance(cp);
    if (cc.left <= 0) break;
    compute_unit(cc, bufB);
    advance(cc);
    load_unit(cl, bufB);
    advance(cl);
    prefetch_unit(cp);
    advance(cp);
  }
  __syncthreads();

  // ---- epilogue: per (activation row, output row), this CTA's partials of
  // the row added in warp order; with a cluster of two, each CTA keeps its
  // K-half totals, and after a cluster barrier the two CTAs finish one half
  // of the rows each, adding rank 0's total then rank 1's (deterministic)
  auto cta_total = [&](int rl, int m, float (&v)[NW]) {
    int j = min(RT - 1, rl * RT / rows);
    while (j > 0 && tstart[j] > rl) --j;
    while (j + 1 < RT && tstart[j + 1] <= rl) ++j;
    const int i = rl - tstart[j];
#pragma unroll
    for (int mat = 0; mat < NW; ++mat) v[mat] = 0.f;
    for (int w = 0; w < MMA_WARPS; ++w) {
      const int w0 = (int)((long)w * U / MMA_WARPS), w1 = (int)((long)(w + 1) * U / MMA_WARPS);
      if (w1 > w0 && w0 < (j + 1) * KB && w1 > j * KB) {
        const float* pp = parts + ((size_t)(w * a.NS + (j - w0 / KB)) * 16 + i) * M * NW + m * NW;
#pragma unroll
        for (int mat = 0; mat < NW; ++mat) v[mat] += pp[mat];
      }
    }
  };
  auto finish = [&](int rl, int m, const float (&v)[NW]) {
    const int n = r_begin + rl;
    float outv;
    if constexpr (KIND == 0) {
      outv = v[0] / (1.0f + expf(-v[0])) * v[NW - 1];  // silu(gate) * up
    } else {
      outv = a.res ? v[0] + bf16f(a.res[(size_t)m * a.res_ld + n]) : v[0];  // + residual or bias
    }
    if (a.out_f32)
      static_cast<float*>(a.out)[(size_t)m * a.N + n] = outv;
    else
      static_cast<uint16_t*>(a.out)[(size_t)m * a.N + n] = f2bf(outv);
  };
  if (a.ck == 1) {
    for (int o = tid; o < rows * M; o += MMA_THREADS) {
      const int m = o / rows, rl = o - m * rows;
      float v[NW];
      cta_total(rl, m, v);
      finish(rl, m, v);
    }
  } else {
    for (int o = tid; o < rows * M; o += MMA_THREADS) {
      const int m = o / rows, rl = o - m * rows;
      float v[NW];
      cta_total(rl, m, v);
#pragma unroll
      for (int mat = 0; mat < NW; ++mat) tot[((size_t)rl * M + m) * NW + mat] = v[mat];
    }
    cluster_sync_all();
    const int half = (rows + 1) >> 1;
    const int rl0 = rank ? half : 0, nr = rank ? rows - half : half;
    for (int o = tid; o < nr * M; o += MMA_THREADS) {
      const int m = o / nr, rl = rl0 + (o - m * nr);
      float v[NW];
#pragma unroll
      for (int mat = 0; mat < NW; ++mat) {
        const float* q = tot + ((size_t)rl * M + m) * NW + mat;
        v[mat] = ld_cluster_f32(q, 0) + ld_cluster_f32(q, 1);
      }
      finish(rl, m, v);
    }
    cluster_sync_all();  // the peer may still read this CTA's totals
  }
}

// Launches a gemv_mma_kernel instantiation: programmatic stream
// serialization when l.pdl is set, clusters of ck CTAs when ck == 2.
template <typename KernelT>
mt_status launch_mma(KernelT kern, int grid, size_t smem, const Launch& l, const MmaArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MMA_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (l.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (a.ck == 2) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return cuda_fail(e);
  return MT_OK;
}

// Host plan and launch of the tensor-core kernel for one (format, kind, load
// width).  Returns MT_ERR_SHAPE when the problem does not fit its layout
// (K not a multiple of a chunk, or the shared arrays over the budget); the
// caller then uses the team kernel.
template <int FMT, int KIND, int WPL>
mt_status run_gemv_mma(const GemvProblem& p, const Launch& l) {
  using C = MmaCfg<FMT, KIND, WPL>;
  constexpr bool AFF = FmtTraits<FMT>::AFFINE;
  constexpr bool MX = FmtTraits<FMT>::MX;
  constexpr bool GRP = AFF || MX;
  constexpr int NW = C::NW;
  static OccCache cache;  // only the attribute flags are used
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  if (!di) return cuda_fail((cudaError_t)derr);
  if (p.M < 1 || p.M > 8 || p.K % C::CW) return MT_ERR_SHAPE;
  if (GRP && (p.group % C::CW || p.K % p.group)) return MT_ERR_SHAPE;

  MmaArgs a = {};
  a.x = p.x;
  a.W0 = static_cast<const uint8_t*>(p.W0);
  a.W1 = static_cast<const uint8_t*>(p.W1);
  a.s0 = p.s0; a.b0 = p.b0; a.s1 = p.s1; a.b1 = p.b1;
  a.res = p.res;
  a.res_ld = p.res_ld;
  a.out = p.out;
  a.out_f32 = p.out_f32 ? 1 : 0;
  a.M = p.M; a.K = p.K; a.N = p.N;
  a.group = GRP ? p.group : 1;
  a.lg_group = GRP ? (p.group == 32 ? 5 : (p.group == 64 ? 6 : 7)) : 0;
  a.G = GRP ? p.K / p.group : 0;
  a.row_bytes = (int)code_bytes<FMT>(p.K);

  // The geometry for ck CTAs per row range (1, or a cluster of 2 that
  // splits K) and `waves` times as many row ranges as fit the SMs at once;
  // returns the dynamic shared memory it needs (0: no tile table).
  const int sms = di->sm_count;
  int grid = 0;
  auto plan = [&](int ck, int waves) -> size_t {
    a.ck = ck;
    a.Kc = p.K / ck;
    a.Gc = a.G / ck;
    const int nrange = std::min(sms / ck * waves, p.N);  // row ranges (clusters)
    grid = nrange * ck;
    a.rows_base = p.N / nrange;
    a.rows_extra = p.N % nrange;
    const int rows_max = a.rows_base + (a.rows_extra ? 1 : 0);
    const int RT = (rows_max + 15) / 16;
    if (RT > 64) return 0;  // the tile-start table holds 65 entries
    a.KB = (a.Kc + C::UK - 1) / C::UK;
    const long U = (long)RT * a.KB;
    const long len = (U + MMA_WARPS - 1) / MMA_WARPS;  // longest warp range
    a.NS = (int)std::min<long>(RT, (len - 1 + a.KB - 1) / a.KB + 1);
    a.xstride = (a.Kc * 2 + 127) / 128 * 128 + mma_row_pad<C::LB>();
    a.raw_vec = (AFF && a.Gc % 8 == 0) || (MX && a.Gc % 16 == 0) ? 1 : 0;
    auto al16 = [](size_t v) { return (v + 15) / 16 * 16; };
    size_t off = al16((size_t)p.M * a.xstride);
    a.off_sbf = (int)off;
    if (GRP) off += (size_t)NW * RT * a.Gc * 8 * (AFF ? 16 : 8);
    a.off_ginv = (int)off;
    if (GRP) off += (size_t)a.Gc * 8 * 4;
    const size_t raw_bytes = AFF ? al16((size_t)NW * 2 * rows_max * a.Gc * 2)
                                 : (MX ? al16((size_t)NW * rows_max * a.Gc) : 0);
    const size_t parts_bytes = (size_t)MMA_WARPS * a.NS * 16 * p.M * NW * 4;
    a.off_raw = (int)off;    // the raw scales/biases are dead once the
    a.off_parts = (int)off;  // mainloop writes its first partial
    off += std::max(raw_bytes, parts_bytes);
    a.off_tstart = (int)al16(off);
    off = a.off_tstart + 80 * 4;  // tile starts
    a.off_tot = (int)al16(off);
    if (ck == 2) off = a.off_tot + (size_t)rows_max * p.M * NW * 4;
    return off;
  };
  // Clusters of two take half of K each when K halves into whole groups and
  // chunks and a row range stays at least a tile high, and either x would
  // not fit one CTA's shared memory or it is large next to the CTA's
  // weights (staging and converting x costs every CTA; measured: a win for
  // the down projection at M = 8, a loss when x is under ~2/3 of the bytes of
  // the CTA's weight rows).
  // A row range too long for the tile table or the shared arrays is cut into
  // more ranges than SMs (CTAs run in waves).
  const size_t budget = (size_t)di->max_smem_optin - 1024;
  const int Kh = p.K / 2;
  const bool can2 = sms % 2 == 0 && p.K % 2 == 0 && Kh % C::CW == 0 &&
                    (!GRP || Kh % p.group == 0) && p.N >= 16 * (sms / 2);
  const double x_bytes = 2.0 * p.M * p.K;
  const double w_bytes = (double)p.N / sms * (double)a.row_bytes * NW;
  size_t smem = 0;
  for (int waves = 1; waves <= 64; ++waves) {
    smem = plan(1, waves);
    if (can2 && (smem == 0 || smem > budget || x_bytes * 3 * waves > w_bytes * 2)) {
      const size_t s2 = plan(2, waves);
      if (s2 != 0 && s2 <= budget) { smem = s2; break; }
      smem = plan(1, waves);
    }
    if (smem != 0 && smem <= budget) break;
    if ((p.N + sms * waves - 1) / (sms * waves) <= 16) break;  // one tile per range already
  }
  if (smem == 0 || smem > budget) return MT_ERR_SHAPE;

  auto kern = gemv_mma_kernel<FMT, KIND, WPL>;
  {
    std::lock_guard<std::mutex> g(cache.mu);
    if (dev < 64 && !cache.attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
      if (e != cudaSuccess) return cuda_fail(e);
      cache.attr_set[dev] = 1;
    }
  }
  return launch_mma(kern, grid, smem, l, a);
}

// The load width for a format and group size: a k step's 16 K indices (4
// lanes x WPL words) must lie in one group.
template <int FMT, int KIND>
mt_status dispatch_mma(const GemvProblem& p, const Launch& l) {
  if constexpr (FMT == FMT_MX8) {
    return run_gemv_mma<FMT, KIND, 2>(p, l);  // blocks of 32: 4 lanes x 8 bytes
  } else if constexpr (FMT == FMT_MX4) {
    return run_gemv_mma<FMT, KIND, 1>(p, l);  // blocks of 32: 4 lanes x 4 bytes
  } else if constexpr (FMT == FMT_A8) {
    if (p.group == 32) return run_gemv_mma<FMT, KIND, 2>(p, l);
    return run_gemv_mma<FMT, KIND, 4>(p, l);
  } else if constexpr (FMT == FMT_A4) {
    if (p.group == 32) return run_gemv_mma<FMT, KIND, 1>(p, l);
    if (p.group == 64) return run_gemv_mma<FMT, KIND, 2>(p, l);
    return run_gemv_mma<FMT, KIND, 4>(p, l);
  } else {
    return run_gemv_mma<FMT, KIND, 4>(p, l);
  }
}

}  // namespace mt
