// k_prefill.cuh - multi-row prefill (M > 8 activation rows) of the gate/up +
// SwiGLU, down + residual and projection + bias GEMMs over affine INT8/INT4
// weights, on the fifth-generation tensor cores (tcgen05, TMEM, TMA).
//
// meTile docs, "MLX-LM Backend", Dispatch Policy (multi-row shapes take a
// row-tiled dual GEMM: the gate and up tiles share each activation tile and
// the SwiGLU is applied in registers before the only store; affine
// w = scale * q + bias per group of 32/64/128 along K, fp32 accumulation);
// "Compute-Graph Fusion", Automatic Gated Epilogues (the residual and bias
// epilogues).
//
// GB300 design:
//  * One CTA computes a tile of 128 A rows x NT activation rows (NT = 64,
//    128 or 256 by M): D[128 x NT] = A[128 x K] . X[NT x K]^T with
//    tcgen05.mma (cta_group::1, M = 128, N = NT, K = 16, fp32 accumulators
//    in tensor memory).  The A rows are 128 output features (down /
//    projection) or 64 gate rows over the same 64 up rows (gate/up), so one
//    MMA per K step covers both matrices.
//  * A operand: affine codes enter exactly as fp16 subnormals (the bit
//    pattern 0x00qq is q * 2^-24: one byte permute per two INT8 codes, a
//    mask and permute for INT4); MX elements as their exact fp16 values
//    (cvt.rn.f16x2.e4m3x2 / .e2m1x2); two converter warps write them into
//    the 128-byte-swizzled K-major layout from TMA-filled code tiles.  Dense
//    bf16 weights go straight from TMA into the A tiles (bf16 MMA).
//  * B operand: the activations, converted once per call (prefill_x_kernel)
//    to fp16 scaled per row by 2^e_m (max|x_m| 2^e_m in [2^14, 2^15): every
//    bf16 value above 2^-28 of its row's maximum is exact) with their group
//    sums X'_g kept in fp32 (bf16 weights take x as stored); TMA
//    (SWIZZLE_128B) brings each 64-element K block.
//  * Each quantisation group accumulates into its own tensor-memory buffer
//    (two, alternating): the epilogue warpgroups read a finished group with
//    tcgen05.ld while the MMA fills the other and add s * D + b * X'_g into
//    fp32 registers (one A row per thread, NT / 2 activation rows per
//    warpgroup).  At the end the row scale 2^-e_m is undone, the up rows
//    hand their totals to the gate rows through shared memory for the
//    SwiGLU (or the residual / bias is added), and the bf16 tile leaves by
//    one TMA store.  With few tiles, K is split into slices whose fp32
//    partial sums prefill_finalize_kernel adds in slice order.
//  * Warp roles and rings: warp 11 lane 0 issues the x-tile copies (ring X),
//    lane 1 the code-tile copies (ring C, deeper: they are freed as soon as
//    converted); warps 8-9 convert ring C into ring B; warp 10 (converged,
//    elect.sync) issues the MMAs and the tcgen05.commits that free ring X,
//    ring B and fill the accumulator buffers; warps 0-7 are the epilogue.
//    Every mbarrier wait is bounded (~1 s): on expiry the thread records
//    MT_ERR_TIMEOUT in the device error word, the CTA stops, drains its
//    outstanding copies and MMAs, frees its tensor memory and returns.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "k_gemv.cuh"

namespace mt {

constexpr int PF_ROWS = 128;       // weight rows per tile (MMA M)
constexpr int PF_COLS = 256;       // largest activation-row tile (MMA N); 64 and 128 for small M
constexpr int PF_KB = 64;          // K per stage (one 128-byte swizzle row of fp16)
constexpr int PF_EPI_WARPS = 8;    // warps 0-7: epilogue, two warpgroups (NT / 2 tile columns each)
constexpr int PF_CONV_WARPS = 2;   // warps 8-9: converters
constexpr int PF_THREADS = 32 * (PF_EPI_WARPS + PF_CONV_WARPS + 2);  // + warp 10: MMA, warp 11: TMA
constexpr int PF_W_TILE = PF_ROWS * PF_KB * 2;   // 16 KB
// Groups whose scale, bias and X'_g the epilogue has in flight ahead of use
// (even): a group's MMAs take well under the latency of a global load under
// the tensor-core stream, so one group ahead left the MMA waiting for the
// epilogue.
constexpr int PF_EPI_AHEAD = 4;

struct PrefillArgs {
  const uint8_t* W0;  // gate (kind 0) or the weight (kind 1): codes [N][row_bytes]
  const uint8_t* W1;  // up (kind 0)
  const uint16_t* s0;
  const uint16_t* b0;
  const uint16_t* s1;
  const uint16_t* b1;
  const float* XgT;   // [G][Mp] group sums of the scaled activations (Mp = 64 n_ctiles)
  const float* einv;  // [M] 2^-e_m
  const uint16_t* res;  // addend (kind 1) or nullptr
  int res_ld;           // its row stride in elements (0: one bias row for all m)
  void* out;            // [M][N]
  int out_f32;
  int M, K, N, group, lg_group, G, KB, row_bytes;
  int n_ctiles;         // ceil(M / NT)
  int Mp;               // row stride of XgT (M rounded up to 256)
  int ks, KBs;          // K slices (split K when the tiles do not fill the GPU) and K blocks per slice
  float* part;          // ks > 1: partial sums [ks][NW][Mp][N] before the row scale and epilogue
  int tma_store;        // 1: bf16 output written by one TMA store per tile (row stride a multiple of 16 B)
  int* err;             // device error word
  const float* tsc;     // dequantising kernel: 2^t_n of each weight row [NW][N]
  const float* tinv;    // and 2^-t_n
};

// ------------------------------------------------------------- PTX wrappers

// Waits until at most N of this thread's committed asynchronous copy groups
// (cp.async) are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared-memory matrix descriptor of a K-major fp16 tile whose rows are 128
// bytes, stored with the 128-byte swizzle (16-byte chunk c of row r at chunk
// c ^ (r & 7)); 8-row core groups 1024 bytes apart.  The tile starts on a
// 1024-byte boundary; a K step of 16 elements advances the start by 32 bytes.
__device__ __forceinline__ uint64_t pf_desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                             // leading offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;                   // stride offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                             // descriptor version
  d |= (uint64_t)2 << 61;                             // 128-byte swizzle
  return d;
}

// Instruction descriptor: fp32 accumulator, fp16 A and B, both K-major,
// N = 64, M = 128.
// Instruction descriptor: fp32 accumulator, A and B fp16 (BF = false) or
// bf16 (BF = true), both K-major, N = NT, M = 128.
template <int NT, bool BF>
__host__ __device__ constexpr uint32_t pf_idesc() {
  return (1u << 4) | ((BF ? 1u : 0u) << 7) | ((BF ? 1u : 0u) << 10) | ((uint32_t)(NT >> 3) << 17) |
         ((uint32_t)(PF_ROWS >> 4) << 24);
}

template <int NT, bool BF>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(pf_idesc<NT, BF>()), "r"(accumulate)
      : "memory");
}

// The mbarrier tracks the completion of every tcgen05.mma this thread issued.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane at taddr,
// the wait for the load inside the same statement so that no use of the
// registers can be scheduled before it.
__device__ __forceinline__ void tc_ld16_wait(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Plain global stores as inline PTX: the compiler then knows they touch no
// shared memory and keeps the loads of the store loops ahead of them.
__device__ __forceinline__ void st_global_f32(float* p, float v) {
  asm volatile("st.global.f32 [%0], %1;" ::"l"(p), "f"(v));
}
__device__ __forceinline__ void st_global_bf16(uint16_t* p, float v) {
  asm volatile("st.global.b16 [%0], %1;" ::"l"(p), "h"(f2bf(v)));
}

// 2D tiled TMA store of a shared-memory tile at (x0, y0); the part outside
// the tensor is not written.  Waits until the tile has been read out of
// shared memory.
__device__ __forceinline__ void tma_store_2d_wait(const CUtensorMap* map, int x0, int y0, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x0),
               "r"(y0), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// 2D tiled TMA load of box {64 elements, 64 rows} at (k0, m0), completing on bar.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int k0, int m0, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(k0), "r"(m0), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------- activations pass

// One CTA per activation row m (grid: M rounded up to the column tile, Mp):
// e_m from the row's maximum magnitude, the row as fp16 x * 2^e_m (round to
// nearest), the group sums of x * 2^e_m (fp32, in a fixed order; [G][Mp]) and
// 2^-e_m.
__global__ void __launch_bounds__(256) prefill_x_kernel(const uint16_t* __restrict__ x, int M, int K, int group,
                                                        __half* __restrict__ x16, float* __restrict__ XgT,
                                                        float* __restrict__ einv);  // defined in k_prefill.cu

// ------------------------------------------------------------- the GEMM

// Codes of weight rows r0, r0 + step, ... (R rows) for one K block of 64
// (INT8: 64 bytes a row, INT4: 32), read from the TMA-filled code tile (rows
// of CB bytes, 64- or 32-byte swizzle: 16-byte chunk u of row r at
// u ^ ((r >> 1) & 3), resp. u ^ ((r >> 2) & 1), so that eight consecutive
// rows read their chunk u from distinct banks), written as fp16 subnormals
// q * 2^-24 into the same rows of the MMA tile (128-byte rows, chunk j at
// j ^ (r & 7)).  Every load of the R rows is issued before the first store.
// MX elements as exact fp16 values: lo = codes (c0, c1), hi = (c2, c3) of a
// word's four E4M3 bytes; or the two E2M1 codes of one byte as one f16x2.
__device__ __forceinline__ void pf_e4m3x4(uint32_t v, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(v));
}
__device__ __forceinline__ void pf_e2m1x8(uint32_t v, uint4& o) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w)
      : "r"(v));
}

// Affine codes become fp16 q * 2^-24 (exact); MX elements (E4M3, E2M1)
// become their exact fp16 values (the E8M0 block scale is applied at the
// group flush).
template <int FMT, int R>
__device__ __forceinline__ void pf_convert_rows(const unsigned char* __restrict__ ctile,
                                                unsigned char* __restrict__ wtile, int r0, int step) {
  constexpr bool W8 = FmtTraits<FMT>::EPW == 4;  // one byte per code (INT8, E4M3)
  constexpr int U = W8 ? 4 : 2;                  // 16-byte code chunks a row
  uint4 v[R][U];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int r = r0 + i * step;
#pragma unroll
    for (int u = 0; u < U; ++u)
      v[i][u] = W8
                    ? *reinterpret_cast<const uint4*>(ctile + r * 64 + ((u ^ ((r >> 1) & 3)) << 4))
                    : *reinterpret_cast<const uint4*>(ctile + r * 32 + ((u ^ ((r >> 2) & 1)) << 4));
  }
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int r = r0 + i * step;
    unsigned char* rowp = wtile + r * 128;
    const int sw = r & 7;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t w[4] = {v[i][u].x, v[i][u].y, v[i][u].z, v[i][u].w};
      if constexpr (FMT == FMT_MX8) {  // 16 E4M3 codes -> chunks 2u, 2u+1
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint4 o;
          pf_e4m3x4(w[2 * h], o.x, o.y);
          pf_e4m3x4(w[2 * h + 1], o.z, o.w);
          *reinterpret_cast<uint4*>(rowp + (((2 * u + h) ^ sw) << 4)) = o;
        }
      } else if constexpr (FMT == FMT_MX4) {  // 32 E2M1 codes -> chunks 4u .. 4u+3
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 o;
          pf_e2m1x8(w[k], o);
          *reinterpret_cast<uint4*>(rowp + (((4 * u + k) ^ sw) << 4)) = o;
        }
      } else if constexpr (FMT == FMT_A8) {  // 16 codes -> chunks 2u, 2u+1
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t a = w[2 * h], b = w[2 * h + 1];
          const uint4 o = make_uint4(__byte_perm(a, 0u, 0x4140), __byte_perm(a, 0u, 0x4342),
                                     __byte_perm(b, 0u, 0x4140), __byte_perm(b, 0u, 0x4342));
          *reinterpret_cast<uint4*>(rowp + (((2 * u + h) ^ sw) << 4)) = o;
        }
      } else {  // 32 codes -> chunks 4u .. 4u+3 (one word each)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // byte j of w holds code 2j (bits 0..3) and 2j+1 (bits 4..7)
          const uint32_t lo = w[k] & 0x0F0F0F0Fu, hi = (w[k] >> 4) & 0x0F0F0F0Fu;
          const uint4 o = make_uint4(__byte_perm(lo, hi, 0x4400) & 0x00FF00FFu, __byte_perm(lo, hi, 0x5511) & 0x00FF00FFu,
                                     __byte_perm(lo, hi, 0x6622) & 0x00FF00FFu, __byte_perm(lo, hi, 0x7733) & 0x00FF00FFu);
          *reinterpret_cast<uint4*>(rowp + (((4 * u + k) ^ sw) << 4)) = o;
        }
      }
    }
  }
}

// Shared-memory plan of one (format, kind).  The MMA's A tile is 128 weight
// rows: 128 output features (down / projection), or the gate rows (0-63) and
// the up rows (64-127) of 64 output features (gate/up), so that one MMA per K
// step covers both matrices.  Three rings: X, the x tiles (256 rows x 128 B,
// 128-byte swizzle; TMA in, freed by the MMA); C, the code tiles (128 rows x
// CB bytes; TMA in, freed by the converters, so they are fetched further
// ahead); B, the fp16 A tiles (converters in, freed by the MMA).
template <int FMT, int KIND, int NT>
struct PfShape {
  static constexpr int XT = NT * PF_KB * 2;             // x tile bytes (8, 16 or 32 KB)
  static constexpr int FT = KIND == 0 ? 64 : 128;       // output features per tile
  static constexpr int CB = FmtTraits<FMT>::EPW == 4 ? 64 : 32;  // code bytes per row and K block
  static constexpr int CTILE = PF_ROWS * CB;            // 8 or 4 KB
  // ring depths: narrow tiles (small M, weights streamed from HBM once) keep
  // more code tiles in flight; wide tiles more x tiles
  // (dense bf16 weights skip the code ring: TMA fills the A ring itself)
  static constexpr bool BFW = FMT == FMT_BF16;
  static constexpr int SX = NT == 128 ? 5 : 4;
  static constexpr int SC = BFW ? 1 : (NT == 64 ? 96 : (NT == 128 ? 64 : 48)) * 1024 / CTILE;
  static constexpr int SB = BFW ? (NT == 256 ? 4 : 6) : (NT == 256 ? 2 : 4);
  static constexpr size_t OFF_C = (size_t)SX * XT;
  static constexpr size_t OFF_B = OFF_C + (size_t)SC * CTILE;
  static constexpr size_t SMEM = 1024 + OFF_B + (size_t)SB * PF_W_TILE;
  static_assert(SMEM <= 218 * 1024, "shared memory plan");
  static_assert(OFF_C >= (size_t)64 * NT * 4 + (size_t)NT * 128 * 2, "final-phase buffers in ring X");
};

// 1 in exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
  return e != 0;
}

template <int FMT, int KIND, int NT>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap0,
                        const __grid_constant__ CUtensorMap wmap1, const __grid_constant__ CUtensorMap omap,
                        const PrefillArgs a) {
  using SH = PfShape<FMT, KIND, NT>;
  constexpr int SX = SH::SX, SC = SH::SC, SB = SH::SB, FT = SH::FT;
  constexpr uint32_t NCOLS = 2 * NT;        // two accumulator buffers of NT columns
  constexpr bool BFW = SH::BFW;              // dense bf16 weights: no codes, no converters
  constexpr int EPI = 32 * PF_EPI_WARPS;    // epilogue threads
  constexpr int HALF = NT / 2;              // tile columns per epilogue warpgroup

  extern __shared__ unsigned char smem_raw[];
  // 1024-byte aligned start, by an offset on the shared array itself (so the
  // compiler keeps shared-space loads and stores)
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bars[2 * (SX + SC + SB) + 5];
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;
  __shared__ __align__(16) float xg_sh[PF_EPI_AHEAD][NT];  // X'_g of the tile's rows, a ring of groups
  __shared__ __align__(16) float einv_sh[NT];   // 2^-e_m of the tile's rows

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x / a.ks, sk = blockIdx.x - tile * a.ks;
  const int rt = tile / a.n_ctiles, ct = tile - rt * a.n_ctiles;
  const int f0 = rt * FT, m0 = ct * NT;  // first output feature and activation row
  // this CTA's K slice: K blocks [kb0, kb0 + KB) and groups [g0, g0 + G)
  const int kb0 = sk * a.KBs, KB = min(a.KB - kb0, a.KBs);
  const int g0 = kb0 * PF_KB / a.group, G = KB * PF_KB / a.group, Gall = a.G, Mp = a.Mp;
  auto x_full = [&](int i) { return smem_u32(&bars[i]); };                  // TMA bytes of x slot i
  auto x_free = [&](int i) { return smem_u32(&bars[SX + i]); };             // MMA done with it
  auto c_full = [&](int i) { return smem_u32(&bars[2 * SX + i]); };         // TMA bytes of code slot i
  auto c_free = [&](int i) { return smem_u32(&bars[2 * SX + SC + i]); };    // converters done with it
  auto w_full = [&](int i) { return smem_u32(&bars[2 * (SX + SC) + i]); };  // converters wrote A slot i
  auto b_free = [&](int i) { return smem_u32(&bars[2 * (SX + SC) + SB + i]); };  // MMA done with it
  auto acc_full = [&](int b) { return smem_u32(&bars[2 * (SX + SC + SB) + b]); };
  auto acc_free = [&](int b) { return smem_u32(&bars[2 * (SX + SC + SB) + 2 + b]); };
  const uint32_t mma_done = smem_u32(&bars[2 * (SX + SC + SB) + 4]);
  auto xslot = [&](int i) { return smem + (size_t)i * SH::XT; };
  auto cslot = [&](int i) { return smem + SH::OFF_C + (size_t)i * SH::CTILE; };
  auto wslot = [&](int i) { return smem + SH::OFF_B + (size_t)i * PF_W_TILE; };
  constexpr int CONV0 = PF_EPI_WARPS;                   // first converter warp
  constexpr int MMA_WARP = PF_EPI_WARPS + PF_CONV_WARPS;
  constexpr int TMA_WARP = MMA_WARP + 1;
  constexpr int CONV = 32 * PF_CONV_WARPS;              // converter threads

  if (tid == 0) {
    for (int i = 0; i < SX; ++i) {
      mbar_init(x_full(i), 1);
      mbar_init(x_free(i), 1);
    }
    for (int i = 0; i < SC; ++i) {
      mbar_init(c_full(i), 1);
      mbar_init(c_free(i), PF_CONV_WARPS);  // one arrival per converter warp
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(w_full(i), BFW ? 1 : PF_CONV_WARPS);  // TMA (bf16 weights) or the converter warps
      mbar_init(b_free(i), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_free(b), PF_EPI_WARPS);  // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    abort_sh = 0;
    mbar_fence_init();
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_sh)),
                 "r"(NCOLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_sh;
  volatile int* abort_flag = &abort_sh;
  auto fail = [&]() {
    atomicExch(a.err, (int)MT_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == TMA_WARP) {
    // ---- producers: lane 0 the x tiles (SX blocks ahead of the MMA), lane 1
    // the code tiles (SC blocks ahead of the converters)
    if (lane < 2) {
      // bf16 weights: lane 1 fills the A ring directly
      const int S = lane == 0 ? SX : (BFW ? SB : SC);
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int i = kb % S;
        const uint32_t full = lane == 0 ? x_full(i) : (BFW ? w_full(i) : c_full(i));
        const uint32_t free_ = lane == 0 ? x_free(i) : (BFW ? b_free(i) : c_free(i));
        if (kb >= S && !mbar_wait_bounded(free_, ((kb / S) + 1) & 1)) { fail(); break; }
        if (*abort_flag) break;
        const int kg = kb0 + kb;  // K block of the tensor
        if (lane == 0) {
          mbar_arrive_expect_tx(full, SH::XT);
          tma_load_2d(smem_u32(xslot(i)), &xmap, kg * PF_KB, m0, full);
        } else if constexpr (BFW) {
          mbar_arrive_expect_tx(full, PF_W_TILE);
          tma_load_2d(smem_u32(wslot(i)), &wmap0, kg * PF_KB, f0, full);
          if constexpr (KIND == 0) tma_load_2d(smem_u32(wslot(i) + 64 * 128), &wmap1, kg * PF_KB, f0, full);
        } else {
          mbar_arrive_expect_tx(full, SH::CTILE);
          tma_load_2d(smem_u32(cslot(i)), &wmap0, kg * SH::CB, f0, full);
          if constexpr (KIND == 0) tma_load_2d(smem_u32(cslot(i) + 64 * SH::CB), &wmap1, kg * SH::CB, f0, full);
        }
        ++issued;
      }
      // copies still in flight (only after an abort) land before the CTA ends
      for (int kb = max(0, issued - S); kb < issued; ++kb)
        (void)mbar_wait_bounded(lane == 0 ? x_full(kb % S) : (BFW ? w_full(kb % S) : c_full(kb % S)), (kb / S) & 1);
    }
    __syncwarp();
  } else if (warp >= CONV0 && warp < MMA_WARP) {
    // ---- converters: rows c, c + CONV of the code tile into the fp16 A tile
    // (none for bf16 weights)
    if constexpr (!BFW) {
    const int c = tid - 32 * CONV0;
    for (int kb = 0; kb < KB; ++kb) {
      const int i = kb % SC, j = kb % SB;
      bool ok = mbar_wait_bounded(c_full(i), (kb / SC) & 1);
      if (ok && kb >= SB) ok = mbar_wait_bounded(b_free(j), ((kb / SB) + 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) { fail(); break; }
      pf_convert_rows<FMT, PF_ROWS / CONV>(cslot(i), wslot(j), c, CONV);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor core reads
      // one arrival per warp (an mbarrier arrival is a shared-memory atomic:
      // 32 of them on one word serialise)
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(w_full(j));
        mbar_arrive(c_free(i));
      }
      if (__any_sync(0xffffffffu, *abort_flag)) break;
    }
    }
  } else if (warp == MMA_WARP) {
    // ---- MMA issuer: the whole warp walks the loop, one elected lane issues
    const int group = a.group;
    bool ok = true;
    for (int kb = 0; kb < KB && ok; ++kb) {
      const int i = kb % SX, jb = kb % SB;
      // one decision for the whole warp (elect.sync below needs every lane)
      const bool got = mbar_wait_bounded(x_full(i), (kb / SX) & 1) && mbar_wait_bounded(w_full(jb), (kb / SB) & 1);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t xd = pf_desc_sw128(smem_u32(xslot(i)));
      const uint64_t wd = pf_desc_sw128(smem_u32(wslot(jb)));
#pragma unroll
      for (int j = 0; j < PF_KB / 16; ++j) {
        const int k = kb * PF_KB + 16 * j;       // K within the slice (slices start on a group)
        const int gi = k >> a.lg_group, b = gi & 1;  // group within the slice
        const bool first = (k & (group - 1)) == 0;
        if (first && gi >= 2) {
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(acc_free(b), ((gi >> 1) - 1) & 1))) { ok = false; break; }
          tc_fence_after();
        }
        if (elect_one()) {
          tc_mma<NT, BFW>(tbase + (uint32_t)(b * NT), wd + 2 * j, xd + 2 * j, first ? 0u : 1u);
          if (((k + 16) & (group - 1)) == 0) tc_commit(acc_full(b));
        }
        __syncwarp();
      }
      if (elect_one()) {
        tc_commit(b_free(jb));
        tc_commit(x_free(i));
      }
      __syncwarp();
      if (__any_sync(0xffffffffu, *abort_flag)) break;
    }
    if (!ok) fail();
    if (elect_one()) tc_commit(mma_done);  // completes when every MMA issued above has
    __syncwarp();
    (void)mbar_wait_bounded(mma_done, 0);
  } else {
    // ---- epilogue: two warpgroups; thread (r, wg) owns A row r (tensor
    // memory lane r) and the tile columns [wg * 128, wg * 128 + 128)
    const int wg = warp >> 2, r = tid & 127;
    const int mat = (KIND == 0 && r >= 64) ? 1 : 0;     // gate/up: rows 64-127 are the up matrix
    const int n = f0 + (KIND == 0 ? (r & 63) : r);      // output feature
    const bool okr = n < a.N;
    const uint16_t* sp = mat ? a.s1 : a.s0;
    const uint16_t* bp = mat ? a.b1 : a.b0;
    const size_t sbo = (size_t)(okr ? n : 0) * Gall + g0;
    float acc[HALF];
#pragma unroll
    for (int j = 0; j < HALF; ++j) acc[j] = 0.f;
    const uint32_t lane_base = tbase + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(wg * HALF);
    // group scale and bias, loaded raw PD groups ahead of their use and
    // converted there: affine s * 2^24 (the codes enter the MMA as
    // q * 2^-24) and b; MX the E8M0 block scale 2^(E - 127) and no bias
    constexpr bool MXF = FmtTraits<FMT>::MX;
    constexpr int PD = PF_EPI_AHEAD;
    auto raw_scale = [&](int gi) -> uint32_t {
      if constexpr (BFW) return 0u;
      else if constexpr (MXF) return (okr && gi < G) ? (uint32_t)__ldg(reinterpret_cast<const uint8_t*>(sp) + sbo + gi) : 0u;
      else return (okr && gi < G) ? (uint32_t)__ldg(sp + sbo + gi) : 0u;
    };
    auto raw_bias = [&](int gi) -> uint32_t {
      if constexpr (MXF || BFW) return 0u;
      else return (okr && gi < G) ? (uint32_t)__ldg(bp + sbo + gi) : 0u;
    };
    auto scale_of = [&](uint32_t raw) -> float {
      if constexpr (BFW) {
        return 1.0f;  // dense bf16 weights: D is the dot product itself
      } else if constexpr (MXF) {
        return raw ? __int_as_float((int)(raw << 23)) : __int_as_float(0x00400000);
      } else {
        return bf16f((uint16_t)raw) * 16777216.f;
      }
    };
    auto bias_of = [&](uint32_t raw) -> float {
      if constexpr (MXF || BFW) return 0.f;
      else return bf16f((uint16_t)raw);
    };
    // X'_g of group gi for the tile's rows comes into xg_sh[gi % PD] by
    // asynchronous copies PD - 1 groups ahead (threads 0-63, 16 bytes each);
    // one commit group per group index, empty past the slice's end
    auto fetch_xg = [&](int gi) {
      if (!BFW && gi < G && tid < NT / 4)
        cp_async16(&xg_sh[gi % PD][4 * tid], a.XgT + (size_t)(g0 + gi) * Mp + m0 + 4 * tid);
      cp_async_commit();
    };
    auto epi_sync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(EPI) : "memory"); };
    // barrier of the epilogue warps that also ORs a flag over them (a uniform decision)
    auto epi_sync_or = [&](bool v) -> bool {
      uint32_t res;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
          "barrier.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(res)
          : "r"((uint32_t)v), "n"(EPI)
          : "memory");
      return res != 0;
    };
    // the tile's row scales (padded rows hold 0), in the first commit group
    if constexpr (BFW) {  // x enters the MMA as stored: no row scale, no group sums
      for (int i = tid; i < NT; i += EPI) einv_sh[i] = 1.0f;
    } else {
      if (tid < NT / 4) cp_async16(&einv_sh[4 * tid], a.einv + m0 + 4 * tid);
    }
    uint32_t sq[PD], bq[PD];  // raw scale and bias of groups gi0 + u (then gi0 + PD + u)
#pragma unroll
    for (int u = 0; u < PD; ++u) {
      sq[u] = raw_scale(u);
      bq[u] = raw_bias(u);
    }
#pragma unroll
    for (int u = 0; u < PD - 1; ++u) fetch_xg(u);
    cp_async_wait_group<PD - 2>();  // group 0's sums and the row scales landed
    epi_sync();
    bool aborted = false;
    for (int gi0 = 0; gi0 < G && !aborted; gi0 += PD) {
#pragma unroll
      for (int u = 0; u < PD; ++u) {
        const int gi = gi0 + u, b = u & 1;  // gi % PD == u, gi & 1 == b (PD even)
        if (gi >= G) break;
        fetch_xg(gi + PD - 1);
        const float sv = scale_of(sq[u]), bv = bias_of(bq[u]);
        sq[u] = raw_scale(gi + PD);
        bq[u] = raw_bias(gi + PD);
        if (!mbar_wait_bounded(acc_full(b), (gi >> 1) & 1)) { fail(); aborted = true; }
        // the tensor-memory loads below are warp-wide: one decision per warp
        aborted = __any_sync(0xffffffffu, aborted);
        if (!aborted) {
          tc_fence_after();
          const float* xg = xg_sh[u] + wg * HALF;
#pragma unroll
          for (int q = 0; q < HALF / 16; ++q) {
            float d[16];
            tc_ld16_wait(lane_base + (uint32_t)(b * NT + q * 16), d);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 X = *reinterpret_cast<const float4*>(xg + q * 16 + 4 * i);
              const float Xv[4] = {X.x, X.y, X.z, X.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int jj = q * 16 + 4 * i + e;
                if constexpr (BFW || MXF)
                  acc[jj] = fmaf(sv, d[4 * i + e], acc[jj]);  // no bias term
                else
                  acc[jj] = fmaf(sv, d[4 * i + e], fmaf(bv, Xv[e], acc[jj]));
              }
            }
          }
        }
        // this warp is done reading the buffer: one arrival for the warp
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_free(b));
        // the next group's X'_g has landed and every thread is done with
        // this one; the decision to stop is the same for every epilogue thread
        cp_async_wait_group<PD - 2>();
        aborted = epi_sync_or(aborted || *abort_flag);
        if (aborted) break;
      }
    }
    cp_async_wait_all();  // nothing left in flight (after an abort: copies of later groups)
    if (!aborted && a.ks > 1) {
      // split K: this slice's sums, before the row scale and the epilogue
      if (okr) {
        float* pp = a.part + ((size_t)(sk * (KIND == 0 ? 2 : 1) + mat) * Mp + m0 + wg * HALF) * a.N + n;
#pragma unroll
        for (int j = 0; j < HALF; ++j) st_global_f32(pp + (size_t)j * a.N, acc[j]);
      }
    } else if (!aborted) {
      const int cbase = wg * HALF;
      const float* ei = einv_sh + cbase;
      const int jmax = min(HALF, a.M - m0 - cbase);
      const size_t obase = (size_t)(m0 + cbase) * a.N + n;
      // bf16 output tile [256 rows][FT features], row-major, for one TMA store
      // (ring A is idle now: every copy and MMA has completed)
      uint16_t* stg = reinterpret_cast<uint16_t*>(smem + (KIND == 0 ? NT * 64 * 4 : 0));
      if constexpr (KIND == 0) {
        // the up rows hand their totals to the gate rows through shared
        // memory, column-major so that consecutive rows hit consecutive banks
        float* xch = reinterpret_cast<float*>(smem);  // [NT][64]
        if (mat == 1) {
#pragma unroll
          for (int j = 0; j < HALF; ++j) xch[(cbase + j) * 64 + (r - 64)] = acc[j];
        }
        epi_sync();
        if (mat == 0 && a.tma_store) {
          // 16 columns at a time: their loads, then their stores
#pragma unroll
          for (int q = 0; q < HALF / 16; ++q) {
            float u[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) u[e] = xch[(cbase + q * 16 + e) * 64 + r];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int j = q * 16 + e;
              const float g = acc[j] * ei[j];
              stg[(cbase + j) * FT + r] = f2bf(g / (1.0f + expf(-g)) * (u[e] * ei[j]));  // silu(gate) * up
            }
          }
        }
        if (mat == 0 && okr && !a.tma_store) {
#pragma unroll
          for (int j = 0; j < HALF; ++j) {
            const float g = acc[j] * ei[j], u = xch[(cbase + j) * 64 + r] * ei[j];
            const float h = g / (1.0f + expf(-g)) * u;  // silu(gate) * up
            if (j < jmax) {
              if (a.out_f32)
                st_global_f32(static_cast<float*>(a.out) + obase + (size_t)j * a.N, h);
              else
                st_global_bf16(static_cast<uint16_t*>(a.out) + obase + (size_t)j * a.N, h);
            }
          }
        }
      } else if (okr || a.tma_store) {
        // down / projection: 16 columns at a time, their addends loaded
        // together, then stored
        const uint16_t* __restrict__ res = a.res;
#pragma unroll
        for (int q = 0; q < HALF / 16; ++q) {
          float add[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = q * 16 + e;
            add[e] = (res && okr && j < jmax) ? bf16f(__ldg(res + (size_t)(m0 + cbase + j) * a.res_ld + n)) : 0.f;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = q * 16 + e;
            const float v = acc[j] * ei[j] + add[e];  // + residual or bias
            if (a.tma_store) {
              stg[(cbase + j) * FT + r] = f2bf(v);
            } else if (j < jmax) {
              if (a.out_f32)
                st_global_f32(static_cast<float*>(a.out) + obase + (size_t)j * a.N, v);
              else
                st_global_bf16(static_cast<uint16_t*>(a.out) + obase + (size_t)j * a.N, v);
            }
          }
        }
      }
      if (a.tma_store) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // tile writes -> TMA reads
        epi_sync();
        if (tid == 0) tma_store_2d_wait(&omap, f0, m0, smem_u32(stg));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == MMA_WARP) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(NCOLS));
}

// Split K: the slices' partial sums added in slice order, the row scales
// (2^-e_m of the activations; 2^-t_n of dequantised weight rows) undone and
// the epilogue applied (one thread per output element).
template <int KIND>
__global__ void __launch_bounds__(256) prefill_finalize_kernel(const float* __restrict__ part, int ks, int Mp,
                                                               const float* __restrict__ einv,
                                                               const float* __restrict__ tinv, int M, int N,
                                                               const uint16_t* __restrict__ res, int res_ld,
                                                               void* out, int out_f32) {
  constexpr int NW = KIND == 0 ? 2 : 1;
  const long total = (long)M * N;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int m = (int)(i / N), n = (int)(i - (long)m * N);
    float v[NW];
#pragma unroll
    for (int mat = 0; mat < NW; ++mat) {
      float t = 0.f;
      for (int s = 0; s < ks; ++s) t += part[((size_t)(s * NW + mat) * Mp + m) * N + n];
      if (einv) t *= einv[m];
      if (tinv) t *= tinv[(size_t)mat * N + n];  // 2^-t_n of the dequantised weight row
      v[mat] = t;
    }
    float o;
    if constexpr (KIND == 0)
      o = v[0] / (1.0f + expf(-v[0])) * v[NW - 1];  // silu(gate) * up
    else
      o = res ? v[0] + bf16f(res[(size_t)m * res_ld + n]) : v[0];  // + residual or bias
    if (out_f32)
      static_cast<float*>(out)[i] = o;
    else
      static_cast<uint16_t*>(out)[i] = f2bf(o);
  }
}

// ---------------------------------------------------------------- host side

namespace {

size_t al1k(size_t v) { return (v + 1023) / 1024 * 1024; }

// The activation-row tile for M rows: the smallest of 64, 128, 256 that holds them.
int prefill_nt(long M) { return M <= 64 ? 64 : (M <= 128 ? 128 : 256); }

// K slices for a grid of `tiles` CTAs on `sms` SMs: split K when the tiles
// fill at most half of the SMs, into whole groups, at most 8 slices and at
// least two groups (and two K blocks) each.  *kbs receives K blocks per slice.
int prefill_ks(long tiles, long K, long group, int sms, int* kbs) {
  const int KB = (int)(K / PF_KB);
  const int gb = group > PF_KB ? (int)(group / PF_KB) : 1;  // K blocks per group (or 1)
  int ks = 1;
  if (tiles * 2 <= sms) ks = (int)std::min<long>(8, sms / tiles);
  ks = std::max(1, std::min(ks, KB / std::max(2, 2 * gb)));
  int per = (KB + ks - 1) / ks;
  per = (per + gb - 1) / gb * gb;
  *kbs = per;
  return (KB + per - 1) / per;
}

// The accumulation group of dense bf16 weights (they have no quantisation
// groups): the largest power of two up to 512 that divides K (K % 64 == 0),
// so that each group's sum is read out of tensor memory while the next one
// accumulates, as for the affine groups.
int prefill_bf16_group(long K) {
  int g = 512;
  while (K % g) g >>= 1;
  return g;
}

// Workspace: x16 [M][K] fp16, XgT [G][Mp] fp32, einv [Mp] fp32, the weight
// rows' 2^t_n and 2^-t_n [2][2][N] fp32 (dequantising kernel), and with split
// K the partial sums [ks][2][Mp][N] fp32 (sized for the largest split of both
// tilings, gate/up and down / projection, and both kernels).
struct PfWs {
  size_t xg, einv, tw, part, total;  // byte offsets (x16 at 0) and the size
};
PfWs prefill_ws_layout(long M, long K, long N, long group, int sms) {
  if (group == 0) group = prefill_bf16_group(K);  // dense bf16 weights
  const long Mp = (M + PF_COLS - 1) / PF_COLS * PF_COLS;
  const long nct = (M + prefill_nt(M) - 1) / prefill_nt(M);
  int kbs = 0, ks = 1;
  for (long g : {group, (long)PF_KB})
    for (long ft : {64L, 128L}) ks = std::max(ks, prefill_ks(nct * ((N + ft - 1) / ft), K, g, sms, &kbs));
  const size_t part = ks > 1 ? (size_t)ks * 2 * Mp * N * 4 : 0;
  PfWs w;
  w.xg = al1k((size_t)M * K * 2);
  w.einv = w.xg + al1k((size_t)(K / group) * Mp * 4);
  w.tw = w.einv + al1k((size_t)Mp * 4);
  w.part = w.tw + al1k((size_t)16 * N);
  w.total = w.part + al1k(part);
  return w;
}
size_t prefill_ws_bytes(long M, long K, long N, long group, int sms) {
  return prefill_ws_layout(M, K, N, group, sms).total;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

template <int FMT, int KIND, int NT>
mt_status run_prefill(const GemvProblem& p, void* ws, const Launch& l) {
  constexpr int NW = KIND == 0 ? 2 : 1;
  constexpr bool BFW = FMT == FMT_BF16;
  const int M = p.M, K = p.K, N = p.N, group = BFW ? prefill_bf16_group(p.K) : p.group;
  using SH = PfShape<FMT, KIND, NT>;
  const int n_ctiles = (M + NT - 1) / NT, Mp = (M + PF_COLS - 1) / PF_COLS * PF_COLS;
  const int n_rtiles = (N + SH::FT - 1) / SH::FT;
  const int G = K / group;
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  if (!di) return cuda_fail((cudaError_t)derr);
  unsigned char* w = static_cast<unsigned char*>(ws);
  const PfWs wl = prefill_ws_layout(M, K, N, group, di->sm_count);
  __half* x16 = reinterpret_cast<__half*>(w);
  float* XgT = reinterpret_cast<float*>(w + wl.xg);
  float* einv = reinterpret_cast<float*>(w + wl.einv);
  float* part = reinterpret_cast<float*>(w + wl.part);
  int kbs = 0;
  const int ks = prefill_ks((long)n_rtiles * n_ctiles, K, group, di->sm_count, &kbs);
  int* err = device_error_ptr();
  if (!err) return MT_ERR_CUDA;

  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cuda_fail(cudaErrorNotSupported);
  CUtensorMap xmap;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)PF_KB, (cuuint32_t)NT};
  const cuuint32_t estr[2] = {1, 1};
  // x: the fp16 rows of the workspace, or (bf16 weights) the bf16 input as stored
  if (enc(&xmap, BFW ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
          BFW ? const_cast<uint16_t*>(p.x) : static_cast<void*>(x16), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return cuda_fail(cudaErrorInvalidValue);
  // code tiles: 128 rows x CB bytes, 64-byte (INT8) or 32-byte (INT4) swizzle;
  // bf16 weights: the A tile itself, 64 elements (128 B) a row, 128-byte swizzle
  CUtensorMap wmap[2];
  for (int mat = 0; mat < 2; ++mat) {
    const void* W = (mat && NW == 2) ? p.W1 : p.W0;
    if constexpr (BFW) {
      const cuuint64_t wdims[2] = {(cuuint64_t)K, (cuuint64_t)N};
      const cuuint64_t wstr[1] = {(cuuint64_t)K * 2};
      const cuuint32_t wbox[2] = {(cuuint32_t)PF_KB, (cuuint32_t)SH::FT};
      if (enc(&wmap[mat], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), wdims, wstr, wbox, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cuda_fail(cudaErrorInvalidValue);
      continue;
    }
    const cuuint64_t wdims[2] = {(cuuint64_t)(SH::CB == 64 ? K : K / 2), (cuuint64_t)N};
    const cuuint64_t wstr[1] = {wdims[0]};
    const cuuint32_t wbox[2] = {(cuuint32_t)SH::CB, (cuuint32_t)SH::FT};  // gate/up: 64 rows of each
    if (enc(&wmap[mat], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), wdims, wstr, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, SH::CB == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cuda_fail(cudaErrorInvalidValue);
  }

  // bf16 output tiles go out by TMA when a row is a multiple of 16 bytes
  CUtensorMap omap = xmap;
  const bool tma_store = !p.out_f32 && N % 8 == 0;
  if (tma_store) {
    const cuuint64_t odims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t ostr[1] = {(cuuint64_t)N * 2};
    const cuuint32_t obox[2] = {(cuuint32_t)SH::FT, (cuuint32_t)NT};
    if (enc(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.out, odims, ostr, obox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cuda_fail(cudaErrorInvalidValue);
  }

  PrefillArgs a = {};
  a.tma_store = tma_store ? 1 : 0;
  a.W0 = static_cast<const uint8_t*>(p.W0);
  a.W1 = static_cast<const uint8_t*>(p.W1);
  a.s0 = p.s0; a.b0 = p.b0; a.s1 = p.s1; a.b1 = p.b1;
  a.XgT = XgT;
  a.einv = BFW ? nullptr : einv;
  a.res = p.res;
  a.res_ld = p.res_ld;
  a.out = p.out;
  a.out_f32 = p.out_f32 ? 1 : 0;
  a.M = M; a.K = K; a.N = N; a.group = group;
  a.lg_group = 31 - __builtin_clz((unsigned)group);
  a.G = G;
  a.KB = K / PF_KB;
  a.row_bytes = SH::CB == 64 ? K : K / 2;
  a.n_ctiles = n_ctiles;
  a.Mp = Mp;
  a.ks = ks;
  a.KBs = ks > 1 ? kbs : K / PF_KB;
  a.part = part;
  a.err = err;

  mt_status st = MT_OK;
  if (!BFW) {  // bf16 weights take x as stored
    st = launch(prefill_x_kernel, dim3(Mp), dim3(256), 0, l, p.x, M, K, group, x16, XgT, einv);
    if (st != MT_OK) return st;
  }
  const size_t smem = SH::SMEM;
  auto kern = prefill_gemm_kernel<FMT, KIND, NT>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev >= 64 || !attr_set[dev]) {
      ce = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (ce != cudaSuccess) return cuda_fail(ce);
      if (dev < 64) attr_set[dev] = true;
    }
  }
  st = launch(kern, dim3((unsigned)(n_rtiles * n_ctiles * ks)), dim3(PF_THREADS), smem, l, xmap, wmap[0], wmap[1],
              omap, a);
  if (st != MT_OK || ks == 1) return st;
  const long total = (long)M * N;
  const unsigned fgrid = (unsigned)std::min<long>((total + 255) / 256, (long)di->sm_count * 16);
  return launch(prefill_finalize_kernel<KIND>, dim3(fgrid), dim3(256), 0, l, (const float*)part, ks, Mp,
                (const float*)a.einv, (const float*)nullptr, M, N, p.res, p.res_ld, p.out, p.out_f32 ? 1 : 0);
}

// The activation-row tile: the smallest of 64, 128, 256 that holds M (a
// narrow tile moves fewer x bytes through shared memory per K block).
template <int FMT, int KIND>
mt_status run_prefill_nt(const GemvProblem& p, void* ws, const Launch& l) {
  if (p.M <= 64) return run_prefill<FMT, KIND, 64>(p, ws, l);
  if (p.M <= 128) return run_prefill<FMT, KIND, 128>(p, ws, l);
  return run_prefill<FMT, KIND, 256>(p, ws, l);
}

}  // namespace mt
