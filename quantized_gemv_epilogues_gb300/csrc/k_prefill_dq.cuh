// k_prefill_dq.cuh - the prefill GEMMs over affine INT8/INT4 weights with
// bf16 outputs: the weights dequantized into fp16 tiles before the
// tensor-core MMA, one accumulator over the whole K range.
//
// meTile docs, "MLX-LM Backend", Dispatch Policy (multi-row shapes run the
// quantised matmul as a tiled GEMM whose weight tiles are dequantised,
// w = scale * q + bias per group, into the activations' floating-point type
// before the matrix multiply, with fp32 accumulation); "Compute-Graph
// Fusion", Automatic Gated Epilogues (SwiGLU, residual and bias epilogues).
//
// GB300 design (against the exact-operand kernel of k_prefill.cuh, which
// keeps every quantisation group in its own tensor-memory sum and pays a
// per-group read-out of 128 fp32 columns per thread):
//  * A prepass (prefill_wscale_kernel) picks per weight row n a power of two
//    2^t_n with max_k |w[n,k]| 2^t_n below 2^15 (the bound taken over the
//    row's groups as |s| (2^b - 1) + |b|), so that every dequantised weight
//    is a normal or subnormal fp16 number.
//  * Warps 0-7 dequantise: each thread owns one weight row and 32 of its
//    codes per K block of 64, computes s 2^t q + b 2^t in fp32 (exact but
//    for one rounding) and rounds it to fp16 (relative error at most 2^-11,
//    3 bits finer than the bf16 tiles of the pages' kernels) into the MMA's
//    128-byte-swizzled K-major tile.  The scale and bias of each thread's
//    group arrive PQ_AHEAD K blocks ahead in registers.
//  * Warp 8 issues tcgen05.mma (M = 128, N = NT, K = 16) into ONE fp32
//    accumulator of NT tensor-memory columns for the whole K slice; warp 9
//    issues the TMA copies of the x tiles (lane 0) and code tiles (lane 1).
//  * After the last MMA, warps 0-7 read the accumulator in 16-column chunks,
//    undo 2^t_n and the activation row scale 2^e_m, and apply the epilogue:
//    gate/up write both halves to shared memory and all 256 threads form
//    silu(gate) * up; down / projection add the residual or bias.  The bf16
//    tile leaves by one TMA store.  With few tiles K is split into slices
//    whose fp32 sums prefill_finalize_kernel adds in slice order.
//  * Every mbarrier wait is bounded (~1 s) as in k_prefill.cuh.
#pragma once
#include "k_prefill.cuh"

namespace mt {

constexpr int PQ_CONV_WARPS = 8;                           // warps 0-7: dequantise, then the epilogue
constexpr int PQ_THREADS = 32 * (PQ_CONV_WARPS + 2);       // + warp 8: MMA, warp 9: TMA
constexpr int PQ_AHEAD = 4;                                // K blocks of scales/biases in flight

// Shared-memory plan: ring X (x tiles, TMA), ring C (code tiles, TMA),
// ring B (fp16 A tiles, written by the dequantising warps, read by the MMA).
// NA: 128-row A sub-tiles per tile, each with its own accumulator of NT
// columns; NA = 2 (with NT = 256) makes one x tile feed twice the MMAs, which
// halves the K-block overhead (waits, commits, TMA latency) per flop.
template <int FMT, int KIND, int NT, int NA = 1>
struct PqShape {
  static_assert(NA == 1 || (NA == 2 && NT == 256), "wide tiles take 256 activation rows");
  static constexpr int XT = NT * PF_KB * 2;
  static constexpr int FT = (KIND == 0 ? 64 : 128) * NA;  // output rows (gate/up: of h) per tile
  static constexpr int CB = FmtTraits<FMT>::EPW == 4 ? 64 : 32;
  static constexpr int CTILE = PF_ROWS * NA * CB;
  static constexpr int BTILE = PF_W_TILE * NA;             // one ring-B slot: NA sub-tiles
  static constexpr int SX = NA == 2 ? 3 : (NT == 256 ? 4 : (NT == 128 ? 6 : 8));
  static constexpr bool BFW = FMT == FMT_BF16;  // dense bf16 weights: no code ring (TMA fills ring B)
  static constexpr int SB = NA == 2 ? (BFW ? 3 : 2) : (BFW ? (NT == 256 ? 5 : 6) : (NT == 256 ? 3 : 4));
  static constexpr int SC0 = (217 * 1024 - SX * XT - SB * BTILE) / CTILE;
  static constexpr int SC = BFW ? 1 : (SC0 > 8 ? 8 : SC0);
  static constexpr size_t OFF_C = (size_t)SX * XT;
  static constexpr size_t OFF_B = OFF_C + (size_t)SC * CTILE;
  static constexpr size_t SMEM = 1024 + OFF_B + (size_t)SB * BTILE;
  // the final phase reuses the rings: narrow gate/up the gate and up sums
  // [NT][64] fp32 each and the bf16 tile [NT][64]; otherwise the bf16 tile
  // [NT][FT]
  static constexpr size_t FINAL = (KIND == 0 && NA == 1) ? (size_t)NT * 64 * 4 * 2 + (size_t)NT * 64 * 2
                                                         : (size_t)NT * FT * 2;
  static_assert(BFW || SC >= 2, "code ring");
  static_assert(SMEM <= 218 * 1024, "shared memory plan");
  static_assert(FINAL + 1024 <= SMEM, "final-phase buffers in the rings");
};

// One weight row's 2^t_n and 2^-t_n: warp per row, max over the row's groups
// of |s| qmax + |b| (a bound on |w|, in binary64 so that it cannot overflow
// for finite scales), t_n = 14 - floor(log2 max) clamped to [-126, 126] (0
// for an all-zero row, and for a row whose scales or biases are not finite:
// its weights are then infinite or NaN and so are its outputs, as in IEEE
// arithmetic).  Every row whose bound is at least 2^-112 is scaled into
// [2^14, 2^15); a smaller row is scaled by 2^126 and keeps full fp16
// precision for every weight above 2^-140.  Rows of both matrices: row
// index i in [0, NW * N), matrix i / N.
__global__ void __launch_bounds__(256) prefill_wscale_kernel(const uint16_t* __restrict__ s0,
                                                             const uint16_t* __restrict__ b0,
                                                             const uint16_t* __restrict__ s1,
                                                             const uint16_t* __restrict__ b1, int N, int G,
                                                             int NW, float qmax, float* __restrict__ tsc,
                                                             float* __restrict__ tinv) {
  const int lane = threadIdx.x & 31;
  const long row = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= (long)NW * N) return;
  const int mat = (int)(row / N), n = (int)(row - (long)mat * N);
  const uint16_t* sp = (mat ? s1 : s0) + (size_t)n * G;
  const uint16_t* bp = (mat ? b1 : b0) + (size_t)n * G;
  double m = 0.0;
  for (int g = lane; g < G; g += 32)
    m = fmax(m, fabs((double)bf16f(sp[g])) * (double)qmax + fabs((double)bf16f(bp[g])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmax(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) {
    int t = 0;
    if (m > 0.0 && isfinite(m)) {
      int e;
      (void)frexp(m, &e);  // m = f 2^e, f in [0.5, 1): floor(log2 m) = e - 1
      t = max(-126, min(126, 14 - (e - 1)));
    }
    tsc[row] = exp2i(t);
    tinv[row] = exp2i(-t);
  }
}

// Four codes of one 32-bit word (bytes 0..3) as floats q (exact): the byte
// placed under the exponent of 2^23, then 2^23 taken away.
__device__ __forceinline__ float pq_byte(uint32_t w, uint32_t sel) {
  return __uint_as_float(__byte_perm(w, 0x4B000000u, sel)) - 8388608.0f;
}

// Eight codes (two words) or the codes of one INT4 word, dequantised to
// one 16-byte chunk of fp16: w = fma(q, s, b) in fp32, rounded to fp16.
__device__ __forceinline__ uint4 pq_chunk8(uint32_t a, uint32_t b, float s, float c) {
  const float q[8] = {pq_byte(a, 0x7440), pq_byte(a, 0x7441), pq_byte(a, 0x7442), pq_byte(a, 0x7443),
                      pq_byte(b, 0x7440), pq_byte(b, 0x7441), pq_byte(b, 0x7442), pq_byte(b, 0x7443)};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __floats2half2_rn(fmaf(q[2 * i], s, c), fmaf(q[2 * i + 1], s, c));
    o[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}
// INT4: byte j of w holds code 2j (bits 0..3) and 2j+1 (bits 4..7)
__device__ __forceinline__ uint4 pq_chunk4(uint32_t w, float s, float c) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
  const uint32_t a = __byte_perm(lo, hi, 0x5140), b = __byte_perm(lo, hi, 0x7362);  // codes 0-3, 4-7
  return pq_chunk8(a, b, s, c);
}

template <int FMT, int KIND, int NT, int NA>
__global__ void __launch_bounds__(PQ_THREADS, 1)
    prefill_dq_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap0,
                      const __grid_constant__ CUtensorMap wmap1, const __grid_constant__ CUtensorMap omap,
                      const PrefillArgs a) {
  using SH = PqShape<FMT, KIND, NT, NA>;
  constexpr uint32_t TCOLS = (uint32_t)(NT * NA);  // tensor-memory columns: NA accumulators
  constexpr int SX = SH::SX, SC = SH::SC, SB = SH::SB, FT = SH::FT, CB = SH::CB;
  constexpr int EPI = 32 * PQ_CONV_WARPS;    // dequantising / epilogue threads
  constexpr int HALF = NT / 2;               // accumulator columns per epilogue warpgroup
  constexpr int MMA_WARP = PQ_CONV_WARPS, TMA_WARP = PQ_CONV_WARPS + 1;
  constexpr bool W8 = CB == 64;              // INT8 codes (else INT4)
  constexpr bool BFW = SH::BFW;              // dense bf16 weights: exact operands, no dequantising

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bars[2 * (SX + SC + SB) + 1];
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;
  __shared__ __align__(16) float einv_sh[NT];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x / a.ks, sk = blockIdx.x - tile * a.ks;
  const int rt = tile / a.n_ctiles, ct = tile - rt * a.n_ctiles;
  const int f0 = rt * FT, m0 = ct * NT;
  const int kb0 = sk * a.KBs, KB = min(a.KB - kb0, a.KBs);
  auto x_full = [&](int i) { return smem_u32(&bars[i]); };
  auto x_free = [&](int i) { return smem_u32(&bars[SX + i]); };
  auto c_full = [&](int i) { return smem_u32(&bars[2 * SX + i]); };
  auto c_free = [&](int i) { return smem_u32(&bars[2 * SX + SC + i]); };
  auto w_full = [&](int i) { return smem_u32(&bars[2 * (SX + SC) + i]); };
  auto b_free = [&](int i) { return smem_u32(&bars[2 * (SX + SC) + SB + i]); };
  const uint32_t acc_full = smem_u32(&bars[2 * (SX + SC + SB)]);
  auto xslot = [&](int i) { return smem + (size_t)i * SH::XT; };
  auto cslot = [&](int i) { return smem + SH::OFF_C + (size_t)i * SH::CTILE; };
  auto wslot = [&](int i) { return smem + SH::OFF_B + (size_t)i * SH::BTILE; };

  if (tid == 0) {
    for (int i = 0; i < SX; ++i) {
      mbar_init(x_full(i), 1);
      mbar_init(x_free(i), 1);
    }
    for (int i = 0; i < SC; ++i) {
      mbar_init(c_full(i), 1);
      mbar_init(c_free(i), PQ_CONV_WARPS);  // one arrival per dequantising warp
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(w_full(i), BFW ? 1 : PQ_CONV_WARPS);  // TMA (bf16 weights) or the dequantising warps
      mbar_init(b_free(i), 1);
    }
    mbar_init(acc_full, 1);
    abort_sh = 0;
    mbar_fence_init();
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_sh)),
                 "r"(TCOLS));
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
    // ---- producers: lane 0 the x tiles, lane 1 the code tiles
    if (lane < 2) {
      // bf16 weights: lane 1 fills ring B directly
      const int S = lane == 0 ? SX : (BFW ? SB : SC);
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int i = kb % S;
        const uint32_t full = lane == 0 ? x_full(i) : (BFW ? w_full(i) : c_full(i));
        const uint32_t free_ = lane == 0 ? x_free(i) : (BFW ? b_free(i) : c_free(i));
        if (kb >= S && !mbar_wait_bounded(free_, ((kb / S) + 1) & 1)) { fail(); break; }
        if (*abort_flag) break;
        const int kg = kb0 + kb;
        if (lane == 0) {
          mbar_arrive_expect_tx(full, SH::XT);
          tma_load_2d(smem_u32(xslot(i)), &xmap, kg * PF_KB, m0, full);
        } else if constexpr (BFW) {
          // gate/up: FT rows of each matrix, the up rows after the gate rows
          mbar_arrive_expect_tx(full, SH::BTILE);
          tma_load_2d(smem_u32(wslot(i)), &wmap0, kg * PF_KB, f0, full);
          if constexpr (KIND == 0) tma_load_2d(smem_u32(wslot(i) + FT * 128), &wmap1, kg * PF_KB, f0, full);
        } else {
          mbar_arrive_expect_tx(full, SH::CTILE);
          tma_load_2d(smem_u32(cslot(i)), &wmap0, kg * CB, f0, full);
          if constexpr (KIND == 0) tma_load_2d(smem_u32(cslot(i) + FT * CB), &wmap1, kg * CB, f0, full);
        }
        ++issued;
      }
      for (int kb = max(0, issued - S); kb < issued; ++kb)
        (void)mbar_wait_bounded(lane == 0 ? x_full(kb % S) : (BFW ? w_full(kb % S) : c_full(kb % S)), (kb / S) & 1);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ---- MMA issuer: one accumulator for the whole slice
    bool ok = true;
    for (int kb = 0; kb < KB; ++kb) {
      const int i = kb % SX, jb = kb % SB;
      // one decision for the whole warp (elect.sync below needs every lane)
      const bool got = mbar_wait_bounded(x_full(i), (kb / SX) & 1) && mbar_wait_bounded(w_full(jb), (kb / SB) & 1);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t xd = pf_desc_sw128(smem_u32(xslot(i)));
      if (elect_one()) {
#pragma unroll
        for (int sa = 0; sa < NA; ++sa) {  // sub-tile sa: A rows 128 sa .. 128 sa + 127, accumulator sa
          const uint64_t wd = pf_desc_sw128(smem_u32(wslot(jb) + sa * PF_W_TILE));
#pragma unroll
          for (int j = 0; j < PF_KB / 16; ++j)
            tc_mma<NT, BFW>(tbase + (uint32_t)(sa * NT), wd + 2 * j, xd + 2 * j, (kb | j) ? 1u : 0u);
        }
        tc_commit(b_free(jb));
        tc_commit(x_free(i));
      }
      __syncwarp();
      if (__any_sync(0xffffffffu, *abort_flag)) break;
    }
    if (!ok) fail();
    // completes when every MMA issued above has (also the epilogue's signal)
    if (elect_one()) tc_commit(acc_full);
    __syncwarp();
    (void)mbar_wait_bounded(acc_full, 0);
  } else {
    // ---- dequantising warps, then the epilogue.  Thread (r, h): row r of
    // each A sub-tile sa (tensor-memory lane r; tile row 128 sa + r), codes
    // [32 h, 32 h + 32) of each K block, and accumulator columns
    // [h * NT / 2, (h + 1) * NT / 2).  Narrow gate/up tiles stack 64 gate rows
    // over the same 64 up rows; wide ones put 128 gate rows in sub-tile 0 and
    // the same 128 up rows in sub-tile 1.
    const int r = tid & 127, h = tid >> 7;
    int mat[NA], n[NA];
    bool okr[NA];
    const uint16_t* sp[NA];
    const uint16_t* bp[NA];
    float tsc[NA];
#pragma unroll
    for (int sa = 0; sa < NA; ++sa) {
      mat[sa] = KIND == 0 ? (NA == 2 ? sa : (r >= 64 ? 1 : 0)) : 0;
      n[sa] = f0 + (KIND == 0 ? (NA == 2 ? r : (r & 63)) : 128 * sa + r);
      okr[sa] = n[sa] < a.N;
      sp[sa] = (mat[sa] ? a.s1 : a.s0) + (size_t)(okr[sa] ? n[sa] : 0) * a.G;
      bp[sa] = (mat[sa] ? a.b1 : a.b0) + (size_t)(okr[sa] ? n[sa] : 0) * a.G;
      tsc[sa] = (okr[sa] && !BFW) ? a.tsc[(size_t)mat[sa] * a.N + n[sa]] : 0.f;
    }
    // raw bf16 scale and bias of sub-tile sa's group in K block kb of the slice
    auto raw_s = [&](int sa, int kb) -> uint32_t {
      return (okr[sa] && !BFW && kb < KB) ? (uint32_t)__ldg(sp[sa] + (((kb0 + kb) * PF_KB + 32 * h) >> a.lg_group))
                                          : 0u;
    };
    auto raw_b = [&](int sa, int kb) -> uint32_t {
      return (okr[sa] && !BFW && kb < KB) ? (uint32_t)__ldg(bp[sa] + (((kb0 + kb) * PF_KB + 32 * h) >> a.lg_group))
                                          : 0u;
    };
    uint32_t sq[NA][PQ_AHEAD], bq[NA][PQ_AHEAD];
#pragma unroll
    for (int sa = 0; sa < NA; ++sa)
#pragma unroll
      for (int u = 0; u < PQ_AHEAD; ++u) {
        sq[sa][u] = raw_s(sa, u);
        bq[sa][u] = raw_b(sa, u);
      }
    bool ok = true;
    for (int kbu = 0; kbu < (BFW ? 0 : KB) && ok; kbu += PQ_AHEAD) {
#pragma unroll
      for (int u = 0; u < PQ_AHEAD; ++u) {
        const int kb = kbu + u;
        if (kb >= KB) break;
        const int i = kb % SC, j = kb % SB;
        float sv[NA], cv[NA];
#pragma unroll
        for (int sa = 0; sa < NA; ++sa) {
          sv[sa] = bf16f((uint16_t)sq[sa][u]) * tsc[sa];
          cv[sa] = bf16f((uint16_t)bq[sa][u]) * tsc[sa];
          sq[sa][u] = raw_s(sa, kb + PQ_AHEAD);
          bq[sa][u] = raw_b(sa, kb + PQ_AHEAD);
        }
        bool w = mbar_wait_bounded(c_full(i), (kb / SC) & 1);
        if (w && kb >= SB) w = mbar_wait_bounded(b_free(j), ((kb / SB) + 1) & 1);
        if (!__all_sync(0xffffffffu, w)) {
          fail();
          ok = false;
          break;
        }
        const unsigned char* ct = cslot(i);
#pragma unroll
        for (int sa = 0; sa < NA; ++sa) {
          const int R = 128 * sa + r;  // row of the code tile
          const float s_ = sv[sa], c_ = cv[sa];
          uint4 o[4];
          if constexpr (W8) {  // chunks 2h, 2h+1 of the 64-byte code row (64-byte swizzle)
            const int swc = (R >> 1) & 3;
            const uint4 v0 = *reinterpret_cast<const uint4*>(ct + R * 64 + (((2 * h) ^ swc) << 4));
            const uint4 v1 = *reinterpret_cast<const uint4*>(ct + R * 64 + (((2 * h + 1) ^ swc) << 4));
            o[0] = pq_chunk8(v0.x, v0.y, s_, c_);
            o[1] = pq_chunk8(v0.z, v0.w, s_, c_);
            o[2] = pq_chunk8(v1.x, v1.y, s_, c_);
            o[3] = pq_chunk8(v1.z, v1.w, s_, c_);
          } else {  // chunk h of the 32-byte code row (32-byte swizzle)
            const uint4 v = *reinterpret_cast<const uint4*>(ct + R * 32 + ((h ^ ((R >> 2) & 1)) << 4));
            o[0] = pq_chunk4(v.x, s_, c_);
            o[1] = pq_chunk4(v.y, s_, c_);
            o[2] = pq_chunk4(v.z, s_, c_);
            o[3] = pq_chunk4(v.w, s_, c_);
          }
          unsigned char* rowp = wslot(j) + sa * PF_W_TILE + r * 128;
#pragma unroll
          for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4*>(rowp + (((4 * h + k) ^ (r & 7)) << 4)) = o[k];
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor core reads
        __syncwarp();
        if (lane == 0) {  // one arrival per warp
          mbar_arrive(w_full(j));
          mbar_arrive(c_free(i));
        }
        if (__any_sync(0xffffffffu, *abort_flag)) {
          ok = false;
          break;
        }
      }
    }
    auto epi_sync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(EPI) : "memory"); };
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
    // (bf16 weights: x enters as stored, no row scales)
    for (int q = tid; q < NT; q += EPI) einv_sh[q] = BFW ? 1.0f : a.einv[m0 + q];  // padded rows hold 0
    bool aborted = epi_sync_or(!ok || *abort_flag);
    if (!aborted && !mbar_wait_bounded(acc_full, 0)) {
      fail();
      aborted = true;
    }
    aborted = epi_sync_or(aborted);
    if (!aborted) {
      tc_fence_after();
      const int wg = h, cbase = wg * HALF;
      const uint32_t lane_base = tbase + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)cbase;
      if constexpr (NA == 1) {
        const float ti = !okr[0] ? 0.f : (BFW ? 1.0f : a.tinv[(size_t)mat[0] * a.N + n[0]]);
        const float* ei = einv_sh + cbase;
        constexpr int NW = KIND == 0 ? 2 : 1;
        if (a.ks > 1) {
          // split K: this slice's sums of the tile, before any scaling
          // (every lane takes part in the warp-wide tensor-memory loads; only
          // rows inside the tensor store)
          float* pp = a.part + ((size_t)(sk * NW + mat[0]) * a.Mp + m0 + cbase) * a.N + (okr[0] ? n[0] : 0);
#pragma unroll 1
          for (int q = 0; q < HALF / 16; ++q) {
            float d[16];
            tc_ld16_wait(lane_base + (uint32_t)(q * 16), d);
            if (okr[0]) {
#pragma unroll
              for (int e = 0; e < 16; ++e) st_global_f32(pp + (size_t)(q * 16 + e) * a.N, d[e]);
            }
          }
        } else if constexpr (KIND == 0) {
          // gate and up sums [NT][64] each in shared memory, then silu(gate) * up
          // over the whole tile by all 256 threads
          float* gsh = reinterpret_cast<float*>(smem);
          float* ush = gsh + NT * 64;
          uint16_t* stg = reinterpret_cast<uint16_t*>(ush + NT * 64);
          float* dst = (mat[0] ? ush : gsh) + (r & 63);
#pragma unroll 1
          for (int q = 0; q < HALF / 16; ++q) {
            float d[16];
            tc_ld16_wait(lane_base + (uint32_t)(q * 16), d);
#pragma unroll
            for (int e = 0; e < 16; ++e) dst[(cbase + q * 16 + e) * 64] = d[e] * ti * ei[q * 16 + e];
          }
          epi_sync();
#pragma unroll 4
          for (int idx = tid; idx < NT * 64; idx += EPI) {
            const int col = idx >> 6, f = idx & 63;
            const float g = gsh[idx], hv = g / (1.0f + __expf(-g)) * ush[idx];  // silu(gate) * up
            if (a.tma_store) {
              stg[idx] = f2bf(hv);
            } else if (m0 + col < a.M && f0 + f < a.N) {
              const size_t o = (size_t)(m0 + col) * a.N + f0 + f;
              if (a.out_f32)
                st_global_f32(static_cast<float*>(a.out) + o, hv);
              else
                st_global_bf16(static_cast<uint16_t*>(a.out) + o, hv);
            }
          }
          if (a.tma_store) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // tile writes -> TMA reads
            epi_sync();
            if (tid == 0) tma_store_2d_wait(&omap, f0, m0, smem_u32(stg));
          }
        } else {
          // down / projection: + residual or bias, 16 columns at a time
          uint16_t* stg = reinterpret_cast<uint16_t*>(smem);  // [NT][128] bf16
          const uint16_t* __restrict__ res = a.res;
          const int jmax = min(HALF, a.M - m0 - cbase);
          const size_t obase = (size_t)(m0 + cbase) * a.N + n[0];
#pragma unroll 1
          for (int q = 0; q < HALF / 16; ++q) {
            float add[16], d[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int jj = q * 16 + e;
              add[e] = (res && okr[0] && jj < jmax) ? bf16f(__ldg(res + (size_t)(m0 + cbase + jj) * a.res_ld + n[0])) : 0.f;
            }
            tc_ld16_wait(lane_base + (uint32_t)(q * 16), d);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int jj = q * 16 + e;
              const float v = d[e] * ti * ei[jj] + add[e];
              if (a.tma_store) {
                stg[(cbase + jj) * FT + r] = f2bf(v);
              } else if (okr[0] && jj < jmax) {
                if (a.out_f32)
                  st_global_f32(static_cast<float*>(a.out) + obase + (size_t)jj * a.N, v);
                else
                  st_global_bf16(static_cast<uint16_t*>(a.out) + obase + (size_t)jj * a.N, v);
              }
            }
          }
          if (a.tma_store) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            epi_sync();
            if (tid == 0) tma_store_2d_wait(&omap, f0, m0, smem_u32(stg));
          }
        }
      } else {
        // wide tile: accumulator sa (columns sa * NT ...) holds sub-tile sa
        const float* ei = einv_sh + cbase;
        constexpr int NW = KIND == 0 ? 2 : 1;
        float ti[NA];
#pragma unroll
        for (int sa = 0; sa < NA; ++sa) ti[sa] = !okr[sa] ? 0.f : (BFW ? 1.0f : a.tinv[(size_t)mat[sa] * a.N + n[sa]]);
        if (a.ks > 1) {
          // split K: this slice's sums of the tile, before any scaling
#pragma unroll
          for (int sa = 0; sa < NA; ++sa) {
            float* pp = a.part + ((size_t)(sk * NW + mat[sa]) * a.Mp + m0 + cbase) * a.N + (okr[sa] ? n[sa] : 0);
#pragma unroll 1
            for (int q = 0; q < HALF / 16; ++q) {
              float d[16];
              tc_ld16_wait(lane_base + (uint32_t)(sa * NT + q * 16), d);
              if (okr[sa]) {
#pragma unroll
                for (int e = 0; e < 16; ++e) st_global_f32(pp + (size_t)(q * 16 + e) * a.N, d[e]);
              }
            }
          }
        } else if constexpr (KIND == 0) {
          // gate (accumulator 0) and up (accumulator 1) of the same row n:
          // silu(gate) * up in registers, into the bf16 tile [NT][FT]
          uint16_t* stg = reinterpret_cast<uint16_t*>(smem);
#pragma unroll 1
          for (int q = 0; q < HALF / 16; ++q) {
            float dg[16], du[16];
            tc_ld16_wait(lane_base + (uint32_t)(q * 16), dg);
            tc_ld16_wait(lane_base + (uint32_t)(NT + q * 16), du);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int col = cbase + q * 16 + e;
              const float g = dg[e] * ti[0] * ei[q * 16 + e], u = du[e] * ti[1] * ei[q * 16 + e];
              const float hv = g / (1.0f + __expf(-g)) * u;  // silu(gate) * up
              if (a.tma_store) {
                stg[col * FT + r] = f2bf(hv);
              } else if (m0 + col < a.M && okr[0]) {
                const size_t o = (size_t)(m0 + col) * a.N + n[0];
                if (a.out_f32)
                  st_global_f32(static_cast<float*>(a.out) + o, hv);
                else
                  st_global_bf16(static_cast<uint16_t*>(a.out) + o, hv);
              }
            }
          }
          if (a.tma_store) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // tile writes -> TMA reads
            epi_sync();
            if (tid == 0) tma_store_2d_wait(&omap, f0, m0, smem_u32(stg));
          }
        } else {
          // down / projection: + residual or bias, 16 columns at a time
          uint16_t* stg = reinterpret_cast<uint16_t*>(smem);  // [NT][FT] bf16
          const uint16_t* __restrict__ res = a.res;
          const int jmax = min(HALF, a.M - m0 - cbase);
#pragma unroll
          for (int sa = 0; sa < NA; ++sa) {
            const size_t obase = (size_t)(m0 + cbase) * a.N + n[sa];
#pragma unroll 1
            for (int q = 0; q < HALF / 16; ++q) {
              float add[16], d[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int jj = q * 16 + e;
                add[e] = (res && okr[sa] && jj < jmax)
                             ? bf16f(__ldg(res + (size_t)(m0 + cbase + jj) * a.res_ld + n[sa]))
                             : 0.f;
              }
              tc_ld16_wait(lane_base + (uint32_t)(sa * NT + q * 16), d);
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int jj = q * 16 + e;
                const float v = d[e] * ti[sa] * ei[jj] + add[e];
                if (a.tma_store) {
                  stg[(cbase + jj) * FT + 128 * sa + r] = f2bf(v);
                } else if (okr[sa] && jj < jmax) {
                  if (a.out_f32)
                    st_global_f32(static_cast<float*>(a.out) + obase + (size_t)jj * a.N, v);
                  else
                    st_global_bf16(static_cast<uint16_t*>(a.out) + obase + (size_t)jj * a.N, v);
                }
              }
            }
          }
          if (a.tma_store) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            epi_sync();
            if (tid == 0) tma_store_2d_wait(&omap, f0, m0, smem_u32(stg));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == MMA_WARP)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TCOLS));
}

// ---------------------------------------------------------------- host side

template <int FMT, int KIND, int NT, int NA>
mt_status run_prefill_dq(const GemvProblem& p, void* ws, const Launch& l) {
  constexpr int NW = KIND == 0 ? 2 : 1;
  using SH = PqShape<FMT, KIND, NT, NA>;
  constexpr bool BFW = SH::BFW;
  // (dense bf16 weights have no groups: group 0 in the workspace layout, and
  // K blocks of 64 stand in for them in the arguments)
  const int M = p.M, K = p.K, N = p.N, group = BFW ? PF_KB : p.group;
  const int n_ctiles = (M + NT - 1) / NT, Mp = (M + PF_COLS - 1) / PF_COLS * PF_COLS;
  const int n_rtiles = (N + SH::FT - 1) / SH::FT;
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  if (!di) return cuda_fail((cudaError_t)derr);
  unsigned char* w = static_cast<unsigned char*>(ws);
  const PfWs wl = prefill_ws_layout(M, K, N, p.group, di->sm_count);
  __half* x16 = reinterpret_cast<__half*>(w);
  float* XgT = reinterpret_cast<float*>(w + wl.xg);
  float* einv = reinterpret_cast<float*>(w + wl.einv);
  float* tsc = reinterpret_cast<float*>(w + wl.tw);
  float* tinv = tsc + 2 * (size_t)N;
  float* part = reinterpret_cast<float*>(w + wl.part);
  int kbs = 0;
  const int ks = prefill_ks((long)n_rtiles * n_ctiles, K, PF_KB, di->sm_count, &kbs);
  int* err = device_error_ptr();
  if (!err) return MT_ERR_CUDA;

  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cuda_fail(cudaErrorNotSupported);
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap xmap;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)PF_KB, (cuuint32_t)NT};
    // x: the fp16 rows of the workspace, or (bf16 weights) the bf16 input as stored
    if (enc(&xmap, BFW ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            BFW ? const_cast<uint16_t*>(p.x) : static_cast<void*>(x16), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cuda_fail(cudaErrorInvalidValue);
  }
  // code tiles: 64 (gate/up: of each matrix) or 128 rows x CB bytes, 64-byte
  // (INT8) or 32-byte (INT4) swizzle
  CUtensorMap wmap[2];
  for (int mat = 0; mat < 2; ++mat) {
    const void* W = (mat && NW == 2) ? p.W1 : p.W0;
    if constexpr (BFW) {  // the A tile itself: 64 elements (128 B) a row, 128-byte swizzle
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
    const cuuint32_t wbox[2] = {(cuuint32_t)SH::CB, (cuuint32_t)SH::FT};
    if (enc(&wmap[mat], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), wdims, wstr, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, SH::CB == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cuda_fail(cudaErrorInvalidValue);
  }
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
  a.G = K / group;
  a.KB = K / PF_KB;
  a.row_bytes = SH::CB == 64 ? K : K / 2;
  a.n_ctiles = n_ctiles;
  a.Mp = Mp;
  a.ks = ks;
  a.KBs = ks > 1 ? kbs : K / PF_KB;
  a.part = part;
  a.err = err;
  a.tsc = tsc;
  a.tinv = tinv;

  mt_status st = MT_OK;
  if (!BFW) {  // bf16 weights take x as stored and have no row scales
    st = launch(prefill_x_kernel, dim3(Mp), dim3(256), 0, l, p.x, M, K, group, x16, XgT, einv);
    if (st != MT_OK) return st;
    const float qmax = SH::CB == 64 ? 255.f : 15.f;
    st = launch(prefill_wscale_kernel, dim3((unsigned)((NW * (long)N + 7) / 8)), dim3(256), 0, l, p.s0, p.b0,
                NW == 2 ? p.s1 : p.s0, NW == 2 ? p.b1 : p.b0, N, K / group, NW, qmax, tsc, tinv);
    if (st != MT_OK) return st;
  }
  const size_t smem = SH::SMEM;
  auto kern = prefill_dq_kernel<FMT, KIND, NT, NA>;
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
  st = launch(kern, dim3((unsigned)(n_rtiles * n_ctiles * ks)), dim3(PQ_THREADS), smem, l, xmap, wmap[0], wmap[1],
              omap, a);
  if (st != MT_OK || ks == 1) return st;
  const long total = (long)M * N;
  const unsigned fgrid = (unsigned)std::min<long>((total + 255) / 256, (long)di->sm_count * 16);
  return launch(prefill_finalize_kernel<KIND>, dim3(fgrid), dim3(256), 0, l, (const float*)part, ks, Mp,
                (const float*)(BFW ? nullptr : einv), (const float*)(BFW ? nullptr : tinv), M, N, p.res, p.res_ld,
                p.out, p.out_f32 ? 1 : 0);
}

template <int FMT, int KIND>
mt_status run_prefill_dq_nt(const GemvProblem& p, void* ws, const Launch& l) {
  if (p.M <= 64) return run_prefill_dq<FMT, KIND, 64, 1>(p, ws, l);
  if (p.M <= 128) return run_prefill_dq<FMT, KIND, 128, 1>(p, ws, l);
  return run_prefill_dq<FMT, KIND, 256, 2>(p, ws, l);  // wide tiles: 256 weight rows
}

}  // namespace mt
