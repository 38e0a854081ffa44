// k_stack.cu - the warmed decode-MLP executor: L one-row layers
//   summed_l = values_l + r_l, x_l = rms_norm(summed_l), h_l = silu(x_l Wg^T) * (x_l Wu^T),
//   y_l = h_l Wd^T + summed_l, r_{l+1} = y_l
// run by ONE persistent cooperative kernel.
//
// meTile docs, "Compute-Graph Fusion", Automatic Gated Epilogues (the gate/up
// stage with its SwiGLU epilogue and the down stage with its residual
// epilogue are combined into a warmed MLP executor that binds the selected
// stages once); "MLX-LM Backend", Dispatch Policy (residual add + RMSNorm
// with the summed residual kept as a second output; steady-state decode does
// not pass through a per-call wrapper).
//
// GB300 design.  The three single-call kernels of a layer each pay a launch,
// a prologue (x staging, scales) and a tail in which the SMs drain; with
// one CTA per SM, programmatic dependent launch cannot overlap them.  Here
// one CTA per SM stays resident for the whole stack and walks, per layer:
//   norm    every CTA rebuilds x_l = rms_norm(summed_l) for the whole vector
//           from summed_l and the per-CTA partial sums of squares,
//   gate/up the CTA's rows of Wg/Wu (warp-task phase, k_phase.cuh),
//           publishing its rows of h,
//   down    the CTA's rows of Wd with x = h; the epilogue adds the residual
//           and publishes its rows of summed_{l+1} = values_{l+1} + y_l and
//           their sum of squares.
// A hand-off between CTAs is a grid barrier split in two halves.  A CTA
// stores its rows (plain stores), passes a CTA barrier, and thread 0 adds
// the CTA's arrival to one counter with a release reduction (no reply is
// awaited); the CTA then requests what its next phase needs that does not
// depend on the hand-off, and thread 0 polls the counter with acquire loads
// until every CTA has arrived; after a second CTA barrier every thread reads
// the published rows from L2.  (Tagged per-word data polled by one warp per
// CTA measured about 2 us slower per hand-off on this two-die part than the
// single counter; letting every thread poll its own words flooded L2.)  The
// counter and an abort flag are zeroed before each run.  Every wait is
// bounded (~1 s): on expiry the thread records MT_ERR_TIMEOUT in the device
// error word and raises the abort flag that every other wait also watches,
// and every CTA returns.
//
// As soon as its task loop ends, a CTA asks L2 for the first rows of its
// next phase's weights with bulk (TMA) prefetches, and it stages that phase's
// scales, biases and RMSNorm gain during the current loop, so HBM keeps
// streaming while the hand-off completes.  x and h are staged in one pass with
// one fixed-point scale per vector: the gate/up CTAs publish the largest |h|
// of their rows next to h, and x's largest |x| is a CTA reduction.
#include <math.h>

#include <new>

#include "k_phase.cuh"

namespace mt {

constexpr int STACK_MAX_GRID = 256;  // CTAs (one per SM)
// Bytes of each weight stream a CTA asks L2 for before a phase: about what
// HBM delivers to one SM during a hand-off and the staging that follows.
constexpr int STACK_PRE_GATEUP = 64 * 1024;  // per gate and per up stream (swept: 0-192 KB)
constexpr int STACK_PRE_DOWN = 160 * 1024;   // (swept: 0-256 KB)

// One layer's device pointers.
struct StackLayerDev {
  const uint16_t* wn;  // RMSNorm gain [d]
  const uint8_t* Wg;
  const uint8_t* Wu;
  const uint8_t* Wd;
  const uint16_t* sg;
  const uint16_t* bg;
  const uint16_t* su;
  const uint16_t* bu;
  const uint16_t* sd;
  const uint16_t* bd;
};

// Run state (one 128-byte line, zeroed before every run).
struct StackCtl {
  unsigned count;  // barrier arrivals so far (barrier k completes at (k + 1) * grid)
  int abort;       // set when a wait expired
  int pad[30];
};

struct StackArgs {
  PhaseGeom gu, dn;
  const StackLayerDev* layers;
  int L, d, f;
  float eps;
  const uint16_t* values;    // [L][d]
  const uint16_t* residual;  // [d]
  uint16_t* out_y;           // [d]
  StackCtl* ctl;
  uint16_t* hbuf;  // [f]    h of the current layer
  uint16_t* sbuf;  // [d]    summed of the next layer
  float* ssq;      // [grid] per-CTA partial sums of squares of sbuf
  float* hmax;     // [grid] per-CTA largest |h| of its gate/up rows
  int* err;
  int pre_g, pre_d;   // bytes per weight stream asked of L2 ahead of a phase
  unsigned bar_extra; // arrivals a barrier waits for beyond the grid (0; > 0 only in tests)
  uint16_t* tr_sum;   // optional [L][d]
  uint16_t* tr_norm;  // optional [L][d]
  uint16_t* tr_h;     // optional [L][f]
  uint16_t* tr_y;     // optional [L][d]
  // shared-memory carve-up (byte offsets)
  int off_xs, off_tail_g, off_tail_d;
  int off_wn, off_ssm;
};

// ---- grid barrier halves

// Thread 0, right after a CTA barrier that follows the CTA's global stores.
__device__ __forceinline__ void grid_arrive(StackCtl* ctl) { red_release_gpu_add(&ctl->count, 1u); }

// Thread 0: polls until all CTAs have arrived at barrier k (bounded).  The
// caller follows with a CTA barrier that also spreads the verdict.
__device__ __forceinline__ bool grid_poll(StackCtl* ctl, unsigned k, unsigned extra, int* err) {
  const unsigned target = (k + 1) * gridDim.x + extra;
  if (ld_acquire_gpu(&ctl->count) >= target) return true;
  const long long t0 = clock64();
  for (unsigned spins = 1;; ++spins) {
    if (ld_acquire_gpu(&ctl->count) >= target) return true;
    if ((spins & 63u) == 0) {
      if (ld_relaxed_gpu(&ctl->abort)) return false;
      if (clock64() - t0 > (1ll << 31)) {
        atomicExch(&ctl->abort, 1);
        atomicExch(err, (int)MT_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ PhaseW gateup_w(const StackLayerDev& L) {
  PhaseW w;
  w.W0 = L.Wg; w.W1 = L.Wu;
  w.s0 = L.sg; w.b0 = L.bg; w.s1 = L.su; w.b1 = L.bu;
  return w;
}
__device__ __forceinline__ PhaseW down_w(const StackLayerDev& L) {
  PhaseW w;
  w.W0 = L.Wd; w.W1 = nullptr;
  w.s0 = L.sd; w.b0 = L.bd; w.s1 = nullptr; w.b1 = nullptr;
  return w;
}

// Sum over the CTA of one float per thread, in a fixed order; thread 0
// receives the total.  red: WARP_TASK_WARPS floats of shared memory, free on
// entry.
__device__ __forceinline__ float cta_sum(float v, float* red, int tid) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if ((tid & 31) == 0) red[tid >> 5] = v;
  __syncthreads();
  float t = 0.f;
  if (tid == 0)
    for (int w = 0; w < WARP_TASK_WARPS; ++w) t += red[w];
  return t;
}

__device__ __forceinline__ uint32_t pack2(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

// RSG: rows per load stream of the gate/up phase (a.gu.RS); the down phase
// always has one.  PL: bytes of the fixed-point x and h (every output of the
// executor, h and y, is bf16: 2 by default, 3 when MT_OPT_ACT_BITS is 24 at
// plan creation).
template <int FMT, int RSG, int PL>
__global__ void __launch_bounds__(WT_THREADS, 1) mlp_stack_kernel(const StackArgs a) {
  constexpr bool AFF = FmtTraits<FMT>::AFFINE;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int task_ctr;
  __shared__ float red[WARP_TASK_WARPS];
  __shared__ float vec_max;  // the staged vector's largest |value|, or its sum of squares
  __shared__ __align__(16) StackLayerDev lay_s[2];  // layers l and l + 1
  static_assert(sizeof(StackLayerDev) % 16 == 0, "layer table entries are copied in 16-byte units");
  constexpr int LAY_UNITS = (int)(sizeof(StackLayerDev) / 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int d = a.d, f = a.f;

  PhaseSmem smG, smD;
  smG.xraw = smD.xraw = reinterpret_cast<uint16_t*>(smem);
  smG.xs = smD.xs = reinterpret_cast<uint4*>(smem + a.off_xs);
  phase_tail_carve<FMT, 0>(a.gu, smem + a.off_tail_g, smG);
  phase_tail_carve<FMT, 1>(a.dn, smem + a.off_tail_d, smD);
  uint16_t* wn = reinterpret_cast<uint16_t*>(smem + a.off_wn);    // [d] RMSNorm gain
  uint16_t* ssm = reinterpret_cast<uint16_t*>(smem + a.off_ssm);  // [d] summed_l

  const PhaseCta cg = phase_cta<0, RSG>(a.gu, cta);
  const PhaseCta cd = phase_cta<1>(a.dn, cta);
  const uint64_t pol = l2_evict_first_policy();
  uint4 bufA[WT_NS][WT_CL], bufB[WT_NS][WT_CL];
  const int tA = warp, tB = warp + WARP_TASK_WARPS;
  unsigned nbar = 0;  // grid barriers passed

  // Copies layer l's pointer table entry into lay_s[l & 1] (cp.async; the
  // caller commits and waits).
  auto fetch_layer = [&](int l) {
    if (tid < LAY_UNITS && l < a.L)
      cp_async16(reinterpret_cast<uint4*>(&lay_s[l & 1]) + tid,
                 reinterpret_cast<const uint4*>(a.layers + l) + tid);
  };
  // Asks L2 for bytes [off, off + n) of the CTA's (contiguous) rows of W,
  // clipped to the rows: one bulk prefetch, issued by the calling thread.
  auto l2_range = [&](const PhaseGeom& g, const PhaseCta& c, const uint8_t* W, int off, int n) {
    const size_t all = (size_t)c.rows * g.row_bytes;
    if (n <= 0 || (size_t)off >= all) return;
    const size_t m = all - (size_t)off < (size_t)n ? all - (size_t)off : (size_t)n;
    bulk_prefetch_l2(W + (size_t)c.r_begin * g.row_bytes + off, (uint32_t)m);
  };
  // A phase's prefetch is split: the first three quarters are issued when the
  // previous task loop ends, the last quarter by thread 0 right after its
  // arrival at the barrier (the arrival's release fence waits for the CTA's
  // bulk prefetches in flight, so a smaller first part shortens it).
  constexpr int pre_g1 = (STACK_PRE_GATEUP * 3 / 4) & ~15, pre_d1 = (STACK_PRE_DOWN * 3 / 4) & ~15;
  // What a phase needs that does not depend on the hand-off is requested
  // early: its scales and biases and (gate/up) the RMSNorm gain go to shared
  // memory at the start of the PREVIOUS phase's task loop (stage_*_smem; the
  // copies are small next to the weight stream), and its first rows' weights
  // go to L2 with bulk prefetches as soon as the previous task loop ends
  // (prefetch_*; issued after the arrival or after the barrier, the hand-off
  // left HBM idle for longer).  lay_s[l & 1] must be complete and visible.
  // The caller commits the copies.
  auto stage_gateup_smem = [&](int l) {
    const StackLayerDev& Ly = lay_s[l & 1];
    if constexpr (AFF) stage_sb<0>(a.gu, gateup_w(Ly), cg, smG.sbr, tid, WT_THREADS);
    for (int i = tid; i < d / 8; i += WT_THREADS) cp_async16(wn + (size_t)i * 8, Ly.wn + (size_t)i * 8);
  };
  auto stage_down_smem = [&](int l) {
    const StackLayerDev& Ly = lay_s[l & 1];
    if constexpr (AFF) stage_sb<1>(a.dn, down_w(Ly), cd, smD.sbr, tid, WT_THREADS);
  };
  auto prefetch_gateup = [&](int l, int n) {
    const StackLayerDev& Ly = lay_s[l & 1];
    if (tid == 32) l2_range(a.gu, cg, Ly.Wg, 0, n);
    if (tid == 64) l2_range(a.gu, cg, Ly.Wu, 0, n);
  };
  auto prefetch_gateup_rest = [&](int l) {  // thread 0, after its arrival
    const StackLayerDev& Ly = lay_s[l & 1];
    l2_range(a.gu, cg, Ly.Wg, pre_g1, a.pre_g - pre_g1);
    l2_range(a.gu, cg, Ly.Wu, pre_g1, a.pre_g - pre_g1);
  };
  auto prefetch_down = [&](int l) {
    const StackLayerDev& Ly = lay_s[l & 1];
    if (tid == 32) l2_range(a.dn, cd, Ly.Wd, 0, pre_d1);
  };
  // Completes barrier nbar: thread 0 polls, then every thread learns the
  // verdict.  (Thread 0 issues no other loads between its arrival and here:
  // polls queued behind loads from HBM took microseconds longer.)
  auto grid_wait = [&]() -> bool {
    int ok = 1;
    if (tid == 0) ok = grid_poll(a.ctl, nbar, a.bar_extra, a.err) ? 1 : 0;
    ++nbar;
    return __syncthreads_and(ok) != 0;
  };
  // This CTA's rows of summed_l = values_l + r (bf16 sum of two bf16, one
  // rounding): pair j (rows 2j, 2j+1 of the CTA's down rows) is computed and
  // stored by thread j, its squares folded into the CTA's partial sum, which
  // thread 0 stores before arriving at the barrier.  r2: the pair of r.
  // next_l >= 0: thread 0 then asks L2 for the rest of that layer's gate/up
  // prefetch.
  auto publish_summed = [&](uint32_t v2, uint32_t r2, bool have, int next_l) {
    float ss = 0.f;
    if (have) {
      const uint16_t s0 = f2bf(bf16lo(v2) + bf16lo(r2));
      const uint16_t s1 = f2bf(bf16hi(v2) + bf16hi(r2));
      *reinterpret_cast<uint32_t*>(a.sbuf + cd.r_begin + 2 * tid) = pack2(s0, s1);
      ss = fmaf(bf16f(s0), bf16f(s0), bf16f(s1) * bf16f(s1));
    }
    ss = cta_sum(ss, red, tid);  // its CTA barrier orders the summed stores
    if (tid == 0) {
      a.ssq[cta] = ss;
      grid_arrive(a.ctl);
      if (next_l >= 0) prefetch_gateup_rest(next_l);
    }
  };

  const int npair_d = cd.rows >> 1, npair_g = cg.rows >> 1;

  // ---- prologue: layer 0's table entry and staging, summed_0
  fetch_layer(0);
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  {
    const bool have = tid < npair_d;
    uint32_t v2 = 0, r2 = 0;
    if (have) {
      v2 = *reinterpret_cast<const uint32_t*>(a.values + cd.r_begin + 2 * tid);
      r2 = *reinterpret_cast<const uint32_t*>(a.residual + cd.r_begin + 2 * tid);
    }
    publish_summed(v2, r2, have, -1);
  }
  prefetch_gateup(0, a.pre_g);  // all of it: nothing waits on this arrival's fence
  if (warp > 0) stage_gateup_smem(0);
  cp_async_commit();
  if (!grid_wait()) { cp_async_wait_all(); return; }
  if (warp == 0) stage_gateup_smem(0);  // warp 0's share, after its polls
  cp_async_commit();

  for (int l = 0; l < a.L; ++l) {
    const StackLayerDev& Ly = lay_s[l & 1];
    fetch_layer(l + 1);  // waited for below
    cp_async_commit();
    // values_{l+1} of this thread's pair of down rows, for the down epilogue
    uint32_t vnx = 0;
    if (l + 1 < a.L && tid < npair_d)
      vnx = *reinterpret_cast<const uint32_t*>(a.values + (size_t)(l + 1) * d + cd.r_begin + 2 * tid);

    // ---- add + RMSNorm of the whole vector (every CTA)
    {
      const int nu = d / 8;  // x units of 8 elements
      // the per-CTA partial sums of squares (warp 0 reads them, in one fixed
      // order; read by every warp they piled up on a few L2 lines) and this
      // thread's first two units of summed_l
      float tot = 0.f;
      if (warp == 0) {
        float q[STACK_MAX_GRID / 32];
#pragma unroll
        for (int k = 0; k < STACK_MAX_GRID / 32; ++k) {
          const int i = lane + 32 * k;
          q[k] = i < (int)gridDim.x ? ldg_cg_f32(a.ssq + i) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < STACK_MAX_GRID / 32; ++k) tot += q[k];
      }
      uint4 u0 = make_uint4(0, 0, 0, 0), u1 = u0;
      if (tid < nu) u0 = ldg_cg(a.sbuf + (size_t)tid * 8);
      if (tid + WT_THREADS < nu) u1 = ldg_cg(a.sbuf + (size_t)(tid + WT_THREADS) * 8);
      if (warp == 0) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
        if (lane == 0) vec_max = tot;
      }
      cp_async_wait_all();
      __syncthreads();  // the sum of squares, the RMSNorm gain, the scales and the next table entry
      const float inv = rsqrtf(vec_max / (float)d + a.eps);
      // x = bf16(summed * inv * w) into xraw, unit by unit, and its largest |x|
      float m = 0.f;
      auto norm_unit = [&](int i, const uint4 sv) {
        const uint4 w = reinterpret_cast<const uint4*>(wn)[i];
        const uint32_t* sp = &sv.x;
        const uint32_t* wp = &w.x;
        uint4 o;
        uint32_t* op = &o.x;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = bf16lo(sp[j]) * inv * bf16lo(wp[j]);
          const float hi = bf16hi(sp[j]) * inv * bf16hi(wp[j]);
          op[j] = pack2(f2bf(lo), f2bf(hi));
        }
        reinterpret_cast<uint4*>(ssm)[i] = sv;
        reinterpret_cast<uint4*>(smG.xraw)[i] = o;
        m = fmaxf(m, unit_absmax(o));
      };
      if (tid < nu) norm_unit(tid, u0);
      if (tid + WT_THREADS < nu) norm_unit(tid + WT_THREADS, u1);
      for (int i = tid + 2 * WT_THREADS; i < nu; i += WT_THREADS)  // d > 8192
        norm_unit(i, ldg_cg(a.sbuf + (size_t)i * 8));
      if (tid == 0) task_ctr = 2 * WARP_TASK_WARPS;  // tasks 0..2W-1 are taken statically
      // the first gate/up task (mostly L2 hits after prefetch_gateup), in
      // flight while x is staged; the second is requested after the staging
      // (loads in flight slow the staging's shared-memory accesses)
      {
        const PhaseW w = gateup_w(Ly);
        wt_load<0, RSG>(a.gu, w, cg, tA, bufA, pol, lane);
        wt_prefetch<0, RSG>(a.gu, w, cg, tA + 2 * WARP_TASK_WARPS, lane);
      }
      // one staging pass with the vector's fixed-point scale
      int ex = 0;
      if constexpr (AFF) ex = fx_exponent<PL>(cta_max(m, red, tid));  // its barrier also publishes xraw
      else __syncthreads();
      const float xscale = exp2i(ex);
      for (int base = warp * 32; base < nu; base += WT_THREADS) {
        const int i = base + lane < nu ? base + lane : -1;
        x_stage_unit<FMT, PL>(a.gu, smG, i, i >= 0 ? reinterpret_cast<const uint4*>(smG.xraw)[i] : make_uint4(0, 0, 0, 0),
                          xscale, false);
      }
      x_set_scale<FMT>(a.gu, smG, ex, tid, WT_THREADS);
      __syncthreads();
      stage_down_smem(l);  // for the next phase, during this one's loop
      cp_async_commit();
      if (a.tr_sum || a.tr_norm)
        for (int rl = tid; rl < cd.rows; rl += WT_THREADS) {
          const int n = cd.r_begin + rl;
          if (a.tr_sum) a.tr_sum[(size_t)l * d + n] = ssm[n];
          if (a.tr_norm) a.tr_norm[(size_t)l * d + n] = smG.xraw[n];
        }
    }
    // ---- gate/up with the SwiGLU epilogue; h rows published in pairs
    {
      wt_load<0, RSG>(a.gu, gateup_w(Ly), cg, tB, bufB, pol, lane);
      wt_prefetch<0, RSG>(a.gu, gateup_w(Ly), cg, tB + 2 * WARP_TASK_WARPS, lane);
      wt_run<FMT, 0, PL, RSG>(a.gu, gateup_w(Ly), cg, smG, bufA, bufB, tA, tB, &task_ctr, pol, lane);
      __syncthreads();
      prefetch_down(l);  // HBM keeps streaming through the hand-off
      float hm = 0.f;
      for (int i0 = 0; i0 < 2 * npair_g; i0 += WT_THREADS) {  // one row per thread, pairs stored by lane pairs
        const int i = i0 + tid;
        const bool ok = i < 2 * npair_g;
        uint16_t hb = 0;
        if (ok) {
          const float g = row_total<2>(a.gu, smG.parts, i, 0);
          const float u = row_total<2>(a.gu, smG.parts, i, 1);
          hb = f2bf(g / (1.0f + expf(-g)) * u);
          hm = fmaxf(hm, fabsf(bf16f(hb)));
        }
        const uint16_t ho = (uint16_t)__shfl_down_sync(0xffffffffu, (uint32_t)hb, 1);
        if (ok && (i & 1) == 0) {
          *reinterpret_cast<uint32_t*>(a.hbuf + cg.r_begin + i) = pack2(hb, ho);
          if (a.tr_h) *reinterpret_cast<uint32_t*>(a.tr_h + (size_t)l * f + cg.r_begin + i) = pack2(hb, ho);
        }
      }
      hm = cta_max(hm, red, tid);  // its barrier also orders the h stores before the release
      if (tid == 0) {
        a.hmax[cta] = hm;
        grid_arrive(a.ctl);  // h and its largest |h| are published
        l2_range(a.dn, cd, Ly.Wd, pre_d1, a.pre_d - pre_d1);  // the rest of the down prefetch
      }
    }
    // ---- down
    {
      if (tid == 0) task_ctr = 2 * WARP_TASK_WARPS;
      if (!grid_wait()) { cp_async_wait_all(); return; }
      // h (every unit of a batch read before it is used) and the largest |h|
      // (warp 0 reads the per-CTA maxima); one staging pass per batch with
      // the vector's fixed-point scale
      const PhaseW w = down_w(Ly);
      const int nu = f / 8;
      constexpr int HB = 4;  // units per thread and batch: f <= 16384 in one batch
      float hm = 0.f;
      if (warp == 0)
        for (int i = lane; i < (int)gridDim.x; i += 32) hm = fmaxf(hm, ldg_cg_f32(a.hmax + i));
      int ex = 0;
      for (int base0 = warp * 32, batch = 0;; base0 += HB * WT_THREADS, ++batch) {
        uint4 hv[HB];
#pragma unroll
        for (int k = 0; k < HB; ++k) {
          const int i = base0 + k * WT_THREADS + lane;
          hv[k] = i < nu ? ldg_cg(a.hbuf + (size_t)i * 8) : make_uint4(0, 0, 0, 0);
        }
        if (batch == 0) {
          if (warp == 0) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, off));
            if (lane == 0) vec_max = hm;
          }
          __syncthreads();
          if constexpr (AFF) ex = fx_exponent<PL>(vec_max);
        }
        const float xscale = exp2i(ex);
#pragma unroll
        for (int k = 0; k < HB; ++k) {
          const int base = base0 + k * WT_THREADS;
          if (base < nu) x_stage_unit<FMT, PL>(a.dn, smD, base + lane < nu ? base + lane : -1, hv[k], xscale, true);
        }
        if (base0 + HB * WT_THREADS >= nu) break;
      }
      x_set_scale<FMT>(a.dn, smD, ex, tid, WT_THREADS);
      cp_async_wait_all();  // scales and biases (long complete)
      // the first two tasks (mostly L2 hits after prefetch_down), then the
      // staged h is published to the CTA
      wt_load<1>(a.dn, w, cd, tA, bufA, pol, lane);
      wt_load<1>(a.dn, w, cd, tB, bufB, pol, lane);
      wt_prefetch<1>(a.dn, w, cd, tA + 2 * WARP_TASK_WARPS, lane);
      wt_prefetch<1>(a.dn, w, cd, tB + 2 * WARP_TASK_WARPS, lane);
      __syncthreads();
      if (l + 1 < a.L) {  // the next gate/up phase's, during this loop
        stage_gateup_smem(l + 1);
        cp_async_commit();
      }
      wt_run<FMT, 1, PL>(a.dn, w, cd, smD, bufA, bufB, tA, tB, &task_ctr, pol, lane);
      __syncthreads();
      if (l + 1 < a.L) prefetch_gateup(l + 1, pre_g1);  // HBM keeps streaming through the hand-off
      // epilogue: y = h . Wd[n] + summed_l[n]; summed_{l+1} = values_{l+1} + y
      const bool last = l + 1 == a.L;
      const bool have = tid < npair_d;
      uint32_t y2 = 0;
      if (have) {
        uint16_t yb[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int n = cd.r_begin + 2 * tid + e;
          yb[e] = f2bf(row_total<1>(a.dn, smD.parts, 2 * tid + e, 0) + bf16f(ssm[n]));
        }
        y2 = pack2(yb[0], yb[1]);
        if (a.tr_y) *reinterpret_cast<uint32_t*>(a.tr_y + (size_t)l * d + cd.r_begin + 2 * tid) = y2;
        if (last) *reinterpret_cast<uint32_t*>(a.out_y + cd.r_begin + 2 * tid) = y2;
      }
      if (last) break;
      publish_summed(vnx, y2, have, l + 1);
      if (!grid_wait()) { cp_async_wait_all(); return; }
    }
  }
}

// ---------------------------------------------------------------- host side

struct StackPlanImpl {
  int dev;
  int L, d, f, group, fmt;
  float eps;
  int grid;
  size_t smem;
  StackArgs base;       // geometry, layer table, workspace and smem offsets
  void* alloc;          // device allocation owned by the plan
  void* run_state;      // what is zeroed before each run (the control line)
  size_t run_state_bytes;
  const void* kernel;   // mlp_stack_kernel<FMT, RSG, PL>
};

template <int FMT>
static bool plan_stack(StackPlanImpl* P, const DeviceInfo* di) {
  size_t pg = 0, pd = 0;
  const int grid = di->sm_count;
  if (grid > STACK_MAX_GRID) return false;
  StackArgs& a = P->base;
  // rows in pairs: every published word has one writer
  if (!plan_phase<FMT, 0>(P->d, P->f, P->group, grid, &a.gu, &pg, 2)) return false;
  if (!plan_phase<FMT, 1>(P->f, P->d, P->group, grid, &a.dn, &pd, 2, 1)) return false;
  if (a.dn.rows_alloc > 2 * WT_THREADS) return false;  // one pair of down rows per thread
  const int Kmax = P->d > P->f ? P->d : P->f;
  size_t off = (size_t)Kmax * 2;  // xraw
  a.off_xs = (int)off; off += xs_bytes<FMT, 3>(Kmax);  // room for either width
  a.off_tail_g = (int)off; off += pg;  // plan_phase's phase_tail_bytes (16-byte multiples)
  a.off_tail_d = (int)off; off += pd;
  a.off_wn = (int)off; off += (size_t)P->d * 2;
  a.off_ssm = (int)off; off += (size_t)P->d * 2;
  P->smem = off;
  P->grid = grid;
  P->kernel = a.gu.RS == 2 ? reinterpret_cast<const void*>(mlp_stack_kernel<FMT, 2, 2>)
                           : reinterpret_cast<const void*>(mlp_stack_kernel<FMT, 1, 2>);
  if constexpr (FmtTraits<FMT>::AFFINE)  // dense bf16 weights stage x as stored
    if (act_bits() == 24)
      P->kernel = a.gu.RS == 2 ? reinterpret_cast<const void*>(mlp_stack_kernel<FMT, 2, 3>)
                               : reinterpret_cast<const void*>(mlp_stack_kernel<FMT, 1, 3>);
  return true;
}

static bool is16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace mt

struct mt_mlp_plan {
  mt::StackPlanImpl impl;
};

using namespace mt;

extern "C" mt_status mt_mlp_plan_create(const mt_mlp_layer* layers, int L, int d, int f,
                                        int group, mt_wfmt fmt, float eps, mt_mlp_plan** plan) {
  if (!plan) return MT_ERR_NULL;
  *plan = nullptr;
  if (!layers) return MT_ERR_NULL;
  if (fmt != MT_W_BF16 && fmt != MT_W_AFFINE8 && fmt != MT_W_AFFINE4) return MT_ERR_FORMAT;
  if (L < 1 || L > 4096 || d < 8 || f < 8 || d > 32768 || f > 32768 || d % 8 || f % 8)
    return MT_ERR_SHAPE;
  if (!(eps >= 0.f) || !isfinite(eps)) return MT_ERR_SHAPE;
  if (fmt == MT_W_BF16) {
    if (group != 0) return MT_ERR_GROUP;
  } else {
    if (group != 32 && group != 64 && group != 128) return MT_ERR_GROUP;
    if (d % group || f % group) return MT_ERR_SHAPE;
  }
  const bool aff = fmt != MT_W_BF16;
  for (int l = 0; l < L; ++l) {
    const mt_mlp_layer& y = layers[l];
    if (!y.norm_weight || !y.Wg || !y.Wu || !y.Wd) return MT_ERR_NULL;
    if (aff && (!y.gu_scales || !y.gu_biases || !y.d_scales || !y.d_biases)) return MT_ERR_NULL;
    if (!is16(y.norm_weight) || !is16(y.Wg) || !is16(y.Wu) || !is16(y.Wd)) return MT_ERR_ALIGN;
    if (aff && (!is16(y.gu_scales) || !is16(y.gu_biases) || !is16(y.d_scales) || !is16(y.d_biases)))
      return MT_ERR_ALIGN;
  }
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  if (!di) return cuda_fail((cudaError_t)derr);

  StackPlanImpl P = {};
  cudaError_t ce = cudaGetDevice(&P.dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  P.L = L; P.d = d; P.f = f; P.group = aff ? group : 0; P.fmt = fmt; P.eps = eps;
  bool ok = false;
  if (fmt == MT_W_AFFINE8) ok = plan_stack<FMT_A8>(&P, di);
  else if (fmt == MT_W_AFFINE4) ok = plan_stack<FMT_A4>(&P, di);
  else ok = plan_stack<FMT_BF16>(&P, di);
  if (!ok) return MT_ERR_SHAPE;
  const size_t budget = (size_t)di->max_smem_optin - 1024;  // static smem and slack
  if (P.smem > budget) return MT_ERR_SHAPE;
  // the opt-in maximum, so that plans of different sizes never shrink it
  ce = cudaFuncSetAttribute(P.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
  if (ce != cudaSuccess) return cuda_fail(ce);
  int occ = 0;
  ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, P.kernel, WT_THREADS, P.smem);
  if (ce != cudaSuccess) return cuda_fail(ce);
  if (occ < 1) return MT_ERR_SHAPE;

  // device memory: [layer table | control line | ssq | hmax | sbuf | hbuf];
  // the control line is zeroed before each run
  const size_t tab = ((size_t)L * sizeof(StackLayerDev) + 127) / 128 * 128;
  const size_t o_ctl = tab, o_ssq = o_ctl + 128;
  const size_t o_hmax = o_ssq + ((size_t)P.grid * 4 + 127) / 128 * 128;
  const size_t o_sbuf = o_hmax + ((size_t)P.grid * 4 + 127) / 128 * 128;
  const size_t o_hbuf = o_sbuf + ((size_t)d * 2 + 127) / 128 * 128;
  const size_t total = o_hbuf + ((size_t)f * 2 + 127) / 128 * 128;
  StackLayerDev* host_tab = new (std::nothrow) StackLayerDev[L];
  if (!host_tab) return MT_ERR_SHAPE;
  for (int l = 0; l < L; ++l) {
    const mt_mlp_layer& y = layers[l];
    StackLayerDev& t = host_tab[l];
    t.wn = (const uint16_t*)y.norm_weight;
    t.Wg = (const uint8_t*)y.Wg; t.Wu = (const uint8_t*)y.Wu; t.Wd = (const uint8_t*)y.Wd;
    if (aff) {
      const size_t plane = (size_t)f * (d / group);
      t.sg = (const uint16_t*)y.gu_scales; t.su = t.sg + plane;
      t.bg = (const uint16_t*)y.gu_biases; t.bu = t.bg + plane;
      t.sd = (const uint16_t*)y.d_scales; t.bd = (const uint16_t*)y.d_biases;
    } else {
      t.sg = t.su = t.bg = t.bu = t.sd = t.bd = nullptr;
    }
  }
  void* mem = nullptr;
  ce = cudaMalloc(&mem, total);
  if (ce != cudaSuccess) { delete[] host_tab; return cuda_fail(ce); }
  ce = cudaMemcpy(mem, host_tab, (size_t)L * sizeof(StackLayerDev), cudaMemcpyHostToDevice);
  delete[] host_tab;
  if (ce == cudaSuccess) ce = cudaMemset(static_cast<char*>(mem) + o_ctl, 0, total - o_ctl);
  if (ce != cudaSuccess) { cudaFree(mem); return cuda_fail(ce); }
  int* err = device_error_ptr();
  if (!err) { cudaFree(mem); return cuda_fail(cudaErrorInvalidSymbol); }

  StackArgs& a = P.base;
  char* base = static_cast<char*>(mem);
  a.layers = reinterpret_cast<const StackLayerDev*>(base);
  a.ctl = reinterpret_cast<StackCtl*>(base + o_ctl);
  a.ssq = reinterpret_cast<float*>(base + o_ssq);
  a.hmax = reinterpret_cast<float*>(base + o_hmax);
  a.sbuf = reinterpret_cast<uint16_t*>(base + o_sbuf);
  a.hbuf = reinterpret_cast<uint16_t*>(base + o_hbuf);
  P.run_state = base + o_ctl;
  P.run_state_bytes = 128;
  a.L = L; a.d = d; a.f = f; a.eps = eps;
  a.pre_g = STACK_PRE_GATEUP;
  a.pre_d = STACK_PRE_DOWN;
  a.err = err;
  P.alloc = mem;

  mt_mlp_plan* out = new (std::nothrow) mt_mlp_plan;
  if (!out) { cudaFree(mem); return MT_ERR_SHAPE; }
  out->impl = P;
  *plan = out;
  return MT_OK;
}

extern "C" mt_status mt_mlp_plan_run(const mt_mlp_plan* plan, const void* values,
                                     const void* residual, void* out_y, const mt_mlp_trace* trace,
                                     void* stream) {
  if (!plan || !values || !residual || !out_y) return MT_ERR_NULL;
  const StackPlanImpl& P = plan->impl;
  if (!is16(values) || !is16(residual) || !is16(out_y)) return MT_ERR_ALIGN;
  StackArgs a = P.base;
  a.values = (const uint16_t*)values;
  a.residual = (const uint16_t*)residual;
  a.out_y = (uint16_t*)out_y;
  a.bar_extra = (unsigned)test_barrier_extra();
  if (trace) {
    a.tr_sum = (uint16_t*)trace->out_sum;
    a.tr_norm = (uint16_t*)trace->out_norm;
    a.tr_h = (uint16_t*)trace->h;
    a.tr_y = (uint16_t*)trace->y;
  }
  // out_y may equal residual; no other overlap among inputs and outputs
  const uintptr_t yb = (uintptr_t)out_y, ye = yb + (size_t)P.d * 2;
  auto hits = [&](const void* p, size_t n) {
    const uintptr_t b = (uintptr_t)p;
    return p && b < ye && yb < b + n;
  };
  if (hits(values, (size_t)P.L * P.d * 2)) return MT_ERR_ALIAS;
  if (hits(residual, (size_t)P.d * 2) && residual != out_y) return MT_ERR_ALIAS;
  if (trace) {
    const void* tr[4] = {trace->out_sum, trace->out_norm, trace->h, trace->y};
    const size_t tn[4] = {(size_t)P.L * P.d * 2, (size_t)P.L * P.d * 2, (size_t)P.L * P.f * 2,
                          (size_t)P.L * P.d * 2};
    for (int i = 0; i < 4; ++i) {
      if (tr[i] && !is16(tr[i])) return MT_ERR_ALIGN;
      if (hits(tr[i], tn[i])) return MT_ERR_ALIAS;
      const uintptr_t b = (uintptr_t)tr[i];
      const uintptr_t vb = (uintptr_t)values, rb = (uintptr_t)residual;
      if (tr[i] && ((b < vb + (size_t)P.L * P.d * 2 && vb < b + tn[i]) ||
                    (b < rb + (size_t)P.d * 2 && rb < b + tn[i])))
        return MT_ERR_ALIAS;
    }
  }
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  if (dev != P.dev) return cuda_fail(cudaErrorInvalidDevice);
  cudaStream_t s = (cudaStream_t)stream;
  ce = cudaMemsetAsync(P.run_state, 0, P.run_state_bytes, s);
  if (ce != cudaSuccess) return cuda_fail(ce);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid);
  cfg.blockDim = dim3(WT_THREADS);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  ce = cudaLaunchKernelExC(&cfg, P.kernel, args);
  if (ce != cudaSuccess) return cuda_fail(ce);
  return MT_OK;
}

extern "C" mt_status mt_mlp_plan_destroy(mt_mlp_plan* plan) {
  if (!plan) return MT_ERR_NULL;
  cudaError_t ce = cudaSuccess;
  if (plan->impl.alloc) ce = cudaFree(plan->impl.alloc);
  delete plan;
  if (ce != cudaSuccess) return cuda_fail(ce);
  return MT_OK;
}

// ------------------------------------------- the stack without any allocation
//
// mt_mlp_stack_run_noalloc runs the same kernel as mt_mlp_plan_run, but its
// layer table and hand-off words live in a file-scope static device array
// instead of memory a plan allocates.  It is for callers that cannot let the
// library allocate device memory: engines that reserve the device's memory up
// front for their own pool (a cudaMalloc by the library would fail, or carve
// memory out of a budget the engine has already planned) and code that must
// not synchronise the device (cudaMalloc and cudaFree may).  The array is
// shared by every call on a device, so calls that overlap in time race.
static __device__ __align__(256) unsigned char g_stack_scratch[MT_STACK_SCRATCH_BYTES];

namespace mt {

// The layer table reaches the device as kernel parameters: a launch copies
// its parameters when it is issued, so nothing on the host has to outlive the
// call and the upload can be captured into a CUDA graph (a cudaMemcpyAsync
// from pageable host memory can be neither).  48 entries of 80 bytes keep the
// parameter block under the classic 4 KB limit.
constexpr int TABLE_CHUNK = 48;
struct TableChunk {
  StackLayerDev t[TABLE_CHUNK];
};
static_assert(sizeof(StackLayerDev) % 8 == 0, "table entries copied as 8-byte words");
static_assert(sizeof(TableChunk) + 32 <= 4096, "table chunk within the parameter limit");

// Writes n entries of the chunk to dst and, when ctl is given, zeroes the
// control line (barrier counter, abort flag) that the stack kernel starts from.
__global__ void __launch_bounds__(256) stack_table_kernel(const TableChunk c, int n,
                                                          StackLayerDev* __restrict__ dst,
                                                          StackCtl* __restrict__ ctl) {
  constexpr int WPE = sizeof(StackLayerDev) / 8;
  const unsigned long long* src = reinterpret_cast<const unsigned long long*>(c.t);
  unsigned long long* out = reinterpret_cast<unsigned long long*>(dst);
  for (int i = threadIdx.x; i < n * WPE; i += blockDim.x) out[i] = src[i];
  if (ctl && threadIdx.x < (int)(sizeof(StackCtl) / 4)) reinterpret_cast<int*>(ctl)[threadIdx.x] = 0;
}

// Set-up done on every call, so that nothing cached outlives a
// cudaDeviceReset (which reloads the module at new addresses and drops the
// kernel's attributes): the scratch's device address and the kernel's
// shared-memory limit.  Neither call allocates or synchronises.
static mt_status noalloc_setup(const void* kernel, size_t smem_limit, void** scratch) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_stack_scratch);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_limit);
  if (e != cudaSuccess) return cuda_fail(e);
  *scratch = p;
  return MT_OK;
}

static size_t round128(size_t n) { return (n + 127) / 128 * 128; }

}  // namespace mt

extern "C" mt_status mt_mlp_stack_run_noalloc(const mt_mlp_layer* layers, int L, int d, int f,
                                              int group, mt_wfmt fmt, float eps,
                                              const void* values, const void* residual,
                                              void* out_y, void* stream) {
  // ---- arguments (nothing touches the device before these pass)
  if (!layers || !values || !residual || !out_y) return MT_ERR_NULL;
  if (fmt != MT_W_BF16 && fmt != MT_W_AFFINE8 && fmt != MT_W_AFFINE4) return MT_ERR_FORMAT;
  if (L < 1 || L > 4096 || d < 8 || f < 8 || d > 32768 || f > 32768 || d % 8 || f % 8)
    return MT_ERR_SHAPE;
  if (!(eps >= 0.f) || !isfinite(eps)) return MT_ERR_SHAPE;
  if (fmt == MT_W_BF16) {
    if (group != 0) return MT_ERR_GROUP;
  } else {
    if (group != 32 && group != 64 && group != 128) return MT_ERR_GROUP;
    if (d % group || f % group) return MT_ERR_SHAPE;
  }
  const bool aff = fmt != MT_W_BF16;
  for (int l = 0; l < L; ++l) {
    const mt_mlp_layer& y = layers[l];
    if (!y.norm_weight || !y.Wg || !y.Wu || !y.Wd) return MT_ERR_NULL;
    if (aff && (!y.gu_scales || !y.gu_biases || !y.d_scales || !y.d_biases)) return MT_ERR_NULL;
    if (!is16(y.norm_weight) || !is16(y.Wg) || !is16(y.Wu) || !is16(y.Wd)) return MT_ERR_ALIGN;
    if (aff && (!is16(y.gu_scales) || !is16(y.gu_biases) || !is16(y.d_scales) || !is16(y.d_biases)))
      return MT_ERR_ALIGN;
  }
  if (!is16(values) || !is16(residual) || !is16(out_y)) return MT_ERR_ALIGN;
  {
    const uintptr_t yb = (uintptr_t)out_y, ye = yb + (size_t)d * 2;
    const uintptr_t vb = (uintptr_t)values, ve = vb + (size_t)L * d * 2;
    const uintptr_t rb = (uintptr_t)residual, re = rb + (size_t)d * 2;
    if (vb < ye && yb < ve) return MT_ERR_ALIAS;
    if (rb < ye && yb < re && residual != out_y) return MT_ERR_ALIAS;
  }

  // ---- geometry (host arithmetic) and the scratch it needs
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  if (!di) return cuda_fail((cudaError_t)derr);
  StackPlanImpl P = {};
  cudaError_t ce = cudaGetDevice(&P.dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  P.L = L; P.d = d; P.f = f; P.group = aff ? group : 0; P.fmt = fmt; P.eps = eps;
  bool ok = false;
  if (fmt == MT_W_AFFINE8) ok = plan_stack<FMT_A8>(&P, di);
  else if (fmt == MT_W_AFFINE4) ok = plan_stack<FMT_A4>(&P, di);
  else ok = plan_stack<FMT_BF16>(&P, di);
  if (!ok) return MT_ERR_SHAPE;
  const size_t budget = (size_t)di->max_smem_optin - 1024;  // static smem and slack
  if (P.smem > budget) return MT_ERR_SHAPE;
  // scratch layout: [layer table | control line | ssq | hmax | sbuf | hbuf]
  const size_t o_ctl = round128((size_t)L * sizeof(StackLayerDev));
  const size_t o_ssq = o_ctl + 128;
  const size_t o_hmax = o_ssq + round128((size_t)P.grid * 4);
  const size_t o_sbuf = o_hmax + round128((size_t)P.grid * 4);
  const size_t o_hbuf = o_sbuf + round128((size_t)d * 2);
  const size_t total = o_hbuf + round128((size_t)f * 2);
  if (total > (size_t)MT_STACK_SCRATCH_BYTES) return MT_ERR_SHAPE;

  // ---- set-up, the table upload, then the launch
  void* scratch = nullptr;
  const mt_status st = noalloc_setup(P.kernel, budget, &scratch);
  if (st != MT_OK) return st;
  int occ = 0;
  ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, P.kernel, WT_THREADS, P.smem);
  if (ce != cudaSuccess) return cuda_fail(ce);
  if (occ < 1) return MT_ERR_SHAPE;
  int* err = device_error_ptr();
  if (!err) return cuda_fail(cudaErrorInvalidSymbol);
  cudaStream_t s = (cudaStream_t)stream;
  char* base = static_cast<char*>(scratch);
  for (int l0 = 0; l0 < L; l0 += TABLE_CHUNK) {
    TableChunk c;
    const int n = L - l0 < TABLE_CHUNK ? L - l0 : TABLE_CHUNK;
    for (int i = 0; i < n; ++i) {
      const mt_mlp_layer& y = layers[l0 + i];
      StackLayerDev& t = c.t[i];
      t.wn = (const uint16_t*)y.norm_weight;
      t.Wg = (const uint8_t*)y.Wg; t.Wu = (const uint8_t*)y.Wu; t.Wd = (const uint8_t*)y.Wd;
      if (aff) {
        const size_t plane = (size_t)f * (d / group);
        t.sg = (const uint16_t*)y.gu_scales; t.su = t.sg + plane;
        t.bg = (const uint16_t*)y.gu_biases; t.bu = t.bg + plane;
        t.sd = (const uint16_t*)y.d_scales; t.bd = (const uint16_t*)y.d_biases;
      } else {
        t.sg = t.su = t.bg = t.bu = t.sd = t.bd = nullptr;
      }
    }
    for (int i = n; i < TABLE_CHUNK; ++i) c.t[i] = StackLayerDev{};
    StackLayerDev* dst = reinterpret_cast<StackLayerDev*>(base) + l0;
    StackCtl* ctl = l0 == 0 ? reinterpret_cast<StackCtl*>(base + o_ctl) : nullptr;
    int cnt = n;
    void* targs[] = {&c, &cnt, &dst, &ctl};
    ce = cudaLaunchKernel((const void*)stack_table_kernel, dim3(1), dim3(256), targs, 0, s);
    if (ce != cudaSuccess) return cuda_fail(ce);
  }

  StackArgs a = P.base;
  a.layers = reinterpret_cast<const StackLayerDev*>(base);
  a.ctl = reinterpret_cast<StackCtl*>(base + o_ctl);
  a.ssq = reinterpret_cast<float*>(base + o_ssq);
  a.hmax = reinterpret_cast<float*>(base + o_hmax);
  a.sbuf = reinterpret_cast<uint16_t*>(base + o_sbuf);
  a.hbuf = reinterpret_cast<uint16_t*>(base + o_hbuf);
  a.L = L; a.d = d; a.f = f; a.eps = eps;
  a.err = err;
  a.pre_g = STACK_PRE_GATEUP;
  a.pre_d = STACK_PRE_DOWN;
  a.values = (const uint16_t*)values;
  a.residual = (const uint16_t*)residual;
  a.out_y = (uint16_t*)out_y;
  a.bar_extra = (unsigned)test_barrier_extra();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid);
  cfg.blockDim = dim3(WT_THREADS);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  ce = cudaLaunchKernelExC(&cfg, P.kernel, args);
  if (ce != cudaSuccess) return cuda_fail(ce);
  return MT_OK;
}
