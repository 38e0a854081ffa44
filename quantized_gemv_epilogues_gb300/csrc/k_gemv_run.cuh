// k_gemv_run.cuh - host-side plan of one GEMV launch: team size, grid and
// shared-memory layout for a (format, kind, rows) instantiation.
#pragma once
#include <atomic>
#include <mutex>

#include "k_gemv.cuh"

namespace mt {

// Occupancy queries are cached per (device, block, smem) for each kernel.
struct OccCache {
  std::mutex mu;
  struct E { int dev, block; size_t smem; int occ; } e[16];
  int n = 0, next = 0;
  int attr_set[64] = {0};
};

template <int FMT, int KIND, int MR, int R>
mt_status run_gemv(const GemvProblem& p, const Launch& l) {
  using T = FmtTraits<FMT>;
  constexpr int EPC = T::EPC;
  constexpr bool AFF = T::AFFINE;
  constexpr int NW = KIND == 0 ? 2 : 1;
  constexpr int V = R * NW * MR;
  constexpr bool FACTOR = AFF && MR == 1;
  static OccCache cache;

  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  int derr = 0;
  const DeviceInfo* di = device_info(&derr);
  if (!di) return cuda_fail((cudaError_t)derr);

  GemvArgs a = {};
  a.x = p.x;
  a.W0 = static_cast<const uint8_t*>(p.W0);
  a.W1 = static_cast<const uint8_t*>(p.W1);
  a.s0 = p.s0; a.b0 = p.b0; a.s1 = p.s1; a.b1 = p.b1;
  a.res = p.res;
  a.res_ld = p.res_ld;
  a.out = p.out;
  a.M = p.M; a.K = p.K; a.N = p.N;
  a.group = AFF ? p.group : 1;
  a.G = AFF ? p.K / p.group : 0;
  a.CPR = p.K / EPC;
  a.row_bytes = FMT == FMT_BF16 ? p.K * 2 : (FMT == FMT_A8 ? p.K : p.K / 2);
  a.out_f32 = p.out_f32 ? 1 : 0;

  // Team size: a multiple of 32 up to 256 that wastes the fewest chunk slots
  // (ties go to the larger team, i.e. fewer chunks per thread).
  int best_w = 1;
  long best_slots = -1;
  for (int w = 1; w <= 8; ++w) {
    const long ts = 32L * w;
    const long slots = ((a.CPR + ts - 1) / ts) * ts;
    if (best_slots < 0 || slots <= best_slots) { best_slots = slots; best_w = w; }
  }
  a.TS = 32 * best_w;
  a.CPT = (a.CPR + a.TS - 1) / a.TS;
  a.NT = 256 / a.TS;
  const int block = a.NT * a.TS;

  const size_t base_smem = (size_t)MR * p.K * 2 + (FACTOR ? (size_t)a.CPR * 4 : 0) +
                           (size_t)2 * (block / 32) * V * 4;
  const size_t sb_row_bytes = AFF ? (size_t)NW * a.G * 4 : 0;
  auto kern = gemv_kernel<FMT, KIND, MR, R>;

  auto occupancy = [&](size_t smem) -> int {
    std::lock_guard<std::mutex> g(cache.mu);
    for (int i = 0; i < cache.n; ++i)
      if (cache.e[i].dev == dev && cache.e[i].block == block && cache.e[i].smem == smem)
        return cache.e[i].occ;
    if (dev < 64 && !cache.attr_set[dev]) {
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di->max_smem_optin);
      cache.attr_set[dev] = 1;
    }
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, block, smem) != cudaSuccess)
      occ = 1;
    if (occ < 1) occ = 1;
    cache.e[cache.next] = {dev, block, smem, occ};
    cache.next = (cache.next + 1) % 16;
    if (cache.n < 16) ++cache.n;
    return occ;
  };

  // Grid: one wave of persistent CTAs (SMs x CTAs per SM), each owning a
  // contiguous row range.  The staged scales/biases grow with the rows of a
  // CTA, so the occupancy is evaluated with the final row count.
  const int N = p.N;
  int grid = di->sm_count;
  int occ = occupancy(base_smem + sb_row_bytes * (size_t)R *
                                      ((N + di->sm_count * 2 * R - 1) / (di->sm_count * 2 * R)));
  grid = di->sm_count * occ;
  const int min_rows = R * a.NT;
  if ((long)grid * min_rows > N) grid = (N + min_rows - 1) / min_rows;
  if (grid < 1) grid = 1;
  int rows_per = (N + grid - 1) / grid;
  const size_t budget = (size_t)di->max_smem_optin;
  if (base_smem + sb_row_bytes * (size_t)((rows_per + R - 1) / R * R) > budget) {
    if (sb_row_bytes == 0 || base_smem + sb_row_bytes * R > budget) return MT_ERR_SHAPE;
    const size_t per_row = sb_row_bytes ? sb_row_bytes : 1;  // nonzero here
    const int cap = (int)((budget - base_smem) / per_row) / R * R;
    grid = (N + cap - 1) / cap;
    rows_per = (N + grid - 1) / grid;
  }
  a.rows_base = N / grid;
  a.rows_extra = N % grid;
  a.sb_rows = AFF ? (rows_per + R - 1) / R * R : 0;
  const size_t smem = base_smem + sb_row_bytes * (size_t)a.sb_rows;
  if (smem > budget) return MT_ERR_SHAPE;
  (void)occupancy(smem);  // sets the smem attribute for this device if needed
  return launch(kern, dim3(grid), dim3(block), smem, l, a);
}

template <int FMT, int KIND>
mt_status run_gemv_warp(const GemvProblem& p, const Launch& l);
template <int FMT, int KIND>
mt_status dispatch_mma(const GemvProblem& p, const Launch& l);

// Chooses the kernel for one (format, kind) by MT_OPT_GEMV: 0 (default) the
// warp-task kernel for one row (and for two rows over affine INT8, where it
// measured faster than the tensor-core kernel) and the tensor-core kernel for
// more rows; 1 the team kernel for every M; 2 the tensor-core kernel for every
// M.  A shape that does not fit the chosen kernel's shared memory falls back
// to the team kernel by row count.
template <int FMT, int KIND>
mt_status dispatch_rows(const GemvProblem& p, const Launch& l) {
  const int choice = gemv_choice();
  if ((p.M == 1 || (p.M == 2 && FMT == FMT_A8)) && choice == 0) {
    const mt_status st = run_gemv_warp<FMT, KIND>(p, l);
    if (st != MT_ERR_SHAPE) return st;
  }
  if ((p.M > 1 && choice == 0) || choice == 2) {
    const mt_status st = dispatch_mma<FMT, KIND>(p, l);
    if (st != MT_ERR_SHAPE) return st;
  }
  if (p.M <= 1) return run_gemv<FMT, KIND, 1, 4>(p, l);
  if (p.M <= 2) return run_gemv<FMT, KIND, 2, 4>(p, l);
  if (p.M <= 4) return run_gemv<FMT, KIND, 4, 2>(p, l);
  return run_gemv<FMT, KIND, 8, 2>(p, l);
}

}  // namespace mt
