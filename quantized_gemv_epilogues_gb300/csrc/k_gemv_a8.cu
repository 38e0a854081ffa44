// k_gemv_a8.cu - instantiations of the GEMV kernels for one weight format
// (compiled as a separate translation unit to build in parallel).
#include "k_gemv_run.cuh"
#include "k_gemv_mma.cuh"
#include "k_gemv_warp.cuh"

namespace mt {

mt_status launch_gemv_a8(const GemvProblem& p, const Launch& l) {
  if (p.kind == Kind::GateUp) return dispatch_rows<FMT_A8, 0>(p, l);
  return dispatch_rows<FMT_A8, 1>(p, l);
}

}  // namespace mt
