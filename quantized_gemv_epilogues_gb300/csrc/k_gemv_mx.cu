// k_gemv_mx.cu - instantiations of the GEMV for MX block-scaled weights
// (MXFP8: E4M3 elements, MXFP4: E2M1 elements, one E8M0 scale per 32 along
// K), every row count on the tensor-core kernel.
//
// meTile docs, "MLX-LM Backend", Block-Scaled MLX Primitive (E8M0 scale
// decode and E2M1 / E4M3 value decode composed into the matmul; BF16 inputs
// and outputs with FP32 accumulation).
#include "k_gemv_mma.cuh"

namespace mt {

mt_status launch_gemv_mx8(const GemvProblem& p, const Launch& l) {
  if (p.kind == Kind::GateUp) return dispatch_mma<FMT_MX8, 0>(p, l);
  return dispatch_mma<FMT_MX8, 1>(p, l);
}

mt_status launch_gemv_mx4(const GemvProblem& p, const Launch& l) {
  if (p.kind == Kind::GateUp) return dispatch_mma<FMT_MX4, 0>(p, l);
  return dispatch_mma<FMT_MX4, 1>(p, l);
}

}  // namespace mt
