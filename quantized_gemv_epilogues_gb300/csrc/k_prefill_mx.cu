// k_prefill_mx.cu - the prefill GEMMs (k_prefill.cuh) for MX block-scaled
// weights (MXFP8: E4M3, MXFP4: E2M1, E8M0 scales per 32), compiled as their
// own translation unit to build in parallel.
//
// meTile docs, "MLX-LM Backend", Block-Scaled MLX Primitive (E8M0 scale and
// E2M1 / E4M3 value decode composed into the matmul).
#include "k_prefill.cuh"

namespace mt {

mt_status launch_prefill_mx(const GemvProblem& p, void* ws, const Launch& l) {
  if (p.fmt == MT_W_MXFP8)
    return p.kind == Kind::GateUp ? run_prefill_nt<FMT_MX8, 0>(p, ws, l) : run_prefill_nt<FMT_MX8, 1>(p, ws, l);
  return p.kind == Kind::GateUp ? run_prefill_nt<FMT_MX4, 0>(p, ws, l) : run_prefill_nt<FMT_MX4, 1>(p, ws, l);
}

}  // namespace mt
