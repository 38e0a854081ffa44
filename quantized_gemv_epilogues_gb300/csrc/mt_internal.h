// mt_internal.h - host-side declarations shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mt.h"

namespace mt {

// Per-device facts, queried once per device.
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;  // bytes of dynamic shared memory a CTA may opt into
};
const DeviceInfo* device_info(int* err);

// Launch configuration shared by the launchers.
struct Launch {
  cudaStream_t stream;
  bool pdl;
};

// Records a CUDA error for mt_last_cuda_error() and returns MT_ERR_CUDA.
mt_status cuda_fail(cudaError_t e);

// Device address of the library's device error word (set by kernels whose
// bounded waits expire); nullptr if it cannot be resolved.
int* device_error_ptr();

// Which GEMV kernel family to use for one-row problems (MT_OPT_GEMV).
int gemv_choice();

// Phantom arrivals the executor's grid barriers wait for
// (MT_OPT_TEST_BARRIER_EXTRA; 0 except in failure-detection tests).
int test_barrier_extra();

// MT_OPT_ACT_BITS: 16 or 24 (fixed-point activation bits for bf16 outputs).
int act_bits();

// Launches `kernel` with (grid, block, smem) on l.stream, adding the
// programmatic-stream-serialization attribute when l.pdl is set.
template <typename... KArgs, typename... Args>
mt_status launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, const Launch& l,
                 Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = l.pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  if (e != cudaSuccess) return cuda_fail(e);
  return MT_OK;
}

// ---- K1: add + RMSNorm
mt_status launch_add_rmsnorm(const uint16_t* v, const uint16_t* r, const uint16_t* w, float eps,
                             uint16_t* out_sum, void* out_norm, int M, int d, bool norm_f32,
                             const Launch& l);

// ---- K2 / K3: affine or bf16 GEMV with an epilogue
// GateUp: silu(x.Wg) * (x.Wu).  Down: x.W plus an optional addend (the residual
// of the down projection, or the bias of an attention or vocabulary projection).
enum class Kind { GateUp = 0, Down = 1 };

struct GemvProblem {
  Kind kind;
  int fmt;         // mt_wfmt
  int M, K, N;     // x is [M][K]; W is [N][K]; out is [M][N]
  int group;       // 0 for bf16
  const uint16_t* x;
  const void* W0;  // gate (GateUp) or down (Down)
  const void* W1;  // up (GateUp) or nullptr
  const uint16_t* s0;
  const uint16_t* b0;
  const uint16_t* s1;
  const uint16_t* b1;
  const uint16_t* res;  // Down: residual [M][N], or a bias [N] (res_ld 0), or nullptr
  int res_ld;           // elements between rows of res: N for a residual, 0 for a bias
  void* out;
  bool out_f32;
};

mt_status launch_gemv(const GemvProblem& p, const Launch& l);

// ---- packer
mt_status launch_pack_affine(const float* W, int N, int K, int group, int bits, uint8_t* q,
                             uint16_t* s, uint16_t* b, const Launch& l);
mt_status launch_pack_mx(const float* W, int N, int K, int bits, uint8_t* q, uint8_t* s,
                         const Launch& l);
mt_status launch_unpack_affine(const uint8_t* q, const uint16_t* s, const uint16_t* b, int N,
                               int K, int group, int bits, float* W, const Launch& l);

}  // namespace mt
