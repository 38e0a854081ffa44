/*
 * synth_dev.cu - device fill kernels of the seeded input generator
 * (definition in synth_core.h).  Each element is computed from its index
 * alone, so the device values equal the host values bit for bit.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include "synth_core.h"

__global__ void syn_fill_f32_kernel(float* out, uint64_t n, uint64_t seed,
                                    uint64_t offset, float mean, float stdv,
                                    uint32_t p32, float oscale) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    out[j] = syn_value(seed, offset + j, mean, stdv, p32, oscale);
}

__global__ void syn_fill_bf16_kernel(uint16_t* out, uint64_t n, uint64_t seed,
                                     uint64_t offset, float mean, float stdv,
                                     uint32_t p32, float oscale) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    out[j] = syn_bf16(syn_value(seed, offset + j, mean, stdv, p32, oscale));
}

static unsigned syn_grid(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 152ull * 16ull) g = 152ull * 16ull;
  if (g == 0) g = 1;
  return (unsigned)g;
}

/* Returns the cudaError_t of the launch (0 on success). */
extern "C" int syn_fill_f32_device(float* out, uint64_t n, uint64_t seed,
                                   uint64_t offset, float mean, float stdv,
                                   uint32_t p32, float oscale, void* stream) {
  if (n == 0) return 0;
  syn_fill_f32_kernel<<<syn_grid(n), 256, 0, (cudaStream_t)stream>>>(
      out, n, seed, offset, mean, stdv, p32, oscale);
  return (int)cudaGetLastError();
}

extern "C" int syn_fill_bf16_device(uint16_t* out, uint64_t n, uint64_t seed,
                                    uint64_t offset, float mean, float stdv,
                                    uint32_t p32, float oscale, void* stream) {
  if (n == 0) return 0;
  syn_fill_bf16_kernel<<<syn_grid(n), 256, 0, (cudaStream_t)stream>>>(
      out, n, seed, offset, mean, stdv, p32, oscale);
  return (int)cudaGetLastError();
}
