/*
 * synth_host.c - host fill routines of the seeded input generator
 * (definition in synth_core.h).  Built with gcc -O2 -ffp-contract=off.
 */
#include <stddef.h>
#include <stdint.h>
#include "synth_core.h"

void syn_fill_f32_host(float* out, uint64_t n, uint64_t seed, uint64_t offset,
                       float mean, float stdv, uint32_t outlier_p32,
                       float outlier_scale) {
  for (uint64_t j = 0; j < n; ++j)
    out[j] = syn_value(seed, offset + j, mean, stdv, outlier_p32, outlier_scale);
}

void syn_fill_bf16_host(uint16_t* out, uint64_t n, uint64_t seed,
                        uint64_t offset, float mean, float stdv,
                        uint32_t outlier_p32, float outlier_scale) {
  for (uint64_t j = 0; j < n; ++j)
    out[j] = syn_bf16(
        syn_value(seed, offset + j, mean, stdv, outlier_p32, outlier_scale));
}
