// Launch of the 3-bit pack (quant.cu): the 4-bit quantiser with levels 0..7,
// stored as three bit planes per 32 levels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace awq {

// planes: [N][K/32][3] uint32 -- word p of a 32-level block holds bit p of
// level i at bit i; scales, zeros: [N][K/128] fp16.
cudaError_t launch_pack_int3(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const float* s,
                             uint32_t* planes, uint16_t* scales, uint16_t* zeros, unsigned* status,
                             int num_sms, cudaStream_t st);

}  // namespace awq
