// The 3-bit variant: its pack (quant.cu), the 4-bit quantiser with levels
// 0..7 stored as three bit planes per 32 levels, and its decode matmul
// (gemv3.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace awq {

// planes: [N][K/32][3] uint32 -- word p of a 32-level block holds bit p of
// level i at bit i; scales, zeros: [N][K/128] fp16.
cudaError_t launch_pack_int3(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const float* s,
                             uint32_t* planes, uint16_t* scales, uint16_t* zeros, unsigned* status,
                             int num_sms, cudaStream_t st);

// Y[M,N] = X[M,K] deq(planes)^T for 1 <= M <= 16; X 16-byte aligned with
// ldx a multiple of 8.
cudaError_t launch_gemv_w3a16(const uint16_t* X, int64_t ldx, int M, const uint32_t* planes,
                              const uint16_t* scales, const uint16_t* zeros, int64_t N, int64_t K,
                              uint16_t* Y, int64_t ldy, int num_sms, cudaStream_t st);

}  // namespace awq
