// Launchers of the dequantisation and transpose kernels (host side, called by
// the C ABI layer).
#pragma once
#include "common.cuh"

namespace mpm {
cudaError_t launch_nvfp4_dequant(const uint8_t* q, const uint8_t* s, const float* outer,
                                 long long rows_per_outer, long long M, int K, void* out,
                                 long long ldo, const int* m_valid, cudaStream_t st);
cudaError_t launch_mxfp8_dequant(const uint8_t* q, const uint8_t* s, long long M, int K, void* out,
                                 long long ldo, const int* m_valid, cudaStream_t st);
cudaError_t launch_transpose_bf16(const void* in, long long R, long long C, long long ldi, void* out,
                                  long long ldo, const int* m_valid, cudaStream_t st);
}  // namespace mpm
