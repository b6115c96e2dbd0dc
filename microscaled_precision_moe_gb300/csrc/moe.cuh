// Launchers of the expert segment / gather / combine kernels.
#pragma once
#include "common.cuh"

namespace mpm {
size_t segments_ws_bytes(long long T, int k, long long E);
cudaError_t launch_build_segments(const int* ids, const float* prob, long long T, int k,
                                  long long E, int pad, int* seg_offsets, int* perm,
                                  int* inv_perm, float* row_prob, long long cap, void* ws,
                                  int* st, cudaStream_t s);
cudaError_t launch_gather(int what, const void* src, const uint8_t* src_s, const float* src_ts,
                          long long K, int k, const int* perm, const int* seg_end,
                          long long cap, void* dst, uint8_t* dst_s, float* dst_ts,
                          float* amax_zero, cudaStream_t s);
cudaError_t launch_combine(const void* y, const int* inv, long long T, int k, long long H,
                           void* out, cudaStream_t s);
}  // namespace mpm
