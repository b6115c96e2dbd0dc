// Launchers of the quantiser kernels (host side, called by the C ABI layer).
#pragma once
#include <cuda.h>
#include "common.cuh"

namespace mpm {
cudaError_t launch_nvfp4_per_token(const void* x, long long M, int K, long long ldx,
                                   const float* amax_in, uint8_t* q, uint8_t* s, float* ts,
                                   const int* m_valid, cudaStream_t st);
cudaError_t launch_nvfp4_weight(const void* const* parts, const long long* part_rows, int nparts,
                                int K, long long E, uint8_t* q, uint8_t* s, float* ts,
                                unsigned* ws, cudaStream_t st);
// tile-by-tile NVFP4 with the running row amax (256-column tiles; K % 256
// == 0): codes, tiled block scales and one outer scale per (row, tile)
cudaError_t launch_nvfp4_online(const void* x, long long M, int K, long long ldx, uint8_t* q,
                                uint8_t* s, float* gs, const int* m_valid, cudaStream_t st);
// per-token NVFP4 of x [T, K] written into the expert-ordered rows (codes,
// tiled scales, outer scales; padding rows below *seg_end zeroed); ws holds
// nvfp4_scatter_ws_bytes(T, K) bytes (4-byte aligned)
size_t nvfp4_scatter_ws_bytes(long long T, int K);
cudaError_t launch_nvfp4_quantize_scatter(const void* x, long long T, int K, long long ldx,
                                          const int* inv, int k, const int* perm,
                                          const int* seg_end, long long cap, uint8_t* q,
                                          uint8_t* s, float* ts, float* amax_zero, void* ws,
                                          int* status, cudaStream_t st);
// x is read through a 2-D bf16 tensor map (box 64 columns x 128 rows); the
// codes of full tiles are stored through trow (row_q, box 64 x 128 bytes)
// and tcol (col_q, box 128 x 64 bytes, 128-byte swizzle)
cudaError_t launch_mxfp8_tma(const CUtensorMap& tx, const CUtensorMap& trow, const CUtensorMap& tcol,
                             long long M, long long K, long long ldx,
                             unsigned flags, uint8_t* row_q, uint8_t* row_s, uint8_t* col_q,
                             long long ldc, uint8_t* col_s, const int* m_valid, int* status,
                             cudaStream_t st);
// the same quantiser over the routed rows of x [T, K]: row r < *seg_end of
// the quantised matrix (cap rows) is token row perm[r] / k, a zero row where
// perm[r] < 0; the tiles are gathered by 16-byte copies instead of the
// tensor-map load
cudaError_t launch_mxfp8_gather(const CUtensorMap& trow, const CUtensorMap& tcol, const void* x,
                                long long T, long long K, long long ldx, const int* perm, int k,
                                const int* seg_end, long long cap, unsigned flags,
                                uint8_t* row_q, uint8_t* row_s, uint8_t* col_q, long long ldc,
                                uint8_t* col_s, int* status, cudaStream_t st);

}  // namespace mpm
