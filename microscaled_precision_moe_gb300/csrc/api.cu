// C ABI of libmpm: host-side validation and launch of the sm_103a kernels.
// Nothing here allocates device memory; every entry point validates its
// arguments before launching anything and returns an mpm_status.
#include <cuda.h>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "quant.cuh"
#include "moe.cuh"
#include "gemm.cuh"
#include "dequant.cuh"

namespace {

__device__ int g_status_word;

constexpr int kMaxDevices = 64;

int* status_ptr() {
  static int* ptrs[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

mpm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MPM_OK : MPM_ERR_CUDA; }

long long pad_to(long long v, long long m) { return (v + m - 1) / m * m; }

// segment paddings: 256 (CTA-pair tiles), 128 (one-CTA tiles), 16 / 32 / 64
// (the small-M kernel, which takes segments of any length)
bool valid_pad(int pad) { return pad == 16 || pad == 32 || pad == 64 || pad == 128 || pad == 256; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D uint8 tensor map over [rows, pitch bytes] with a 128 x 128 box and the
// 128-byte swizzle (the K-major operand layout of the MMA).
// box_rows = 64: the MN-major bf16 staging (128 bytes of M/N x 64 K rows).
bool make_tmap(CUtensorMap* m, const void* base, long long pitch, long long rows,
               unsigned box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)pitch, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)pitch};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D view of a 128x4-tiled scale buffer as [atoms, 128] 32-bit words (one
// 512-byte tile per row); a box of `atoms_per_box` consecutive tiles.
bool make_sf_tmap(CUtensorMap* m, const void* base, long long atoms, int atoms_per_box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)atoms};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, (cuuint32_t)atoms_per_box};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [rows, cols] bf16 input with row pitch `ld` elements, box_cols x box_rows
// boxes (rows land 2 * box_cols bytes apart in shared memory; a 128-byte wide
// box with the 128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r % 8));
// out-of-range elements read as zero
bool make_bf16_tmap(CUtensorMap* m, const void* base, long long cols, long long rows, long long ld,
                    unsigned box_cols, unsigned box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  box_cols * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [rows, cols] uint8 matrix with row pitch `ld` bytes, box_cols x box_rows
// boxes, optionally with the 128-byte swizzle (box_cols = 128): the code
// stores of the MXFP8 quantiser
bool make_u8_tmap(CUtensorMap* m, const void* base, long long cols, long long rows, long long ld,
                  unsigned box_cols, unsigned box_rows, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [rows, cols] bf16 or fp32 output with row pitch `ld` elements: 128-row boxes
// of 128 bytes per row (64 bf16 or 32 fp32 columns), 128-byte swizzle (the
// staging layout of the TMA-store epilogues)
bool make_out_tmap(CUtensorMap* m, const void* base, long long cols, long long rows, long long ld,
                   bool f32 = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int esz = f32 ? 4 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * esz)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / esz), 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

const char* mpm_status_string(int s) {
  switch (s) {
    case MPM_OK: return "MPM_OK";
    case MPM_ERR_NULL: return "MPM_ERR_NULL";
    case MPM_ERR_SHAPE: return "MPM_ERR_SHAPE";
    case MPM_ERR_ALIGN: return "MPM_ERR_ALIGN";
    case MPM_ERR_UNSUPPORTED: return "MPM_ERR_UNSUPPORTED";
    case MPM_ERR_CUDA: return "MPM_ERR_CUDA";
    case MPM_ERR_DEVICE_TIMEOUT: return "MPM_ERR_DEVICE_TIMEOUT";
    case MPM_ERR_DEVICE_BOUNDS: return "MPM_ERR_DEVICE_BOUNDS";
    default: return "MPM_ERR_UNKNOWN";
  }
}

int mpm_version(void) { return 101; }

size_t mpm_scale_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return (size_t)(pad_to(rows, 128) * pad_to(cols, 4));
}

mpm_status mpm_mxfp8_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, unsigned flags,
                              uint8_t* row_q, uint8_t* row_s, uint8_t* col_q, int64_t ldc,
                              uint8_t* col_s, const int32_t* m_valid, cudaStream_t stream) {
  if (!x) return MPM_ERR_NULL;
  if ((flags & (MPM_ROWWISE | MPM_COLWISE)) == 0 || (flags & ~3u)) return MPM_ERR_SHAPE;
  if (M < 1 || K < 32 || K % 32 != 0 || ldx < K) return MPM_ERR_SHAPE;
  if (M > (1ll << 31) - 256 || K > (1ll << 31) - 256) return MPM_ERR_SHAPE;
  if (!aligned(x, 16) || ldx % 8 != 0) return MPM_ERR_ALIGN;
  if (flags & MPM_ROWWISE) {
    if (!row_q || !row_s) return MPM_ERR_NULL;
    if (!aligned(row_q, 16)) return MPM_ERR_ALIGN;
  }
  if (flags & MPM_COLWISE) {
    if (!col_q || !col_s) return MPM_ERR_NULL;
    if (ldc < M) return MPM_ERR_SHAPE;
    if (!aligned(col_q, 16) || ldc % 16 != 0) return MPM_ERR_ALIGN;
  }
  CUtensorMap tx, trow, tcol;
  std::memset(&trow, 0, sizeof(trow));
  std::memset(&tcol, 0, sizeof(tcol));
  if (!make_bf16_tmap(&tx, x, K, M, ldx, 64, 128)) return MPM_ERR_CUDA;
  if ((flags & MPM_ROWWISE) && !make_u8_tmap(&trow, row_q, K, M, K, 64, 128, false))
    return MPM_ERR_CUDA;
  if ((flags & MPM_COLWISE) && !make_u8_tmap(&tcol, col_q, M, K, ldc, 128, 64, true))
    return MPM_ERR_CUDA;
  return cuda_status(mpm::launch_mxfp8_tma(tx, trow, tcol, M, K, ldx, flags, row_q, row_s, col_q,
                                           ldc, col_s, m_valid, status_ptr(), stream));
}

mpm_status mpm_mxfp8_quantize_gather(const void* x, int64_t T, int64_t K, int64_t ldx,
                                     const int32_t* perm, int k, const int32_t* seg, int64_t E,
                                     int64_t cap, unsigned flags, uint8_t* row_q, uint8_t* row_s,
                                     uint8_t* col_q, int64_t ldc, uint8_t* col_s,
                                     cudaStream_t stream) {
  if (!x || !perm || !seg) return MPM_ERR_NULL;
  if ((flags & (MPM_ROWWISE | MPM_COLWISE)) == 0 || (flags & ~3u)) return MPM_ERR_SHAPE;
  if (T < 1 || cap < 1 || E < 1 || k < 1 || k > 64) return MPM_ERR_SHAPE;
  if (K < 32 || K % 32 != 0 || ldx < K) return MPM_ERR_SHAPE;
  if (cap > (1ll << 31) - 256 || K > (1ll << 31) - 256 || T * k > (1ll << 31) - 1 ||
      ldx > (1ll << 31) - 1)
    return MPM_ERR_SHAPE;
  if (!aligned(x, 16) || ldx % 8 != 0) return MPM_ERR_ALIGN;
  if (flags & MPM_ROWWISE) {
    if (!row_q || !row_s) return MPM_ERR_NULL;
    if (!aligned(row_q, 16)) return MPM_ERR_ALIGN;
  }
  if (flags & MPM_COLWISE) {
    if (!col_q || !col_s) return MPM_ERR_NULL;
    if (ldc < cap) return MPM_ERR_SHAPE;
    if (!aligned(col_q, 16) || ldc % 16 != 0) return MPM_ERR_ALIGN;
  }
  CUtensorMap trow, tcol;
  std::memset(&trow, 0, sizeof(trow));
  std::memset(&tcol, 0, sizeof(tcol));
  if ((flags & MPM_ROWWISE) && !make_u8_tmap(&trow, row_q, K, cap, K, 64, 128, false))
    return MPM_ERR_CUDA;
  if ((flags & MPM_COLWISE) && !make_u8_tmap(&tcol, col_q, cap, K, ldc, 128, 64, true))
    return MPM_ERR_CUDA;
  return cuda_status(mpm::launch_mxfp8_gather(trow, tcol, x, T, K, ldx, perm, k, seg + E, cap,
                                              flags, row_q, row_s, col_q, ldc, col_s,
                                              status_ptr(), stream));
}

mpm_status mpm_nvfp4_quantize_per_token(const void* x, int64_t M, int64_t K, int64_t ldx,
                                        const float* amax_in, uint8_t* q, uint8_t* s,
                                        float* ts, const int32_t* m_valid,
                                        cudaStream_t stream) {
  if (!x || !q || !s || !ts) return MPM_ERR_NULL;
  if (M < 1 || K < 64 || K % 64 != 0 || K > 8192 || ldx < K) return MPM_ERR_SHAPE;
  if (M > (1ll << 31) - 256) return MPM_ERR_SHAPE;
  if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(q, 16) || !aligned(ts, 4)) return MPM_ERR_ALIGN;
  if (amax_in && !aligned(amax_in, 4)) return MPM_ERR_ALIGN;
  return cuda_status(mpm::launch_nvfp4_per_token(x, M, (int)K, ldx, amax_in, q, s, ts, m_valid,
                                                 stream));
}

mpm_status mpm_nvfp4_quantize_online(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                                     uint8_t* s, float* gs, const int32_t* m_valid,
                                     cudaStream_t stream) {
  if (!x || !q || !s || !gs) return MPM_ERR_NULL;
  if (M < 1 || K < 256 || K % 256 != 0 || K > 8192 || ldx < K) return MPM_ERR_SHAPE;
  if (M > (1ll << 31) - 256) return MPM_ERR_SHAPE;
  if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(q, 16) || !aligned(gs, 4)) return MPM_ERR_ALIGN;
  return cuda_status(mpm::launch_nvfp4_online(x, M, (int)K, ldx, q, s, gs, m_valid, stream));
}

size_t mpm_nvfp4_weight_workspace_bytes(int64_t E) {
  return E > 0 ? (size_t)pad_to(E * 4, 256) : 0;
}

mpm_status mpm_nvfp4_quantize_weight(const void* const* parts, const int64_t* part_rows,
                                     int nparts, int64_t K, int64_t E, uint8_t* q, uint8_t* s,
                                     float* ts, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!parts || !part_rows || !q || !s || !ts || !ws) return MPM_ERR_NULL;
  if (nparts < 1 || nparts > 4 || E < 1 || K < 64 || K % 64 != 0 || K > 8192) return MPM_ERR_SHAPE;
  long long R = 0;
  long long rows[4];
  for (int i = 0; i < nparts; ++i) {
    if (!parts[i]) return MPM_ERR_NULL;
    if (part_rows[i] < 1) return MPM_ERR_SHAPE;
    if (!aligned(parts[i], 16)) return MPM_ERR_ALIGN;
    rows[i] = part_rows[i];
    R += part_rows[i];
  }
  if (R % 128 != 0 || E * R > (1ll << 31) - 256) return MPM_ERR_SHAPE;
  if (ws_bytes < mpm_nvfp4_weight_workspace_bytes(E)) return MPM_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(ws, 4) || !aligned(ts, 4)) return MPM_ERR_ALIGN;
  return cuda_status(mpm::launch_nvfp4_weight(parts, rows, nparts, (int)K, E, q, s, ts,
                                              static_cast<unsigned*>(ws), stream));
}

int64_t mpm_moe_row_capacity(int64_t T, int k, int64_t E, int pad) {
  if (T < 1 || k < 1 || E < 1 || !valid_pad(pad)) return 0;
  return pad_to(T * k, pad) + (int64_t)pad * E;
}

size_t mpm_moe_segments_workspace_bytes(int64_t T, int k, int64_t E) {
  if (T < 1 || k < 1 || E < 1) return 0;
  return mpm::segments_ws_bytes(T, k, E);
}

mpm_status mpm_moe_build_segments(const int32_t* ids, const float* prob, int64_t T, int k,
                                  int64_t E, int pad, int32_t* seg, int32_t* perm, int32_t* inv,
                                  float* row_prob, void* ws, size_t ws_bytes,
                                  cudaStream_t stream) {
  if (!ids || !prob || !seg || !perm || !inv || !row_prob || !ws) return MPM_ERR_NULL;
  if (T < 1 || k < 1 || k > 64 || E < 1 || E > 1024) return MPM_ERR_SHAPE;
  if (!valid_pad(pad)) return MPM_ERR_SHAPE;
  if (T * k > (1ll << 30)) return MPM_ERR_SHAPE;
  if (ws_bytes < mpm::segments_ws_bytes(T, k, E)) return MPM_ERR_SHAPE;
  if (!aligned(ws, 4)) return MPM_ERR_ALIGN;
  return cuda_status(mpm::launch_build_segments(ids, prob, T, k, E, pad, seg, perm, inv,
                                                row_prob, mpm_moe_row_capacity(T, k, E, pad), ws,
                                                status_ptr(), stream));
}

mpm_status mpm_moe_gather(int what, const void* src, const uint8_t* src_s, const float* src_ts,
                          int64_t T, int64_t K, int k, const int32_t* perm, const int32_t* seg,
                          int64_t E, int64_t capacity, void* dst, uint8_t* dst_s,
                          float* dst_ts, float* amax_zero, cudaStream_t stream) {
  if (!src || !perm || !seg || !dst) return MPM_ERR_NULL;
  if (what != MPM_GATHER_BF16 && what != MPM_GATHER_NVFP4) return MPM_ERR_UNSUPPORTED;
  if (T < 1 || K < 64 || K % 64 != 0 || k < 1 || E < 1 || capacity < 1) return MPM_ERR_SHAPE;
  if (what == MPM_GATHER_NVFP4) {
    if (!src_s || !src_ts || !dst_s || !dst_ts) return MPM_ERR_NULL;
    if (!aligned(src_s, 4) || !aligned(dst_s, 4)) return MPM_ERR_ALIGN;
  }
  if (!aligned(src, 16) || !aligned(dst, 16)) return MPM_ERR_ALIGN;
  if (amax_zero && !aligned(amax_zero, 4)) return MPM_ERR_ALIGN;
  return cuda_status(mpm::launch_gather(what, src, src_s, src_ts, K, k, perm, seg + E, capacity,
                                        dst, dst_s, dst_ts, amax_zero, stream));
}

size_t mpm_nvfp4_quantize_scatter_workspace_bytes(int64_t T, int64_t K) {
  if (T < 1 || K < 64 || K % 64 != 0 || K > 8192) return 0;
  return mpm::nvfp4_scatter_ws_bytes(T, (int)K);
}

mpm_status mpm_nvfp4_quantize_scatter(const void* x, int64_t T, int64_t K, int64_t ldx,
                                      const int32_t* inv, int k, const int32_t* perm,
                                      const int32_t* seg, int64_t E, int64_t capacity,
                                      uint8_t* q, uint8_t* s, float* ts, float* amax_zero,
                                      void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!x || !inv || !perm || !seg || !q || !s || !ts || !ws) return MPM_ERR_NULL;
  if (T < 1 || K < 64 || K % 64 != 0 || K > 8192 || ldx < K || k < 1 || k > 64 || E < 1 ||
      capacity < 1)
    return MPM_ERR_SHAPE;
  if (T > (1ll << 31) - 256 || T * k > (1ll << 30)) return MPM_ERR_SHAPE;
  if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(q, 16) || !aligned(s, 4) || !aligned(ts, 4))
    return MPM_ERR_ALIGN;
  if (amax_zero && !aligned(amax_zero, 4)) return MPM_ERR_ALIGN;
  if (ws_bytes < mpm::nvfp4_scatter_ws_bytes(T, (int)K)) return MPM_ERR_SHAPE;
  if (!aligned(ws, 4)) return MPM_ERR_ALIGN;
  return cuda_status(mpm::launch_nvfp4_quantize_scatter(x, T, (int)K, ldx, inv, k, perm, seg + E,
                                                        capacity, q, s, ts, amax_zero, ws,
                                                        status_ptr(), stream));
}

mpm_status mpm_moe_combine(const void* y, const int32_t* inv, int64_t T, int k, int64_t H,
                           void* out, cudaStream_t stream) {
  if (!y || !inv || !out) return MPM_ERR_NULL;
  if (T < 1 || k < 1 || H < 8 || H % 8 != 0) return MPM_ERR_SHAPE;
  if (!aligned(y, 16) || !aligned(out, 16)) return MPM_ERR_ALIGN;
  return cuda_status(mpm::launch_combine(y, inv, T, k, H, out, stream));
}

mpm_status mpm_nvfp4_dequantize(const uint8_t* q, const uint8_t* s, const float* outer,
                                int64_t rows_per_outer, int64_t M, int64_t K, void* out,
                                int64_t ldo, const int32_t* m_valid, cudaStream_t stream) {
  if (!q || !s || !outer || !out) return MPM_ERR_NULL;
  if (M < 1 || K < 64 || K % 64 != 0 || K > (1LL << 30) || rows_per_outer < 1 || ldo < K ||
      ldo % 8 != 0)
    return MPM_ERR_SHAPE;
  if ((M + 3) / 4 > 0x7FFFFFFFLL) return MPM_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(s, 16) || !aligned(out, 16) || !aligned(outer, 4))
    return MPM_ERR_ALIGN;
  return cuda_status(mpm::launch_nvfp4_dequant(q, s, outer, rows_per_outer, M, (int)K, out, ldo,
                                               m_valid, stream));
}

mpm_status mpm_mxfp8_dequantize(const uint8_t* q, const uint8_t* s, int64_t M, int64_t K,
                                void* out, int64_t ldo, const int32_t* m_valid,
                                cudaStream_t stream) {
  if (!q || !s || !out) return MPM_ERR_NULL;
  if (M < 1 || K < 32 || K % 32 != 0 || K > (1LL << 30) || ldo < K || ldo % 8 != 0)
    return MPM_ERR_SHAPE;
  if ((M + 3) / 4 > 0x7FFFFFFFLL) return MPM_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(s, 16) || !aligned(out, 16)) return MPM_ERR_ALIGN;
  return cuda_status(mpm::launch_mxfp8_dequant(q, s, M, (int)K, out, ldo, m_valid, stream));
}

mpm_status mpm_transpose_bf16(const void* in, int64_t R, int64_t C, int64_t ldi, void* out,
                              int64_t ldo, const int32_t* m_valid, cudaStream_t stream) {
  if (!in || !out) return MPM_ERR_NULL;
  if (R < 1 || C < 1 || ldi < C || ldo < R) return MPM_ERR_SHAPE;
  if ((C + 63) / 64 > 0x7FFFFFFFLL || (R + 63) / 64 > 65535) return MPM_ERR_SHAPE;
  if (!aligned(in, 2) || !aligned(out, 2)) return MPM_ERR_ALIGN;
  return cuda_status(mpm::launch_transpose_bf16(in, R, C, ldi, out, ldo, m_valid, stream));
}

mpm_status mpm_moe_grouped_gemm(const mpm_grouped_gemm_desc* d, cudaStream_t stream) {
  if (!d) return MPM_ERR_NULL;
  if (d->kind != MPM_KIND_NVFP4 && d->kind != MPM_KIND_MXFP8 && d->kind != MPM_KIND_BF16)
    return MPM_ERR_UNSUPPORTED;
  const bool bf16 = d->kind == MPM_KIND_BF16;
  if (d->group != MPM_GROUP_M && d->group != MPM_GROUP_K) return MPM_ERR_UNSUPPORTED;
  const int tile_m = d->tile_m == 0 ? 128 : d->tile_m;
  if (tile_m != 128 && tile_m != 256 && tile_m != MPM_TILE_SMALL_M) return MPM_ERR_UNSUPPORTED;
  const bool small = tile_m == MPM_TILE_SMALL_M;
  if (small && (bf16 || d->group != MPM_GROUP_M ||
                (d->epilogue != MPM_EPI_F32 && d->epilogue != MPM_EPI_BF16 &&
                 d->epilogue != MPM_EPI_SWIGLU)))
    return MPM_ERR_UNSUPPORTED;
  if (tile_m == 256 && d->group == MPM_GROUP_K && d->a_rows % 256 != 0) return MPM_ERR_SHAPE;
  if (bf16 && tile_m != 256) return MPM_ERR_UNSUPPORTED;
  const int a_mn = d->a_mn_major ? 1 : 0, b_mn = d->b_mn_major ? 1 : 0;
  const int maj = a_mn | (b_mn << 1);
  if (maj != 0) {
    if (!bf16) return MPM_ERR_UNSUPPORTED;
    const bool ok_m = d->group == MPM_GROUP_M && maj == 2 &&
                      (d->epilogue == MPM_EPI_BF16 || d->epilogue == MPM_EPI_F32 ||
                       d->epilogue == MPM_EPI_DSWIGLU);
    const bool ok_k = d->group == MPM_GROUP_K && maj == 3 && d->epilogue == MPM_EPI_F32;
    if (!ok_m && !ok_k) return MPM_ERR_UNSUPPORTED;
  }
  if (d->epilogue < MPM_EPI_F32 || d->epilogue > MPM_EPI_BF16_ONLINE) return MPM_ERR_UNSUPPORTED;
  if (d->epilogue == MPM_EPI_BF16_ONLINE) {
    // FC2 of the single-pass FFN: NVFP4, CTA pairs, row segments only
    if (d->kind != MPM_KIND_NVFP4 || tile_m != 256 || d->group != MPM_GROUP_M || maj != 0)
      return MPM_ERR_UNSUPPORTED;
    if (!d->seg_dev || !d->aux_dev) return MPM_ERR_NULL;
    if (d->alpha_a_dev) return MPM_ERR_UNSUPPORTED;      // the outer scales are per tile, in aux
    if (d->K % 256 != 0 || d->ld_aux < d->K / 256) return MPM_ERR_SHAPE;
    if (!aligned(d->aux_dev, 4)) return MPM_ERR_ALIGN;
  }
  if (!d->a_dev || !d->b_dev || !d->out_dev) return MPM_ERR_NULL;
  if (!bf16 && (!d->sfa_dev || !d->sfb_dev)) return MPM_ERR_NULL;
  if (d->E < 1 || d->E > 65535 || d->N < 256 || d->N % 256 != 0 || d->a_rows < 1)
    return MPM_ERR_SHAPE;
  const bool swiglu = d->epilogue == MPM_EPI_SWIGLU || d->epilogue == MPM_EPI_SWIGLU_SAVE;
  const int elems_per_kb = d->kind == MPM_KIND_NVFP4 ? 256 : (bf16 ? 64 : 128);
  const int vec = d->kind == MPM_KIND_NVFP4 ? 16 : 32;
  if (d->group == MPM_GROUP_M) {
    if (d->K < elems_per_kb || d->K % elems_per_kb != 0) return MPM_ERR_SHAPE;
    if (!d->seg_dev && d->E != 1) return MPM_ERR_NULL;
    if (d->b_k_per_expert < 0 || d->b_k_per_expert % (d->kind == MPM_KIND_NVFP4 ? 64 : elems_per_kb))
      return MPM_ERR_SHAPE;
  } else {
    if (d->kind == MPM_KIND_NVFP4 || d->epilogue != MPM_EPI_F32) return MPM_ERR_UNSUPPORTED;
    if (!d->seg_dev) return MPM_ERR_NULL;
    if (d->a_rows % 128 != 0) return MPM_ERR_SHAPE;
  }
  if (d->b_rows_per_expert < 0 || d->b_rows_per_expert % 128 != 0) return MPM_ERR_SHAPE;
  if (d->a_total_rows < 1 || d->b_total_rows < 1) return MPM_ERR_SHAPE;
  if (d->lda_bytes < 128 || d->lda_bytes % 16 || d->ldb_bytes < 128 || d->ldb_bytes % 16)
    return MPM_ERR_ALIGN;
  if (!aligned(d->a_dev, 16) || !aligned(d->b_dev, 16) || !aligned(d->out_dev, 16))
    return MPM_ERR_ALIGN;
  if (!bf16) {
    if (!aligned(d->sfa_dev, 16) || !aligned(d->sfb_dev, 16)) return MPM_ERR_ALIGN;
    if (d->sfa_cols < 1 || d->sfb_cols < 1) return MPM_ERR_SHAPE;
  }
  if (d->group == MPM_GROUP_M) {
    // bytes = elems * this / 2
    const int bytes_per_elem2 = d->kind == MPM_KIND_NVFP4 ? 1 : (bf16 ? 4 : 2);
    if (d->K * bytes_per_elem2 / 2 > d->lda_bytes) return MPM_ERR_SHAPE;
    if (b_mn && 2 * d->N > d->ldb_bytes) return MPM_ERR_SHAPE;
    if (!bf16 && d->sfa_cols < d->K / vec) return MPM_ERR_SHAPE;
  }
  if (swiglu) {
    if (!d->out2_dev || !d->row_prob_dev) return MPM_ERR_NULL;
    if ((d->N / 2) % 128 != 0) return MPM_ERR_SHAPE;
    if (!aligned(d->out2_dev, 16) || d->ldo2 % 8 || d->ldo2 < d->N / 2) return MPM_ERR_ALIGN;
    if (d->epilogue == MPM_EPI_SWIGLU_SAVE && (d->ldo % 8 || d->ldo < d->N)) return MPM_ERR_ALIGN;
  } else if (d->epilogue == MPM_EPI_DSWIGLU) {
    if (!d->aux_dev || !d->row_prob_dev) return MPM_ERR_NULL;
    if (!aligned(d->aux_dev, 16) || d->ld_aux % 8 || d->ld_aux < 2 * d->N) return MPM_ERR_ALIGN;
    if (d->ldo % 8 || d->ldo < 2 * d->N) return MPM_ERR_ALIGN;
  } else {
    const int q = d->epilogue == MPM_EPI_F32 ? 4 : 8;
    if (d->ldo % q || d->ldo < d->N) return MPM_ERR_ALIGN;
  }

  if (d->group == MPM_GROUP_K && a_mn &&
      (2 * d->a_rows > d->lda_bytes || 2 * d->N > d->ldb_bytes))
    return MPM_ERR_SHAPE;

  CUtensorMap ta, tb;
  if (!make_tmap(&ta, d->a_dev, d->lda_bytes, d->a_total_rows, a_mn ? 64 : 128))
    return MPM_ERR_CUDA;
  if (!make_tmap(&tb, d->b_dev, d->ldb_bytes, d->b_total_rows, b_mn ? 64 : 128))
    return MPM_ERR_CUDA;

  mpm::GemmArgs a{};
  a.group = d->group;
  a.E = (int)d->E;
  a.a_rows = d->a_rows;
  a.N = d->N;
  a.K = d->K;
  a.M_out = d->a_rows;
  a.seg = d->seg_dev;
  a.b_rows_per_e = d->b_rows_per_expert;
  a.b_k_per_e = d->b_k_per_expert;
  a.sfa = d->sfa_dev; a.sfa_cols_pad = pad_to(d->sfa_cols, 4);
  a.sfb = d->sfb_dev; a.sfb_cols_pad = pad_to(d->sfb_cols, 4);
  a.alpha_a = d->alpha_a_dev;
  a.alpha_b = d->alpha_b_dev;
  a.row_prob = d->row_prob_dev;
  a.out = d->out_dev; a.ldo = d->ldo;
  a.out2 = d->out2_dev; a.ldo2 = d->ldo2;
  a.aux = d->aux_dev; a.ld_aux = d->ld_aux;
  a.amax = d->amax_dev;
  a.row_perm = d->row_perm_dev;
  a.status = status_ptr();

  if (small) {
    // weights (B) on the MMA's M side: 128-row weight tiles, 128-row chunks
    // of the routed rows (A) on its N side
    const long long n_out = d->epilogue == MPM_EPI_SWIGLU ? d->N / 2 : d->N;
    if (n_out % 128 != 0) return MPM_ERR_SHAPE;
    const int n_wt = (int)(n_out / 128);
    // one dense group of at most 128 rows (the single-expert GEMM): split K
    // over a cluster of CTAs per weight tile instead of giving only n_wt
    // CTAs the whole K chain
    const int nkb = (int)(d->K / elems_per_kb);
    if (!d->seg_dev && d->a_rows <= 128 && nkb >= 2 &&
        (d->epilogue == MPM_EPI_F32 || d->epilogue == MPM_EPI_BF16)) {
      int ks = 1;
      for (int c = 8; c >= 2; c >>= 1)
        if (nkb >= c) { ks = c; break; }
      return cuda_status(mpm::launch_gemm_splitk(d->kind, d->epilogue, ta, tb, a, n_wt, ks, stream));
    }
    const long long n_tasks = (long long)n_wt * ((d->a_rows + 127) / 128);
    return cuda_status(mpm::launch_grouped_gemm_small(d->kind, d->epilogue, ta, tb, a, n_wt, n_tasks,
                                                      stream));
  }
  if (d->epilogue == MPM_EPI_BF16_ONLINE) {
    CUtensorMap tb64, tsa, tsb, tout;
    if (!make_tmap(&tb64, d->b_dev, d->ldb_bytes, d->b_total_rows, 64)) return MPM_ERR_CUDA;
    const long long atoms_a = pad_to(d->a_total_rows, 128) * pad_to(d->sfa_cols, 4) / 512;
    const long long atoms_b = pad_to(d->b_total_rows, 128) * pad_to(d->sfb_cols, 4) / 512;
    if (!make_sf_tmap(&tsa, d->sfa_dev, atoms_a, 4)) return MPM_ERR_CUDA;
    if (!make_sf_tmap(&tsb, d->sfb_dev, atoms_b, 4)) return MPM_ERR_CUDA;
    if (!make_out_tmap(&tout, d->out_dev, d->N, d->a_rows, d->ldo)) return MPM_ERR_CUDA;
    const int n_tiles = (int)(d->N / 128);
    const long long n_tasks = (long long)n_tiles * ((d->a_rows + 255) / 256);
    return cuda_status(mpm::launch_fc2_online(ta, tb64, tsa, tsb, tout, a, n_tiles, n_tasks, stream));
  }
  if (tile_m == 256) {
    const int kind_atoms = d->kind == MPM_KIND_NVFP4 ? 4 : 1;
    const long long atoms_a = pad_to(d->a_total_rows, 128) * pad_to(d->sfa_cols, 4) / 512;
    const long long atoms_b = pad_to(d->b_total_rows, 128) * pad_to(d->sfb_cols, 4) / 512;
    CUtensorMap tsa, tsb;
    std::memset(&tsa, 0, sizeof(tsa));
    std::memset(&tsb, 0, sizeof(tsb));
    if (!bf16) {
      if (!make_sf_tmap(&tsa, d->sfa_dev, atoms_a, kind_atoms)) return MPM_ERR_CUDA;
      if (!make_sf_tmap(&tsb, d->sfb_dev, atoms_b, kind_atoms)) return MPM_ERR_CUDA;
    }
    CUtensorMap tout, taux;
    std::memset(&tout, 0, sizeof(tout));
    std::memset(&taux, 0, sizeof(taux));
    if (d->epilogue == MPM_EPI_DSWIGLU) {
      if (!make_out_tmap(&tout, d->out_dev, 2 * d->N, d->a_rows, d->ldo)) return MPM_ERR_CUDA;
      if (!make_out_tmap(&taux, d->aux_dev, 2 * d->N, d->a_rows, d->ld_aux)) return MPM_ERR_CUDA;
    } else if (d->epilogue == MPM_EPI_BF16) {
      if (!make_out_tmap(&tout, d->out_dev, d->N, d->a_rows, d->ldo)) return MPM_ERR_CUDA;
    } else if (d->epilogue == MPM_EPI_F32) {
      const long long rows = d->group == MPM_GROUP_K ? d->E * d->a_rows : d->a_rows;
      if (!make_out_tmap(&tout, d->out_dev, d->N, rows, d->ldo, true)) return MPM_ERR_CUDA;
    } else if (swiglu) {
      if (!make_out_tmap(&tout, d->out2_dev, d->N / 2, d->a_rows, d->ldo2)) return MPM_ERR_CUDA;
      if (d->epilogue == MPM_EPI_SWIGLU_SAVE &&
          !make_out_tmap(&taux, d->out_dev, d->N, d->a_rows, d->ldo))
        return MPM_ERR_CUDA;
    }
    const int n_tiles = (int)(swiglu ? (d->N / 2) / 128 : d->N / 256);
    long long n_tasks = (long long)n_tiles * ((d->a_rows + 255) / 256);
    if (d->group == MPM_GROUP_K) n_tasks *= d->E;
    return cuda_status(mpm::launch_grouped_gemm_pair(d->kind, d->epilogue, maj, ta, tb, tsa, tsb, tout,
                                                     taux, a, n_tiles, n_tasks, stream));
  }
  dim3 grid;
  if (d->group == MPM_GROUP_M) {
    grid = dim3((unsigned)(swiglu ? (d->N / 2) / 128 : d->N / 256),
                (unsigned)((d->a_rows + 127) / 128), 1);
  } else {
    grid = dim3((unsigned)(d->N / 256), (unsigned)(d->a_rows / 128), (unsigned)d->E);
  }
  if (grid.y > 65535 && d->group == MPM_GROUP_M) return MPM_ERR_SHAPE;
  return cuda_status(mpm::launch_grouped_gemm(d->kind, d->epilogue, ta, tb, a, grid, stream));
}

mpm_status mpm_moe_grouped_gemm_wgrad(const mpm_grouped_gemm_desc* d, cudaStream_t stream) {
  if (!d) return MPM_ERR_NULL;
  mpm_grouped_gemm_desc w = *d;
  w.group = MPM_GROUP_K;
  return mpm_moe_grouped_gemm(&w, stream);
}

mpm_status mpm_get_device_status(int32_t* host_out, cudaStream_t stream) {
  if (!host_out) return MPM_ERR_NULL;
  int* p = status_ptr();
  if (!p) return MPM_ERR_CUDA;
  int zero = 0;
  if (cudaMemcpyAsync(host_out, p, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MPM_ERR_CUDA;
  if (cudaMemcpyAsync(p, &zero, sizeof(int), cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return MPM_ERR_CUDA;
  return cuda_status(cudaStreamSynchronize(stream));
}

}  // extern "C"
