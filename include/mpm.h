/*
 * mpm.h -- C ABI of libmpm: microscaled-precision (MXFP8 / NVFP4) quantisers
 * and block-scaled MoE grouped GEMMs for sm_103a (GB300).
 *
 * Every call is asynchronous on the caller's CUDA stream, allocates no device
 * memory, and validates its arguments on the host before launching anything:
 * a call that returns a status other than MPM_OK has launched nothing.  The
 * caller owns every buffer.  Pointers named *_dev are device pointers; all
 * other pointers are host pointers.  Identical inputs always give identical
 * output bytes (no floating-point atomics, fixed reduction orders).
 *
 * Formats (source: "Towards Blackwell-native 8-bit and 4-bit RL", section
 * "Format background"; "miniTE technical report", section 2.2):
 *   MXFP8  32 consecutive E4M3 values share one E8M0 power-of-two scale,
 *          rounded up so the block max never clips.
 *   NVFP4  E2M1 codes, one E4M3 scale per 16 values (round to nearest), and an
 *          FP32 outer scale; decode x_hat = q * s_b * s_g.
 *
 * Layouts shared by all calls:
 *   - bf16 inputs are row-major with a leading dimension in elements.
 *   - FP4 codes are packed two per byte, element 2j in the low nibble.
 *   - Scale matrices [rows, cols] are stored in 128x4 tiles: rows padded to a
 *     multiple of 128 and cols to a multiple of 4 with zero bytes; tile
 *     (rt, ct) starts at byte (rt * pad4(cols) / 4 + ct) * 512 and holds entry
 *     (r, c) at (r % 32) * 16 + (r / 32 % 4) * 4 + c % 4.  Size:
 *     mpm_scale_bytes(rows, cols).  This is the operand layout the sm_100
 *     family block-scaled tensor-core MMA reads its scale factors in.
 *
 * Errors: host-side validation failures return MPM_ERR_NULL / _SHAPE /
 * _ALIGN / _UNSUPPORTED; a failed launch returns MPM_ERR_CUDA.  Sizes must
 * be at least 1: an empty input (no rows, no tokens, no experts) is a shape
 * error, not a no-op, so a caller never mistakes unwritten outputs for
 * results.  Experts that receive no rows are not an empty input: the
 * segment, gather and GEMM calls handle them inside one call.  When several
 * requirements are broken at once, which of their statuses is returned is
 * not specified.  Problems only visible on the device (an expert offset
 * table that is not monotone or that exceeds the row capacity, a pipeline
 * wait that ran out of time) set a per-device status word and make the
 * kernel skip the affected work (no trap, no hang); read it with
 * mpm_get_device_status().
 */
#ifndef MPM_H
#define MPM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MPM_OK = 0,
  MPM_ERR_NULL = 1,          /* a required pointer is NULL                     */
  MPM_ERR_SHAPE = 2,         /* a size is zero/negative/inconsistent           */
  MPM_ERR_ALIGN = 3,         /* a pointer or leading dimension is misaligned   */
  MPM_ERR_UNSUPPORTED = 4,   /* valid request this build does not implement    */
  MPM_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed              */
  MPM_ERR_DEVICE_TIMEOUT = 6,/* (device status) a bounded pipeline wait expired */
  MPM_ERR_DEVICE_BOUNDS = 7  /* (device status) bad offsets / row indices       */
} mpm_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* mpm_status_string(int status);

/* Library version, e.g. 101 for 1.0.1 (101: mpm_grouped_gemm_desc.row_perm_dev). */
int mpm_version(void);

/* Bytes of a 128x4-tiled scale matrix: pad128(rows) * pad4(cols). */
size_t mpm_scale_bytes(int64_t rows, int64_t cols);

/* ------------------------------------------------------------------------ */
/* Quantisers                                                               */
/* ------------------------------------------------------------------------ */

#define MPM_ROWWISE 1u
#define MPM_COLWISE 2u

/*
 * MXFP8 quantisation of x_dev (bf16 [M, K], leading dimension ldx elements)
 * into a row-wise 1x32 copy and/or a column-wise 32x1 copy, each quantised
 * independently from the bf16 input in one pass over it.
 * Source: "Towards Blackwell-native 8-bit and 4-bit RL", sections "Format
 * background / MXFP8" (E8M0 scale rounded up) and "Recipe 1 / Training"
 * (row-wise and column-wise copies materialised by one quantisation).
 *
 * Per block of 32 values v: a = max|v|; e = smallest integer with
 * a <= 448 * 2^e, clamped to [-127, 127] (a = 0 gives -127); scale byte
 * e + 127; code = E4M3(v * 2^-e), round to nearest even, saturating.
 *
 * flags: MPM_ROWWISE and/or MPM_COLWISE.
 * ROWWISE: row_q_dev  u8 [M, K] (leading dim K),
 *          row_s_dev  scales [M, K/32] in 128x4 tiles (mpm_scale_bytes(M, K/32)).
 * COLWISE: col_q_dev  u8 [K, ldc] -- the copy is stored TRANSPOSED, so each
 *          column block is 32 contiguous bytes; ldc >= M, columns >= M of
 *          each row are not written,
 *          col_s_dev  scales [K, ceil(M/32)] in 128x4 tiles.
 * The last column block of a partial 32-row group behaves as zero padded.
 * m_valid_dev (nullable): device int32; if given, only rows < min(M, *m_valid)
 * are quantised and rows at or beyond it read as zero (used for buffers whose
 * used row count is known only on the device).
 * Requirements: M >= 1, K >= 32, K % 32 == 0, ldx >= K, ldx % 8 == 0,
 * x_dev 16-byte aligned, ldc % 16 == 0, all output pointers 16-byte aligned.
 * The kernel is launched with programmatic stream serialization: it may
 * start while the previous kernel on the stream finishes, and it touches
 * global memory only after that kernel has completed (stream order holds
 * for the caller as for any other launch).
 */
mpm_status mpm_mxfp8_quantize(const void* x_dev, int64_t M, int64_t K, int64_t ldx,
                              unsigned flags,
                              uint8_t* row_q_dev, uint8_t* row_s_dev,
                              uint8_t* col_q_dev, int64_t ldc, uint8_t* col_s_dev,
                              const int32_t* m_valid_dev, cudaStream_t stream);

/*
 * Per-token NVFP4 quantisation: one call returns the packed FP4 codes, the
 * E4M3 block scales and the per-token FP32 outer scales.
 * Source: "Towards Blackwell-native 8-bit and 4-bit RL", section "Per-token
 * activation scaling" (one online FP32 scale per token, returned by the same
 * call that emits the codes and block scales); "miniTE technical report",
 * section 5.6 (s_g = amax / 2688) and section 5.3 (reuse of an amax computed
 * by the producer of the activation).
 *
 * Per row, every step IEEE binary32 round-to-nearest (no FMA contraction):
 *   a   = max_j |x_j|  (or amax_in_dev[row] when given)
 *   s_g = a / 2688, raised to 2^-116 if it is below that; a = 0 -> s_g = 0
 *   per 16-block: s_b = E4M3_rn_satfinite(bmax / (6 * s_g))
 *   s_b = 0 -> codes 0; else r = 1 / (s_b * s_g), q_j = E2M1_rn_satfinite(x_j * r)
 *
 * x_dev: bf16 [M, K], leading dimension ldx elements.
 * amax_in_dev (nullable): fp32 [M] row amax computed by the producer.
 * q_dev: u8 [M, K/2] (leading dim K/2).  s_dev: scales [M, K/16] in 128x4
 * tiles.  token_scale_dev: fp32 [M] (the s_g above).
 * m_valid_dev (nullable): as for mpm_mxfp8_quantize; rows at or beyond the
 * device row count are left untouched (their scale tiles are not written).
 * Requirements: M >= 1, K % 64 == 0, 64 <= K <= 8192, ldx >= K,
 * ldx % 8 == 0, all pointers 16-byte aligned (token_scale_dev and
 * amax_in_dev 4-byte).
 */
mpm_status mpm_nvfp4_quantize_per_token(const void* x_dev, int64_t M, int64_t K,
                                        int64_t ldx, const float* amax_in_dev,
                                        uint8_t* q_dev, uint8_t* s_dev,
                                        float* token_scale_dev,
                                        const int32_t* m_valid_dev,
                                        cudaStream_t stream);

/*
 * NVFP4 quantisation with a running row amax, tile by tile: the activation
 * side of the single-pass FC2.  Source: "miniTE technical report", section
 * 5.6 (a row is consumed in K tiles; the row amax seen so far sets the outer
 * scale gs = gamax / 2688 each tile is encoded against; the FC2 partial sum
 * is compensated when gs grows; see MPM_EPI_BF16_ONLINE).
 *
 * Per row, tiles t = 0, 1, ... of 256 columns in order:
 *   gamax_t = max(gamax_{t-1}, max |x| over tile t)   (gamax_{-1} = 0)
 *   gs_t    = gamax_t / 2688 with the 2^-116 floor; gamax_t = 0 -> gs_t = 0
 *   the tile's 16-blocks: the steps of mpm_nvfp4_quantize_per_token with
 *   gs_t in place of s_g.
 * x_dev: bf16 [M, K] (leading dimension ldx).  q_dev: u8 [M, K/2];
 * s_dev: scales [M, K/16] in 128x4 tiles; tile_scale_dev: fp32 [M, K/256]
 * (gs_t of row r at r * K/256 + t).  m_valid_dev (nullable) as for
 * mpm_nvfp4_quantize_per_token.
 * Requirements: M >= 1, K % 256 == 0, 256 <= K <= 8192, ldx >= K,
 * ldx % 8 == 0, pointers 16-byte aligned (tile_scale_dev 4-byte).
 */
mpm_status mpm_nvfp4_quantize_online(const void* x_dev, int64_t M, int64_t K, int64_t ldx,
                                     uint8_t* q_dev, uint8_t* s_dev, float* tile_scale_dev,
                                     const int32_t* m_valid_dev, cudaStream_t stream);

/*
 * NVFP4 weight quantisation with one FP32 outer scale per expert shared by
 * all given parts (gate and up quantised jointly so that the fused gate|up
 * GEMM sees one weight scale).
 * Source: "Towards Blackwell-native 8-bit and 4-bit RL", section "Per-token
 * activation scaling" (gate/up paired quantisation with a shared FP32 scale);
 * block and element rules as for mpm_nvfp4_quantize_per_token.
 *
 * parts_dev: host array of nparts device pointers; part p is bf16
 * [E, part_rows[p], K] contiguous.  The quantised expert e holds the parts'
 * rows concatenated in order: R = sum(part_rows) rows.
 * q_dev: u8 [E, R, K/2].  s_dev: E consecutive scale matrices [R, K/16] in
 * 128x4 tiles, expert e at byte e * mpm_scale_bytes(R, K/16).
 * tensor_scale_dev: fp32 [E] (s_g of each expert).
 * ws_dev: workspace of at least mpm_nvfp4_weight_workspace_bytes(E) bytes.
 * Requirements: nparts in 1..4, E >= 1, K % 64 == 0, 64 <= K <= 8192,
 * each part_rows[p] >= 1, R % 128 == 0, ws_bytes at least
 * mpm_nvfp4_weight_workspace_bytes(E); parts and q_dev 16-byte aligned,
 * ws_dev and tensor_scale_dev 4-byte.
 */
size_t mpm_nvfp4_weight_workspace_bytes(int64_t E);
mpm_status mpm_nvfp4_quantize_weight(const void* const* parts_dev, const int64_t* part_rows,
                                     int nparts, int64_t K, int64_t E,
                                     uint8_t* q_dev, uint8_t* s_dev, float* tensor_scale_dev,
                                     void* ws_dev, size_t ws_bytes, cudaStream_t stream);

/*
 * Allocation-free variant of mpm_nvfp4_quantize_weight (the pages have no
 * counterpart: this is an interface convenience of this library).  For
 * callers that cannot allocate device memory where they quantise weights --
 * code whose device memory belongs to a pool it cannot reach there, or a
 * latency-critical loop where a cudaMalloc, which may synchronise the device,
 * is not allowed.  Same inputs, outputs, rules and requirements as
 * mpm_nvfp4_quantize_weight, but no workspace argument: the per-expert amax
 * scratch lives in a fixed device array declared by the library (16 KiB, room
 * for E <= 4096 experts; every GPU that loads the library keeps it until the
 * process exits).  E > 4096 returns MPM_ERR_SHAPE before any launch.
 * Each call made outside stream capture looks up that array's device address
 * on the current device (so a device reset, after which the library's device
 * memory lives elsewhere, is picked up by the next such call); a call made
 * while the stream is capturing reuses the address the last uncaptured call
 * on that device found, so make one call on each device (and one after any
 * device reset) before capturing; a first call under capture returns
 * MPM_ERR_CUDA.  The call allocates nothing and clears the slots it uses before
 * reducing into them.  All calls share the one array: calls whose work can
 * overlap on the GPU (other streams, other host threads) race on it, so
 * order them on one stream or synchronise between them.
 */
mpm_status mpm_nvfp4_quantize_weight_noalloc(const void* const* parts_dev,
                                             const int64_t* part_rows, int nparts,
                                             int64_t K, int64_t E, uint8_t* q_dev,
                                             uint8_t* s_dev, float* tensor_scale_dev,
                                             cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Expert segments, permutation, combine                                    */
/* ------------------------------------------------------------------------ */

/*
 * Row capacity of the permuted buffers for T tokens, top-k and E experts with
 * segments padded to `pad` rows (16, 32, 64, 128 or 256): pad(T*k) + pad*E;
 * 0 for an invalid argument.
 */
int64_t mpm_moe_row_capacity(int64_t T, int k, int64_t E, int pad);
size_t mpm_moe_segments_workspace_bytes(int64_t T, int k, int64_t E);

/*
 * Counting sort of the T*k routed (token, slot) pairs by expert into one
 * contiguous buffer, each expert's segment padded to `pad` rows (128: one
 * MMA tile; 256: one CTA-pair tile, required by the tile_m = 256 GEMM;
 * 16 / 32 / 64 for the small-M GEMM, which takes segments of any length).
 * Source: "miniTE technical report", section 5.2 (contiguous buffer with
 * expert boundaries given by offsets kept on the device; zero-token experts
 * and padding handled in the same path).
 *
 * topk_ids_dev: int32 [T, k] expert ids in [0, E); topk_prob_dev: fp32 [T, k].
 * Outputs (device): seg_offsets int32 [E+1] (seg_offsets[0] = 0, segment e is
 * rows [seg_offsets[e], seg_offsets[e+1]), a multiple of pad long); perm
 * int32 [capacity] (row -> flat index t*k + j, -1 for padding rows and rows
 * beyond seg_offsets[E]); inv_perm int32 [T*k] (flat index -> row); row_prob
 * fp32 [capacity] (0 for padding).  Rows of one expert are in ascending flat
 * index order (stable).  An id outside [0, E) sets MPM_ERR_DEVICE_BOUNDS and
 * the pair is dropped.  Requirements: T >= 1, 1 <= k <= 64, 1 <= E <= 1024,
 * T * k <= 2^30, pad one of the values above, ws_bytes at least
 * mpm_moe_segments_workspace_bytes(T, k, E), ws_dev 4-byte aligned.
 */
mpm_status mpm_moe_build_segments(const int32_t* topk_ids_dev, const float* topk_prob_dev,
                                  int64_t T, int k, int64_t E, int pad,
                                  int32_t* seg_offsets_dev, int32_t* perm_dev,
                                  int32_t* inv_perm_dev, float* row_prob_dev,
                                  void* ws_dev, size_t ws_bytes, cudaStream_t stream);

/*
 * Gather rows into the permuted layout: dst[row] = src[perm[row] / k] for
 * rows < seg_offsets[E] with perm[row] >= 0, zero for padding rows.
 * MPM_GATHER_BF16:  src bf16 [T, K] (ld K) -> dst bf16 [capacity, K].
 * MPM_GATHER_NVFP4: src codes u8 [T, K/2], scales (128x4 tiles of [T, K/16])
 *   and token scales fp32 [T] -> the same three for [capacity] rows
 *   (src_s / dst_s / src_ts / dst_ts used only here).
 * amax_zero_dev (nullable): fp32 [capacity]; entries of the gathered rows are
 * set to 0, ready for the row-amax reduction of the FC1 epilogue.
 * Source: "miniTE technical report", section 5.3 (dispatch/permute before the
 * FC1 quantised GEMM; the padding step handles the activation and its amax
 * together).  Requirements: T, k, E, capacity >= 1, K % 64 == 0, src and
 * dst 16-byte aligned, the NVFP4 scale pointers 4-byte aligned (amax_zero_dev
 * too); `what` other than the two kinds is MPM_ERR_UNSUPPORTED.
 */
#define MPM_GATHER_BF16 0
#define MPM_GATHER_NVFP4 1
mpm_status mpm_moe_gather(int what, const void* src_dev, const uint8_t* src_s_dev,
                          const float* src_ts_dev, int64_t T, int64_t K, int k,
                          const int32_t* perm_dev, const int32_t* seg_offsets_dev,
                          int64_t E, int64_t capacity,
                          void* dst_dev, uint8_t* dst_s_dev, float* dst_ts_dev,
                          float* amax_zero_dev, cudaStream_t stream);

/*
 * Per-token NVFP4 quantisation of x_dev (bf16 [T, K], leading dimension ldx
 * elements) written straight into the expert-ordered rows: the same bytes as
 * mpm_nvfp4_quantize_per_token of x followed by mpm_moe_gather
 * (MPM_GATHER_NVFP4) with the same segments, without the token-ordered copy.
 * Row r < seg_offsets[E] with perm[r] >= 0 gets the codes, block scales and
 * outer scale of token perm[r] / k; a padding row (perm[r] < 0) gets zeros;
 * amax_zero_dev[r] (nullable) is set to 0 for every such row; rows at or
 * beyond seg_offsets[E] are not written.
 * Sources: "Towards Blackwell-native 8-bit and 4-bit RL", section
 * "Per-token activation scaling" (one scale per token, so a token's bytes do
 * not depend on where its rows go), and "miniTE technical report", section
 * 5.3 (dispatch/permute ahead of the FC1 quantised GEMM, the activation and
 * its amax padded together).
 * Layouts: q_dev u8 [capacity, K/2]; s_dev 128x4 tiles of [capacity, K/16]
 * (mpm_scale_bytes(capacity, K/16)); ts_dev fp32 [capacity]; inv_perm_dev
 * int32 [T*k] and perm_dev int32 [capacity] as written by
 * mpm_moe_build_segments.  A row index outside [0, seg_offsets[E]) in
 * inv_perm sets MPM_ERR_DEVICE_BOUNDS and that write is dropped.
 * Two launches: the codes go to the routed rows while each token's block
 * scales and outer scale go to ws_dev (token order); the second writes the
 * scale tiles, outer scales, amax slots and padding rows from it.  ws_dev:
 * caller-owned, at least mpm_nvfp4_quantize_scatter_workspace_bytes(T, K)
 * bytes, 4-byte aligned; its contents need no initialisation.
 * Requirements: T >= 1, 64 <= K <= 8192, K % 64 == 0, ldx >= K, ldx % 8 == 0,
 * 1 <= k <= 64, E >= 1, capacity >= 1; x_dev and q_dev 16-byte aligned,
 * s_dev, ts_dev and amax_zero_dev 4-byte aligned.
 */
size_t mpm_nvfp4_quantize_scatter_workspace_bytes(int64_t T, int64_t K);
mpm_status mpm_nvfp4_quantize_scatter(const void* x_dev, int64_t T, int64_t K, int64_t ldx,
                                      const int32_t* inv_perm_dev, int k,
                                      const int32_t* perm_dev, const int32_t* seg_offsets_dev,
                                      int64_t E, int64_t capacity, uint8_t* q_dev,
                                      uint8_t* s_dev, float* ts_dev, float* amax_zero_dev,
                                      void* ws_dev, size_t ws_bytes, cudaStream_t stream);

/*
 * MXFP8 quantisation of the expert-ordered rows of x_dev (bf16 [T, K],
 * leading dimension ldx elements) without the gathered bf16 copy: the same
 * bytes as mpm_moe_gather (MPM_GATHER_BF16) with the same segments followed
 * by mpm_mxfp8_quantize of the gathered [capacity, K] matrix with
 * m_valid = seg_offsets + E.  Row r < seg_offsets[E] of the quantised matrix
 * is token row perm[r] / k of x, a zero row where perm[r] < 0; rows at or
 * beyond seg_offsets[E] are not written.
 * Sources: "Towards Blackwell-native 8-bit and 4-bit RL", sections "Format
 * background / MXFP8" and "Recipe 1 / Training" (row-wise and column-wise
 * copies of each GEMM operand from one quantisation), and "miniTE technical
 * report", section 5.3 (dispatch/permute ahead of the quantised expert
 * GEMMs).
 * flags, row_q_dev, row_s_dev, col_q_dev, ldc, col_s_dev: as for
 * mpm_mxfp8_quantize with M = capacity.  perm_dev int32 [capacity] as written
 * by mpm_moe_build_segments.  A token index perm[r] / k >= T sets
 * MPM_ERR_DEVICE_BOUNDS and that row reads as zero.
 * Requirements: T >= 1, capacity >= 1, E >= 1, 1 <= k <= 64, T * k < 2^31,
 * K >= 32, K % 32 == 0, K <= ldx < 2^31, ldx % 8 == 0, x_dev 16-byte aligned,
 * ldc >= capacity,
 * ldc % 16 == 0, output pointers 16-byte aligned.  Launched with programmatic
 * stream serialization, as mpm_mxfp8_quantize.
 */
mpm_status mpm_mxfp8_quantize_gather(const void* x_dev, int64_t T, int64_t K, int64_t ldx,
                                     const int32_t* perm_dev, int k,
                                     const int32_t* seg_offsets_dev, int64_t E,
                                     int64_t capacity, unsigned flags,
                                     uint8_t* row_q_dev, uint8_t* row_s_dev,
                                     uint8_t* col_q_dev, int64_t ldc, uint8_t* col_s_dev,
                                     cudaStream_t stream);

/*
 * out[t] = sum over j = 0..k-1 (in that order, fp32) of y_perm[inv_perm[t*k+j]],
 * rounded once to bf16.  y_perm bf16 [capacity, H]; out bf16 [T, H].
 * Source: "miniTE technical report", section 5.3 (expert outputs, weighted by
 * the router, summed back per token); the router weight is applied earlier in
 * the FC1 epilogue.  Requirements: T, k >= 1, H >= 8, H % 8 == 0, y_perm and
 * out 16-byte aligned.
 */
mpm_status mpm_moe_combine(const void* y_perm_dev, const int32_t* inv_perm_dev,
                           int64_t T, int k, int64_t H, void* out_dev,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Dequantisation and transpose: operands of the BF16 backward              */
/* ------------------------------------------------------------------------ */

/*
 * NVFP4 -> bf16:
 *   out[r, c] = bf16_rn( e2m1(q[r, c]) * e4m3(s_b[r, c/16]) * s_g[r / rows_per_outer] ),
 * the product rounded ONCE (to nearest, ties to even) to bf16.
 * Source: "Towards Blackwell-native 8-bit and 4-bit RL", section
 * "High-precision and dequantized backward" (the backward GEMMs run in BF16
 * on the BF16 dequantisation of the exact low-precision forward operands);
 * "miniTE technical report", section 2.2 (x_hat = q * s_b * s_g).
 *
 * q_dev: packed codes u8 [M, K/2] (element 2j in the low nibble); s_dev: E4M3
 * scales [M, K/16] in 128x4 tiles; outer_dev: fp32 outer scales, one per
 * rows_per_outer consecutive rows (1 for per-token activations, the rows of
 * one expert for a weight).  out_dev: bf16 [M, K], leading dimension ldo
 * elements.  m_valid_dev (nullable): device row count; rows at or beyond it
 * are not written.  Requirements: M >= 1, K % 64 == 0, rows_per_outer >= 1,
 * ldo >= K, ldo % 8 == 0, q / s / out 16-byte aligned, outer 4-byte.
 */
mpm_status mpm_nvfp4_dequantize(const uint8_t* q_dev, const uint8_t* s_dev,
                                const float* outer_dev, int64_t rows_per_outer,
                                int64_t M, int64_t K, void* out_dev, int64_t ldo,
                                const int32_t* m_valid_dev, cudaStream_t stream);

/*
 * MXFP8 (row-wise copy) -> bf16:
 *   out[r, c] = bf16_rn( e4m3(q[r, c]) * 2^(s[r, c/32] - 127) ).
 * Source: as above, and "Towards Blackwell-native 8-bit and 4-bit RL",
 * section "Format background / MXFP8" (blocks of 32 with an E8M0
 * power-of-two scale).  q_dev u8 [M, K]; s_dev [M, K/32] in 128x4 tiles.
 * Requirements: M >= 1, K % 32 == 0, ldo >= K, ldo % 8 == 0, pointers 16-byte
 * aligned.
 */
mpm_status mpm_mxfp8_dequantize(const uint8_t* q_dev, const uint8_t* s_dev, int64_t M,
                                int64_t K, void* out_dev, int64_t ldo,
                                const int32_t* m_valid_dev, cudaStream_t stream);

/*
 * out[c, r] = in[r, c] for bf16 matrices: the K-major copies that the BF16
 * weight-gradient and input-gradient GEMMs read.  in [R, C] with leading
 * dimension ldi; out [C, >= R] with leading dimension ldo >= R.
 * m_valid_dev (nullable): device row count R' <= R; input rows at or beyond
 * it are not read and the matching output columns are not written.  Bit
 * copies, no arithmetic.  Requirements: R, C >= 1, ldi >= C, ldo >= R,
 * R <= 64 * 65535; in and out do not overlap.
 */
mpm_status mpm_transpose_bf16(const void* in_dev, int64_t R, int64_t C, int64_t ldi,
                              void* out_dev, int64_t ldo, const int32_t* m_valid_dev,
                              cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Block-scaled grouped GEMM (tcgen05)                                      */
/* ------------------------------------------------------------------------ */

#define MPM_KIND_NVFP4 0   /* E2M1 x E2M1, E4M3 scales per 16, fp32 accumulate */
#define MPM_KIND_MXFP8 1   /* E4M3 x E4M3, E8M0 scales per 32, fp32 accumulate */
#define MPM_KIND_BF16 2    /* bf16 x bf16, fp32 accumulate, no scales (tile_m 256
                              only): the high-precision / dequantized backward */

/* tile_m value selecting the small-M (decode / rollout) kernel: one CTA per
   128 weight rows x 128 routed rows, weights on the MMA's M side */
#define MPM_TILE_SMALL_M 1

#define MPM_GROUP_M 0      /* rows of A split into expert segments (fprop, dgrad) */
#define MPM_GROUP_K 1      /* reduction split into expert segments (wgrad)        */

#define MPM_EPI_F32 0            /* out fp32 [rows, N]                             */
#define MPM_EPI_BF16 1           /* out bf16 [rows, N]                             */
#define MPM_EPI_SWIGLU 2         /* out2 = D bf16 [rows, N/2], amax atomically max'd */
#define MPM_EPI_SWIGLU_SAVE 3    /* SWIGLU and out = C bf16 [rows, N] (gate|up)     */
#define MPM_EPI_DSWIGLU 4        /* out = dH bf16 [rows, 2N] from aux = C bf16       */
#define MPM_EPI_BF16_ONLINE 5    /* out bf16 [rows, N] = alpha_b[e] * sum_t aux[row, t] *
                                    (the product over reduction tile t of 256): the
                                    FC2 of the single-pass FFN (NVFP4, tile_m 256)   */

/*
 * Descriptor of one grouped GEMM  C_e = A_e * B_e^T  (both operands K-major,
 * i.e. row-major with the reduction dimension contiguous).
 *
 * GROUP_M: rows [seg[e], seg[e+1]) of A (a [capacity, K] matrix) multiply
 *   expert e's B, rows e*b_rows_per_expert .. +N of the B matrix, reduction
 *   columns e*b_k_per_expert .. +K.  Output rows = A rows.  seg_dev may be
 *   NULL for one dense group of a_rows rows.
 * GROUP_K: for expert e, A is the [M_out, .] matrix and B the [N, .] matrix
 *   restricted to reduction columns [seg[e], seg[e+1]); output expert e is
 *   [M_out, N] at out + e * M_out * ldo (fp32 only).  Empty experts give 0.
 *
 * a_dev / b_dev: codes (NVFP4: packed, K/2 bytes per row; MXFP8: K bytes;
 * BF16: the bf16 values, 2K bytes per row, sfa_dev / sfb_dev unused),
 * lda_bytes / ldb_bytes their row pitches (multiples of 16).
 * sfa_dev / sfb_dev: their scale matrices in 128x4 tiles, sfa_cols / sfb_cols
 * the UNPADDED scale column counts of the whole A / B matrices
 * (row pitch/16 or /32 elements); B's per-expert rows are addressed
 * directly inside one tiled matrix (b_rows_per_expert % 128 == 0).
 * alpha_a_dev (NVFP4, GROUP_M): fp32 per-row outer scale of A; alpha_b_dev:
 * fp32 [E] outer scale of each expert's B (either may be NULL = 1).
 * Epilogue: acc * alpha_a[row] * alpha_b[e], then
 *   F32/BF16: store;  SWIGLU: D[r, j] = silu(g) * u * row_prob[r] with
 *   g = column j, u = column N/2 + j, rounded to bf16, and amax_dev[r] =
 *   max(amax_dev[r], max_j |D[r, j]|) (fp32 bits, caller zeroes it first);
 *   DSWIGLU: dD = acc, with (g, u) read from aux (bf16 C, [rows, 2N]):
 *   dH[r, j] = dD*p*u*silu'(g), dH[r, N+j] = dD*p*silu(g), bf16.
 *   BF16_ONLINE (NVFP4, tile_m 256, GROUP_M): A quantised tile by tile with
 *   a running row amax (mpm_nvfp4_quantize_online); aux = its fp32 outer
 *   scales [rows, ld_aux] (ld_aux >= K/256), alpha_a_dev must be NULL:
 *   out[r, n] = bf16( alpha_b[e] * sum_t aux[r, t] * P_t[r, n] ), P_t the
 *   block-scaled product over reduction columns [256 t, 256 t + 256).  This
 *   is the compensated partial sum of "miniTE technical report", section 5.6
 *   (O <- O * gs_prev / gs_t + P_t, Y = O * gs_last * s_g(W2)) written as
 *   its closed form; CTA pairs on 256 x 128 output tiles, N % 128 == 0.
 * Source: "miniTE technical report", section 5.2 (grouped GEMM over a
 * contiguous buffer with device offsets), section 5.4 (FC1 epilogue:
 * ACC x alpha_a[m] (x alpha_b), C = gate|up, D = act(gate, up) x prob, amax
 * of D); "Towards Blackwell-native 8-bit and 4-bit RL", section "Recipe 1 /
 * Training" (dgrad with the column-wise weight copy, wgrad with column-wise
 * activation and gradient copies).
 * tile_m = 256 runs the tile on a pair of CTAs (tcgen05 cta_group::2): each
 * SM stages its 128 rows of A and half of B, so B moves through shared
 * memory once per 256 output rows instead of once per 128.
 * BF16 (kind::f16 on the tensor cores): "Towards Blackwell-native 8-bit and
 * 4-bit RL", section "High-precision and dequantized backward" (backward
 * GEMMs in BF16 on original or dequantised operands).
 * Requirements: K % 256 == 0 (NVFP4), % 128 == 0 (MXFP8) or % 64 == 0 (BF16)
 * in GROUP_M; N % 256 == 0 (SwiGLU: N/2 % 128 == 0); GROUP_K (MXFP8 or
 * BF16, F32 epilogue): M_out % 128 == 0, segments multiples of 128 rows.
 * BF16 requires tile_m = 256.
 * tile_m = MPM_TILE_SMALL_M computes the same result with the roles swapped
 * inside the MMA: 128 weight rows on its M side, a chunk of 128 routed rows
 * of one segment on its N side, persistent CTAs over (chunk, weight tile),
 * for batches where each expert receives few rows and the layer is bound by
 * reading the active experts' weights once ("Towards Blackwell-native 8-bit
 * and 4-bit RL", the rollout side of section "Per-token activation
 * scaling").  MN-major operands (a_mn_major / b_mn_major,
 * BF16 only) let the backward GEMMs read the row-major activations, gradients
 * and weights as they are, with no transposed copies: GROUP_M with
 * b_mn_major (epilogue BF16, F32 or DSWIGLU), GROUP_K with both (F32).
 * Pitches of MN-major operands: lda_bytes >= 2 * M_out, ldb_bytes >= 2 * N.
 * Zero-initialise the two fields (memset of the whole descriptor) when they
 * are not used.
 */
typedef struct {
  int kind;                    /* MPM_KIND_*                                   */
  int tile_m;                  /* 128: one CTA per 128x256 tile; 256: a CTA pair
                                  per 256x256 tile, persistent (GROUP_M: the
                                  expert segments must be multiples of 256
                                  rows, checked on the device; GROUP_K: the
                                  output rows a_rows % 256 == 0);
                                  MPM_TILE_SMALL_M: the small-M kernel
                                  (GROUP_M, NVFP4 or MXFP8, epilogue F32, BF16
                                  or SWIGLU, 128-row segments, N (SWIGLU: N/2)
                                  % 128 == 0)                                */
  int group;                   /* MPM_GROUP_*                                  */
  int epilogue;                /* MPM_EPI_*                                    */
  int64_t E;                   /* experts (groups)                             */
  int64_t a_rows;              /* GROUP_M: row capacity of A (grid bound);
                                  GROUP_K: M_out                               */
  int64_t N;                   /* output columns per expert                    */
  int64_t K;                   /* reduction length (GROUP_M); GROUP_K: unused  */
  const int32_t* seg_dev;      /* [E+1] device offsets (rows of A, or the
                                  reduction for GROUP_K)                        */
  const uint8_t* a_dev; int64_t lda_bytes; int64_t a_total_rows;
  const uint8_t* b_dev; int64_t ldb_bytes; int64_t b_total_rows;
  int64_t b_rows_per_expert;   /* row offset of expert e's B is e * this       */
  int64_t b_k_per_expert;      /* reduction-column offset of expert e's B      */
  const uint8_t* sfa_dev; int64_t sfa_cols;
  const uint8_t* sfb_dev; int64_t sfb_cols;
  const float* alpha_a_dev;
  const float* alpha_b_dev;
  const float* row_prob_dev;   /* SWIGLU / DSWIGLU                             */
  void* out_dev; int64_t ldo;  /* elements                                     */
  void* out2_dev; int64_t ldo2;/* SWIGLU(_SAVE): D                             */
  const void* aux_dev; int64_t ld_aux; /* DSWIGLU: C (gate|up)                 */
  float* amax_dev;             /* SWIGLU: fp32 [rows]                          */
  int a_mn_major;              /* BF16, GROUP_K: 1 = A given as the [rows, M_out]
                                  matrix (M_out contiguous, rows = the reduction)
                                  instead of its K-major transpose            */
  int b_mn_major;              /* BF16: 1 = B given as [K rows, N] (N contiguous):
                                  GROUP_M: expert e's reduction rows start at
                                  e * b_k_per_expert and its columns at
                                  e * b_rows_per_expert; GROUP_K: the [rows, N]
                                  matrix (with a_mn_major)                    */
  const int32_t* row_perm_dev; /* nullable; GROUP_M: the row map of the segment
                                  build ([a_rows], -1 for a segment's padding
                                  rows).  When given, padding rows are not part
                                  of the result: their output rows may be left
                                  unwritten (the small-M kernel's F32 / BF16
                                  epilogues skip them; the combine never reads
                                  them)                                       */
} mpm_grouped_gemm_desc;

mpm_status mpm_moe_grouped_gemm(const mpm_grouped_gemm_desc* desc, cudaStream_t stream);

/*
 * The weight-gradient grouped GEMM: dW_e = dY_e^T * X_e, the contraction
 * running over expert e's own rows [seg[e], seg[e+1]) of the permuted
 * buffers.  Source: "Towards Blackwell-native 8-bit and 4-bit RL", section
 * "Recipe 1 / Training" (wgrad reads the column-wise 32x1 copies of the
 * activation and of the output gradient); "miniTE technical report",
 * section 5.2 (segments given by device offsets, zero-token experts handled
 * in the same path).
 * The same descriptor and rules as mpm_moe_grouped_gemm in GROUP_K mode; the
 * call sets group = MPM_GROUP_K itself (the field is ignored).  a_dev is
 * the [M_out, R] operand (MXFP8: the column-wise copy of dY, stored
 * transposed; BF16: with a_mn_major, dY_perm as it is), b_dev the [N, R]
 * operand (X's column-wise copy; BF16: X_perm with b_mn_major); out_dev
 * fp32 [E, M_out, N] (ldo elements per row), written whole: an expert with
 * no rows gets zeros.  Kinds MXFP8 and BF16, epilogue F32 only (anything
 * else returns MPM_ERR_UNSUPPORTED before any launch).
 */
mpm_status mpm_moe_grouped_gemm_wgrad(const mpm_grouped_gemm_desc* desc, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Device status                                                            */
/* ------------------------------------------------------------------------ */

/*
 * Copies the current device's status word to *host_out (0 = MPM_OK, else an
 * mpm_status from a kernel) and resets it to 0.  Synchronises the stream.
 */
mpm_status mpm_get_device_status(int32_t* host_out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MPM_H */
