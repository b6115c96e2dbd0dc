// Dequantisation to bf16 and a bf16 transpose: the operand preparation of the
// dequantized / high-precision backward.
//
// "Towards Blackwell-native 8-bit and 4-bit RL", section "High-precision and
// dequantized backward": the backward GEMMs run in BF16, either on the
// original BF16 operands or on the BF16 dequantisation of the exact
// low-precision operands the forward pass produced.  Decode ("miniTE
// technical report", section 2.2): x_hat = q * s_b * s_g.
#include "dequant.cuh"

namespace mpm {

// q * s_b is exact in fp32 (at most 2 + 4 significant bits, never below
// 2^-10 unless zero); its product with the fp32 outer scale is rounded ONCE
// to bf16.  The product is first formed with round-to-odd in fp32: truncate,
// then set the last bit if anything was dropped (the dropped part is exact by
// an FMA); rounding the round-to-odd value to bf16 then equals rounding the
// exact product, since fp32 carries at least two more bits than the bf16
// result (Boldo and Melquiond, "Emulation of FMA and correctly rounded sums:
// proved algorithms using rounding to odd", 2008).
//
// The FMA residual is exact only while the product's 30 significant bits sit
// above fp32's subnormal spacing 2^-149, i.e. for |product| >= 2^-120.  Below
// that the product is formed scaled by 2^64 (normal, exact residual) and the
// bf16 rounding of (scaled value) x 2^-64 is done on the integer significand,
// which covers bf16's own subnormal range.
MPM_DEV uint16_t bf16_bits_of_scaled(float v, int k) {
  // v > 0 normal, round-to-odd (its last bit is a sticky bit); returns the
  // bf16 bits of v * 2^-k, rounded to nearest even
  const uint32_t u = __float_as_uint(v);
  const int te = (int)((u >> 23) & 0xFFu) - k;           // biased exponent of the result
  const uint32_t man = (u & 0x7FFFFFu) | 0x800000u;      // 24-bit significand
  if (te >= 1) {
    const uint32_t w = ((uint32_t)te << 23) | (man & 0x7FFFFFu);
    return (uint16_t)((w + 0x7FFFu + ((w >> 16) & 1u)) >> 16);
  }
  const int drop = 16 + (1 - te);                        // bits below bf16's 2^-133
  if (drop >= 25) return 0;                              // below half the least subnormal
  const uint32_t q = man >> drop, rem = man & ((1u << drop) - 1u), half = 1u << (drop - 1);
  return (uint16_t)(q + ((rem > half || (rem == half && (q & 1u))) ? 1u : 0u));
}

MPM_DEV __nv_bfloat16 mul_to_bf16_once(float a, float b) {
  const float rz = __fmul_rz(a, b);
  if (!isfinite(rz) || a == 0.0f || b == 0.0f) return __float2bfloat16_rn(__fmul_rn(a, b));
  if (fabsf(rz) >= 0x1p-120f) {
    const float err = __fmaf_rn(a, b, -rz);
    uint32_t bits = __float_as_uint(rz);
    if (err != 0.0f) bits |= 1u;
    return __float2bfloat16_rn(__uint_as_float(bits));
  }
  const float a2 = __fmul_rn(fabsf(a), 0x1p64f);          // exact
  const float b2 = fabsf(b);
  const float rz2 = __fmul_rz(a2, b2);                    // >= 2^-95: normal
  const float err2 = __fmaf_rn(a2, b2, -rz2);
  uint32_t bits = __float_as_uint(rz2);
  if (err2 != 0.0f) bits |= 1u;
  uint16_t h = bf16_bits_of_scaled(__uint_as_float(bits), 64);
  if ((a < 0.0f) != (b < 0.0f)) h |= 0x8000u;
  return __ushort_as_bfloat16(h);
}

MPM_DEV float e2m1_value(uint32_t c) {
  // magnitudes of codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6
  const uint32_t m = c & 7u;
  const float mag = m < 4u ? 0.5f * (float)m : (float)(1u << ((m >> 1) - 1u)) * (1.0f + 0.5f * (float)(m & 1u));
  return (c & 8u) ? -mag : mag;
}

// one warp per row; each lane expands 16-element blocks (8 packed bytes)
__global__ void __launch_bounds__(128) nvfp4_dequant_kernel(const uint8_t* __restrict__ q,
                                                           const uint8_t* __restrict__ s,
                                                           const float* __restrict__ outer,
                                                           long long rows_per_outer, long long M,
                                                           int K, __nv_bfloat16* out, long long ldo,
                                                           const int* m_valid) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  long long M_eff = M;
  if (m_valid) { const long long mv = *m_valid; M_eff = mv < M_eff ? mv : M_eff; }
  if (row >= M_eff) return;
  const int nblk = K >> 4;                 // K % 64 == 0: no column padding
  const float sg = outer[row / rows_per_outer];
  const uint8_t* qr = q + row * (long long)(K >> 1);
  for (int b = lane; b < nblk; b += 32) {
    const uint2 w = *reinterpret_cast<const uint2*>(qr + (long long)b * 8);
    const float sb = e4m3_to_f32(s[sf_offset(row, b, nblk)]);
    uint32_t packed[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t byte = ((j < 4 ? w.x : w.y) >> (8 * (j & 3))) & 0xFFu;
      const __nv_bfloat16 h0 = mul_to_bf16_once(__fmul_rn(e2m1_value(byte & 0xFu), sb), sg);
      const __nv_bfloat16 h1 = mul_to_bf16_once(__fmul_rn(e2m1_value(byte >> 4), sb), sg);
      packed[j] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + row * ldo + (long long)b * 16);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  }
}

// MXFP8: E4M3 value x 2^(byte - 127) is exact in fp32; one rounding to bf16
__global__ void __launch_bounds__(128) mxfp8_dequant_kernel(const uint8_t* __restrict__ q,
                                                           const uint8_t* __restrict__ s, long long M,
                                                           int K, __nv_bfloat16* out, long long ldo,
                                                           const int* m_valid) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  long long M_eff = M;
  if (m_valid) { const long long mv = *m_valid; M_eff = mv < M_eff ? mv : M_eff; }
  if (row >= M_eff) return;
  const int nblk = K >> 5;
  const long long cpad = (nblk + 3) / 4 * 4;
  const uint8_t* qr = q + row * (long long)K;
  for (int c = lane; c < (K >> 3); c += 32) {          // 8 codes per step
    const uint2 w = *reinterpret_cast<const uint2*>(qr + (long long)c * 8);
    const uint32_t e8 = s[sf_offset(row, c >> 2, cpad)];
    // 2^(e8 - 127) as an fp32 (e8 in 0..254; 0 is 2^-127, a subnormal)
    const float scale = e8 == 0 ? 0x1p-127f : __uint_as_float(e8 << 23);
    uint32_t packed[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t pair = ((j < 2 ? w.x : w.y) >> (16 * (j & 1))) & 0xFFFFu;
      const float v0 = __fmul_rn(e4m3_to_f32(pair & 0xFFu), scale);
      const float v1 = __fmul_rn(e4m3_to_f32(pair >> 8), scale);
      packed[j] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v0)) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v1)) << 16);
    }
    *reinterpret_cast<uint4*>(out + row * ldo + (long long)c * 8) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

// out[c, r] = in[r, c] for r below the (device) row count; 64 x 64 tiles
// through shared memory so that both the reads and the writes are row runs
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* __restrict__ in,
                                                            long long R, long long C, long long ldi,
                                                            uint16_t* __restrict__ out,
                                                            long long ldo, const int* m_valid) {
  __shared__ uint16_t tile[64][66];
  long long R_eff = R;
  if (m_valid) { const long long mv = *m_valid; R_eff = mv < R_eff ? mv : R_eff; }
  const long long r0 = (long long)blockIdx.y * 64, c0 = (long long)blockIdx.x * 64;
  if (r0 >= R_eff) return;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;   // 64 x 4
  for (int i = ty; i < 64; i += 4) {
    const long long r = r0 + i, c = c0 + tx;
    tile[i][tx] = (r < R_eff && c < C) ? in[r * ldi + c] : (uint16_t)0;
  }
  __syncthreads();
  for (int i = ty; i < 64; i += 4) {
    const long long c = c0 + i, r = r0 + tx;
    if (c < C && r < R_eff) out[c * ldo + r] = tile[tx][i];
  }
}

cudaError_t launch_nvfp4_dequant(const uint8_t* q, const uint8_t* s, const float* outer,
                                 long long rows_per_outer, long long M, int K, void* out,
                                 long long ldo, const int* m_valid, cudaStream_t st) {
  nvfp4_dequant_kernel<<<(unsigned)((M + 3) / 4), 128, 0, st>>>(
      q, s, outer, rows_per_outer, M, K, static_cast<__nv_bfloat16*>(out), ldo, m_valid);
  return cudaGetLastError();
}

cudaError_t launch_mxfp8_dequant(const uint8_t* q, const uint8_t* s, long long M, int K, void* out,
                                 long long ldo, const int* m_valid, cudaStream_t st) {
  mxfp8_dequant_kernel<<<(unsigned)((M + 3) / 4), 128, 0, st>>>(
      q, s, M, K, static_cast<__nv_bfloat16*>(out), ldo, m_valid);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const void* in, long long R, long long C, long long ldi, void* out,
                                  long long ldo, const int* m_valid, cudaStream_t st) {
  const dim3 grid((unsigned)((C + 63) / 64), (unsigned)((R + 63) / 64));
  transpose_bf16_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(in), R, C, ldi,
                                              static_cast<uint16_t*>(out), ldo, m_valid);
  return cudaGetLastError();
}

}  // namespace mpm
