// MXFP8 and NVFP4 quantisers for sm_103a.
//
// NVFP4 (E2M1 codes, E4M3 scale per 16, FP32 outer scale; "Towards
// Blackwell-native 8-bit and 4-bit RL", sections "Format background / NVFP4"
// and "Per-token activation scaling"; "miniTE technical report", section 5.6
// for s_g = amax / 2688).  One warp per row: the row is read once with 128-bit
// loads and kept in registers, the row amax is reduced with warp shuffles, and
// codes plus 128x4-tiled scales are written directly in the operand layout of
// the block-scaled MMA.
//
// MXFP8 (E4M3 codes, E8M0 scale per 32 rounded up; same post, sections
// "Format background / MXFP8" and "Recipe 1 / Training").  A CTA reads a
// 128 x 64 bf16 tile once, writes the row-wise 1x32 copy from registers and the
// column-wise 32x1 copy, transposed, from a shared-memory copy of the tile.
#include <cstring>
#include "quant.cuh"

namespace mpm {

// ============================================================================
// NVFP4
// ============================================================================

// Canonical per-row fp32 sequence, step 2: s_g = a / 2688 with the 2^-116 floor.
MPM_DEV float nvfp4_outer(float a) {
  if (!(a > 0.0f)) return 0.0f;
  float sg = __fdiv_rn(a, 2688.0f);
  const float floor_sg = 0x1p-116f;
  return sg < floor_sg ? floor_sg : sg;
}

struct Nvfp4Rows {
  const __nv_bfloat16* part[4];
  long long part_rows[4];   // rows per group in each part
  int nparts;
  long long R;              // rows per group (sum of part_rows)
  long long ldx;            // elements (single-part activation mode)
  long long rows;           // total rows to quantise (= groups * R)
  long long rows_pad;       // rows whose scale bytes are written (zeros past rows)
  int K;
  int amax_mode;            // 0 = own row max, 1 = amax_in[row], 2 = group amax bits
  const float* amax_in;
  const unsigned* group_amax;
  uint8_t* q;
  uint8_t* s;
  float* ts;                // per row (modes 0/1) or per group (mode 2)
  const int* m_valid;
};

MPM_DEV const __nv_bfloat16* nvfp4_row_ptr(const Nvfp4Rows& p, long long row) {
  if (p.nparts == 1 && p.amax_mode != 2) return p.part[0] + row * p.ldx;
  long long g = row / p.R, lr = row - g * p.R;
  int k = 0;
#pragma unroll
  for (int i = 0; i < 3; ++i)
    if (k < p.nparts - 1 && lr >= p.part_rows[k]) { lr -= p.part_rows[k]; ++k; }
  return p.part[k] + (g * p.part_rows[k] + lr) * (long long)p.K;
}

// {s, s} as the operand of a packed f32x2 multiply
MPM_DEV uint64_t f32x2_splat(float s) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %1};" : "=l"(v) : "f"(s));
  return v;
}
// the bf16 pair in w (low half first) times a power of two, then packed to
// E4M3 (RN, satfinite, low byte first).  Both lanes go through one packed
// f32x2 multiply: per lane the same IEEE product as a scalar multiply (exact
// here), so the codes are those of the scalar path.
MPM_DEV uint32_t e4m3x2_scaled(uint32_t w, uint64_t sc2) {
  uint64_t v, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(bf16lo(w)), "f"(bf16hi(w)));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(v), "l"(sc2));
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(out) : "f"(lo), "f"(hi));
  return out;
}

// the bf16 pair in w times r (one packed f32x2 multiply, per lane the IEEE
// RN product of the scalar path), then packed to one E2M1 byte (RN,
// satfinite, low nibble first)
MPM_DEV uint32_t e2m1x2_scaled(uint32_t w, uint64_t r2) {
  uint64_t v, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(bf16lo(w)), "f"(bf16hi(w)));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(v), "l"(r2));
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
  uint32_t out;
  asm("{\n\t.reg .b8 b;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b, %2, %1;\n\t"
      "cvt.u32.u8 %0, b;\n\t}"
      : "=r"(out) : "f"(lo), "f"(hi));
  return out;
}

// One 16-element block of the canonical NVFP4 sequence: its E4M3 scale byte
// sb = E4M3(bmax / (6 s_g)) and its eight code bytes from x * 1/(E4M3(sb) s_g),
// every step one IEEE binary32 operation (s_g = 0: zero scale and codes).
MPM_DEV uint2 nvfp4_encode_block(const uint4 (&vb)[2], uint32_t bmax16, float sg, float six_sg,
                                 uint32_t& sb) {
  sb = 0;
  if (sg > 0.0f) {
    const float sbf = __fdiv_rn(__uint_as_float(bmax16 << 16), six_sg);
    sb = cvt_e4m3x2(sbf, 0.0f) & 0xFFu;
  }
  const float sbv = e4m3_to_f32(sb);
  uint2 out = make_uint2(0, 0);
  if (sbv > 0.0f) {
    const float r = __frcp_rn(__fmul_rn(sbv, sg));
    const uint32_t w[8] = {vb[0].x, vb[0].y, vb[0].z, vb[0].w, vb[1].x, vb[1].y, vb[1].z, vb[1].w};
    const uint64_t r2 = f32x2_splat(r);
    uint32_t bytes[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) bytes[j] = e2m1x2_scaled(w[j], r2);
    out.x = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
    out.y = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
  }
  return out;
}

// One row of the NVFP4 quantisers, by W lanes of a warp (32: one row per
// warp; 16: one row per half-warp, for rows of at most 64 blocks): the row
// is read once into registers (NB x W lanes x 16 elements), then encoded.
// amax_mode 0 takes the row's own max, 1 amax_in[row], 2 the group amax
// `group_bits` (fp32 bits).  `sub` is the lane within the row's W lanes; a
// row that is not `live` reads and writes nothing but still takes part in
// the warp's shuffles.
template <int NB, int W>
MPM_DEV void nvfp4_quant_row(const Nvfp4Rows& p, long long row, int sub, bool live,
                             uint32_t group_bits) {
  static_assert(W == 32 || W == 16, "a row takes a warp or a half-warp");
  const int nblk = p.K >> 4;
  const long long cols_pad = nblk;          // K % 64 == 0 -> nblk % 4 == 0
  const __nv_bfloat16* xr = nvfp4_row_ptr(p, live ? row : 0);

  uint4 v[NB][2];
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const int b = i * W + sub;
    if (live && b < nblk) {
      const uint4* src = reinterpret_cast<const uint4*>(xr + (long long)b * 16);
      v[i][0] = __ldcs(src);
      v[i][1] = __ldcs(src + 1);
    } else {
      v[i][0] = make_uint4(0, 0, 0, 0);
      v[i][1] = make_uint4(0, 0, 0, 0);
    }
  }
  // per-block |x| max (as bf16 bit patterns) and the lane max
  uint32_t bmax16[NB];
  uint32_t lmax = 0;
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    uint32_t m = 0;
    m = absmax_bf16x2(m, v[i][0].x); m = absmax_bf16x2(m, v[i][0].y);
    m = absmax_bf16x2(m, v[i][0].z); m = absmax_bf16x2(m, v[i][0].w);
    m = absmax_bf16x2(m, v[i][1].x); m = absmax_bf16x2(m, v[i][1].y);
    m = absmax_bf16x2(m, v[i][1].z); m = absmax_bf16x2(m, v[i][1].w);
    m = max(m & 0xFFFFu, m >> 16);
    bmax16[i] = m;
    lmax = max(lmax, m);
  }
  float a;
  if (p.amax_mode == 0) {
    // xor offsets below W stay within the row's lanes
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) lmax = max(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
    a = __uint_as_float(lmax << 16);
  } else if (p.amax_mode == 1) {
    a = live ? p.amax_in[row] : 0.0f;
  } else {
    a = __uint_as_float(group_bits);
  }
  const float sg = nvfp4_outer(a);
  if (!live) return;
  if (sub == 0) {
    if (p.amax_mode != 2) p.ts[row] = sg;
    else if (row % p.R == 0) p.ts[row / p.R] = sg;
  }
  const float six_sg = __fmul_rn(6.0f, sg);
  uint8_t* qr = p.q + row * (long long)(p.K >> 1);
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const int b = i * W + sub;
    if (b >= nblk) continue;
    uint32_t sb;
    const uint2 out = nvfp4_encode_block(v[i], bmax16[i], sg, six_sg, sb);
    *reinterpret_cast<uint2*>(qr + (long long)b * 8) = out;
    p.s[sf_offset(row, b, cols_pad)] = (uint8_t)sb;
  }
}

template <int NB>
__global__ void __launch_bounds__(128) nvfp4_quant_rows_kernel(const Nvfp4Rows p) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  long long rows_eff = p.rows;
  if (p.m_valid) {
    long long mv = *p.m_valid;
    rows_eff = mv < rows_eff ? mv : rows_eff;
    if (row >= rows_eff) return;
  }
  const int nblk = p.K >> 4;
  if (row >= rows_eff) {
    if (row < p.rows_pad) {                 // padding rows of the last tile
      for (int b = lane; b < nblk; b += 32) p.s[sf_offset(row, b, nblk)] = 0;
    }
    return;
  }
  nvfp4_quant_row<NB, 32>(p, row, lane, true, p.amax_mode == 2 ? p.group_amax[row / p.R] : 0u);
}

// Rows of at most 64 blocks (K <= 1024): two rows per warp, one per
// half-warp, so every lane holds blocks (one warp per row left a quarter of
// the lanes idle at K = 768 and kept half as many bytes in flight).
template <int NB>
__global__ void __launch_bounds__(128) nvfp4_quant_rows_half_kernel(const Nvfp4Rows p) {
  const int lane = threadIdx.x & 31, sub = lane & 15;
  const long long row0 = ((long long)blockIdx.x * 4 + (threadIdx.x >> 5)) * 2;   // the warp's rows
  const long long row = row0 + (lane >> 4);
  long long rows_eff = p.rows;
  if (p.m_valid) {
    const long long mv = *p.m_valid;
    rows_eff = mv < rows_eff ? mv : rows_eff;
  }
  const int nblk = p.K >> 4;
  const bool live = row < rows_eff;
  if (row0 < rows_eff)                      // warp-uniform: both halves shuffle together
    nvfp4_quant_row<NB, 16>(p, row, sub, live,
                            (p.amax_mode == 2 && live) ? p.group_amax[row / p.R] : 0u);
  if (!live && !p.m_valid && row < p.rows_pad) {   // padding rows of the last tile
    for (int b = sub; b < nblk; b += 16) p.s[sf_offset(row, b, nblk)] = 0;
  }
}

// ---------------------------------------------------------------- NVFP4, into routed rows
// Per-token quantisation written straight into the expert-ordered rows: the
// bytes of the per-token quantiser followed by the NVFP4 gather, without the
// token-ordered codes in between.  Two launches.  The first takes one token
// per warp: the row is read once and encoded once (the same per-block
// sequence as the per-token quantiser); its codes go to each of its k rows
// inv_perm[t k + j], its scale bytes (four blocks' bytes gathered into one
// word by shuffles) and outer scale to a token-ordered workspace.  The second
// takes 128 rows per block and writes whole 512-byte scale tiles from the
// workspace, the outer scales and zeroed amax slots, and zeros the padding
// rows (perm < 0) below the segment end.  (Writing each token's scale words
// straight into the shared tiles from the first launch, each word in a
// sector the other 127 rows of the tile also write, took 0.44 ms at the
// headline size against 0.25 ms for the codes alone.)
struct NvScatter {
  const __nv_bfloat16* x; long long T; int K; long long ldx;
  const int* inv; int k; const int* perm; const int* seg_end; long long cap;
  uint8_t* q; uint8_t* s; float* ts; float* amax_zero; int* status;
  uint32_t* ws_s;           // [T][K/64] words: the token's scale bytes, 4 blocks per word
  float* ws_ts;             // [T]
};

template <int NB>
__global__ void __launch_bounds__(128) nvfp4_scatter_codes_kernel(const NvScatter a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long t = (long long)blockIdx.x * 4 + warp;
  if (t >= a.T) return;
  long long rend = *a.seg_end;
  if (rend > a.cap) rend = a.cap;
  const int nblk = a.K >> 4;
  const __nv_bfloat16* xr = a.x + t * a.ldx;
  uint4 v[NB][2];
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const int b = i * 32 + lane;
    if (b < nblk) {
      const uint4* src = reinterpret_cast<const uint4*>(xr + (long long)b * 16);
      v[i][0] = __ldcs(src);
      v[i][1] = __ldcs(src + 1);
    } else {
      v[i][0] = make_uint4(0, 0, 0, 0);
      v[i][1] = make_uint4(0, 0, 0, 0);
    }
  }
  uint32_t bmax16[NB];
  uint32_t lmax = 0;
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    uint32_t m = 0;
    m = absmax_bf16x2(m, v[i][0].x); m = absmax_bf16x2(m, v[i][0].y);
    m = absmax_bf16x2(m, v[i][0].z); m = absmax_bf16x2(m, v[i][0].w);
    m = absmax_bf16x2(m, v[i][1].x); m = absmax_bf16x2(m, v[i][1].y);
    m = absmax_bf16x2(m, v[i][1].z); m = absmax_bf16x2(m, v[i][1].w);
    m = max(m & 0xFFFFu, m >> 16);
    bmax16[i] = m;
    lmax = max(lmax, m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lmax = max(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
  const float sg = nvfp4_outer(__uint_as_float(lmax << 16));
  const float six_sg = __fmul_rn(6.0f, sg);
  uint2 codes[NB];
  uint32_t* wsr = a.ws_s + t * (long long)(nblk >> 2);
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    uint32_t sb = 0;
    codes[i] = nvfp4_encode_block(v[i], bmax16[i], sg, six_sg, sb);
    const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sb, 1);
    const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
    const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sb, 3);
    const int b = i * 32 + lane;
    if (b < nblk && (lane & 3) == 0) wsr[b >> 2] = sb | (b1 << 8) | (b2 << 16) | (b3 << 24);
  }
  if (lane == 0) a.ws_ts[t] = sg;
  for (int j = 0; j < a.k; ++j) {
    const long long row = a.inv[t * a.k + j];
    if (row < 0 || row >= rend) {
      if (lane == 0) set_status(a.status, MPM_ERR_DEVICE_BOUNDS);
      continue;
    }
    uint8_t* qr = a.q + row * (long long)(a.K >> 1);
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int b = i * 32 + lane;
      if (b < nblk) *reinterpret_cast<uint2*>(qr + (long long)b * 8) = codes[i];
    }
  }
}

__global__ void __launch_bounds__(128) nvfp4_scatter_rows_kernel(const NvScatter a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long rend = *a.seg_end;
  if (rend > a.cap) rend = a.cap;
  const long long rbase = (long long)blockIdx.x * 128;
  if (rbase >= rend) return;
  const int nrows = (int)min(128LL, rend - rbase);
  __shared__ long long tok[128];            // source token of each row, -1 for padding
  {
    const int i = threadIdx.x;
    long long tk = -1;
    if (i < nrows) {
      const int f = a.perm[rbase + i];
      if (f >= 0) tk = f / a.k;
      if (tk >= a.T) {                      // a slot past the tokens: report, write zeros
        set_status(a.status, MPM_ERR_DEVICE_BOUNDS);
        tk = -1;
      }
      a.ts[rbase + i] = tk >= 0 ? a.ws_ts[tk] : 0.0f;
      if (a.amax_zero) a.amax_zero[rbase + i] = 0.0f;
    }
    tok[i] = tk;
  }
  __syncthreads();
  const long long q16 = a.K / 32;           // 16-byte chunks of codes per row
  for (int i = warp; i < nrows; i += 4) {
    if (tok[i] >= 0) continue;              // real rows: codes written by the first launch
    uint4* d = reinterpret_cast<uint4*>(a.q) + (rbase + i) * q16;
    for (long long c = lane; c < q16; c += 32) d[c] = make_uint4(0, 0, 0, 0);
  }
  // scale tiles: word w of a tile holds row (w % 4) * 32 + w / 4
  const long long ngroups = a.K / 64;       // 4-column groups = tiles per 128 rows
  const long long rt = rbase >> 7;
  const int w = threadIdx.x;
  const int r = (w & 3) * 32 + (w >> 2);
  if (r < nrows) {
    const long long tk = tok[r];
    const uint32_t* src = tk >= 0 ? a.ws_s + tk * ngroups : nullptr;
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.s + rt * ngroups * 512) + w;
    long long g = 0;
    // the token's words four at a time when they are 16-byte aligned, eight
    // such loads in flight before their stores (the rows are L2 hits whose
    // latency, not bandwidth, paces this launch)
    if (src && (ngroups & 3) == 0 && (reinterpret_cast<uintptr_t>(a.ws_s) & 15) == 0) {
      for (; g + 32 <= ngroups; g += 32) {
        uint4 v4[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v4[u] = __ldg(reinterpret_cast<const uint4*>(src + g) + u);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          dst[(g + 4 * u + 0) * 128] = v4[u].x;
          dst[(g + 4 * u + 1) * 128] = v4[u].y;
          dst[(g + 4 * u + 2) * 128] = v4[u].z;
          dst[(g + 4 * u + 3) * 128] = v4[u].w;
        }
      }
      for (; g < ngroups; g += 4) {
        const uint4 v4 = __ldg(reinterpret_cast<const uint4*>(src + g));
        dst[(g + 0) * 128] = v4.x;
        dst[(g + 1) * 128] = v4.y;
        dst[(g + 2) * 128] = v4.z;
        dst[(g + 3) * 128] = v4.w;
      }
    }
    for (; g < ngroups; ++g) dst[g * 128] = src ? src[g] : 0u;
  }
}

// ---------------------------------------------------------------- NVFP4, running amax
// The quantisation of the single-pass FC2 ("miniTE technical report",
// section 5.6): a row of D is consumed in tiles of 256 columns, in order;
// tile t is encoded against gs_t = outer(max |x| over tiles 0 .. t), the
// running row amax, so a tile never waits for the rest of its row.  Same
// canonical fp32 sequence as the per-token quantiser, with gs_t in place of
// s_g.  One warp per row: lane l holds blocks i*32 + l (16 elements each),
// so tile t = 2i + (l >= 16) is the 16 lanes of one half-warp at index i.
template <int NB>
__global__ void __launch_bounds__(128) nvfp4_quant_online_kernel(const Nvfp4Rows p, float* gs_out,
                                                                 int n_tiles) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  long long rows_eff = p.rows;
  if (p.m_valid) {
    long long mv = *p.m_valid;
    rows_eff = mv < rows_eff ? mv : rows_eff;
    if (row >= rows_eff) return;
  }
  const int nblk = p.K >> 4;
  const long long cols_pad = nblk;
  if (row >= rows_eff) {
    if (row < p.rows_pad) {
      for (int b = lane; b < nblk; b += 32) p.s[sf_offset(row, b, cols_pad)] = 0;
    }
    return;
  }
  const __nv_bfloat16* xr = p.part[0] + row * p.ldx;
  uint4 v[NB][2];
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const int b = i * 32 + lane;
    if (b < nblk) {
      const uint4* src = reinterpret_cast<const uint4*>(xr + (long long)b * 16);
      v[i][0] = __ldcs(src);
      v[i][1] = __ldcs(src + 1);
    } else {
      v[i][0] = make_uint4(0, 0, 0, 0);
      v[i][1] = make_uint4(0, 0, 0, 0);
    }
  }
  uint32_t bmax16[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    uint32_t m = 0;
    m = absmax_bf16x2(m, v[i][0].x); m = absmax_bf16x2(m, v[i][0].y);
    m = absmax_bf16x2(m, v[i][0].z); m = absmax_bf16x2(m, v[i][0].w);
    m = absmax_bf16x2(m, v[i][1].x); m = absmax_bf16x2(m, v[i][1].y);
    m = absmax_bf16x2(m, v[i][1].z); m = absmax_bf16x2(m, v[i][1].w);
    bmax16[i] = max(m & 0xFFFFu, m >> 16);
  }
  // tile maxima (bf16 patterns of |x| order like unsigned integers), then
  // the running maximum in tile order: tile 2i, then 2i + 1, then 2i + 2 ...
  const bool upper = lane >= 16;
  uint32_t run = 0;
  float gs_mine[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    uint32_t t = bmax16[i];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) t = max(t, __shfl_xor_sync(0xFFFFFFFFu, t, o));
    const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, t, 16);
    const uint32_t t_lo = upper ? other : t, t_hi = upper ? t : other;
    const uint32_t run_lo = max(run, t_lo);
    run = max(run_lo, t_hi);
    gs_mine[i] = nvfp4_outer(__uint_as_float((upper ? run : run_lo) << 16));
    const int tile = 2 * i + (upper ? 1 : 0);
    if ((lane & 15) == 0 && tile < n_tiles) gs_out[row * n_tiles + tile] = gs_mine[i];
  }
  uint8_t* qr = p.q + row * (long long)(p.K >> 1);
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const int b = i * 32 + lane;
    if (b >= nblk) continue;
    const float sg = gs_mine[i];
    uint32_t sb = 0;
    if (sg > 0.0f) {
      const float sbf = __fdiv_rn(__uint_as_float(bmax16[i] << 16), __fmul_rn(6.0f, sg));
      sb = cvt_e4m3x2(sbf, 0.0f) & 0xFFu;
    }
    const float sbv = e4m3_to_f32(sb);
    uint2 out = make_uint2(0, 0);
    if (sbv > 0.0f) {
      const float r = __frcp_rn(__fmul_rn(sbv, sg));
      const uint32_t w[8] = {v[i][0].x, v[i][0].y, v[i][0].z, v[i][0].w,
                             v[i][1].x, v[i][1].y, v[i][1].z, v[i][1].w};
      const uint64_t r2 = f32x2_splat(r);
      uint32_t bytes[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) bytes[j] = e2m1x2_scaled(w[j], r2);
      out.x = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
      out.y = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
    }
    *reinterpret_cast<uint2*>(qr + (long long)b * 8) = out;
    p.s[sf_offset(row, b, cols_pad)] = (uint8_t)sb;
  }
}

// Per-group amax for the joint weight scale: |x| max over a group's rows of
// all parts, as fp32 bits, reduced with an integer atomicMax (order-free).
struct GroupAmax {
  const __nv_bfloat16* part[4];
  long long part_elems[4];  // elements per group in each part
  int nparts;
  unsigned* out;            // [groups]
};

__global__ void __launch_bounds__(256) group_amax_kernel(const GroupAmax p, int chunks_per_group) {
  const int g = blockIdx.y;
  const int c = blockIdx.x;
  uint32_t m = 0;
  for (int k = 0; k < p.nparts; ++k) {
    const long long n = p.part_elems[k];
    const uint4* src = reinterpret_cast<const uint4*>(p.part[k] + g * n);
    const long long nv = n >> 3;
    const long long per = (nv + chunks_per_group - 1) / chunks_per_group;
    const long long lo = c * per, hi = min(nv, lo + per);
    for (long long i = lo + threadIdx.x; i < hi; i += blockDim.x) {
      uint4 w = __ldcs(src + i);
      m = absmax_bf16x2(m, w.x); m = absmax_bf16x2(m, w.y);
      m = absmax_bf16x2(m, w.z); m = absmax_bf16x2(m, w.w);
    }
  }
  m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ uint32_t wm[8];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = max(r, wm[i]);
    atomicMax(p.out + g, r << 16);
  }
}

// ============================================================================
// MXFP8
// ============================================================================

// Scale exponent e of a block whose |max| has the fp32 bit pattern `bits`:
// the smallest e with a <= 448 * 2^e, clamped to [-127, 127].  For
// a = 1.f * 2^p:  e = p - 8 + [1.f > 1.75].  Zero and subnormal a clamp to -127.
MPM_DEV int mx_exponent(uint32_t bits) {
  const int E = (int)(bits >> 23) & 0xFF;
  if (E == 0) return -127;
  const int e = (E - 127) - 8 + (((bits & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 32 bf16 values (16 words) -> 32 E4M3 codes (8 words) scaled by 2^-e
MPM_DEV void mx_encode32(const uint32_t (&w)[16], float scale, uint32_t (&o)[8]) {
  const uint64_t sc2 = f32x2_splat(scale);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    o[j] = e4m3x2_scaled(w[2 * j], sc2) | (e4m3x2_scaled(w[2 * j + 1], sc2) << 16);
}

MPM_DEV float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

struct Mxfp8Args {
  const __nv_bfloat16* x;
  long long M, K, ldx;
  unsigned flags;
  uint8_t* row_q; uint8_t* row_s; long long row_s_cols_pad;
  uint8_t* col_q; long long ldc; uint8_t* col_s; long long col_s_cols_pad;
  const int* m_valid;
  int pad_blocks;           // 1: zero the scale padding (host-sized buffers)
  int* status;
  // gather form: row r of the quantised matrix is token row perm[r] / kk of
  // x (T rows, stride ldx); perm[r] < 0 marks a zero padding row.  The
  // division is a multiply by div_m with shifts div_s1, div_s2 (see
  // div_magic below); T, ldx < 2^31.
  const int* perm; int kk; long long T;
  uint32_t div_m; int div_s1, div_s2;
};

// Unsigned 32-bit division by an invariant d >= 1 as a multiply and two
// shifts (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, the round-up multiplier with the add-and-shift
// step that keeps it within 32 bits): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (t + ((n - t) >> s1)) >> s2
// for t = mulhi(m, n), s1 = min(l, 1), s2 = max(l - 1, 0), every n < 2^32.
static void div_magic(uint32_t d, uint32_t& m, int& s1, int& s2) {
  int l = 0;
  while ((1ull << l) < d) ++l;
  m = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
  s1 = l < 1 ? l : 1;
  s2 = l > 1 ? l - 1 : 0;
}
MPM_DEV uint32_t div_by_magic(uint32_t n, uint32_t m, int s1, int s2) {
  const uint32_t t = __umulhi(m, n);
  return (t + ((n - t) >> s1)) >> s2;
}

MPM_DEV void zero_scale_padding(uint8_t* s, long long rows, long long cols, long long tid,
                                long long nthreads);

// max |x| over bf16 pairs with packed bf16 abs / max (finite inputs), as the
// 16-bit pattern of the larger magnitude in the low half
template <int N>
MPM_DEV uint32_t absmax_bf16x2_packed(const uint32_t (&w)[N]) {
  __nv_bfloat162 acc = __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[0]));
#pragma unroll
  for (int j = 1; j < N; ++j) acc = __hmax2(acc, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[j])));
  const uint32_t m = *reinterpret_cast<uint32_t*>(&acc);
  return max(m & 0xFFFFu, m >> 16);
}

// ---------------------------------------------------------------- MXFP8, TMA-staged
// Persistent CTAs walk 128 x 64 tiles of x; a 2-deep ring of TMA loads keeps
// the next tiles in flight while a tile is encoded from shared memory (two
// 16 KB input stages and two 16 KB code-staging buffers, 66.6 KB per CTA:
// three CTAs per SM; deeper rings, and one staging buffer at four CTAs per
// SM, measured slower).
// Row pass: one thread per 32-element row block (its 64 bytes in four
// 16-byte loads).  Column pass: a pair of adjacent columns x 16 rows per thread
// (two threads per pair of 32-row column blocks, see below).  The tile is
// staged with the 128-byte swizzle.
constexpr int MQ_TM = 128, MQ_TK = 64, MQ_STAGES = 2;
constexpr int MQ_TILE_BYTES = MQ_TM * MQ_TK * 2;     // 16 KB

// Codes of a full tile (all 128 rows below the valid row count, all 64
// columns inside K) leave through shared memory by TMA stores: the
// row-wise codes as a 128 x 64-byte box, the transposed column-wise codes as
// a 64 x 128-byte box (128-byte swizzle), double-buffered so a tile's
// stores drain while the next tile is encoded.  Measured without any code
// stores the kernel ran in 56 % of its time: the per-thread stores (each
// warp's column-copy store touching 32 lines) were the bound.  Edge tiles
// keep the per-thread stores, and the scale bytes always use them.
constexpr int MQ_OUT_BYTES = MQ_TM * MQ_TK + MQ_TK * MQ_TM;     // 8 KB rows + 8 KB columns

// 16-byte global -> shared copy, zero-filled past n bytes (n = 0 or 16)
MPM_DEV void cp_async_16(uint32_t dst, const void* src, uint32_t n) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
MPM_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
MPM_DEV void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
MPM_DEV void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Tile cursor: tile (mt, kt) of the row-major tile order (kt fastest), moved
// by the grid stride without a division per step.
struct MqCursor {
  int mt, kt;
  MPM_DEV void init(int ti, int n_kt) { mt = ti / n_kt; kt = ti - mt * n_kt; }
  MPM_DEV void step(int dq, int dr, int n_kt) {
    kt += dr; mt += dq;
    if (kt >= n_kt) { kt -= n_kt; ++mt; }
  }
};

// Gather form of the tile load: the 128 routed rows of a tile come from
// their tokens' rows of x.  Thread t copies 16-byte chunk t % 8 of rows
// t / 8 + 32 j (j < 4) to the 128-byte-swizzled offset a TMA load of the
// gathered matrix would have used, so the encode passes read the stage
// unchanged; rows past the valid count, padding rows and columns past K are
// zero-filled.  A warp's 16 rows are looked up once each, by lanes 0-15
// (lane 4 j + q: row 4 w + q + 32 j), one tile before the copies are issued,
// and handed to the copying lanes by shuffle.
MPM_DEV int mq_lookup(const Mxfp8Args& p, const MqCursor& c, int n_mt, int M_eff, int warp,
                      int lane) {
  if (lane >= 16 || c.mt >= n_mt) return -1;
  const int row = c.mt * MQ_TM + warp * 4 + (lane & 3) + 32 * (lane >> 2);
  return row < M_eff ? __ldg(p.perm + row) : -1;
}

// One copy group per tile (committed even when empty, so the group count
// stays uniform).  dst_off: this thread's offset for j = 0 (rows j > 0 sit
// 4096 bytes apart with the same swizzle phase).  A zero-filled copy still
// names an address inside x: token 0 at the chunk's column, or column 0 when
// the chunk lies past K.
MPM_DEV void mq_gather_issue(const Mxfp8Args& p, uint32_t dst, const MqCursor& c, int f,
                             uint32_t dst_off, int lane) {
  int tok = -1;
  if (f >= 0) {
    tok = (int)div_by_magic((uint32_t)f, p.div_m, p.div_s1, p.div_s2);
    if (tok >= (int)p.T) { set_status(p.status, MPM_ERR_DEVICE_BOUNDS); tok = -1; }
  }
  const int col = c.kt * MQ_TK + (lane & 7) * 8;
  const bool col_ok = col < (int)p.K;
  const __nv_bfloat16* xc = p.x + (col_ok ? col : 0);
  const uint32_t ldx = (uint32_t)p.ldx;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tj = __shfl_sync(0xffffffffu, tok, 4 * j + (lane >> 3));
    const bool on = col_ok && tj >= 0;
    const __nv_bfloat16* src = xc + (size_t)((uint32_t)max(tj, 0)) * ldx;
    cp_async_16(dst + dst_off + 4096u * j, src, on ? 16u : 0u);
  }
  cp_async_commit();
}

template <bool GATHER>
__global__ void __launch_bounds__(256) mxfp8_quant_tma_kernel(const __grid_constant__ CUtensorMap tx,
                                                             const __grid_constant__ CUtensorMap trow,
                                                             const __grid_constant__ CUtensorMap tcol,
                                                             const Mxfp8Args p, int n_kt) {
  extern __shared__ uint8_t mq_smem[];
  const uint32_t raw = smem_u32(mq_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint8_t* gbase = mq_smem + (base - raw);
  const uint32_t sOut = base + MQ_STAGES * MQ_TILE_BYTES;        // two output buffers
  const uint32_t bar = sOut + 2 * MQ_OUT_BYTES;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // launched as a programmatic dependent: no global access before this wait;
  // the grid is persistent (every CTA resident), so the next launch may
  // begin its prologue on the SMs this grid's CTAs leave
  pdl_wait();
  pdl_launch_dependents();
  long long M_eff = p.M;
  if (p.m_valid) { const long long mv = *p.m_valid; M_eff = mv < M_eff ? mv : M_eff; }
  const long long n_tiles = (M_eff + MQ_TM - 1) / MQ_TM * n_kt;
  if (t == 0) {
    if (!GATHER) {
      for (int s = 0; s < MQ_STAGES; ++s) mbar_init(bar + 8 * s, 1);
      fence_mbar_init();
      prefetch_tmap(&tx);
    }
    if (p.flags & MPM_ROWWISE) prefetch_tmap(&trow);
    if (p.flags & MPM_COLWISE) prefetch_tmap(&tcol);
    for (int i = 0; i < MQ_STAGES && !GATHER; ++i) {
      const long long ti = blockIdx.x + (long long)i * gridDim.x;
      if (ti >= n_tiles) break;
      mbar_arrive_expect_tx(bar + 8 * i, MQ_TILE_BYTES);
      tma_load_2d(base + i * MQ_TILE_BYTES, &tx, (int)((ti % n_kt) * MQ_TK), (int)((ti / n_kt) * MQ_TM),
                  bar + 8 * i);
    }
  }
  // gather form: tile cursors (no division per tile); the first MQ_STAGES
  // tiles in flight, nxt left on tile MQ_STAGES with its row lookup loaded
  const int n_mt = (int)((M_eff + MQ_TM - 1) / MQ_TM);   // tile counts fit 31 bits (host-checked)
  const int dq = (int)gridDim.x / n_kt, dr = (int)gridDim.x - dq * n_kt;
  MqCursor cur, nxt;                                // this tile; the next tile to load
  int fn = -1;                                      // row lookup of tile nxt
  const uint32_t dst_off = (uint32_t)((t >> 3) * 128 + (((t & 7) ^ ((t >> 3) & 7)) << 4));
  if (GATHER) {
    cur.init((int)blockIdx.x, n_kt);
    nxt = cur;
    for (int i = 0; i < MQ_STAGES; ++i) {
      fn = mq_lookup(p, nxt, n_mt, (int)M_eff, warp, lane);
      if (nxt.mt < n_mt) mq_gather_issue(p, base + i * MQ_TILE_BYTES, nxt, fn, dst_off, lane);
      else cp_async_commit();
      nxt.step(dq, dr, n_kt);
    }
    fn = mq_lookup(p, nxt, n_mt, (int)M_eff, warp, lane);
  }
  __syncthreads();
  int it = 0, last_buf = -1;                        // last_buf: thread 0's newest store group
  for (long long ti = blockIdx.x; ti < n_tiles; ti += gridDim.x, ++it) {
    const int s = it % MQ_STAGES;
    bool ok = true;
    if (GATHER) cp_async_wait1();                   // this thread's copies of tile it (two groups ring)
    else ok = mbar_wait(bar + 8 * s, (uint32_t)(it / MQ_STAGES) & 1u, p.status);
    // output buffer it % 2 is free once the store groups that read it have:
    // all but the newest group, or all of them when the newest used it too
    // (only full tiles commit a group)
    if (t == 0) {
      if (last_buf == (it & 1)) bulk_wait_group_read0();
      else bulk_wait_group_read1();
    }
    if (__syncthreads_or(!ok)) break;
    const uint8_t* tile = gbase + s * MQ_TILE_BYTES;          // row r at r * 128 bytes
    const long long m0 = GATHER ? (long long)cur.mt * MQ_TM : (ti / n_kt) * MQ_TM;
    const long long k0 = GATHER ? (long long)cur.kt * MQ_TK : (ti % n_kt) * MQ_TK;
    const bool full = (m0 + MQ_TM <= M_eff) && (k0 + MQ_TK <= p.K);
    const uint32_t orow = sOut + (it & 1) * MQ_OUT_BYTES;     // [128 rows][64 B]
    const uint32_t ocol = orow + MQ_TM * MQ_TK;               // [64 columns][128 B], swizzled
    if (p.flags & MPM_ROWWISE) {
      // one thread per 32-element row block: warp w takes rows 16 w .. 16 w + 15,
      // lanes 2 i and 2 i + 1 the two blocks of row 16 w + i; with the swizzle
      // each of the four 16-byte loads is four conflict-free wavefronts
      const int rr = warp * 16 + (lane >> 1), bl = lane & 1;
      const long long row = m0 + rr, col = k0 + bl * 32;
      uint32_t w[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(
            tile + rr * 128 + ((((bl << 2) | c) ^ (rr & 7)) << 4));
        w[4 * c] = u.x; w[4 * c + 1] = u.y; w[4 * c + 2] = u.z; w[4 * c + 3] = u.w;
      }
      if (row < M_eff && col < p.K) {
        const int e = mx_exponent(absmax_bf16x2_packed(w) << 16);
        uint32_t o[8];
        mx_encode32(w, pow2_neg(e), o);
        if (full) {
          const uint32_t a = orow + rr * MQ_TK + bl * 32;
          st_shared_v4(a, o[0], o[1], o[2], o[3]);
          st_shared_v4(a + 16, o[4], o[5], o[6], o[7]);
        } else {
          uint4* d = reinterpret_cast<uint4*>(p.row_q + row * p.K + col);
          d[0] = make_uint4(o[0], o[1], o[2], o[3]);
          d[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
        p.row_s[sf_offset(row, col >> 5, p.row_s_cols_pad)] = (uint8_t)(e + 127);
      }
    }
    if (p.flags & MPM_COLWISE) {
      // Thread = a pair of adjacent columns x 16 of a 32-row block: warp w
      // takes row block w / 2 and column pairs 16 (w % 2) .. + 15; the two
      // lanes of a pair split the block's rows by bit 2 (rows 8a + b and
      // 8a + 4 + b, b < 4), so at each load the warp's two halves read rows
      // whose 128-byte swizzle differs by 4 chunks: 32 lanes, 32 banks.
      const int g = warp >> 1, half = lane & 1;
      const int cp = (warp & 1) * 16 + (lane >> 1);      // column pair 0..31
      const long long mb = m0 + g * 32;
      const long long nvalid = M_eff - mb;
      const int chunk = cp >> 2, within = (cp & 3) * 4;
      // row 32 g + 8 a + 4 half + b sits at lane_base + 1024 a + 128 b +
      // swizzled chunk offset; the four offsets (b = 0..3) are fixed per lane
      const uint8_t* lane_base = tile + g * 4096 + half * 512 + within;
      int off[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) off[b] = ((chunk ^ (half * 4 + b)) << 4) + b * 128;
      uint32_t wv[16];                                  // row r: (col 2cp, col 2cp + 1)
#pragma unroll
      for (int j = 0; j < 16; ++j)
        wv[j] = *reinterpret_cast<const uint32_t*>(lane_base + (j >> 2) * 1024 + off[j & 3]);
      if (nvalid < 32) {                                // rows past the valid count
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if ((j >> 2) * 8 + half * 4 + (j & 3) >= nvalid) wv[j] = 0;
      }
      uint32_t m = 0;
      {
        __nv_bfloat162 acc = __habs2(*reinterpret_cast<const __nv_bfloat162*>(&wv[0]));
#pragma unroll
        for (int j = 1; j < 16; ++j)
          acc = __hmax2(acc, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&wv[j])));
        m = *reinterpret_cast<uint32_t*>(&acc);
      }
      const uint32_t mo = __shfl_xor_sync(0xffffffffu, m, 1);
      // this lane's column (2cp + half) exponent; the partner's by shuffle
      const uint32_t mine = half ? max(m >> 16, mo >> 16) : max(m & 0xFFFFu, mo & 0xFFFFu);
      const int e_own = mx_exponent(mine << 16);
      const int e_oth = __shfl_xor_sync(0xffffffffu, e_own, 1);
      const int e0 = half ? e_oth : e_own, e1 = half ? e_own : e_oth;
      const uint64_t s0 = f32x2_splat(pow2_neg(e0)), s1 = f32x2_splat(pow2_neg(e1));
      // codes of four consecutive rows per word: column 2cp in p0, 2cp + 1 in p1
      uint32_t p0[4], p1[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const uint32_t x0 = wv[4 * a], x1 = wv[4 * a + 1], x2 = wv[4 * a + 2], x3 = wv[4 * a + 3];
        p0[a] = e4m3x2_scaled(__byte_perm(x0, x1, 0x5410), s0) |
                (e4m3x2_scaled(__byte_perm(x2, x3, 0x5410), s0) << 16);
        p1[a] = e4m3x2_scaled(__byte_perm(x0, x1, 0x7632), s1) |
                (e4m3x2_scaled(__byte_perm(x2, x3, 0x7632), s1) << 16);
      }
      // lane 0 of the pair ends with all 32 rows of column 2cp, lane 1 with
      // column 2cp + 1: each passes the other column's words to its partner
      uint32_t o[8];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const uint32_t got = __shfl_xor_sync(0xffffffffu, half ? p0[a] : p1[a], 1);
        o[2 * a] = half ? got : p0[a];
        o[2 * a + 1] = half ? p1[a] : got;
      }
      const long long col = k0 + 2 * cp + half;
      if (full) {
        // column c of the tile is row c of the staged box; this thread's 32
        // codes are 16-byte chunks 2g and 2g + 1 of it, 128-byte swizzled
        const int cr = 2 * cp + half;
        const uint32_t rowa = ocol + cr * MQ_TM;
        st_shared_v4(rowa + (((2 * g) ^ (cr & 7)) << 4), o[0], o[1], o[2], o[3]);
        st_shared_v4(rowa + (((2 * g + 1) ^ (cr & 7)) << 4), o[4], o[5], o[6], o[7]);
        p.col_s[sf_offset(col, mb >> 5, p.col_s_cols_pad)] = (uint8_t)(e_own + 127);
      } else if (col < p.K && mb < M_eff) {
        uint8_t* dst = p.col_q + col * p.ldc + mb;
        if (nvalid >= 32) {
          uint4* d4 = reinterpret_cast<uint4*>(dst);
          d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
          d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nvalid) dst[j] = (uint8_t)(o[j >> 2] >> (8 * (j & 3)));
        }
        p.col_s[sf_offset(col, mb >> 5, p.col_s_cols_pad)] = (uint8_t)(e_own + 127);
      }
    }
    if (full) fence_proxy_async();                    // staged codes visible to the TMA stores
    __syncthreads();                                  // stage s fully read
    if (t == 0) {
      if (full) {
        if (p.flags & MPM_ROWWISE) tma_store_2d(&trow, (int)k0, (int)m0, orow);
        if (p.flags & MPM_COLWISE) tma_store_2d(&tcol, (int)m0, (int)k0, ocol);
        bulk_commit_group();
        last_buf = it & 1;
      }
      const long long tn = ti + (long long)MQ_STAGES * gridDim.x;
      if (!GATHER && tn < n_tiles) {
        mbar_arrive_expect_tx(bar + 8 * s, MQ_TILE_BYTES);
        tma_load_2d(base + s * MQ_TILE_BYTES, &tx, (int)((tn % n_kt) * MQ_TK),
                    (int)((tn / n_kt) * MQ_TM), bar + 8 * s);
      }
    }
    if (GATHER) {
      if (nxt.mt < n_mt) mq_gather_issue(p, base + s * MQ_TILE_BYTES, nxt, fn, dst_off, lane);
      else cp_async_commit();
      nxt.step(dq, dr, n_kt);
      fn = mq_lookup(p, nxt, n_mt, (int)M_eff, warp, lane);
      cur.step(dq, dr, n_kt);
    }
  }
  if (GATHER) cp_async_wait0();                     // no copy outlives the CTA (loop left early)
  if (t == 0) bulk_wait_group0();                   // the code stores have completed
  if (p.pad_blocks) {
    // host-sized buffers: zero the padding entries of the scale tiles
    const long long tid = (long long)blockIdx.x * blockDim.x + t;
    const long long nth = (long long)gridDim.x * blockDim.x;
    if (p.flags & MPM_ROWWISE) zero_scale_padding(p.row_s, p.M, p.K / 32, tid, nth);
    if (p.flags & MPM_COLWISE) zero_scale_padding(p.col_s, p.K, (p.M + 31) / 32, tid, nth);
  }
}

MPM_DEV void zero_scale_padding(uint8_t* s, long long rows, long long cols, long long tid,
                                long long nthreads) {
  const long long rows_pad = (rows + 127) / 128 * 128, cols_pad = (cols + 3) / 4 * 4;
  const long long ncp = cols_pad - cols;
  const long long nA = rows * ncp;
  const long long nB = (rows_pad - rows) * cols_pad;
  for (long long i = tid; i < nA + nB; i += nthreads) {
    long long r, c;
    if (i < nA) { r = i / ncp; c = cols + i % ncp; }
    else { long long j = i - nA; r = rows + j / cols_pad; c = j % cols_pad; }
    s[sf_offset(r, c, cols_pad)] = 0;
  }
}


// ============================================================================
// launchers
// ============================================================================

static int nb_for(int nblk) {
  const int need = (nblk + 31) / 32;
  const int opts[] = {1, 2, 4, 8, 14, 16};
  for (int o : opts) if (o >= need) return o;
  return -1;
}

static cudaError_t launch_nvfp4_rows(const Nvfp4Rows& p, cudaStream_t st) {
  const int nblk = p.K >> 4;
  const long long rows = p.rows_pad > p.rows ? p.rows_pad : p.rows;
  if (nblk <= 64) {                          // two rows per warp, eight per block
    const dim3 grid((unsigned)((rows + 7) / 8)), block(128);
    switch ((nblk + 15) / 16) {
      case 1: nvfp4_quant_rows_half_kernel<1><<<grid, block, 0, st>>>(p); break;
      case 2: nvfp4_quant_rows_half_kernel<2><<<grid, block, 0, st>>>(p); break;
      case 3: nvfp4_quant_rows_half_kernel<3><<<grid, block, 0, st>>>(p); break;
      case 4: nvfp4_quant_rows_half_kernel<4><<<grid, block, 0, st>>>(p); break;
      default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  const int nb = nb_for(nblk);
  const long long warps = rows;
  const dim3 grid((unsigned)((warps + 3) / 4)), block(128);
  switch (nb) {
    case 1: nvfp4_quant_rows_kernel<1><<<grid, block, 0, st>>>(p); break;
    case 2: nvfp4_quant_rows_kernel<2><<<grid, block, 0, st>>>(p); break;
    case 4: nvfp4_quant_rows_kernel<4><<<grid, block, 0, st>>>(p); break;
    case 8: nvfp4_quant_rows_kernel<8><<<grid, block, 0, st>>>(p); break;
    case 14: nvfp4_quant_rows_kernel<14><<<grid, block, 0, st>>>(p); break;
    case 16: nvfp4_quant_rows_kernel<16><<<grid, block, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_per_token(const void* x, long long M, int K, long long ldx,
                                   const float* amax_in, uint8_t* q, uint8_t* s, float* ts,
                                   const int* m_valid, cudaStream_t st) {
  Nvfp4Rows p{};
  p.part[0] = static_cast<const __nv_bfloat16*>(x);
  p.part_rows[0] = M;
  p.nparts = 1;
  p.R = M;
  p.ldx = ldx;
  p.rows = M;
  p.rows_pad = m_valid ? M : (M + 127) / 128 * 128;
  p.K = K;
  p.amax_mode = amax_in ? 1 : 0;
  p.amax_in = amax_in;
  p.q = q; p.s = s; p.ts = ts;
  p.m_valid = m_valid;
  return launch_nvfp4_rows(p, st);
}

cudaError_t launch_nvfp4_weight(const void* const* parts, const long long* part_rows, int nparts,
                                int K, long long E, uint8_t* q, uint8_t* s, float* ts,
                                unsigned* ws, cudaStream_t st) {
  cudaError_t err = cudaMemsetAsync(ws, 0, (size_t)E * sizeof(unsigned), st);
  if (err != cudaSuccess) return err;
  GroupAmax ga{};
  long long R = 0;
  for (int i = 0; i < nparts; ++i) {
    ga.part[i] = static_cast<const __nv_bfloat16*>(parts[i]);
    ga.part_elems[i] = part_rows[i] * K;
    R += part_rows[i];
  }
  ga.nparts = nparts;
  ga.out = ws;
  const long long per_group = R * K;
  int chunks = (int)((per_group + (1 << 20) - 1) >> 20);   // ~1M elements per CTA
  if (chunks < 1) chunks = 1;
  if (chunks > 1024) chunks = 1024;
  group_amax_kernel<<<dim3(chunks, (unsigned)E), 256, 0, st>>>(ga, chunks);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  Nvfp4Rows p{};
  for (int i = 0; i < nparts; ++i) {
    p.part[i] = ga.part[i];
    p.part_rows[i] = part_rows[i];
  }
  p.nparts = nparts;
  p.R = R;
  p.ldx = K;
  p.rows = E * R;
  p.rows_pad = E * R;
  p.K = K;
  p.amax_mode = 2;
  p.group_amax = ws;
  p.q = q; p.s = s; p.ts = ts;
  p.m_valid = nullptr;
  return launch_nvfp4_rows(p, st);
}

cudaError_t launch_nvfp4_online(const void* x, long long M, int K, long long ldx, uint8_t* q,
                                uint8_t* s, float* gs, const int* m_valid, cudaStream_t st) {
  Nvfp4Rows p{};
  p.part[0] = static_cast<const __nv_bfloat16*>(x);
  p.part_rows[0] = M;
  p.nparts = 1;
  p.R = M;
  p.ldx = ldx;
  p.rows = M;
  p.rows_pad = m_valid ? M : (M + 127) / 128 * 128;
  p.K = K;
  p.q = q; p.s = s;
  p.m_valid = m_valid;
  const int n_tiles = K / 256;
  const dim3 grid((unsigned)((p.rows_pad + 3) / 4)), block(128);
  switch (nb_for(K >> 4)) {
    case 1: nvfp4_quant_online_kernel<1><<<grid, block, 0, st>>>(p, gs, n_tiles); break;
    case 2: nvfp4_quant_online_kernel<2><<<grid, block, 0, st>>>(p, gs, n_tiles); break;
    case 4: nvfp4_quant_online_kernel<4><<<grid, block, 0, st>>>(p, gs, n_tiles); break;
    case 8: nvfp4_quant_online_kernel<8><<<grid, block, 0, st>>>(p, gs, n_tiles); break;
    case 14: nvfp4_quant_online_kernel<14><<<grid, block, 0, st>>>(p, gs, n_tiles); break;
    case 16: nvfp4_quant_online_kernel<16><<<grid, block, 0, st>>>(p, gs, n_tiles); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

size_t nvfp4_scatter_ws_bytes(long long T, int K) {
  return (size_t)T * (size_t)(K / 16) + (size_t)T * sizeof(float) + 16;
}

cudaError_t launch_nvfp4_quantize_scatter(const void* x, long long T, int K, long long ldx,
                                          const int* inv, int k, const int* perm,
                                          const int* seg_end, long long cap, uint8_t* q,
                                          uint8_t* s, float* ts, float* amax_zero, void* ws,
                                          int* status, cudaStream_t st) {
  NvScatter a{};
  a.x = static_cast<const __nv_bfloat16*>(x); a.T = T; a.K = K; a.ldx = ldx;
  a.inv = inv; a.k = k; a.perm = perm; a.seg_end = seg_end; a.cap = cap;
  a.q = q; a.s = s; a.ts = ts; a.amax_zero = amax_zero; a.status = status;
  a.ws_s = static_cast<uint32_t*>(ws);
  a.ws_ts = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + (size_t)T * (size_t)(K / 16));
  const dim3 g1((unsigned)((T + 3) / 4)), block(128);
  switch (nb_for(K >> 4)) {
    case 1: nvfp4_scatter_codes_kernel<1><<<g1, block, 0, st>>>(a); break;
    case 2: nvfp4_scatter_codes_kernel<2><<<g1, block, 0, st>>>(a); break;
    case 4: nvfp4_scatter_codes_kernel<4><<<g1, block, 0, st>>>(a); break;
    case 8: nvfp4_scatter_codes_kernel<8><<<g1, block, 0, st>>>(a); break;
    case 14: nvfp4_scatter_codes_kernel<14><<<g1, block, 0, st>>>(a); break;
    case 16: nvfp4_scatter_codes_kernel<16><<<g1, block, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  nvfp4_scatter_rows_kernel<<<(unsigned)((cap + 127) / 128), block, 0, st>>>(a);
  return cudaGetLastError();
}

template <bool GATHER>
static cudaError_t launch_mxfp8_impl(const CUtensorMap& tx, const CUtensorMap& trow,
                                     const CUtensorMap& tcol, const Mxfp8Args& p,
                                     cudaStream_t st) {
  const int n_kt = (int)((p.K + MQ_TK - 1) / MQ_TK);
  const long long n_tiles = (p.M + MQ_TM - 1) / MQ_TM * n_kt;
  if (n_tiles > (1ll << 30)) return cudaErrorInvalidValue;   // tile cursors are 32-bit
  constexpr int smem = 1024 + MQ_STAGES * MQ_TILE_BYTES + 2 * MQ_OUT_BYTES + 64;
  static int ctas[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && ctas[dev] == 0) {
    err = cudaFuncSetAttribute(mxfp8_quant_tma_kernel<GATHER>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    int sms = 0, per = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, mxfp8_quant_tma_kernel<GATHER>, 256, smem);
    ctas[dev] = (sms > 0 ? sms : 1) * (per > 0 ? per : 1);
  }
  long long grid = dev < 64 ? ctas[dev] : 1;
  if (grid > n_tiles) grid = n_tiles;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mxfp8_quant_tma_kernel<GATHER>, tx, trow, tcol, p, n_kt);
}

static Mxfp8Args mxfp8_args(long long M, long long K, long long ldx, unsigned flags,
                            uint8_t* row_q, uint8_t* row_s, uint8_t* col_q, long long ldc,
                            uint8_t* col_s, const int* m_valid, int* status) {
  Mxfp8Args p{};
  p.M = M; p.K = K; p.ldx = ldx; p.flags = flags;
  p.row_q = row_q; p.row_s = row_s; p.row_s_cols_pad = (K / 32 + 3) / 4 * 4;
  p.col_q = col_q; p.ldc = ldc; p.col_s = col_s;
  p.col_s_cols_pad = ((M + 31) / 32 + 3) / 4 * 4;
  p.m_valid = m_valid;
  p.pad_blocks = m_valid ? 0 : 1;
  p.status = status;
  return p;
}

cudaError_t launch_mxfp8_tma(const CUtensorMap& tx, const CUtensorMap& trow, const CUtensorMap& tcol,
                             long long M, long long K, long long ldx,
                             unsigned flags, uint8_t* row_q, uint8_t* row_s, uint8_t* col_q,
                             long long ldc, uint8_t* col_s, const int* m_valid, int* status,
                             cudaStream_t st) {
  const Mxfp8Args p = mxfp8_args(M, K, ldx, flags, row_q, row_s, col_q, ldc, col_s, m_valid, status);
  return launch_mxfp8_impl<false>(tx, trow, tcol, p, st);
}

cudaError_t launch_mxfp8_gather(const CUtensorMap& trow, const CUtensorMap& tcol, const void* x,
                                long long T, long long K, long long ldx, const int* perm, int k,
                                const int* seg_end, long long cap, unsigned flags,
                                uint8_t* row_q, uint8_t* row_s, uint8_t* col_q, long long ldc,
                                uint8_t* col_s, int* status, cudaStream_t st) {
  Mxfp8Args p = mxfp8_args(cap, K, ldx, flags, row_q, row_s, col_q, ldc, col_s, seg_end, status);
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.perm = perm; p.kk = k; p.T = T;
  div_magic((uint32_t)k, p.div_m, p.div_s1, p.div_s2);
  CUtensorMap none;
  std::memset(&none, 0, sizeof(none));
  return launch_mxfp8_impl<true>(none, trow, tcol, p, st);
}

}  // namespace mpm
