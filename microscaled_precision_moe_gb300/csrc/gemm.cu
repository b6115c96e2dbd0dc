// Block-scaled grouped GEMM on the 5th-generation tensor cores (sm_103a).
//
// C_e = A_e * B_e^T with A and B K-major, NVFP4 (kind::mxf4nvf4, E2M1 with an
// E4M3 scale per 16 values) or MXFP8 (kind::mxf8f6f4, E4M3 with an E8M0 scale
// per 32 values), fp32 accumulation in tensor memory.
//
// "miniTE technical report", section 5.2: the quantised operands of all
// experts sit in one contiguous buffer with expert offsets on the device, so
// one launch covers every expert without host synchronisation; section 5.4:
// the FC1 epilogue applies alpha_a[m] (x alpha_b), forms gate|up,
// D = act(gate, up) x prob and reduces the row amax of D.  "Towards
// Blackwell-native 8-bit and 4-bit RL", section "Recipe 1 / Training": dgrad
// uses the column-wise weight copy and wgrad the column-wise activation and
// gradient copies (the GROUP_K mode below contracts over each expert's rows).
//
// One CTA computes one 128 x 256 output tile:
//   warp 0 lane 0  TMA producer: A/B tiles (128-byte swizzle) and the 128x4
//                  scale tiles (bulk copies) into a 4-stage shared-memory ring
//   warp 3 lane 0  copies each stage's scale tiles into TMEM (tcgen05.cp)
//   warp 1 lane 0  MMA issuer: tcgen05.mma with block scaling once a stage's
//                  scale tiles are in TMEM; commits free ring slots
//   warp 2         allocates / frees the 512 TMEM columns
//   warps 0-3      epilogue: tcgen05.ld of the fp32 accumulator (one row per
//                  thread), outer scales, optional SwiGLU / SwiGLU backward,
//                  stores
// Every mbarrier wait is bounded; a timeout sets the device status word and
// the CTA skips the rest of its work.
#include "gemm.cuh"

namespace mpm {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BKB = 128;             // bytes of K per stage (one swizzle row)
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BKB;    // 16 KB
constexpr int B_STAGE = BN * BKB;    // 32 KB
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_TMEM_BASE = 256;

template <int KIND> struct KindCfg;
template <> struct KindCfg<MPM_KIND_NVFP4> {
  static constexpr int kElemsPerKB = 256;     // FP4 elements per 128 bytes
  static constexpr int kAtomsPerKB = 4;       // 128x4 scale tiles per 128 rows
  static constexpr int kSfaBytes = 4 * 512;
  static constexpr int kSfbBytes = 2 * 4 * 512;
  static constexpr int kSfTmemPerStage = 16 + 32;
  static constexpr uint32_t kFmt = 1, kUe8m0 = 0;
};
template <> struct KindCfg<MPM_KIND_MXFP8> {
  static constexpr int kElemsPerKB = 128;
  static constexpr int kAtomsPerKB = 1;
  static constexpr int kSfaBytes = 512;
  static constexpr int kSfbBytes = 2 * 512;
  static constexpr int kSfTmemPerStage = 4 + 8;
  static constexpr uint32_t kFmt = 0, kUe8m0 = 1;
};

template <int KIND>
constexpr int smem_bytes() {
  return 1024 /*alignment slack*/ +
         STAGES * (A_STAGE + B_STAGE + KindCfg<KIND>::kSfaBytes + KindCfg<KIND>::kSfbBytes) +
         (3 * STAGES + 1) * 8 + 16;
}

MPM_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

template <int KIND, int EPI>
__global__ void __launch_bounds__(128, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tma_a,
                    const __grid_constant__ CUtensorMap tma_b, const GemmArgs p) {
  using Cfg = KindCfg<KIND>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ------------------------------------------------------------ tile -> work
  int e = 0;
  long long row0 = 0;        // first row of A / of the output tile
  int num_kb = 0;
  long long ka_elem = 0;     // reduction offset (elements) of A
  long long kb_elem = 0;     // reduction offset (elements) of B
  long long brow[2];         // global B rows of the two 128-row halves
  long long out_row_base = 0;
  const long long n0 = (long long)blockIdx.x * ((EPI == MPM_EPI_SWIGLU || EPI == MPM_EPI_SWIGLU_SAVE) ? BN / 2 : BN);
  if (p.group == MPM_GROUP_M) {
    row0 = (long long)blockIdx.y * BM;
    long long seg_end = p.a_rows;
    if (p.seg) {
      seg_end = p.seg[p.E];
      if (seg_end > p.a_rows || seg_end < 0) {
        if (threadIdx.x == 0) set_status(p.status, MPM_ERR_DEVICE_BOUNDS);
        return;
      }
      if (row0 >= seg_end) return;
      int lo = 0, hi = p.E - 1;                 // last e with seg[e] <= row0
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seg[mid] <= row0) lo = mid; else hi = mid - 1;
      }
      e = lo;
    } else if (row0 >= seg_end) {
      return;
    }
    num_kb = p.K / Cfg::kElemsPerKB;
    ka_elem = 0;
    kb_elem = (long long)e * p.b_k_per_e;
    out_row_base = row0;
  } else {
    e = blockIdx.z;
    row0 = (long long)blockIdx.y * BM;          // output row (rows of A)
    const long long s0 = p.seg[e], s1 = p.seg[e + 1];
    if (s1 < s0 || s0 < 0 || ((s1 - s0) % Cfg::kElemsPerKB) != 0) {
      if (threadIdx.x == 0) set_status(p.status, MPM_ERR_DEVICE_BOUNDS);
      return;
    }
    num_kb = (int)((s1 - s0) / Cfg::kElemsPerKB);
    ka_elem = s0;
    kb_elem = s0;
    out_row_base = (long long)e * p.M_out + row0;
  }
  if (EPI == MPM_EPI_SWIGLU || EPI == MPM_EPI_SWIGLU_SAVE) {
    brow[0] = (long long)e * p.b_rows_per_e + n0;               // gate rows
    brow[1] = (long long)e * p.b_rows_per_e + p.N / 2 + n0;     // up rows
  } else {
    brow[0] = (long long)e * p.b_rows_per_e + n0;
    brow[1] = brow[0] + 128;
  }

  // ------------------------------------------------------------ empty reduction
  if (num_kb == 0) {
    // wgrad of an expert without rows: the gradient is zero
    if (EPI == MPM_EPI_F32) {
      float* o = static_cast<float*>(p.out) + (out_row_base + threadIdx.x) * p.ldo + n0;
      for (int c = 0; c < BN; c += 4) *reinterpret_cast<float4*>(o + c) = make_float4(0, 0, 0, 0);
    }
    return;
  }

  // ------------------------------------------------------------ shared memory
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = sA + STAGES * A_STAGE;
  const uint32_t sSFA = sB + STAGES * B_STAGE;
  const uint32_t sSFB = sSFA + STAGES * Cfg::kSfaBytes;
  const uint32_t sBar = sSFB + STAGES * Cfg::kSfbBytes;
  const uint32_t bar_full = sBar, bar_empty = sBar + 8 * STAGES, bar_acc = sBar + 16 * STAGES;
  const uint32_t sTmemHolder = bar_acc + 8;
  const uint32_t bar_sf = sTmemHolder + 8;     // scale tiles of a stage are in TMEM
  volatile uint32_t* tmem_holder =
      reinterpret_cast<volatile uint32_t*>(gbase + (sTmemHolder - base));

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    for (int s = 0; s < STAGES; ++s) mbar_init(bar_sf + 8 * s, 1);
    fence_mbar_init();
    fence_proxy_async();
    prefetch_tmap(&tma_a);
    prefetch_tmap(&tma_b);
  }
  if (warp == 2) {
    tmem_alloc(sTmemHolder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const long long sfa_rt = row0 >> 7;                        // A row tile
  const int stage_tx = A_STAGE + B_STAGE + Cfg::kSfaBytes + Cfg::kSfbBytes;

  if (warp == 0 && lane == 0) {
    // ======================================================== TMA producer
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
      if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, p.status)) break;
      mbar_arrive_expect_tx(bar_full + 8 * s, stage_tx);
      const long long ka = ka_elem + (long long)kb * Cfg::kElemsPerKB;   // elements
      const long long kbb = kb_elem + (long long)kb * Cfg::kElemsPerKB;
      const int xa = (int)(KIND == MPM_KIND_NVFP4 ? ka / 2 : ka);
      const int xb = (int)(KIND == MPM_KIND_NVFP4 ? kbb / 2 : kbb);
      tma_load_2d(sA + s * A_STAGE, &tma_a, xa, (int)row0, bar_full + 8 * s);
      tma_load_2d(sB + s * B_STAGE, &tma_b, xb, (int)brow[0], bar_full + 8 * s);
      tma_load_2d(sB + s * B_STAGE + 128 * BKB, &tma_b, xb, (int)brow[1], bar_full + 8 * s);
      // scale tiles: atoms are 512 bytes = 128 rows x 4 scale columns
      const long long atom_a = (KIND == MPM_KIND_NVFP4) ? ka / 64 : ka / 128;
      const long long atom_b = (KIND == MPM_KIND_NVFP4) ? kbb / 64 : kbb / 128;
      const uint8_t* srcA = p.sfa + ((sfa_rt * (p.sfa_cols_pad >> 2)) + atom_a) * 512;
      bulk_load(sSFA + s * Cfg::kSfaBytes, srcA, Cfg::kSfaBytes, bar_full + 8 * s);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const long long rt = brow[nt] >> 7;
        const uint8_t* srcB = p.sfb + ((rt * (p.sfb_cols_pad >> 2)) + atom_b) * 512;
        bulk_load(sSFB + s * Cfg::kSfbBytes + nt * (Cfg::kSfbBytes / 2), srcB,
                  Cfg::kSfbBytes / 2, bar_full + 8 * s);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ======================================================== MMA issuer
    // Waits until the copy thread (warp 3) has put the stage's scale tiles in
    // tensor memory; copies and MMAs come from different threads so that the
    // copies of one stage can run alongside the MMAs of the previous one.
    bool ok = true;
    for (int kb = 0; ok && kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      if (!mbar_wait(bar_sf + 8 * s, (uint32_t)(kb / STAGES) & 1u, p.status)) break;
      tc_fence_after();
      const uint32_t sf_col = tmem + SF_TMEM_BASE + s * Cfg::kSfTmemPerStage;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t adesc = sdesc_sw128(sA + s * A_STAGE + ks * 32);
        const uint64_t bdesc = sdesc_sw128(sB + s * B_STAGE + ks * 32);
        const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
        if (KIND == MPM_KIND_NVFP4) {
          const uint32_t idesc = idesc_block_scaled(Cfg::kFmt, BN, Cfg::kUe8m0, 0);
          mma_nvf4(tmem, adesc, bdesc, idesc, sf_col + ks * 4, sf_col + 16 + ks * 8, acc);
        } else {
          const uint32_t idesc = idesc_block_scaled(Cfg::kFmt, BN, Cfg::kUe8m0, (uint32_t)ks);
          mma_mxf8(tmem, adesc, bdesc, idesc, sf_col, sf_col + 4, acc);
        }
      }
      tc_commit(bar_empty + 8 * s);
    }
    tc_commit(bar_acc);
  } else if (warp == 3 && lane == 0) {
    // ======================================================== scale-tile copies
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      if (!mbar_wait(bar_full + 8 * s, (uint32_t)(kb / STAGES) & 1u, p.status)) break;
      tc_fence_after();
      const uint32_t sf_col = tmem + SF_TMEM_BASE + s * Cfg::kSfTmemPerStage;
      if (KIND == MPM_KIND_NVFP4) {
        // SFA: atom ks -> 4 columns; SFB: (ks, half) -> 4 columns
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          tc_cp_32x128b_x4(sf_col + ks * 4, sdesc_sf(sSFA + s * Cfg::kSfaBytes + ks * 512));
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            tc_cp_32x128b_x4(sf_col + 16 + ks * 8 + nt * 4,
                             sdesc_sf(sSFB + s * Cfg::kSfbBytes + nt * 2048 + ks * 512));
        }
      } else {
        tc_cp_32x128b_x4(sf_col, sdesc_sf(sSFA + s * Cfg::kSfaBytes));
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          tc_cp_32x128b_x4(sf_col + 4 + nt * 4, sdesc_sf(sSFB + s * Cfg::kSfbBytes + nt * 512));
      }
      tc_commit(bar_sf + 8 * s);
    }
  }
  __syncwarp();

  // ======================================================== epilogue
  const bool acc_ok = mbar_wait(bar_acc, 0, p.status);
  tc_fence_after();
  const int r = warp * 32 + lane;                       // row within the tile
  const long long grow = row0 + r;                      // row of A / output
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  const bool row_ok = (p.group == MPM_GROUP_K) || (grow < p.a_rows);
  if (acc_ok) {
    float alpha = 1.0f;
    if (p.group == MPM_GROUP_M && row_ok) {
      if (p.alpha_a) alpha = p.alpha_a[grow];
      if (p.alpha_b) alpha = __fmul_rn(alpha, p.alpha_b[e]);
    }
    uint32_t v[32], u[32];
    if (EPI == MPM_EPI_F32 || EPI == MPM_EPI_BF16) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        tmem_ld_32x32b_x32(trow + c * 32, v);
        tmem_ld_wait();
        if (!row_ok) continue;
        if (EPI == MPM_EPI_F32) {
          float* o = static_cast<float*>(p.out) + out_row_base * p.ldo + (long long)r * p.ldo + n0 + c * 32;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(o + j) = make_float4(
                __fmul_rn(__uint_as_float(v[j]), alpha), __fmul_rn(__uint_as_float(v[j + 1]), alpha),
                __fmul_rn(__uint_as_float(v[j + 2]), alpha), __fmul_rn(__uint_as_float(v[j + 3]), alpha));
        } else {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + (out_row_base + r) * p.ldo + n0 + c * 32;
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 w;
            w.x = pack_bf16(__fmul_rn(__uint_as_float(v[j]), alpha), __fmul_rn(__uint_as_float(v[j + 1]), alpha));
            w.y = pack_bf16(__fmul_rn(__uint_as_float(v[j + 2]), alpha), __fmul_rn(__uint_as_float(v[j + 3]), alpha));
            w.z = pack_bf16(__fmul_rn(__uint_as_float(v[j + 4]), alpha), __fmul_rn(__uint_as_float(v[j + 5]), alpha));
            w.w = pack_bf16(__fmul_rn(__uint_as_float(v[j + 6]), alpha), __fmul_rn(__uint_as_float(v[j + 7]), alpha));
            *reinterpret_cast<uint4*>(o + j) = w;
          }
        }
      }
    } else if (EPI == MPM_EPI_SWIGLU || EPI == MPM_EPI_SWIGLU_SAVE) {
      const float prob = row_ok ? p.row_prob[grow] : 0.0f;
      const long long half = p.N / 2;
      float amax = 0.0f;
#pragma unroll 1
      for (int c = 0; c < (BN / 2) / 32; ++c) {
        tmem_ld_32x32b_x32(trow + c * 32, v);                 // gate
        tmem_ld_32x32b_x32(trow + BN / 2 + c * 32, u);        // up
        tmem_ld_wait();
        if (!row_ok) continue;
        uint32_t dw[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float d2[2];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const float g = __fmul_rn(__uint_as_float(v[j + q]), alpha);
            const float uu = __fmul_rn(__uint_as_float(u[j + q]), alpha);
            d2[q] = swiglu_fwd(g, uu, prob);
          }
          const uint32_t pk = pack_bf16(d2[0], d2[1]);
          dw[j / 2] = pk;
          amax = fmaxf(amax, fmaxf(fabsf(bf16lo(pk)), fabsf(bf16hi(pk))));
        }
        __nv_bfloat16* od = static_cast<__nv_bfloat16*>(p.out2) + grow * p.ldo2 + n0 + c * 32;
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<uint4*>(od + 2 * j) = make_uint4(dw[j], dw[j + 1], dw[j + 2], dw[j + 3]);
        if (EPI == MPM_EPI_SWIGLU_SAVE) {
          __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.out) + grow * p.ldo + n0 + c * 32;
          __nv_bfloat16* ou = og + half;
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 wg, wu;
            wg.x = pack_bf16(__fmul_rn(__uint_as_float(v[j]), alpha), __fmul_rn(__uint_as_float(v[j + 1]), alpha));
            wg.y = pack_bf16(__fmul_rn(__uint_as_float(v[j + 2]), alpha), __fmul_rn(__uint_as_float(v[j + 3]), alpha));
            wg.z = pack_bf16(__fmul_rn(__uint_as_float(v[j + 4]), alpha), __fmul_rn(__uint_as_float(v[j + 5]), alpha));
            wg.w = pack_bf16(__fmul_rn(__uint_as_float(v[j + 6]), alpha), __fmul_rn(__uint_as_float(v[j + 7]), alpha));
            wu.x = pack_bf16(__fmul_rn(__uint_as_float(u[j]), alpha), __fmul_rn(__uint_as_float(u[j + 1]), alpha));
            wu.y = pack_bf16(__fmul_rn(__uint_as_float(u[j + 2]), alpha), __fmul_rn(__uint_as_float(u[j + 3]), alpha));
            wu.z = pack_bf16(__fmul_rn(__uint_as_float(u[j + 4]), alpha), __fmul_rn(__uint_as_float(u[j + 5]), alpha));
            wu.w = pack_bf16(__fmul_rn(__uint_as_float(u[j + 6]), alpha), __fmul_rn(__uint_as_float(u[j + 7]), alpha));
            *reinterpret_cast<uint4*>(og + j) = wg;
            *reinterpret_cast<uint4*>(ou + j) = wu;
          }
        }
      }
      if (row_ok && p.amax && amax > 0.0f)
        atomicMax(reinterpret_cast<unsigned*>(p.amax) + grow, __float_as_uint(amax));
    } else if (EPI == MPM_EPI_DSWIGLU) {
      const float prob = row_ok ? p.row_prob[grow] : 0.0f;
      const long long Nh = p.N;        // dH has 2N columns: [dg | du]
      const __nv_bfloat16* cg = static_cast<const __nv_bfloat16*>(p.aux) + grow * p.ld_aux;
      const __nv_bfloat16* cu = cg + Nh;
      __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.out) + grow * p.ldo;
      __nv_bfloat16* ou = og + Nh;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        tmem_ld_32x32b_x32(trow + c * 32, v);
        tmem_ld_wait();
        if (!row_ok) continue;
        const long long col = n0 + c * 32;
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          const uint4 gw = *reinterpret_cast<const uint4*>(cg + col + j);
          const uint4 uw = *reinterpret_cast<const uint4*>(cu + col + j);
          const uint32_t ga[4] = {gw.x, gw.y, gw.z, gw.w};
          const uint32_t ua[4] = {uw.x, uw.y, uw.z, uw.w};
          uint32_t og4[4], ou4[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float dg2[2], du2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float g = h ? bf16hi(ga[q]) : bf16lo(ga[q]);
              const float uu = h ? bf16hi(ua[q]) : bf16lo(ua[q]);
              const float dd = __fmul_rn(__uint_as_float(v[j + 2 * q + h]), alpha);
              swiglu_bwd(g, uu, dd, prob, dg2[h], du2[h]);
            }
            og4[q] = pack_bf16(dg2[0], dg2[1]);
            ou4[q] = pack_bf16(du2[0], du2[1]);
          }
          *reinterpret_cast<uint4*>(og + col + j) = make_uint4(og4[0], og4[1], og4[2], og4[3]);
          *reinterpret_cast<uint4*>(ou + col + j) = make_uint4(ou4[0], ou4[1], ou4[2], ou4[3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- launcher
template <int KIND, int EPI>
static cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                              dim3 grid, cudaStream_t s) {
  constexpr int smem = smem_bytes<KIND>();
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<KIND, EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  grouped_gemm_kernel<KIND, EPI><<<grid, 128, smem, s>>>(ta, tb, a);
  return cudaGetLastError();
}

template <int KIND>
static cudaError_t dispatch_epi(int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                                const GemmArgs& a, dim3 grid, cudaStream_t s) {
  switch (epi) {
    case MPM_EPI_F32: return launch_one<KIND, MPM_EPI_F32>(ta, tb, a, grid, s);
    case MPM_EPI_BF16: return launch_one<KIND, MPM_EPI_BF16>(ta, tb, a, grid, s);
    case MPM_EPI_SWIGLU: return launch_one<KIND, MPM_EPI_SWIGLU>(ta, tb, a, grid, s);
    case MPM_EPI_SWIGLU_SAVE: return launch_one<KIND, MPM_EPI_SWIGLU_SAVE>(ta, tb, a, grid, s);
    case MPM_EPI_DSWIGLU: return launch_one<KIND, MPM_EPI_DSWIGLU>(ta, tb, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_grouped_gemm(int kind, int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                                const GemmArgs& a, dim3 grid, cudaStream_t s) {
  if (kind == MPM_KIND_NVFP4) return dispatch_epi<MPM_KIND_NVFP4>(epi, ta, tb, a, grid, s);
  return dispatch_epi<MPM_KIND_MXFP8>(epi, ta, tb, a, grid, s);
}

}  // namespace mpm
