// Small-M grouped GEMM for decode / rollout batches: the expert's weights on
// the MMA's M side, the expert's routed rows on its N side.
//
// When each expert receives few rows (tens of tokens), the layer is bound by
// reading every active expert's weights once from HBM.  Here one CTA computes
// a 128 (weight rows) x 128 (routed rows of one segment chunk) tile of the
// transposed output with tcgen05.mma.cta_group::1 (M = 128, N = 128,
// block-scaled NVFP4 or MXFP8), so a weight tile feeds a whole chunk of rows
// per pass and the MMA work per weight byte stays small next to the stream.
// Persistent CTAs walk (chunk, weight tile) tasks; a 4-6 stage TMA ring keeps
// the weight stream going across tasks, and (without SwiGLU) two TMEM
// accumulators let a task's epilogue overlap the next task's MMAs.
//
// Operands: the weight matrix is the descriptor's B ([E * b_rows_per_expert,
// K] codes, tiled scales), the routed rows its A ([capacity, K], segments
// multiples of 128 rows so that a chunk's scale tile is one 128-row tile).
// The epilogue reads the accumulator with lane = weight row and column =
// routed row, and writes out[row, feature] (fp32 / bf16), or for SwiGLU the
// D = silu(gate) * up * prob row with its row amax, exactly as the
// large-tile kernels do.
//
// Sources: "Towards Blackwell-native 8-bit and 4-bit RL", section "Per-token
// activation scaling" (NVFP4 rollout of the MoE experts) and the small-M
// rollout path it names; "miniTE technical report", sections 5.2 and 5.4
// (grouped GEMM over a contiguous buffer with device offsets; FC1 epilogue).
#include "gemm.cuh"

namespace mpm {
namespace smallk {

constexpr int BW = 128;               // weight rows per tile (MMA M)
constexpr int BR = 128;               // routed rows per chunk (MMA N)
constexpr int BKB = 128;              // bytes of K per stage
constexpr int NTHREADS = 192;         // split K: warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
// grouped kernel: warp 0 TMA, warp 1 MMA, warps 2-5 epilogue, warps 6-9 the
// scale tiles into TMEM (one per lane quarter)
constexpr int NTHREADS_G = 320;
constexpr int TILE = 128 * BKB;       // 16 KB operand tile
constexpr uint32_t TMEM_COLS = 512;

template <int KIND> struct KCfg;
template <> struct KCfg<MPM_KIND_NVFP4> {
  static constexpr int kElemsPerKB = 256, kAtoms = 4;       // 4 scale tiles per stage
  static constexpr uint32_t kFmt = 1, kUe8m0 = 0;
};
template <> struct KCfg<MPM_KIND_MXFP8> {
  static constexpr int kElemsPerKB = 128, kAtoms = 1;       // one scale tile, sf_id = k step
  static constexpr uint32_t kFmt = 0, kUe8m0 = 1;
};

template <int KIND, int EPI> struct Cfg {
  static constexpr bool kDual = (EPI == MPM_EPI_SWIGLU);   // gate and up weight tiles
  static constexpr int kWT = kDual ? 2 : 1;
  static constexpr int kSfBytes = KCfg<KIND>::kAtoms * 512;
  static constexpr int kStage = kWT * TILE + TILE + (kWT + 1) * kSfBytes;
  static constexpr int kStages = kDual ? 4 : 5;
  static constexpr int kNacc = kDual ? 1 : 2;               // accumulator buffers
  static constexpr int kAccCols = kWT * BR;                  // TMEM columns per buffer
  static constexpr int kSfCols = (kWT + 1) * 4 * KCfg<KIND>::kAtoms;   // per stage
  static constexpr uint32_t kSfBase = kNacc * kAccCols;
  static_assert(kSfBase + kStages * kSfCols <= TMEM_COLS, "TMEM budget");
};

template <int KIND, int EPI>
constexpr int smem_bytes() {
  return 1024 + Cfg<KIND, EPI>::kStages * Cfg<KIND, EPI>::kStage + (4 * Cfg<KIND, EPI>::kStages + 8) * 8;
}

struct SmallMaps {
  CUtensorMap a, b;   // routed rows (A) and weights (B), 128 x 128-byte boxes
};

// A role's cached view of the segment offsets: its tasks come in increasing
// row order, so a cursor moving forward over the offsets finds each task's
// expert (every offset read once per role, instead of a binary search of
// dependent global reads per task).
struct SegCursor {
  int e = -1;
  long long lo = 0, hi = 0, end = -1;
};

// Expert offsets up to this many (E + 1) are copied to shared memory once
// per CTA: at decode sizes a CTA's next task usually lies several experts
// (many of them empty) further on, and walking the offsets in global memory
// put a chain of dependent L2 reads in front of every task's first load.
constexpr int SEG_SMEM = 1025;

// task t -> chunk of 128 routed rows and weight tile; false past the last row
// (seg: the expert offsets, in shared or global memory; null for dense A)
MPM_DEV bool small_task(const GemmArgs& p, const int* seg, long long t, int n_wt, long long* r0,
                        int* e, int* wt, int* bad, SegCursor& cur) {
  const long long ci = t / n_wt;
  *wt = (int)(t - ci * n_wt);
  *r0 = ci * BR;
  if (cur.end < 0) {
    cur.end = seg ? seg[p.E] : p.a_rows;
    if (seg) {
      cur.e = 0;
      cur.lo = seg[0];
      cur.hi = seg[1];
    }
  }
  if (*r0 >= cur.end || *r0 >= p.a_rows) return false;
  int lo = 0;
  if (seg) {
    while (cur.e + 1 < p.E && cur.hi <= *r0) {
      ++cur.e;
      cur.lo = cur.hi;
      cur.hi = seg[cur.e + 1];
    }
    lo = cur.e;
    if ((cur.lo & (BR - 1)) != 0 || (cur.hi & (BR - 1)) != 0) *bad = 1;
  }
  *e = lo;
  return true;
}

template <int KIND, int EPI>
__global__ void __launch_bounds__(NTHREADS_G, 1)
grouped_gemm_small_kernel(const __grid_constant__ SmallMaps maps, const GemmArgs p, const int n_wt,
                          const long long n_tasks) {
  using C = Cfg<KIND, EPI>;
  using KC = KCfg<KIND>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  // stage s: [weight tile(s) | routed-row tile | weight scale tiles | row scale tiles]
  const uint32_t sStage = base;
  const uint32_t sBar = sStage + S * C::kStage;
  const uint32_t bar_full = sBar, bar_empty = sBar + 8 * S;
  const uint32_t bar_acc = sBar + 16 * S;                 // full at + 16 b, empty at + 16 b + 8
  const uint32_t sTmem = bar_acc + 32;
  const uint32_t sFlag = sTmem + 8;
  const uint32_t bar_sf = sFlag + 8;                      // a stage's scale tiles are in TMEM
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(gbase + (sTmem - base));
  volatile int* fail_flag = reinterpret_cast<volatile int*>(gbase + (sFlag - base));

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_sf + 8 * s, 4);                       // one arrive per scale warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc + 16 * b, 1);
      mbar_init(bar_acc + 16 * b + 8, 4);                // one arrive per epilogue warp
    }
    *fail_flag = 0;
    fence_mbar_init();
    fence_proxy_async();
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.b);
  }
  if (warp == 1) {
    tmem_alloc(sTmem, TMEM_COLS);
    tmem_relinquish();
  }
  __shared__ int s_seg[SEG_SMEM];
  const bool seg_smem = p.seg && p.E < SEG_SMEM;
  if (seg_smem)
    for (int i = threadIdx.x; i <= p.E; i += NTHREADS_G) s_seg[i] = p.seg[i];
  const int* seg = seg_smem ? s_seg : p.seg;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int num_kb = (int)(p.K / KC::kElemsPerKB);
  int bad = 0;

  if (warp == 0 && lane == 0) {
    // ======================================================== TMA producer
    uint32_t it = 0;
    bool ok = true;
    SegCursor cur;
    for (long long t = blockIdx.x; ok && t < n_tasks; t += gridDim.x) {
      long long r0; int e, wt;
      if (!small_task(p, seg, t, n_wt, &r0, &e, &wt, &bad, cur)) break;
      const long long wrow0 = (long long)e * p.b_rows_per_e + (long long)wt * BW;
      const long long wrow1 = wrow0 + p.N / 2;                // up rows (SwiGLU)
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % S;
        if (!mbar_wait(bar_empty + 8 * s, ((it / S) & 1u) ^ 1u, p.status)) { ok = false; break; }
        const uint32_t st = sStage + s * C::kStage;
        mbar_arrive_expect_tx(bar_full + 8 * s, C::kStage);
        const long long ke = (long long)kb * KC::kElemsPerKB;                  // elements
        const int xb = (int)(KIND == MPM_KIND_NVFP4 ? ke / 2 : ke);            // bytes
        const long long kbw = (long long)e * p.b_k_per_e + ke;
        const int xw = (int)(KIND == MPM_KIND_NVFP4 ? kbw / 2 : kbw);
        tma_load_2d(st, &maps.b, xw, (int)wrow0, bar_full + 8 * s);
        if (C::kDual) tma_load_2d(st + TILE, &maps.b, xw, (int)wrow1, bar_full + 8 * s);
        tma_load_2d(st + C::kWT * TILE, &maps.a, xb, (int)r0, bar_full + 8 * s);
        // scale tiles: KC::kAtoms consecutive 512-byte tiles per 128 rows
        const long long atom_w = (KIND == MPM_KIND_NVFP4) ? kbw / 64 : kbw / 128;
        const long long atom_a = (KIND == MPM_KIND_NVFP4) ? ke / 64 : ke / 128;
        const uint32_t sf0 = st + (C::kWT + 1) * TILE;
        bulk_load(sf0, p.sfb + ((wrow0 >> 7) * (p.sfb_cols_pad >> 2) + atom_w) * 512, C::kSfBytes,
                  bar_full + 8 * s);
        if (C::kDual)
          bulk_load(sf0 + C::kSfBytes, p.sfb + ((wrow1 >> 7) * (p.sfb_cols_pad >> 2) + atom_w) * 512,
                    C::kSfBytes, bar_full + 8 * s);
        bulk_load(sf0 + C::kWT * C::kSfBytes,
                  p.sfa + ((r0 >> 7) * (p.sfa_cols_pad >> 2) + atom_a) * 512, C::kSfBytes,
                  bar_full + 8 * s);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ======================================================== MMA issue
    // It waits for a stage's scale barrier only: the scale warps arrive on it
    // after they have seen the stage's TMA loads land and written its scale
    // tiles into TMEM.  A TMEM scale slot is rewritten only after the stage
    // was refilled, i.e. after the MMAs that read it completed.
    uint32_t it = 0, j = 0;
    bool ok = true;
    const uint32_t idesc_base = idesc_block_scaled(KC::kFmt, BR, KC::kUe8m0, 0, 128);
    SegCursor cur;
    for (long long t = blockIdx.x; ok && t < n_tasks; t += gridDim.x) {
      long long r0; int e, wt;
      if (!small_task(p, seg, t, n_wt, &r0, &e, &wt, &bad, cur)) break;
      const uint32_t ab = (C::kNacc > 1) ? (j & 1u) : 0u;
      const uint32_t use = (C::kNacc > 1) ? (j >> 1) : j;
      if (!mbar_wait(bar_acc + 16 * ab + 8, (use & 1u) ^ 1u, p.status)) break;
      ++j;
      tc_fence_after();
      const uint32_t dacc = tmem + ab * C::kAccCols;
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % S;
        if (!mbar_wait(bar_sf + 8 * s, (it / S) & 1u, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t st = sStage + s * C::kStage;
        // TMEM scale columns of this stage: weight tile(s) then the row tile,
        // 4 columns per 512-byte scale tile
        const uint32_t sfcol = tmem + C::kSfBase + s * C::kSfCols;
        const uint32_t sfrow = sfcol + C::kWT * KC::kAtoms * 4;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bdesc = sdesc_sw128(st + C::kWT * TILE + ks * 32);
          const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
#pragma unroll
          for (int w = 0; w < C::kWT; ++w) {
            const uint64_t adesc = sdesc_sw128(st + w * TILE + ks * 32);
            if (KIND == MPM_KIND_NVFP4) {
              mma_nvf4(dacc + w * BR, adesc, bdesc, idesc_base,
                       sfcol + (w * KC::kAtoms + ks) * 4, sfrow + ks * 4, acc);
            } else {
              const uint32_t idesc = idesc_block_scaled(KC::kFmt, BR, KC::kUe8m0, (uint32_t)ks, 128);
              mma_mxf8(dacc + w * BR, adesc, bdesc, idesc, sfcol + w * 4, sfrow, acc);
            }
          }
        }
        tc_commit(bar_empty + 8 * s);
        if (kb + 1 == num_kb) tc_commit(bar_acc + 16 * ab);
      }
    }
  } else if (warp >= 6) {
    // ======================================================== scale tiles, tcgen05.st
    // Warp w writes TMEM lane quarter w % 4 (warps 6-9: quarters 2, 3, 0, 1):
    // lane l of each 512-byte scale tile (its 16-byte row l) goes to lane
    // 32 q + l, four columns — the replicated layout the block-scaled MMA
    // reads, as a 32x128b.warpx4 copy would leave it.  As copies issued by
    // the MMA thread these ran on the tensor pipe between the MMAs (decode
    // FC2 0.301 against 0.231 ms with no copies at all).
    const int q = warp & 3;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    constexpr int NT = (C::kWT + 1) * KC::kAtoms;           // scale tiles per stage
    uint32_t it = 0;
    bool ok = true;
    SegCursor cur;
    for (long long t = blockIdx.x; ok && t < n_tasks; t += gridDim.x) {
      long long r0; int e, wt;
      if (!small_task(p, seg, t, n_wt, &r0, &e, &wt, &bad, cur)) break;
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % S;
        if (!mbar_wait(bar_full + 8 * s, (it / S) & 1u, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint8_t* sf = gbase + (sStage - base) + s * C::kStage + (C::kWT + 1) * TILE + lane * 16;
        const uint32_t col = tq + C::kSfBase + s * C::kSfCols;
#pragma unroll
        for (int i = 0; i < NT; ++i)
          tmem_st_32x32b_x4(col + i * 4, *reinterpret_cast<const uint4*>(sf + i * 512));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sf + 8 * s);
      }
    }
  } else if (warp >= 2) {
    // ======================================================== epilogue (4 warps)
    const int q = warp & 3;                       // TMEM lane quarter
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    uint32_t j = 0;
    SegCursor cur;
    for (long long t = blockIdx.x; t < n_tasks; t += gridDim.x) {
      long long r0; int e, wt;
      if (!small_task(p, seg, t, n_wt, &r0, &e, &wt, &bad, cur)) break;
      const uint32_t ab = (C::kNacc > 1) ? (j & 1u) : 0u;
      const uint32_t use = (C::kNacc > 1) ? (j >> 1) : j;
      // F32 / BF16: the 128 rows' scales and row map (lane = row within each
      // 32-row block) loaded before the accumulator wait, so their latency
      // is not part of the epilogue
      float a_pre[4];
      int m_pre[4];
      if (!C::kDual) {
        const float ab_pre = p.alpha_b ? p.alpha_b[e] : 1.0f;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          const long long rl = r0 + cb * 32 + lane;
          const bool in = rl < p.a_rows;
          a_pre[cb] = (p.alpha_a && in) ? __fmul_rn(p.alpha_a[rl], ab_pre) : ab_pre;
          m_pre[cb] = (p.row_perm && in) ? p.row_perm[rl] : 0;
        }
      }
      const bool w_ok = mbar_wait(bar_acc + 16 * ab, use & 1u, p.status);
      ++j;
      if (!w_ok) *fail_flag = 1;
      named_sync(1, 128);
      if (*fail_flag) break;
      tc_fence_after();
      const uint32_t tacc = tmem + lane_off + ab * C::kAccCols;
      const long long f = (long long)wt * BW + q * 32 + lane;   // this thread's output feature
      const float ab_e = p.alpha_b ? p.alpha_b[e] : 1.0f;
      if (!C::kDual) {
        // all 128 routed rows of this feature in registers, then the
        // accumulator goes back to the MMA
        uint32_t v0[32], v1[32], v2[32], v3[32];
        tmem_ld_32x32b_x32(tacc + 0, v0);
        tmem_ld_32x32b_x32(tacc + 32, v1);
        tmem_ld_32x32b_x32(tacc + 64, v2);
        tmem_ld_32x32b_x32(tacc + 96, v3);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acc + 16 * ab + 8);
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          const uint32_t* v = cb == 0 ? v0 : (cb == 1 ? v1 : (cb == 2 ? v2 : v3));
          // the 32 rows' scales, one coalesced load, broadcast by shuffles;
          // with a row map, a segment's padding rows are not stored (at
          // decode sizes most rows of a 128-row chunk)
          const float a_lane = a_pre[cb];
          const unsigned keep = __ballot_sync(0xffffffffu, m_pre[cb] >= 0);
          // the arithmetic runs for every row and only the store is
          // predicated (a branch per row measured slower than storing all)
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const long long row = r0 + cb * 32 + c;
            const float alpha = __shfl_sync(0xffffffffu, a_lane, c);
            const float val = __fmul_rn(__uint_as_float(v[c]), alpha);
            const bool st = (keep >> c) & 1u;
            if (EPI == MPM_EPI_F32) {
              float* o = static_cast<float*>(p.out) + row * p.ldo + f;
              asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t"
                           "@q st.global.f32 [%0], %1;\n\t}"
                           :: "l"(o), "f"(val), "r"((uint32_t)st) : "memory");
            } else {
              __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + row * p.ldo + f;
              const __nv_bfloat16 b = __float2bfloat16_rn(val);
              asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t"
                           "@q st.global.b16 [%0], %1;\n\t}"
                           :: "l"(o), "h"(*reinterpret_cast<const uint16_t*>(&b)),
                              "r"((uint32_t)st) : "memory");
            }
          }
        }
      } else {
        // SwiGLU: gate accumulator in columns [0, 128), up in [128, 256)
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(tacc + cb * 32, g);
          tmem_ld_32x32b_x32(tacc + BR + cb * 32, u);
          // the 32 rows' scales and router weights: coalesced loads issued
          // under the TMEM loads, broadcast by shuffles
          const long long rl = r0 + cb * 32 + lane;
          const float a_lane = p.alpha_a ? __fmul_rn(p.alpha_a[rl], ab_e) : ab_e;
          const float p_lane = p.row_prob[rl];
          tmem_ld_wait();
          // A block whose gate and up accumulators are all +-0 (the padding
          // rows of a segment, whose operand rows are zero) gives D = +-0
          // exactly: silu(+-0) = +-0, and the products keep the xor of the
          // operands' signs.  Those 32 rows are written from the sign bits
          // alone and add nothing to the row max (decode batches: most of
          // a 128-row chunk), so the accumulator is held for less time.
          uint32_t nz = 0;
#pragma unroll
          for (int c = 0; c < 32; ++c) nz |= (g[c] | u[c]) & 0x7FFFFFFFu;
          if (!__any_sync(0xffffffffu, nz != 0)) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const long long row = r0 + cb * 32 + c;
              const uint32_t sp = __float_as_uint(__shfl_sync(0xffffffffu, p_lane, c));
              const uint32_t sgn = (g[c] ^ u[c] ^ sp) & 0x80000000u;   // alpha's sign cancels
              reinterpret_cast<uint16_t*>(p.out2)[row * p.ldo2 + f] = (uint16_t)(sgn >> 16);
            }
            continue;
          }
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const long long row = r0 + cb * 32 + c;
            const float alpha = __shfl_sync(0xffffffffu, a_lane, c);
            const float gv = __fmul_rn(__uint_as_float(g[c]), alpha);
            const float uv = __fmul_rn(__uint_as_float(u[c]), alpha);
            const float prob = __shfl_sync(0xffffffffu, p_lane, c);
            const __nv_bfloat16 d = __float2bfloat16_rn(swiglu_fwd(gv, uv, prob));
            static_cast<__nv_bfloat16*>(p.out2)[row * p.ldo2 + f] = d;
            g[c] = __float_as_uint(fabsf(__bfloat162float(d)));
          }
          // row amax over this warp's 32 features for the 32 rows at once:
          // a butterfly that halves the rows a lane holds at each step (31
          // shuffles), leaving the max of row cb*32 + lane in lane `lane`
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < off; ++i) {
              const float lo = __uint_as_float(g[i]), hi = __uint_as_float(g[i + off]);
              const float recv = __shfl_xor_sync(0xffffffffu, upper ? lo : hi, off);
              g[i] = __float_as_uint(fmaxf(upper ? hi : lo, recv));
            }
          }
          const float rmax = __uint_as_float(g[0]);
          if (p.amax && rmax > 0.0f)
            atomicMax(reinterpret_cast<unsigned*>(p.amax) + (r0 + cb * 32 + lane), __float_as_uint(rmax));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acc + 16 * ab + 8);
      }
    }
  }
  if (bad && threadIdx.x == 0) set_status(p.status, MPM_ERR_DEVICE_BOUNDS);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace smallk

// ---------------------------------------------------------------- split K
// One dense group of at most 128 rows (no segment offsets): the
// single-expert case.  The kernel above gives it only N / 128 CTAs, each
// running the whole K chain.  Here a cluster of ks CTAs shares one tile of
// 128 weight rows: CTA c accumulates k-blocks [c nkb / ks, (c + 1) nkb / ks)
// in its own TMEM and parks the fp32 partial [128 rows x 128 features] in
// its shared memory; after a cluster barrier CTA c sums rows
// [c 128 / ks, (c + 1) 128 / ks) over the ks partials in CTA order 0 .. ks-1
// (reading its peers' shared memory), applies alpha and writes the output.
// The order is fixed, so the result is deterministic; it rounds in another
// order than the unsplit accumulation (both fp32, within the GEMM
// tolerance).
namespace splitk {
using namespace smallk;

constexpr int KS_MAX = 8;              // portable cluster size
constexpr int S = 4;                   // ring stages
constexpr uint32_t TMEM_COLS = 256;    // accumulator 128 + scale slots 4 x 32

template <int KIND>
constexpr int stage_bytes() { return 2 * TILE + 2 * KCfg<KIND>::kAtoms * 512; }
constexpr int PART_BYTES = BR * BW * 4;        // fp32 [128 rows][128 features]
template <int KIND>
constexpr int ring_bytes() {
  return S * stage_bytes<KIND>() > PART_BYTES ? S * stage_bytes<KIND>() : PART_BYTES;
}
template <int KIND>
constexpr int smem_bytes() { return 1024 + ring_bytes<KIND>() + (2 * S + 2) * 8 + 16; }

template <int KIND, int EPI>
__global__ void __launch_bounds__(NTHREADS, 1)
gemm_splitk_kernel(const __grid_constant__ SmallMaps maps, const GemmArgs p, const int ks) {
  using KC = KCfg<KIND>;
  constexpr int STB = stage_bytes<KIND>();
  constexpr int SFC = 2 * 4 * KC::kAtoms;        // TMEM scale columns per stage (weights, rows)
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sRing = base;                   // the ring; after the MMAs the partial
  const uint32_t sBar = base + ring_bytes<KIND>();
  const uint32_t bar_full = sBar, bar_empty = sBar + 8 * S, bar_acc = sBar + 16 * S;
  const uint32_t sTmem = bar_acc + 16;
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(gbase + (sTmem - base));
  const int c = (int)cluster_ctarank();          // this CTA's part of K
  const int wt = (int)(blockIdx.x / ks);         // weight tile
  const int nkb = (int)(p.K / KC::kElemsPerKB);
  const int kb0 = c * nkb / ks, kb1 = (c + 1) * nkb / ks;
  const long long wrow0 = (long long)wt * BW;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    fence_mbar_init();
    fence_proxy_async();
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.b);
  }
  if (warp == 1) {
    tmem_alloc(sTmem, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    // ======================================================== TMA producer
    for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
      const int s = it % S;
      if (!mbar_wait(bar_empty + 8 * s, ((it / S) & 1u) ^ 1u, p.status)) break;
      const uint32_t st = sRing + s * STB;
      mbar_arrive_expect_tx(bar_full + 8 * s, STB);
      const long long ke = (long long)kb * KC::kElemsPerKB;
      const int xb = (int)(KIND == MPM_KIND_NVFP4 ? ke / 2 : ke);
      tma_load_2d(st, &maps.b, xb, (int)wrow0, bar_full + 8 * s);
      tma_load_2d(st + TILE, &maps.a, xb, 0, bar_full + 8 * s);
      const long long atom = (KIND == MPM_KIND_NVFP4) ? ke / 64 : ke / 128;
      const uint32_t sf0 = st + 2 * TILE;
      bulk_load(sf0, p.sfb + ((wrow0 >> 7) * (p.sfb_cols_pad >> 2) + atom) * 512,
                KC::kAtoms * 512, bar_full + 8 * s);
      bulk_load(sf0 + KC::kAtoms * 512, p.sfa + atom * 512, KC::kAtoms * 512, bar_full + 8 * s);
    }
  } else if (warp == 1 && lane == 0) {
    // ======================================================== scale copies + MMA issue
    const uint32_t idesc_base = idesc_block_scaled(KC::kFmt, BR, KC::kUe8m0, 0, 128);
    for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
      const int s = it % S;
      if (!mbar_wait(bar_full + 8 * s, (it / S) & 1u, p.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t st = sRing + s * STB;
      const uint32_t sf0 = st + 2 * TILE;
      const uint32_t sfcol = tmem + BR + s * SFC;
#pragma unroll
      for (int w = 0; w < 2; ++w)
#pragma unroll
        for (int a = 0; a < KC::kAtoms; ++a)
          tc_cp_32x128b_x4(sfcol + (w * KC::kAtoms + a) * 4, sdesc_sf(sf0 + (w * KC::kAtoms + a) * 512));
      const uint32_t sfrow = sfcol + KC::kAtoms * 4;
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const uint64_t adesc = sdesc_sw128(st + k4 * 32);
        const uint64_t bdesc = sdesc_sw128(st + TILE + k4 * 32);
        const uint32_t acc = (it > 0 || k4 > 0) ? 1u : 0u;
        if (KIND == MPM_KIND_NVFP4) {
          mma_nvf4(tmem, adesc, bdesc, idesc_base, sfcol + k4 * 4, sfrow + k4 * 4, acc);
        } else {
          const uint32_t idesc = idesc_block_scaled(KC::kFmt, BR, KC::kUe8m0, (uint32_t)k4, 128);
          mma_mxf8(tmem, adesc, bdesc, idesc, sfcol, sfrow, acc);
        }
      }
      tc_commit(bar_empty + 8 * s);
    }
    if (ok && kb1 > kb0) tc_commit(bar_acc);
  } else if (warp >= 2) {
    // ======================================================== partial -> shared memory
    const int q = warp & 3;                      // TMEM lane quarter = 32 weight rows
    const int f = q * 32 + lane;                 // this thread's feature within the tile
    float* part = reinterpret_cast<float*>(gbase + (sRing - base));
    bool w_ok = true;
    if (kb1 > kb0) w_ok = mbar_wait(bar_acc, 0u, p.status);
    if (kb1 > kb0 && w_ok) {
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tacc + cb * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int r = 0; r < 32; ++r) part[(cb * 32 + r) * BW + f] = __uint_as_float(v[r]);
      }
    } else {
      // no k-blocks for this CTA, or a failed wait: a zero partial
      for (int r = 0; r < BR; ++r) part[r * BW + f] = 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                                // every partial is in place
  if (warp >= 2) {
    // ======================================================== fixed-order reduction
    // a warp takes one row's 128 features (512 contiguous bytes) per step
    const int t = threadIdx.x - 64;              // 0 .. 127
    const int rows_per = BR / ks;                // ks divides 128
    for (int i = 0; i < rows_per / 4; ++i) {
      const int idx = (i * 128 + t) * 4;         // within this CTA's row slice
      const int row = c * rows_per + idx / BW;
      const int feat = idx % BW;
      const uint32_t off = (uint32_t)((row * BW + feat) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < ks; ++j) {
        const uint32_t src = map_to_rank(sRing + off, (uint32_t)j);
        float4 v;
        asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(src));
        if (j == 0) {
          acc = v;
        } else {
          acc.x = __fadd_rn(acc.x, v.x);
          acc.y = __fadd_rn(acc.y, v.y);
          acc.z = __fadd_rn(acc.z, v.z);
          acc.w = __fadd_rn(acc.w, v.w);
        }
      }
      if (row < p.a_rows) {
        const float ab = p.alpha_b ? p.alpha_b[0] : 1.0f;
        const float alpha = p.alpha_a ? __fmul_rn(p.alpha_a[row], ab) : ab;
        const long long o = (long long)row * p.ldo + wrow0 + feat;
        const float4 y = make_float4(__fmul_rn(acc.x, alpha), __fmul_rn(acc.y, alpha),
                                     __fmul_rn(acc.z, alpha), __fmul_rn(acc.w, alpha));
        if (EPI == MPM_EPI_F32) {
          *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o) = y;
        } else {
          __nv_bfloat162 lo = __floats2bfloat162_rn(y.x, y.y), hi = __floats2bfloat162_rn(y.z, y.w);
          uint2 w;
          w.x = *reinterpret_cast<uint32_t*>(&lo);
          w.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + o) = w;
        }
      }
    }
  }
  cluster_sync();                                // the peers are done reading this partial
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace splitk

template <int KIND, int EPI>
static cudaError_t launch_small_one(const smallk::SmallMaps& maps, const GemmArgs& a, int n_wt,
                                    long long n_tasks, cudaStream_t s) {
  constexpr int smem = smallk::smem_bytes<KIND, EPI>();
  static_assert(smem <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
  static_assert(smem > 114 * 1024, "one CTA per SM (each allocates all TMEM columns)");
  auto kern = smallk::grouped_gemm_small_kernel<KIND, EPI>;
  static int sms[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && sms[dev] == 0) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = n > 0 ? n : 1;
  }
  long long grid = dev < 64 ? sms[dev] : 1;
  if (grid > n_tasks) grid = n_tasks;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, smallk::NTHREADS_G, smem, s>>>(maps, a, n_wt, n_tasks);
  return cudaGetLastError();
}

template <int KIND, int EPI>
static cudaError_t launch_splitk_one(const smallk::SmallMaps& maps, const GemmArgs& a, int n_wt,
                                     int ks, cudaStream_t s) {
  constexpr int smem = splitk::smem_bytes<KIND>();
  static_assert(smem <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
  static_assert(smem > 114 * 1024, "one CTA per SM (TMEM allocation never waits)");
  auto kern = splitk::gemm_splitk_kernel<KIND, EPI>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !attr_set[dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(n_wt * ks), 1, 1);
  cfg.blockDim = dim3(smallk::NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, maps, a, ks);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_gemm_splitk(int kind, int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                               const GemmArgs& a, int n_wt, int ks, cudaStream_t s) {
  smallk::SmallMaps maps;
  maps.a = ta;
  maps.b = tb;
  if (ks < 1 || ks > splitk::KS_MAX || (smallk::BR % ks) != 0) return cudaErrorInvalidValue;
  if (kind == MPM_KIND_NVFP4) {
    if (epi == MPM_EPI_F32) return launch_splitk_one<MPM_KIND_NVFP4, MPM_EPI_F32>(maps, a, n_wt, ks, s);
    if (epi == MPM_EPI_BF16) return launch_splitk_one<MPM_KIND_NVFP4, MPM_EPI_BF16>(maps, a, n_wt, ks, s);
  } else if (kind == MPM_KIND_MXFP8) {
    if (epi == MPM_EPI_F32) return launch_splitk_one<MPM_KIND_MXFP8, MPM_EPI_F32>(maps, a, n_wt, ks, s);
    if (epi == MPM_EPI_BF16) return launch_splitk_one<MPM_KIND_MXFP8, MPM_EPI_BF16>(maps, a, n_wt, ks, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_grouped_gemm_small(int kind, int epi, const CUtensorMap& ta,
                                      const CUtensorMap& tb, const GemmArgs& a, int n_wt,
                                      long long n_tasks, cudaStream_t s) {
  smallk::SmallMaps maps;
  maps.a = ta;
  maps.b = tb;
  if (kind == MPM_KIND_NVFP4) {
    switch (epi) {
      case MPM_EPI_F32: return launch_small_one<MPM_KIND_NVFP4, MPM_EPI_F32>(maps, a, n_wt, n_tasks, s);
      case MPM_EPI_BF16: return launch_small_one<MPM_KIND_NVFP4, MPM_EPI_BF16>(maps, a, n_wt, n_tasks, s);
      case MPM_EPI_SWIGLU:
        return launch_small_one<MPM_KIND_NVFP4, MPM_EPI_SWIGLU>(maps, a, n_wt, n_tasks, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (kind == MPM_KIND_MXFP8) {
    switch (epi) {
      case MPM_EPI_F32: return launch_small_one<MPM_KIND_MXFP8, MPM_EPI_F32>(maps, a, n_wt, n_tasks, s);
      case MPM_EPI_BF16: return launch_small_one<MPM_KIND_MXFP8, MPM_EPI_BF16>(maps, a, n_wt, n_tasks, s);
      case MPM_EPI_SWIGLU:
        return launch_small_one<MPM_KIND_MXFP8, MPM_EPI_SWIGLU>(maps, a, n_wt, n_tasks, s);
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace mpm
