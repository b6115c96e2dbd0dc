// FC2 of the single-pass NVFP4 expert FFN: the grouped GEMM whose activation
// was quantised tile by tile against a running row amax, with the partial
// sum compensated as the outer scale grows.
//
// Source: "miniTE technical report", section 5.6.  FC2 walks its reduction
// (the expert intermediate I) in tiles; tile i of a row is encoded against
// gs_i = (running row amax up to tile i) / 2688 (mpm_nvfp4_quantize_online),
// and the section keeps the partial output on the current scale by
// O <- O * gs_prev / gs_i + dO_i with dO_i the tile's product taken with the
// block scales only; at the end Y = O * gs_last * s_g(W2).  Unrolled, that
// compensation is the closed form O * gs_last = sum_i gs_i * dO_i: every tile
// weighed by its own outer scale.  This kernel accumulates that sum directly,
// Y = s_g(W2_e) * sum_i gs_i * dO_i (one fp32 FMA per tile and element), so
// no rescale of earlier partial sums is needed.
//
// Layout on GB300: the reduction tile is one ring stage (256 FP4 elements),
// so every stage produces its own dO_i.  A CTA pair computes a 256-row x
// 128-column output tile with tcgen05.mma.cta_group::2 (M = 256, N = 128);
// dO_i goes to one of three 128-column TMEM accumulators (the MMAs of the
// next two tiles run while the epilogue drains tile i); the epilogue warps keep O in
// registers (one row per thread, 64 columns), fold each dO_i in with packed
// f32x2 FMAs, and after the last tile write bf16 Y through a 128-byte-swizzled
// staging box with TMA stores.  TMEM: three accumulators (384 columns) and
// four stages' scale tiles (32 columns each).  Expert segments are multiples of
// 256 rows (mpm_moe_build_segments with pad = 256), as for the CTA-pair GEMM.
#include "gemm.cuh"

namespace mpm {
namespace onlinek {

constexpr int BM = 128;              // rows per CTA; 256 per pair
constexpr int BN = 128;              // output columns per tile (64 B rows per CTA)
constexpr int BKB = 128;             // bytes of K per stage (256 FP4 elements)
constexpr int KT = 256;              // reduction tile of the online quantisation
constexpr int S = 4;                 // ring stages (and TMEM scale slots)
constexpr int A_STAGE = BM * BKB;            // 16 KB
constexpr int B_STAGE = (BN / 2) * BKB;      // this CTA's 64 rows of B: 8 KB
constexpr int SFA_BYTES = 4 * 512;           // 4 K-steps x one 128-row tile
constexpr int SFB_BYTES = 4 * 512;           // 4 K-steps x the tile's 128 B rows
constexpr int STAGE_BYTES = A_STAGE + B_STAGE + SFA_BYTES + SFB_BYTES;
constexpr int OUT_BOX_COLS = 64;
constexpr int OUT_BOX_BYTES = BM * OUT_BOX_COLS * 2;    // 16 KB
constexpr int OUT_BYTES = 2 * OUT_BOX_BYTES;            // the 128 x 128 bf16 tile
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t NACC = 3;                // accumulators of 128 columns
constexpr uint32_t SF_TMEM_BASE = NACC * BN;  // after the accumulators
constexpr uint32_t SF_COLS = 16 + 16;        // SFA 4 tiles + SFB 4 tiles, 4 columns each
static_assert(SF_TMEM_BASE + S * SF_COLS <= TMEM_COLS, "TMEM budget");
constexpr int EPI_WARP0 = 3;
constexpr int EPI_THREADS = 256;
constexpr int NTHREADS = 14 * 32;    // 0 TMA, 1 MMA, 2 + 11..13 scale stores, 3..10 epilogue

constexpr int smem_bytes() { return 2048 + S * STAGE_BYTES + OUT_BYTES + (4 * S + 2 * NACC) * 8 + 32; }

struct OnlineMaps {
  CUtensorMap a, b, sfa, sfb, out;
};

MPM_DEV bool named_sync_or(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(n) : "memory");
  return r != 0;
}
// (o0, o1) <- (g * d0 + o0, g * d1 + o1), one packed f32x2 FMA (per lane the
// IEEE fused multiply-add of the scalar form)
MPM_DEV void fma2(float& o0, float& o1, float g, float d0, float d1) {
  uint64_t o, d, gg, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(o) : "f"(o0), "f"(o1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(d0), "f"(d1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(gg) : "f"(g));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(gg), "l"(d), "l"(o));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(o0), "=f"(o1) : "l"(r));
}
MPM_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

struct Task {
  bool valid;
  int e;
  long long row_pair, n0, brow;
};

struct SegCursor {
  int e = -1;
  long long lo = 0, hi = 0, end = -1;
};

// tasks = (256-row pair of A rows) x (128-column N tile); the pair's expert
// is the segment holding its first row (found by a forward cursor)
MPM_DEV Task task_of(const GemmArgs& p, long long t, int n_tiles, int* bad, SegCursor& cur) {
  Task k{};
  const long long mp = t / n_tiles, nt = t - mp * n_tiles;
  k.row_pair = mp * 2 * BM;
  if (cur.end < 0) {
    cur.end = p.seg[p.E];
    cur.e = 0;
    cur.lo = p.seg[0];
    cur.hi = p.seg[1];
  }
  if (k.row_pair >= cur.end || k.row_pair >= p.a_rows) { k.valid = false; return k; }
  while (cur.e + 1 < p.E && cur.hi <= k.row_pair) {
    ++cur.e;
    cur.lo = cur.hi;
    cur.hi = p.seg[cur.e + 1];
  }
  if ((cur.lo & 255) != 0 || (cur.hi & 255) != 0) *bad = 1;      // not pair-aligned
  k.e = cur.e;
  k.n0 = nt * BN;
  k.brow = (long long)cur.e * p.b_rows_per_e + k.n0;
  k.valid = true;
  return k;
}

__global__ void __launch_bounds__(NTHREADS, 1)
fc2_online_kernel(const __grid_constant__ OnlineMaps maps, const GemmArgs p, const int n_tiles,
                  const long long n_tasks) {
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const long long cid = cluster_id_x(), ncl = nclusters_x();
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = sA + S * A_STAGE;
  const uint32_t sSFA = sB + S * B_STAGE;
  const uint32_t sSFB = sSFA + S * SFA_BYTES;
  const uint32_t sOut = (sSFB + S * SFB_BYTES + 1023u) & ~1023u;
  const uint32_t sBar = sOut + OUT_BYTES;
  const uint32_t bar_full = sBar, bar_empty = sBar + 8 * S;
  const uint32_t bar_acc = sBar + 16 * S;      // buffer b: full at + 16 b, empty at + 16 b + 8
  const uint32_t sTmem = bar_acc + 16 * NACC;
  const uint32_t sFlag = sTmem + 8;
  const uint32_t bar_sf = sTmem + 16;          // scale tiles of a stage in TMEM (leader)
  const uint32_t bar_sfull = bar_sf + 8 * S;   // scale tiles of a stage in shared memory
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(gbase + (sTmem - base));
  volatile int* fail_flag = reinterpret_cast<volatile int*>(gbase + (sFlag - base));
  const int n_kt = (int)(p.K / KT);            // reduction tiles = ring stages per task

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_sf + 8 * s, 2);            // one arrive per CTA (after its store warps)
      mbar_init(bar_sfull + 8 * s, 1);
    }
    for (uint32_t b = 0; b < NACC; ++b) {
      mbar_init(bar_acc + 16 * b, 1);
      mbar_init(bar_acc + 16 * b + 8, 16);     // one arrive per epilogue warp of both CTAs
    }
    *fail_flag = 0;
    fence_mbar_init();
    fence_proxy_async();
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.b);
    prefetch_tmap(&maps.sfa);
    prefetch_tmap(&maps.sfb);
    prefetch_tmap(&maps.out);
  }
  if (warp == 1) {
    tmem_alloc_pair(sTmem, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  int bad = 0;

  if (warp == 0 && lane == 0) {
    // ======================================================== TMA producer (both CTAs)
    uint32_t it = 0;
    bool ok = true;
    SegCursor cur;
    for (long long t = cid; ok && t < n_tasks; t += ncl) {
      const Task k = task_of(p, t, n_tiles, &bad, cur);
      if (!k.valid) break;
      const long long a_row = k.row_pair + rank * BM;
      for (int kb = 0; kb < n_kt; ++kb, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1u;
        if (!mbar_wait_cluster(bar_empty + 8 * s, ph ^ 1u, p.status)) { ok = false; break; }
        mbar_arrive_expect_tx(bar_sfull + 8 * s, SFA_BYTES + SFB_BYTES);
        if (rank == 0) mbar_arrive_expect_tx(bar_full + 8 * s, 2 * (A_STAGE + B_STAGE));
        const uint32_t fb = map_to_rank(bar_full + 8 * s, 0);
        const long long ka = (long long)kb * KT;
        const long long kbb = (long long)k.e * p.b_k_per_e + ka;
        tma_load_2d(sSFA + s * SFA_BYTES, &maps.sfa, 0,
                    (int)((a_row >> 7) * (p.sfa_cols_pad >> 2) + ka / 64), bar_sfull + 8 * s);
        tma_load_2d(sSFB + s * SFB_BYTES, &maps.sfb, 0,
                    (int)((k.brow >> 7) * (p.sfb_cols_pad >> 2) + kbb / 64), bar_sfull + 8 * s);
        tma_load_2d_pair(sA + s * A_STAGE, &maps.a, (int)(ka / 2), (int)a_row, fb);
        tma_load_2d_pair(sB + s * B_STAGE, &maps.b, (int)(kbb / 2), (int)(k.brow + rank * (BN / 2)),
                         fb);
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ======================================================== MMA issuer (leader only)
    // every stage is a reduction tile of its own: a fresh accumulation into
    // accumulator j % 2, committed to the epilogue when the stage's four
    // MMAs complete
    uint32_t j = 0;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    const uint32_t idesc = idesc_block_scaled(1, BN, 0, 0, 256);
    SegCursor cur;
    for (long long t = cid; ok && t < n_tasks; t += ncl) {
      const Task k = task_of(p, t, n_tiles, &bad, cur);
      if (!k.valid) break;
      for (int kb = 0; kb < n_kt; ++kb, ++j) {
        const uint32_t ab = j % NACC, use = j / NACC;
        if (!mbar_wait_cluster(bar_acc + 16 * ab + 8, (use & 1u) ^ 1u, p.status)) { ok = false; break; }
        if (!mbar_wait(bar_sf + 8 * s, ph, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dacc = tmem + ab * BN;
        const uint32_t sf_col = tmem + SF_TMEM_BASE + s * SF_COLS;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t adesc = sdesc_sw128(sA + s * A_STAGE + ks * 32);
          const uint64_t bdesc = sdesc_sw128(sB + s * B_STAGE + ks * 32);
          mma_nvf4_pair(dacc, adesc, bdesc, idesc, sf_col + ks * 4, sf_col + 16 + ks * 4,
                        ks > 0 ? 1u : 0u);
        }
        tc_commit_pair(bar_empty + 8 * s, (uint16_t)3);
        tc_commit_pair(bar_acc + 16 * ab, (uint16_t)3);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
  } else if (warp == 2 || warp >= 11) {
    // ======================================================== scale tiles -> TMEM (both CTAs)
    // Warp w writes TMEM lane quarter w % 4: lane l of each 512-byte tile goes
    // to lane 32 q + l, four columns (the replicated layout of the block-
    // scaled MMA).  The leader's arriver also waits for the stage's A and B,
    // so its arrive tells the MMA thread that the whole stage is ready; the
    // arrives are CTA-scoped (the TMEM stores completed before them).
    const int q = warp & 3;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t sf_leader = map_to_rank(bar_sf, 0);
    const bool arriver = (warp == 2 && lane == 0);
    uint32_t it = 0;
    bool ok = true;
    SegCursor cur;
    for (long long t = cid; ok && t < n_tasks; t += ncl) {
      const Task k = task_of(p, t, n_tiles, &bad, cur);
      if (!k.valid) break;
      for (int kb = 0; kb < n_kt; ++kb, ++it) {
        const int s = it % S;
        const bool w_ok = mbar_wait_cluster(bar_sfull + 8 * s, (it / S) & 1u, p.status);
        if (w_ok) {
          const uint32_t col = tq + SF_TMEM_BASE + s * SF_COLS;
          const uint8_t* sa = gbase + (sSFA - base) + s * SFA_BYTES + lane * 16;
          const uint8_t* sb = gbase + (sSFB - base) + s * SFB_BYTES + lane * 16;
#pragma unroll
          for (int a = 0; a < 4; ++a)
            tmem_st_32x32b_x4(col + a * 4, *reinterpret_cast<const uint4*>(sa + a * 512));
#pragma unroll
          for (int a = 0; a < 4; ++a)
            tmem_st_32x32b_x4(col + 16 + a * 4, *reinterpret_cast<const uint4*>(sb + a * 512));
          tmem_st_wait();
        }
        bool a_ok = true;
        if (arriver && rank == 0) a_ok = mbar_wait(bar_full + 8 * s, (it / S) & 1u, p.status);
        tc_fence_before();
        if (named_sync_or(3, 128, !(w_ok && a_ok))) { ok = false; break; }
        if (arriver) {
          if (rank == 0) mbar_arrive(bar_sf + 8 * s);
          else mbar_arrive_cluster(sf_leader + 8 * s);
        }
      }
    }
  } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + 8) {
    // ======================================================== epilogue (both CTAs)
    // thread = one row of this CTA's 128 and 64 of the tile's 128 columns
    const int q = warp & 3;
    const int half = (warp - EPI_WARP0) >> 2;
    const int r = q * 32 + lane;
    const uint32_t trow0 = tmem + ((uint32_t)(q * 32) << 16) + half * 64;
    const uint32_t acce_leader0 = map_to_rank(bar_acc + 8, 0);   // buffer b: + 16 b
    const bool leader_thread = (threadIdx.x == EPI_WARP0 * 32);
    const float* gs_rows = static_cast<const float*>(p.aux);    // [rows, n_kt]
    uint32_t j = 0;
    SegCursor cur;
    for (long long t = cid; t < n_tasks; t += ncl) {
      const Task k = task_of(p, t, n_tiles, &bad, cur);
      if (!k.valid) break;
      const long long grow = k.row_pair + rank * BM + r;
      const float* gsr = gs_rows + grow * p.ld_aux;
      float o[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) o[c] = 0.0f;
      float g_next = gsr[0];
      bool failed = false;
      for (int kb = 0; kb < n_kt; ++kb, ++j) {
        const uint32_t ab = j % NACC, use = j / NACC;
        const float g = g_next;
        if (kb + 1 < n_kt) g_next = gsr[kb + 1];
        const bool w_ok = mbar_wait_cluster(bar_acc + 16 * ab, use & 1u, p.status);
        if (!w_ok) *fail_flag = 1;
        tc_fence_after();
        // the two 32-column halves one after the other (32 registers in
        // flight, not 64); the other accumulator keeps the MMAs busy meanwhile
        uint32_t v[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tmem_ld_32x32b_x32(trow0 + ab * BN + h * 32, v);
          tmem_ld_wait();
          if (h == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce_leader0 + 16 * ab);
          }
#pragma unroll
          for (int c = 0; c < 32; c += 2)
            fma2(o[h * 32 + c], o[h * 32 + c + 1], g, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
        }
        if (*fail_flag) { failed = true; break; }
      }
      named_sync(1, EPI_THREADS);
      if (failed || *fail_flag) break;
      // Y = s_g(W2_e) * O, bf16, through the two staging boxes (this thread's
      // 64 columns are box `half`)
      const float ag = p.alpha_b ? p.alpha_b[k.e] : 1.0f;
      if (leader_thread) bulk_wait_group_read0();     // the previous tile's boxes were read
      named_sync(2, EPI_THREADS);
      {
        const uint32_t box = sOut + half * OUT_BOX_BYTES + r * 128;
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
          const int c = c16 * 8;
          st_shared_v4(box + ((c16 ^ (r & 7)) << 4),
                       pack_bf16(__fmul_rn(o[c], ag), __fmul_rn(o[c + 1], ag)),
                       pack_bf16(__fmul_rn(o[c + 2], ag), __fmul_rn(o[c + 3], ag)),
                       pack_bf16(__fmul_rn(o[c + 4], ag), __fmul_rn(o[c + 5], ag)),
                       pack_bf16(__fmul_rn(o[c + 6], ag), __fmul_rn(o[c + 7], ag)));
        }
      }
      fence_proxy_async();
      named_sync(2, EPI_THREADS);
      if (leader_thread) {
        const int y = (int)(k.row_pair + rank * BM);
#pragma unroll
        for (int b = 0; b < 2; ++b)
          tma_store_2d(&maps.out, (int)k.n0 + b * OUT_BOX_COLS, y, sOut + b * OUT_BOX_BYTES);
        bulk_commit_group();
      }
    }
  }
  if (threadIdx.x == EPI_WARP0 * 32) bulk_wait_group0();    // output stores complete
  if (bad && threadIdx.x == 0) set_status(p.status, MPM_ERR_DEVICE_BOUNDS);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

}  // namespace onlinek

cudaError_t launch_fc2_online(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsfa,
                              const CUtensorMap& tsfb, const CUtensorMap& tout, const GemmArgs& a,
                              int n_tiles, long long n_tasks, cudaStream_t s) {
  constexpr int smem = onlinek::smem_bytes();
  static_assert(smem <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
  auto kern = onlinek::fc2_online_kernel;
  static int max_clusters[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  onlinek::OnlineMaps maps;
  maps.a = ta;
  maps.b = tb;
  maps.sfa = tsfa;
  maps.sfb = tsfb;
  maps.out = tout;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(onlinek::NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dev < 64 && max_clusters[dev] == 0) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    int ncl = 0;
    err = cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg);
    if (err != cudaSuccess || ncl < 1) ncl = sms / 2;
    max_clusters[dev] = ncl;
  }
  long long ncl = dev < 64 ? max_clusters[dev] : 1;
  if (ncl > n_tasks) ncl = n_tasks;
  if (ncl < 1) ncl = 1;
  cfg.gridDim = dim3((unsigned)(2 * ncl), 1, 1);
  err = cudaLaunchKernelEx(&cfg, kern, maps, a, n_tiles, n_tasks);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace mpm
