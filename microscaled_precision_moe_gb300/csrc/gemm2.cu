// Block-scaled grouped GEMM on CTA pairs (tcgen05 cta_group::2), persistent.
//
// Same contract as the one-CTA kernel in gemm.cu (C_e = A_e * B_e^T, NVFP4 or
// MXFP8 operands, fp32 accumulation, the same epilogues), for row-segmented
// GEMMs whose expert segments are multiples of 256 rows.  A cluster of two
// CTAs computes one 256 x 256 output tile at a time:
//
//   * each CTA stages its own 128 rows of A and its own half of B (128 of the
//     256 B rows) plus the scale tiles of its A rows and of all 256 B rows;
//     the A and B loads, the peer's included, complete on the leader CTA's
//     barriers (cp.async.bulk.tensor .cta_group::2).  A stage's scale tiles
//     are loaded first, on a barrier of their own, so they reach TMEM while
//     the A and B tiles are still in flight (the ring is bound by the latency
//     of one stage's round trip, not by bandwidth);
//   * NVFP4: in each CTA four warps, one per TMEM lane quarter, write the
//     stage's twelve scale tiles into TMEM with tcgen05.st and signal the
//     leader's per-stage barrier; MXFP8: two warps of the leader move both
//     CTAs' three tiles with tcgen05.cp.cta_group::2.  The leader's MMA
//     thread waits for A, B and the scales and issues tcgen05.mma.cta_group::2
//     (M = 256, N = 256); each SM reads only half of B from its shared memory;
//   * each CTA's eight epilogue warps (two per TMEM lane quarter, each taking
//     half of the columns) drain its 128 x 256 accumulator; in the SwiGLU and
//     bf16 epilogues the accumulator is released to the next tile as soon as
//     it is in registers, so the activation math and the stores overlap the
//     next tile's MMAs;
//   * clusters loop over tiles (expert-segment M pairs x N tiles) in a fixed
//     stride, so the shared-memory ring never drains between tiles.
//
// Sources: "miniTE technical report", sections 5.2 and 5.4 (grouped GEMM over
// a contiguous buffer with device offsets; FC1 epilogue); "Towards
// Blackwell-native 8-bit and 4-bit RL", section "Recipe 1 / Training".
#include "gemm.cuh"

namespace mpm {
namespace pairk {

constexpr int BM = 128;              // rows per CTA; 256 per pair
constexpr int BN = 256;
constexpr int BKB = 128;             // bytes of K per stage
// warp 0 TMA, warp 1 MMA + TMEM allocation, warp 2 and warps 11, 12, ...
// the scale tiles (Cfg::kSfWarps warps), warps 3-10 epilogue (two warps per
// TMEM lane quarter, each half the columns)
constexpr int EPI_WARP0 = 3;
constexpr int EPI_THREADS = 256;
constexpr int A_STAGE = BM * BKB;    // 16 KB
constexpr int B_STAGE = 128 * BKB;   // this CTA's half of B: 16 KB
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_TMEM_BASE = 256;

template <int KIND> struct Cfg;
// Stage counts: the ring holds as many stages as shared memory allows next to
// the 32 KB output staging.  Scale tiles into TMEM: an NVFP4 stage has twelve
// 512-byte tiles, each needed replicated in all four TMEM lane quarters.  As
// tcgen05.cp instructions (about 50 cycles of tensor-pipe issue each) they
// held the pipe back; instead four warps, one per lane quarter, load them
// from shared memory and write them with tcgen05.st, which leaves the MMA rate
// untouched (kSfStore).  MXFP8's three tiles per stage stay tcgen05.cp from
// two warps (fully hidden behind the MMAs).
template <> struct Cfg<MPM_KIND_NVFP4> {
  static constexpr int kElemsPerKB = 256;
  static constexpr int kAtomsPerKB = 4;
  static constexpr int kSfaBytes = 4 * 512;
  static constexpr int kSfbBytes = 2 * 4 * 512;
  static constexpr int kSfTmemPerStage = 16 + 32;
  static constexpr int kStages = 5;
  static constexpr int kSfWarps = 4;       // one per TMEM lane quarter, both CTAs
  static constexpr bool kSfStore = true;
  static constexpr uint32_t kFmt = 1, kUe8m0 = 0;
};
template <> struct Cfg<MPM_KIND_MXFP8> {
  static constexpr int kElemsPerKB = 128;
  static constexpr int kAtomsPerKB = 1;
  static constexpr int kSfaBytes = 512;
  static constexpr int kSfbBytes = 2 * 512;
  static constexpr int kSfTmemPerStage = 4 + 8;
  static constexpr int kStages = 5;
  static constexpr int kSfWarps = 2;       // tcgen05.cp issuers, leader only
  static constexpr bool kSfStore = false;
  static constexpr uint32_t kFmt = 0, kUe8m0 = 1;
};
// bf16 operands (the high-precision / dequantized backward): 64 elements per
// 128-byte stage row, no scale tiles, one more stage in the freed space
template <> struct Cfg<MPM_KIND_BF16> {
  static constexpr int kElemsPerKB = 64;
  static constexpr int kAtomsPerKB = 0;
  static constexpr int kSfaBytes = 0;
  static constexpr int kSfbBytes = 0;
  static constexpr int kSfTmemPerStage = 0;
  static constexpr int kStages = 6;
  static constexpr int kSfWarps = 2;       // idle: no scale tiles
  static constexpr bool kSfStore = false;
  static constexpr uint32_t kFmt = 0, kUe8m0 = 0;
};

template <int KIND>
constexpr int stage_bytes() {
  return A_STAGE + B_STAGE + Cfg<KIND>::kSfaBytes + Cfg<KIND>::kSfbBytes;
}
// output staging for the TMA-store epilogues: two boxes of 128 rows x 128
// bytes (64 bf16 or 32 fp32 columns, 128-byte swizzle); a CTA's 128 x 256
// tile goes out in rounds of two boxes
constexpr int OUT_BOX_COLS = 64;
constexpr int OUT_BOX_BYTES = BM * OUT_BOX_COLS * 2;    // 16 KB
constexpr int STAGE_OUT_BYTES = 2 * OUT_BOX_BYTES;      // 32 KB

// The SwiGLU-backward epilogue streams C in and dH out through two staging
// buffers of 32 KB (one 64-column chunk of gate and of up each), so its ring
// has one stage less than the kind's default (the bf16 kind: two less).
// (Staging a whole 128 x 256 bf16 output tile the same way, to store it in
// one round instead of two, was measured slower for FC2: the ring stage it
// costs outweighs the second round, 1.86 against 1.70 ms.)
template <int KIND, int EPI>
constexpr bool staging64() {
  return EPI == MPM_EPI_DSWIGLU;
}
template <int KIND, int EPI>
constexpr int stages() {
  return EPI == MPM_EPI_DSWIGLU ? (KIND == MPM_KIND_BF16 ? 5 : 4)
                                : (staging64<KIND, EPI>() ? 4 : Cfg<KIND>::kStages);
}
// The SwiGLU-backward epilogue parks the second half of a CTA's dD tile
// (128 columns) in TMEM columns [DSW_SPARE, 512) when the accumulator and the
// scale slots leave them free, so it can hand the accumulator back before C
// streams in (only with one accumulator: the bf16 kind has two).
constexpr uint32_t DSW_SPARE = 384;
template <int KIND, int EPI>
constexpr bool dsw_park() {
  return EPI == MPM_EPI_DSWIGLU && KIND != MPM_KIND_BF16 &&
         SF_TMEM_BASE + stages<KIND, EPI>() * Cfg<KIND>::kSfTmemPerStage <= DSW_SPARE;
}
template <int KIND, int EPI>
constexpr int out_staging_bytes() {
  return staging64<KIND, EPI>() ? 2 * STAGE_OUT_BYTES : STAGE_OUT_BYTES;
}
template <int KIND, int EPI>
constexpr int smem_bytes() {
  return 2048 + stages<KIND, EPI>() * stage_bytes<KIND>() + out_staging_bytes<KIND, EPI>() +
         (4 * stages<KIND, EPI>() + 4) * 8 + 32 + 16;
}

MPM_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

struct Task {
  bool valid;
  int e;
  long long row_pair;   // first row (of A / of the expert's output) of the pair tile
  long long out_row;    // first output row of this pair tile in the output matrix
  long long n0;         // first output column (D columns for SwiGLU)
  long long brow[2];    // global B rows of the two 128-row halves
  long long ka0, kb0;   // reduction offsets (elements) of A and B
  int num_kb;
};

// Each role of a CTA walks its tasks in increasing order, so it finds a
// task's expert by moving a cursor forward over the device segment offsets
// (each offset is read from global memory once per role, not the ~log2(E)
// dependent reads of a binary search for every task).
struct SegCursor {
  int e = -1;               // expert whose [lo, hi) row range is cached
  long long lo = 0, hi = 0;
  long long end = -1;       // seg[E] (GROUP_M) once read
};

// GROUP_M: tasks = (256-row pair of A rows) x (N tile); the pair's expert is
// the segment holding its first row.  GROUP_K: tasks = expert x (256-row pair
// of output rows) x (N tile); the reduction runs over the expert's segment.
template <int KIND, int EPI>
MPM_DEV Task task_of(const GemmArgs& p, long long t, int n_tiles, int* bad, SegCursor& cur) {
  Task k{};
  const bool swiglu = (EPI == MPM_EPI_SWIGLU || EPI == MPM_EPI_SWIGLU_SAVE);
  int e = 0;
  long long mp, nt;
  if (p.group == MPM_GROUP_K) {
    const long long n_mp = p.M_out / (2 * BM);
    const long long per_e = n_mp * n_tiles;
    e = (int)(t / per_e);
    if (e >= p.E) { k.valid = false; return k; }
    const long long rem = t - (long long)e * per_e;
    mp = rem / n_tiles;
    nt = rem - mp * n_tiles;
    if (e != cur.e) {
      cur.e = e;
      cur.lo = p.seg[e];
      cur.hi = p.seg[e + 1];
    }
    const long long s0 = cur.lo, s1 = cur.hi;
    if (s1 < s0 || ((s1 - s0) % Cfg<KIND>::kElemsPerKB) != 0) *bad = 1;
    k.num_kb = s1 > s0 ? (int)((s1 - s0) / Cfg<KIND>::kElemsPerKB) : 0;
    k.row_pair = mp * 2 * BM;
    k.out_row = (long long)e * p.M_out + k.row_pair;
    k.ka0 = s0;
    k.kb0 = s0;
    k.n0 = nt * BN;
    k.brow[0] = k.n0;
    k.brow[1] = k.n0 + 128;
  } else {
    mp = t / n_tiles;
    nt = t - mp * n_tiles;
    k.row_pair = mp * 2 * BM;
    if (p.seg) {
      if (cur.end < 0) {
        cur.end = p.seg[p.E];
        cur.e = 0;
        cur.lo = p.seg[0];
        cur.hi = p.seg[1];
      }
      if (k.row_pair >= cur.end) { k.valid = false; return k; }
      while (cur.e + 1 < p.E && cur.hi <= k.row_pair) {
        ++cur.e;
        cur.lo = cur.hi;
        cur.hi = p.seg[cur.e + 1];
      }
      e = cur.e;
      if ((cur.lo & 255) != 0 || (cur.hi & 255) != 0) *bad = 1;   // not pair-aligned
    } else if (k.row_pair >= p.a_rows) {
      k.valid = false;
      return k;
    }
    k.out_row = k.row_pair;
    k.n0 = nt * (swiglu ? BN / 2 : BN);
    if (swiglu) {
      k.brow[0] = (long long)e * p.b_rows_per_e + k.n0;
      k.brow[1] = (long long)e * p.b_rows_per_e + p.N / 2 + k.n0;
    } else {
      k.brow[0] = (long long)e * p.b_rows_per_e + k.n0;
      k.brow[1] = k.brow[0] + 128;
    }
    k.ka0 = 0;
    k.kb0 = (long long)e * p.b_k_per_e;
    k.num_kb = (int)(p.K / Cfg<KIND>::kElemsPerKB);
  }
  k.e = e;
  k.valid = true;
  return k;
}

struct PairMaps {
  CUtensorMap a, b, sfa, sfb;
  CUtensorMap out;    // bf16 output of the BF16 epilogue / D of the SwiGLU epilogues / dH
  CUtensorMap aux;    // C = gate|up: read by the SwiGLU-backward epilogue, written by SWIGLU_SAVE
};

// MAJ (bf16 only): bit 0 = A stored MN-major ([K rows, M] with M contiguous:
// the weight-gradient A), bit 1 = B stored MN-major ([K rows, N]).  An
// MN-major operand is staged as two 64-element-wide boxes of 64 K rows each
// (128 bytes x 64 rows, 128-byte swizzle) per 128 rows of M or N.
template <int KIND>
constexpr int nthreads() { return 32 * (10 + Cfg<KIND>::kSfWarps); }

// named barrier over `n` threads that also ORs a predicate across them
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

template <int KIND, int EPI, int MAJ>
__global__ void __launch_bounds__(nthreads<KIND>(), 1)
grouped_gemm_pair_kernel(const __grid_constant__ PairMaps maps, const GemmArgs p, const int n_tiles,
                         const long long n_tasks) {
  using C = Cfg<KIND>;
  constexpr bool A_MN = (MAJ & 1) != 0, B_MN = (MAJ & 2) != 0;
  static_assert(MAJ == 0 || KIND == MPM_KIND_BF16, "MN-major operands are bf16 only");
  constexpr int S = stages<KIND, EPI>();
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();          // 0 = leader of the pair
  const long long cid = cluster_id_x(), ncl = nclusters_x();

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = sA + S * A_STAGE;
  const uint32_t sSFA = sB + S * B_STAGE;
  const uint32_t sSFB = sSFA + S * C::kSfaBytes;
  // the 128-byte-swizzled staging boxes need a 1024-byte-aligned base
  const uint32_t sOut = (sSFB + S * C::kSfbBytes + 1023u) & ~1023u;
  const uint32_t sBar = sOut + out_staging_bytes<KIND, EPI>();
  const uint32_t bar_full = sBar, bar_empty = sBar + 8 * S;
  // accumulator buffer b: full barrier at bar_acc + 16 b, empty at + 8.  The
  // bf16 kind keeps two accumulators in TMEM (columns 0-255 and 256-511, no
  // scale factors there) so a tile's epilogue overlaps the next tile's MMAs.
  constexpr uint32_t NACC = (KIND == MPM_KIND_BF16) ? 2u : 1u;
  const uint32_t bar_acc = sBar + 16 * S;
  const uint32_t sTmem = bar_acc + 32;
  const uint32_t sFlag = sTmem + 8;
  const uint32_t bar_sf = bar_acc + 48;        // scale tiles of a stage are in TMEM
  const uint32_t bar_sfull = bar_sf + 8 * S;   // scale tiles of a stage are in shared memory
  const uint32_t bar_c = bar_sfull + 8 * S;    // SwiGLU backward: C chunk in staging buffer b (+8 b)
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(gbase + (sTmem - base));
  volatile int* fail_flag = reinterpret_cast<volatile int*>(gbase + (sFlag - base));

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(bar_acc + 16 * b, 1);
      mbar_init(bar_acc + 16 * b + 8, 16);  // one arrive per epilogue warp of both CTAs
    }
    for (int s = 0; s < S; ++s) {
      // NVFP4: one arrive per CTA (its four store warps, after a named
      // barrier); MXFP8: one commit per copy warp
      mbar_init(bar_sf + 8 * s, C::kSfStore ? 2 : C::kSfWarps);
      mbar_init(bar_sfull + 8 * s, 1);
    }
    if (EPI == MPM_EPI_DSWIGLU) {
      mbar_init(bar_c, 1);
      mbar_init(bar_c + 8, 1);
    }
    *fail_flag = 0;
    fence_mbar_init();
    fence_proxy_async();
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.b);
    if (KIND != MPM_KIND_BF16) {
      prefetch_tmap(&maps.sfa);
      prefetch_tmap(&maps.sfb);
    }
    prefetch_tmap(&maps.out);
    if (EPI == MPM_EPI_DSWIGLU || EPI == MPM_EPI_SWIGLU_SAVE) prefetch_tmap(&maps.aux);
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
    SegCursor cur;
    for (long long t = cid; t < n_tasks; t += ncl) {
      const Task k = task_of<KIND, EPI>(p, t, n_tiles, &bad, cur);
      if (!k.valid) break;
      const long long a_row = k.row_pair + rank * BM;
      const long long sfa_rt = a_row >> 7;
      bool ok = true;
      for (int kb = 0; kb < k.num_kb; ++kb, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1u;
        if (!mbar_wait_cluster(bar_empty + 8 * s, ph ^ 1u, p.status)) { ok = false; break; }
        // the stage's scale tiles go first, on their own barrier: they move
        // into TMEM while A and B are still in flight.  NVFP4: each CTA loads
        // its own tiles on its own barrier (its store warps read them);
        // MXFP8: the leader's barrier (its copy warps move both CTAs' tiles)
        if (KIND != MPM_KIND_BF16 && C::kSfStore)
          mbar_arrive_expect_tx(bar_sfull + 8 * s, C::kSfaBytes + C::kSfbBytes);
        if (rank == 0) {
          if (KIND != MPM_KIND_BF16 && !C::kSfStore)
            mbar_arrive_expect_tx(bar_sfull + 8 * s, 2 * (C::kSfaBytes + C::kSfbBytes));
          mbar_arrive_expect_tx(bar_full + 8 * s, 2 * (A_STAGE + B_STAGE));
        }
        const uint32_t fb = map_to_rank(bar_full + 8 * s, 0);   // the leader's barriers
        const long long ka = k.ka0 + (long long)kb * C::kElemsPerKB;
        const long long kbb = k.kb0 + (long long)kb * C::kElemsPerKB;
        if (KIND != MPM_KIND_BF16) {
          const long long atom_a = (KIND == MPM_KIND_NVFP4) ? ka / 64 : ka / 128;
          const long long atom_b = (KIND == MPM_KIND_NVFP4) ? kbb / 64 : kbb / 128;
          const int ya = (int)(sfa_rt * (p.sfa_cols_pad >> 2) + atom_a);
          if (C::kSfStore) {
            tma_load_2d(sSFA + s * C::kSfaBytes, &maps.sfa, 0, ya, bar_sfull + 8 * s);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_2d(sSFB + s * C::kSfbBytes + h * (C::kSfbBytes / 2), &maps.sfb, 0,
                          (int)((k.brow[h] >> 7) * (p.sfb_cols_pad >> 2) + atom_b), bar_sfull + 8 * s);
          } else {
            const uint32_t fsb = map_to_rank(bar_sfull + 8 * s, 0);
            tma_load_2d_pair(sSFA + s * C::kSfaBytes, &maps.sfa, 0, ya, fsb);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_2d_pair(sSFB + s * C::kSfbBytes + h * (C::kSfbBytes / 2), &maps.sfb, 0,
                               (int)((k.brow[h] >> 7) * (p.sfb_cols_pad >> 2) + atom_b), fsb);
          }
        }
        // x coordinates in bytes: 128-byte multiples for every kind
        const int xa = (int)(KIND == MPM_KIND_NVFP4 ? ka / 2 : (KIND == MPM_KIND_BF16 ? ka * 2 : ka));
        const int xb =
            (int)(KIND == MPM_KIND_NVFP4 ? kbb / 2 : (KIND == MPM_KIND_BF16 ? kbb * 2 : kbb));
        if (A_MN) {
          // A stored [K rows, M]: this CTA's 128 M columns from K row ka
          tma_load_2d_pair(sA + s * A_STAGE, &maps.a, (int)(a_row * 2), (int)ka, fb);
          tma_load_2d_pair(sA + s * A_STAGE + A_STAGE / 2, &maps.a, (int)((a_row + 64) * 2),
                           (int)ka, fb);
        } else {
          tma_load_2d_pair(sA + s * A_STAGE, &maps.a, xa, (int)a_row, fb);
        }
        if (B_MN) {
          // B stored [K rows, N]: this CTA's 128 N columns from K row kbb
          tma_load_2d_pair(sB + s * B_STAGE, &maps.b, (int)(k.brow[rank] * 2), (int)kbb, fb);
          tma_load_2d_pair(sB + s * B_STAGE + B_STAGE / 2, &maps.b,
                           (int)((k.brow[rank] + 64) * 2), (int)kbb, fb);
        } else {
          tma_load_2d_pair(sB + s * B_STAGE, &maps.b, xb, (int)k.brow[rank], fb);
        }
      }
      if (!ok) break;
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ======================================================== MMA issuer (leader only)
    uint32_t j = 0;
    int s = 0;                                 // ring stage and its phase, kept incrementally
    uint32_t ph = 0;
    bool ok = true;
    SegCursor cur;
    for (long long t = cid; ok && t < n_tasks; t += ncl) {
      const Task k = task_of<KIND, EPI>(p, t, n_tiles, &bad, cur);
      if (!k.valid) break;
      if (k.num_kb == 0) continue;             // empty reduction: nothing to accumulate
      const uint32_t ab = j % NACC, use = j / NACC;
      if (!mbar_wait_cluster(bar_acc + 16 * ab + 8, (use & 1u) ^ 1u, p.status)) break;
      ++j;
      const uint32_t dacc = tmem + ab * 256;
      tc_fence_after();
      for (int kb = 0; kb < k.num_kb; ++kb) {
        // This thread's instruction stream paces the ring (each tcgen05.mma
        // takes ~70 cycles to issue), so it waits on one barrier per stage
        // where it can: NVFP4 — the scale barrier, which the leader's store
        // warps signal only after the stage's A and B have landed too;
        // MXFP8 — A/B and the copies' barrier; bf16 — A/B.  CTA-scoped
        // acquire on the leader's own barriers; tcgen05.fence::after_thread_sync
        // orders the MMAs after the wait.
        if (!C::kSfStore && !mbar_wait(bar_full + 8 * s, ph, p.status)) { ok = false; break; }
        if (KIND != MPM_KIND_BF16 && !mbar_wait(bar_sf + 8 * s, ph, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sf_col = tmem + SF_TMEM_BASE + s * C::kSfTmemPerStage;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          // K step of one MMA: 32 bytes along a K-major row, or 16 rows
          // (2048 bytes) of an MN-major tile
          const uint64_t adesc = A_MN ? sdesc_sw128_mn(sA + s * A_STAGE + ks * 2048, A_STAGE / 2)
                                      : sdesc_sw128(sA + s * A_STAGE + ks * 32);
          const uint64_t bdesc = B_MN ? sdesc_sw128_mn(sB + s * B_STAGE + ks * 2048, B_STAGE / 2)
                                      : sdesc_sw128(sB + s * B_STAGE + ks * 32);
          const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
          if (KIND == MPM_KIND_BF16) {
            mma_bf16_pair(dacc, adesc, bdesc, idesc_bf16(BN, 256, A_MN ? 1u : 0u, B_MN ? 1u : 0u), acc);
          } else if (KIND == MPM_KIND_NVFP4) {
            const uint32_t idesc = idesc_block_scaled(C::kFmt, BN, C::kUe8m0, 0, 256);
            mma_nvf4_pair(dacc, adesc, bdesc, idesc, sf_col + ks * 4, sf_col + 16 + ks * 8, acc);
          } else {
            const uint32_t idesc = idesc_block_scaled(C::kFmt, BN, C::kUe8m0, (uint32_t)ks, 256);
            mma_mxf8_pair(dacc, adesc, bdesc, idesc, sf_col, sf_col + 4, acc);
          }
        }
        tc_commit_pair(bar_empty + 8 * s, (uint16_t)3);
        if (kb + 1 == k.num_kb) tc_commit_pair(bar_acc + 16 * ab, (uint16_t)3);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
  } else if ((warp == 2 || warp >= 11) && C::kSfStore) {
    // ======================================================== scale tiles, tcgen05.st (both CTAs)
    // Warp w writes TMEM lane quarter w % 4 (warps 2, 11, 12, 13: quarters
    // 2, 3, 0, 1): lane l of each 512-byte tile (its 16-byte row l) goes to
    // lane 32 q + l, four columns — the replicated layout the block-scaled
    // MMA reads.  After the stores complete, the four warps meet on a named
    // barrier and one thread arrives on the leader's stage barrier.  That
    // arrive (from the peer CTA too) is CTA-scoped: tcgen05.wait::st has
    // completed the TMEM stores before it executes, so it publishes no memory
    // operation; a cluster-scoped release there cost about 2k cycles per stage
    // and held the whole ring back (dense NVFP4 2.4 PFLOP/s instead of 6.2).
    const int q = warp & 3;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t sf_leader = map_to_rank(bar_sf, 0);
    const bool arriver = (warp == 2 && lane == 0);
    uint32_t it = 0;
    bool ok = true;
    SegCursor cur;
    for (long long t = cid; ok && t < n_tasks; t += ncl) {
      const Task k = task_of<KIND, EPI>(p, t, n_tiles, &bad, cur);
      if (!k.valid) break;
      for (int kb = 0; kb < k.num_kb; ++kb, ++it) {
        const int s = it % S;
        const bool w_ok = mbar_wait_cluster(bar_sfull + 8 * s, (it / S) & 1u, p.status);
        if (w_ok) {
          const uint32_t col = tq + SF_TMEM_BASE + s * C::kSfTmemPerStage;
          const uint8_t* sa = gbase + (sSFA - base) + s * C::kSfaBytes + lane * 16;
          const uint8_t* sb = gbase + (sSFB - base) + s * C::kSfbBytes + lane * 16;
#pragma unroll
          for (int a = 0; a < 4; ++a)
            tmem_st_32x32b_x4(col + a * 4, *reinterpret_cast<const uint4*>(sa + a * 512));
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const int h = b >> 2, ks = b & 3;
            tmem_st_32x32b_x4(col + 16 + ks * 8 + h * 4,
                              *reinterpret_cast<const uint4*>(sb + h * 2048 + ks * 512));
          }
          tmem_st_wait();
        }
        // the leader's arriver also waits for the stage's A and B, so its
        // arrive tells the MMA thread that the whole stage is ready
        bool a_ok = true;
        if (arriver && rank == 0) a_ok = mbar_wait(bar_full + 8 * s, (it / S) & 1u, p.status);
        tc_fence_before();
        // every store warp takes part in the barrier, failed wait or not
        if (named_sync_or(3, 128, !(w_ok && a_ok))) { ok = false; break; }
        if (arriver) {
          if (rank == 0) mbar_arrive(bar_sf + 8 * s);
          else mbar_arrive_cluster(sf_leader + 8 * s);
        }
      }
    }
  } else if ((warp == 2 || warp >= 11) && lane == 0 && rank == 0 && KIND != MPM_KIND_BF16) {
    // ======================================================== scale-tile copies (MXFP8, leader only)
    // kSfWarps threads in as many warps each copy a share of a stage's scale
    // tiles with tcgen05.cp and commit to the stage's barrier.
    constexpr int NCP = C::kSfWarps;
    const int part = (warp == 2) ? 0 : warp - 10;    // 0 .. NCP-1
    uint32_t it = 0;
    bool ok = true;
    SegCursor cur;
    for (long long t = cid; ok && t < n_tasks; t += ncl) {
      const Task k = task_of<KIND, EPI>(p, t, n_tiles, &bad, cur);
      if (!k.valid) break;
      for (int kb = 0; kb < k.num_kb; ++kb, ++it) {
        const int s = it % S;
        if (!mbar_wait_cluster(bar_sfull + 8 * s, (it / S) & 1u, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sf_col = tmem + SF_TMEM_BASE + s * C::kSfTmemPerStage;
        // three atoms: SFA, SFB h = 0, 1
#pragma unroll
        for (int a = 0; a < 3; ++a)
          if (a % NCP == part) {
            if (a == 0)
              tc_cp_32x128b_x4_pair(sf_col, sdesc_sf(sSFA + s * C::kSfaBytes));
            else
              tc_cp_32x128b_x4_pair(sf_col + 4 + (a - 1) * 4,
                                    sdesc_sf(sSFB + s * C::kSfbBytes + (a - 1) * 512));
          }
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     :: "r"(bar_sf + 8 * s) : "memory");
      }
    }
  } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + 8) {
    // ======================================================== epilogue (both CTAs)
    const int q = warp & 3;                     // TMEM lane quarter of this warp
    const int half = (warp - EPI_WARP0) >> 2;   // which half of the columns
    const int r = q * 32 + lane;                // row within this CTA's 128 rows
    const uint32_t trow0 = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t acce_leader0 = map_to_rank(bar_acc + 8, 0);
    const uint32_t acce_leader1 = NACC > 1 ? map_to_rank(bar_acc + 16 + 8, 0) : acce_leader0;
    const bool leader_thread = (threadIdx.x == EPI_WARP0 * 32);
    // SwiGLU backward: staging loads not yet waited for, and the phase parity
    // each one completes
    uint32_t c_pending = 0, c_parity = 0;
    uint32_t j = 0;
    SegCursor cur;
    for (long long t = cid; t < n_tasks; t += ncl) {
      const Task k = task_of<KIND, EPI>(p, t, n_tiles, &bad, cur);
      if (!k.valid) break;
      const long long orow = k.out_row + rank * BM;          // this CTA's first output row
      if (k.num_kb == 0) {
        // empty reduction (an expert without rows in the wgrad mode): zeros
        if (EPI == MPM_EPI_F32) {
          float* o = static_cast<float*>(p.out) + (orow + r) * p.ldo + k.n0 + half * 128;
          for (int c = 0; c < 128; c += 4) *reinterpret_cast<float4*>(o + c) = make_float4(0, 0, 0, 0);
        }
        continue;
      }
      // the row's scales come from global memory: load them before waiting
      // for the accumulator so their latency is not part of the hand-off
      const long long grow = k.row_pair + rank * BM + r;     // row of A (GROUP_M)
      const bool row_ok = (p.group == MPM_GROUP_K) || grow < p.a_rows;
      float alpha_a = 1.0f, alpha_b = 1.0f, prob_r = 0.0f;
      if (row_ok && p.group == MPM_GROUP_M) {
        if (p.alpha_a) alpha_a = p.alpha_a[grow];
        if (p.alpha_b) alpha_b = p.alpha_b[k.e];
        if ((EPI == MPM_EPI_SWIGLU || EPI == MPM_EPI_SWIGLU_SAVE || EPI == MPM_EPI_DSWIGLU) &&
            p.row_prob)
          prob_r = p.row_prob[grow];
      }
      // SwiGLU backward: the tile's first two 64-column chunks of C (gate
      // and up boxes of this CTA's 128 rows) are requested before the
      // accumulator wait, into the two staging buffers
      if (EPI == MPM_EPI_DSWIGLU && leader_thread) {
        bulk_wait_group_read0();                 // the previous tile's dH stores have read them
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint32_t buf = sOut + b * STAGE_OUT_BYTES;
          mbar_arrive_expect_tx(bar_c + 8 * b, STAGE_OUT_BYTES);
          tma_load_2d(buf, &maps.aux, (int)k.n0 + b * OUT_BOX_COLS, (int)orow, bar_c + 8 * b);
          tma_load_2d(buf + OUT_BOX_BYTES, &maps.aux, (int)(p.N + k.n0) + b * OUT_BOX_COLS,
                      (int)orow, bar_c + 8 * b);
        }
        c_pending = 3u;
        c_parity = 0u;                          // first load of each buffer in the tile
      }
      const uint32_t ab = NACC > 1 ? (j & 1u) : 0u, use = NACC > 1 ? (j >> 1) : j;
      const bool w_ok = mbar_wait_cluster(bar_acc + 16 * ab, use & 1u, p.status);
      ++j;
      const uint32_t trow = NACC > 1 ? trow0 + ab * 256 : trow0;
      const uint32_t acce_leader = (NACC > 1 && ab) ? acce_leader1 : acce_leader0;
      if (!w_ok) *fail_flag = 1;
      named_sync(1, EPI_THREADS);
      if (*fail_flag) break;
      tc_fence_after();
      const float alpha = (p.alpha_b && p.group == MPM_GROUP_M) ? __fmul_rn(alpha_a, alpha_b) : alpha_a;
      uint32_t v[32], u[32];
      if (EPI == MPM_EPI_SWIGLU || EPI == MPM_EPI_SWIGLU_SAVE) {
        // this thread: D columns [64*half, 64*half + 64) of the tile
        const uint64_t alpha2 = f32x2(alpha, alpha), prob2 = f32x2(prob_r, prob_r);
        uint32_t dw[32];
        uint32_t cgw[EPI == MPM_EPI_SWIGLU_SAVE ? 32 : 1], cuw[EPI == MPM_EPI_SWIGLU_SAVE ? 32 : 1];
        uint32_t amax2 = 0;
        uint32_t v2[32], u2[32];
        // the thread's whole share of the accumulator in flight at once, one
        // wait, then the accumulator goes back to the MMA before any math
        tmem_ld_32x32b_x32(trow + (half * 2) * 32, v);
        tmem_ld_32x32b_x32(trow + 128 + (half * 2) * 32, u);
        tmem_ld_32x32b_x32(trow + (half * 2 + 1) * 32, v2);
        tmem_ld_32x32b_x32(trow + 128 + (half * 2 + 1) * 32, u2);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acce_leader);   // this warp's share is read
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint32_t* gv = cc ? v2 : v;
          const uint32_t* uv = cc ? u2 : u;
          // two elements per step with packed f32x2 products (the same
          // per-lane results as swiglu_fwd); the row amax over |D| as bf16
          // bit patterns (non-negative bf16 order like unsigned integers)
#pragma unroll
          for (int jj = 0; jj < 32; jj += 2) {
            // swiglu_fwd2 written out, so SWIGLU_SAVE keeps the scaled gate
            // and up values as the bf16 words of C
            float g0, g1, d0, d1;
            f32x2_split(mul_f32x2(f32x2(__uint_as_float(gv[jj]), __uint_as_float(gv[jj + 1])), alpha2),
                        g0, g1);
            const uint64_t uu = mul_f32x2(f32x2(__uint_as_float(uv[jj]), __uint_as_float(uv[jj + 1])),
                                          alpha2);
            if (EPI == MPM_EPI_SWIGLU_SAVE) {
              float u0, u1;
              f32x2_split(uu, u0, u1);
              cgw[cc * 16 + jj / 2] = pack_bf16(g0, g1);
              cuw[cc * 16 + jj / 2] = pack_bf16(u0, u1);
            }
            const uint64_t su = mul_f32x2(f32x2(swiglu_silu(g0), swiglu_silu(g1)), uu);
            f32x2_split(mul_f32x2(su, prob2), d0, d1);
            const uint32_t pk = pack_bf16(d0, d1);
            dw[cc * 16 + jj / 2] = pk;
            amax2 = absmax_bf16x2(amax2, pk);
          }
        }
        // D tile (128 rows x 128 columns) -> staging box `half`, then TMA store
        if (leader_thread) bulk_wait_group_read0();     // previous tile's boxes read
        named_sync(2, EPI_THREADS);
        {
          const uint32_t box = sOut + half * OUT_BOX_BYTES + r * 128;
#pragma unroll
          for (int c16 = 0; c16 < 8; ++c16)
            st_shared_v4(box + ((c16 ^ (r & 7)) << 4), dw[4 * c16], dw[4 * c16 + 1],
                         dw[4 * c16 + 2], dw[4 * c16 + 3]);
        }
        fence_proxy_async();
        named_sync(2, EPI_THREADS);
        if (leader_thread) {
          const int y = (int)orow;
#pragma unroll
          for (int b = 0; b < 2; ++b)
            tma_store_2d(&maps.out, (int)k.n0 + b * OUT_BOX_COLS, y, sOut + b * OUT_BOX_BYTES);
          bulk_commit_group();
        }
        if (EPI == MPM_EPI_SWIGLU_SAVE) {
          // C = gate | up (alpha applied, bf16) for the backward: this
          // thread's 64 gate columns, then its 64 up columns, each round
          // through staging box `half` and out by TMA stores (the same bits
          // as the FC1 output the SwiGLU was computed from)
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint32_t* cw = part ? cuw : cgw;
            if (leader_thread) bulk_wait_group_read0();   // the previous boxes were read
            named_sync(2, EPI_THREADS);
            const uint32_t box = sOut + half * OUT_BOX_BYTES + r * 128;
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16)
              st_shared_v4(box + ((c16 ^ (r & 7)) << 4), cw[4 * c16], cw[4 * c16 + 1],
                           cw[4 * c16 + 2], cw[4 * c16 + 3]);
            fence_proxy_async();
            named_sync(2, EPI_THREADS);
            if (leader_thread) {
              const int x0 = (int)k.n0 + (part ? (int)(p.N / 2) : 0);
#pragma unroll
              for (int b = 0; b < 2; ++b)
                tma_store_2d(&maps.aux, x0 + b * OUT_BOX_COLS, (int)orow, sOut + b * OUT_BOX_BYTES);
              bulk_commit_group();
            }
          }
        }
        const float amax = bf16lo(max(amax2 & 0xFFFFu, amax2 >> 16));
        if (row_ok && p.amax && amax > 0.0f)
          atomicMax(reinterpret_cast<unsigned*>(p.amax) + grow, __float_as_uint(amax));
      } else if (EPI == MPM_EPI_BF16) {
        // this thread: columns [128*half, 128*half + 128)
        uint32_t ow[64];
        uint32_t v2[32], v3[32], v4[32];
        tmem_ld_32x32b_x32(trow + (half * 4 + 0) * 32, v);
        tmem_ld_32x32b_x32(trow + (half * 4 + 1) * 32, v2);
        tmem_ld_32x32b_x32(trow + (half * 4 + 2) * 32, v3);
        tmem_ld_32x32b_x32(trow + (half * 4 + 3) * 32, v4);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acce_leader);   // this warp's share is read
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint32_t* vv = cc == 0 ? v : (cc == 1 ? v2 : (cc == 2 ? v3 : v4));
#pragma unroll
          for (int jj = 0; jj < 32; jj += 2)
            ow[cc * 16 + jj / 2] = pack_bf16(__fmul_rn(__uint_as_float(vv[jj]), alpha),
                                             __fmul_rn(__uint_as_float(vv[jj + 1]), alpha));
        }
        // two rounds: the warps of column half `round` write their 128
        // columns into the two staging boxes, then one TMA store each
#pragma unroll 1
        for (int round = 0; round < 2; ++round) {
          if (leader_thread) bulk_wait_group_read0();
          named_sync(2, EPI_THREADS);
          if (half == round) {
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
              const uint32_t box = sOut + bb * OUT_BOX_BYTES + r * 128;
#pragma unroll
              for (int c16 = 0; c16 < 8; ++c16) {
                const int w = bb * 32 + 4 * c16;
                st_shared_v4(box + ((c16 ^ (r & 7)) << 4), ow[w], ow[w + 1], ow[w + 2], ow[w + 3]);
              }
            }
          }
          fence_proxy_async();
          named_sync(2, EPI_THREADS);
          if (leader_thread) {
#pragma unroll
            for (int b = 0; b < 2; ++b)
              tma_store_2d(&maps.out, (int)k.n0 + round * 128 + b * OUT_BOX_COLS, (int)orow,
                           sOut + b * OUT_BOX_BYTES);
            bulk_commit_group();
          }
        }
      } else if (EPI == MPM_EPI_F32) {
        // the thread's 128 fp32 columns are loaded at once and the
        // accumulator handed back; then fp32 boxes of 32 columns (128 bytes)
        // x 128 rows go out in four rounds of two boxes
        uint32_t v2[32], v3[32], v4[32];
        tmem_ld_32x32b_x32(trow + (half * 4 + 0) * 32, v);
        tmem_ld_32x32b_x32(trow + (half * 4 + 1) * 32, v2);
        tmem_ld_32x32b_x32(trow + (half * 4 + 2) * 32, v3);
        tmem_ld_32x32b_x32(trow + (half * 4 + 3) * 32, v4);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acce_leader);   // this warp's share is read
#pragma unroll
        for (int round = 0; round < 4; ++round) {
          if (leader_thread) bulk_wait_group_read0();
          named_sync(2, EPI_THREADS);
          if (half == (round >> 1)) {
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
              const int cc = (round & 1) * 2 + bb;
              const uint32_t* vv = cc == 0 ? v : (cc == 1 ? v2 : (cc == 2 ? v3 : v4));
              const uint32_t box = sOut + bb * OUT_BOX_BYTES + r * 128;
#pragma unroll
              for (int c16 = 0; c16 < 8; ++c16)
                st_shared_v4(box + ((c16 ^ (r & 7)) << 4),
                             __float_as_uint(__fmul_rn(__uint_as_float(vv[4 * c16]), alpha)),
                             __float_as_uint(__fmul_rn(__uint_as_float(vv[4 * c16 + 1]), alpha)),
                             __float_as_uint(__fmul_rn(__uint_as_float(vv[4 * c16 + 2]), alpha)),
                             __float_as_uint(__fmul_rn(__uint_as_float(vv[4 * c16 + 3]), alpha)));
            }
          }
          fence_proxy_async();
          named_sync(2, EPI_THREADS);
          if (leader_thread) {
#pragma unroll
            for (int b = 0; b < 2; ++b)
              tma_store_2d(&maps.out, (int)(k.n0 + (round >> 1) * 128 + ((round & 1) * 2 + b) * 32),
                           (int)orow, sOut + b * OUT_BOX_BYTES);
            bulk_commit_group();
          }
        }
      } else {   // MPM_EPI_DSWIGLU
        // dD = acc * alpha (fp32, not rounded); with (g, u) from C:
        //   dH[:, j] = dD p u silu'(g),  dH[:, N + j] = dD p silu(g)   (bf16)
        // The tile goes through in four 64-column chunks.  Chunk cq's gate and
        // up columns of C arrive by TMA in staging buffer cq % 2 (two 16 KB
        // boxes, 128-byte swizzle); each thread takes 32 columns of its row
        // (this warp's half of the chunk), reads dD for them from TMEM,
        // overwrites the C values in place with dg / du, and the two boxes
        // go out to dH by TMA stores; the buffer is then refilled with chunk
        // cq + 2.  Where TMEM has room (dsw_park), the thread's columns of
        // chunks 2 and 3 are first copied to spare TMEM columns and those of
        // chunks 0 and 1 loaded into registers, and the accumulator goes back
        // to the MMA before any C is waited for; otherwise it is handed back
        // once the last chunk's columns are in registers.
        const float prob = prob_r;
        constexpr bool kPark = dsw_park<KIND, EPI>();
        const uint32_t park = trow0 + DSW_SPARE + half * 64;   // this thread's 64 parked columns
        if (kPark) {
          tmem_ld_32x32b_x32(trow + 2 * 64 + half * 32, v);
          tmem_ld_32x32b_x32(trow + 3 * 64 + half * 32, u);
          tmem_ld_wait();
          tmem_st_32x32b_x32(park, v);
          tmem_st_32x32b_x32(park + 32, u);
          tmem_ld_32x32b_x32(trow + 0 * 64 + half * 32, v);
          tmem_ld_32x32b_x32(trow + 1 * 64 + half * 32, u);
          tmem_ld_wait();
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acce_leader);     // this warp's share is read
        }
#pragma unroll 1
        for (int cq = 0; cq < 4; ++cq) {
          if (kPark) {
            // v holds the even chunk's columns, u the odd one's: move this
            // chunk's into v (registers cannot be selected by a runtime index)
            if (cq == 1) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = u[i];
            } else if (cq == 2) {
              tmem_ld_32x32b_x32(park, v);
              tmem_ld_32x32b_x32(park + 32, u);
              tmem_ld_wait();
            } else if (cq == 3) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = u[i];
            }
          } else {
            tmem_ld_32x32b_x32(trow + cq * 64 + half * 32, v);
            tmem_ld_wait();
            if (cq == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(acce_leader);   // this warp's share is read
            }
          }
          const int b = cq & 1;
          const uint32_t buf = sOut + b * STAGE_OUT_BYTES;
          const bool c_ok = mbar_wait(bar_c + 8 * b, (uint32_t)(cq >> 1) & 1u, p.status);
          if (leader_thread && c_ok) c_pending &= ~(1u << b);
          if (!c_ok) *fail_flag = 1;
          const uint32_t rg = buf + r * 128, ru = rg + OUT_BOX_BYTES;
#pragma unroll
          for (int c16 = 0; c16 < 4; ++c16) {
            const uint32_t off = (uint32_t)(((half * 4 + c16) ^ (r & 7)) << 4);
            uint32_t ga[4], ua[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(ga[0]), "=r"(ga[1]), "=r"(ga[2]), "=r"(ga[3]) : "r"(rg + off));
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(ua[0]), "=r"(ua[1]), "=r"(ua[2]), "=r"(ua[3]) : "r"(ru + off));
            uint32_t og4[4], ou4[4];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              float dg2[2], du2[2];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const float g = h ? bf16hi(ga[qq]) : bf16lo(ga[qq]);
                const float uu = h ? bf16hi(ua[qq]) : bf16lo(ua[qq]);
                const float dd = __fmul_rn(__uint_as_float(v[c16 * 8 + 2 * qq + h]), alpha);
                swiglu_bwd(g, uu, dd, prob, dg2[h], du2[h]);
              }
              og4[qq] = pack_bf16(dg2[0], dg2[1]);
              ou4[qq] = pack_bf16(du2[0], du2[1]);
            }
            st_shared_v4(rg + off, og4[0], og4[1], og4[2], og4[3]);
            st_shared_v4(ru + off, ou4[0], ou4[1], ou4[2], ou4[3]);
          }
          fence_proxy_async();
          named_sync(2, EPI_THREADS);
          if (*fail_flag) break;
          if (leader_thread) {
            tma_store_2d(&maps.out, (int)k.n0 + cq * OUT_BOX_COLS, (int)orow, buf);
            tma_store_2d(&maps.out, (int)(p.N + k.n0) + cq * OUT_BOX_COLS, (int)orow,
                         buf + OUT_BOX_BYTES);
            bulk_commit_group();
            if (cq + 2 < 4) {
              bulk_wait_group_read0();             // the stores have read the buffer
              mbar_arrive_expect_tx(bar_c + 8 * b, STAGE_OUT_BYTES);
              tma_load_2d(buf, &maps.aux, (int)k.n0 + (cq + 2) * OUT_BOX_COLS, (int)orow,
                          bar_c + 8 * b);
              tma_load_2d(buf + OUT_BOX_BYTES, &maps.aux,
                          (int)(p.N + k.n0) + (cq + 2) * OUT_BOX_COLS, (int)orow, bar_c + 8 * b);
              c_pending |= 1u << b;
              c_parity |= 1u << b;          // the buffer's second load of the tile
            }
          }
        }
        if (*fail_flag) break;
      }
    }
    // a failed wait left staging loads in flight: let them land before exit
    if (EPI == MPM_EPI_DSWIGLU && leader_thread) {
      for (int b = 0; b < 2; ++b)
        if (c_pending & (1u << b)) mbar_wait(bar_c + 8 * b, (c_parity >> b) & 1u, p.status);
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

}  // namespace pairk

// ---------------------------------------------------------------- launcher
template <int KIND, int EPI, int MAJ = 0>
static cudaError_t launch_pair_one(const pairk::PairMaps& maps, const GemmArgs& a, int n_tiles,
                                   long long n_tasks, cudaStream_t s) {
  constexpr int smem = pairk::smem_bytes<KIND, EPI>();
  static_assert(smem <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
  auto kern = pairk::grouped_gemm_pair_kernel<KIND, EPI, MAJ>;
  static int max_clusters[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(pairk::nthreads<KIND>(), 1, 1);
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

template <int KIND>
static cudaError_t pair_dispatch(int epi, const pairk::PairMaps& maps, const GemmArgs& a,
                                 int n_tiles, long long n_tasks, cudaStream_t s) {
  switch (epi) {
    case MPM_EPI_F32: return launch_pair_one<KIND, MPM_EPI_F32>(maps, a, n_tiles, n_tasks, s);
    case MPM_EPI_BF16: return launch_pair_one<KIND, MPM_EPI_BF16>(maps, a, n_tiles, n_tasks, s);
    case MPM_EPI_SWIGLU: return launch_pair_one<KIND, MPM_EPI_SWIGLU>(maps, a, n_tiles, n_tasks, s);
    case MPM_EPI_SWIGLU_SAVE:
      return launch_pair_one<KIND, MPM_EPI_SWIGLU_SAVE>(maps, a, n_tiles, n_tasks, s);
    case MPM_EPI_DSWIGLU: return launch_pair_one<KIND, MPM_EPI_DSWIGLU>(maps, a, n_tiles, n_tasks, s);
    default: return cudaErrorInvalidValue;
  }
}

// bf16 with MN-major operands: B MN-major for the input gradients (bf16 out,
// or the SwiGLU backward), A and B MN-major for the weight gradients (fp32)
static cudaError_t pair_dispatch_bf16_mn(int maj, int epi, const pairk::PairMaps& maps,
                                         const GemmArgs& a, int n_tiles, long long n_tasks,
                                         cudaStream_t s) {
  constexpr int K = MPM_KIND_BF16;
  if (maj == 2) {
    switch (epi) {
      case MPM_EPI_F32: return launch_pair_one<K, MPM_EPI_F32, 2>(maps, a, n_tiles, n_tasks, s);
      case MPM_EPI_BF16: return launch_pair_one<K, MPM_EPI_BF16, 2>(maps, a, n_tiles, n_tasks, s);
      case MPM_EPI_DSWIGLU:
        return launch_pair_one<K, MPM_EPI_DSWIGLU, 2>(maps, a, n_tiles, n_tasks, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (maj == 3 && epi == MPM_EPI_F32)
    return launch_pair_one<K, MPM_EPI_F32, 3>(maps, a, n_tiles, n_tasks, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_grouped_gemm_pair(int kind, int epi, int maj, const CUtensorMap& ta,
                                     const CUtensorMap& tb, const CUtensorMap& tsfa,
                                     const CUtensorMap& tsfb, const CUtensorMap& tout,
                                     const CUtensorMap& taux, const GemmArgs& a, int n_tiles,
                                     long long n_tasks, cudaStream_t s) {
  pairk::PairMaps maps;
  maps.a = ta;
  maps.b = tb;
  maps.sfa = tsfa;
  maps.sfb = tsfb;
  maps.out = tout;
  maps.aux = taux;
  if (kind == MPM_KIND_NVFP4) return pair_dispatch<MPM_KIND_NVFP4>(epi, maps, a, n_tiles, n_tasks, s);
  if (kind == MPM_KIND_BF16) {
    if (maj != 0) return pair_dispatch_bf16_mn(maj, epi, maps, a, n_tiles, n_tasks, s);
    return pair_dispatch<MPM_KIND_BF16>(epi, maps, a, n_tiles, n_tasks, s);
  }
  return pair_dispatch<MPM_KIND_MXFP8>(epi, maps, a, n_tiles, n_tasks, s);
}

}  // namespace mpm
