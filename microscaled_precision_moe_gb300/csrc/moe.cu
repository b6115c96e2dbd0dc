// Expert segments, permutation gather and combine for sm_103a.
//
// "miniTE technical report", section 5.2: the routed rows of all experts sit
// in one contiguous buffer whose expert boundaries are offsets kept on the
// device; zero-token experts and the padding of each segment (to 128 rows, one
// MMA tile, 256, one CTA-pair tile, or 16-64 rows for the small-M kernel) are
// handled in the same path.  Section 5.3: the permute gathers each routed
// (token, slot) row; the combine sums a token's expert outputs.
//
// The counting sort is stable: rows of one expert appear in ascending flat
// index t*k + j.  Every step is integer work, so results are bit-identical
// run to run.
#include "moe.cuh"

namespace mpm {

constexpr int kSegChunk = 512;    // flat (token, slot) pairs per chunk (one warp each)

// 1) per-chunk expert histogram: hist[chunk][e]
__global__ void __launch_bounds__(256) seg_hist_kernel(const int* ids, long long n, int E,
                                                      int* hist, int* st) {
  extern __shared__ int h[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const long long base = (long long)blockIdx.x * kSegChunk;
  for (int i = threadIdx.x; i < kSegChunk; i += blockDim.x) {
    const long long f = base + i;
    if (f >= n) break;
    const int e = ids[f];
    if (e >= 0 && e < E) atomicAdd(&h[e], 1);
    else set_status(st, MPM_ERR_DEVICE_BOUNDS);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(long long)blockIdx.x * E + e] = h[e];
}

// 2a) one CTA per expert: exclusive prefix of the expert's column of the
//     histogram over the chunks (each thread sums a run of chunks, then a
//     block scan of the thread sums): base[chunk][e] relative to the
//     segment start, and the expert's total
__global__ void __launch_bounds__(256) seg_colscan_kernel(const int* __restrict__ hist, int nchunks,
                                                         int E, int* __restrict__ base,
                                                         int* __restrict__ totals) {
  __shared__ int warp_sum[8];
  const int e = blockIdx.x;
  const int per = (nchunks + 255) / 256;
  const int c0 = threadIdx.x * per;
  const int c1 = min(c0 + per, nchunks);
  int local = 0;
  for (int c = c0; c < c1; ++c) local += hist[(long long)c * E + e];
  // block exclusive scan of the 256 thread sums
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[w] = incl;
  __syncthreads();
  int woff = 0;
  for (int i = 0; i < w; ++i) woff += warp_sum[i];
  int run = woff + incl - local;                 // exclusive prefix of this thread's run
  for (int c = c0; c < c1; ++c) {
    const int v = hist[(long long)c * E + e];
    base[(long long)c * E + e] = run;
    run += v;
  }
  if (threadIdx.x == 255) totals[e] = woff + incl;
}

// 2b) one CTA: padded segment offsets from the expert totals (exclusive scan)
__global__ void __launch_bounds__(1024) seg_offsets_kernel(const int* __restrict__ totals, int E,
                                                          int pad, int* __restrict__ seg_offsets) {
  __shared__ int padded[1024];
  const int e = threadIdx.x;
  const int mine = (e < E) ? (totals[e] + pad - 1) / pad * pad : 0;
  padded[e] = mine;
  __syncthreads();
  // Hillis-Steele inclusive scan over padded sizes
  for (int o = 1; o < 1024; o <<= 1) {
    const int v = (e >= o) ? padded[e - o] : 0;
    __syncthreads();
    padded[e] += v;
    __syncthreads();
  }
  if (e < E) seg_offsets[e] = padded[e] - mine;
  if (e == E - 1) seg_offsets[E] = padded[e];
}

// 3) stable scatter: one warp walks its chunk in order, 32 pairs at a time
__global__ void __launch_bounds__(32) seg_scatter_kernel(const int* ids, const float* prob,
                                                        long long n, int E, const int* base,
                                                        const int* seg_offsets, int* perm,
                                                        int* inv_perm, float* row_prob) {
  extern __shared__ int cnt[];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) cnt[e] = base[(long long)blockIdx.x * E + e] + seg_offsets[e];
  __syncwarp();
  const long long c0 = (long long)blockIdx.x * kSegChunk;
  for (int s = 0; s < kSegChunk; s += 32) {
    const long long f = c0 + s + lane;
    int e = -1;
    if (f < n) {
      e = ids[f];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned grp = __match_any_sync(0xFFFFFFFFu, e);
    const unsigned lt = (1u << lane) - 1u;
    const int rank = __popc(grp & lt);
    int row = -1;
    if (e >= 0) row = cnt[e] + rank;
    __syncwarp();
    if (e >= 0 && (grp >> lane) == 1u) cnt[e] += __popc(grp);   // highest lane of group
    __syncwarp();
    if (f < n) {
      inv_perm[f] = row;
      if (row >= 0) {
        perm[row] = (int)f;
        row_prob[row] = prob[f];
      }
    }
    if (c0 + s + 32 >= n) break;
  }
}

// ---------------------------------------------------------------- one cooperative kernel
// The same four steps (histogram, per-expert column scan, padded offsets,
// stable scatter) in one persistent launch whose CTAs meet at two grid
// barriers: at these sizes the separate launches cost more than their work
// (about 46 us for any T).  The kernel is launched cooperatively, so every
// CTA is resident; a barrier wait is bounded and, past the limit, records
// MPM_ERR_DEVICE_TIMEOUT and leaves the kernel.  The results are those of the
// four kernels above, bit for bit: the same chunks, the same scans, the same
// per-chunk stable scatter.
struct SegFused {
  const int* ids; const float* prob;
  long long n; int E; int pad; int nchunks;
  int* hist; int* base; int* totals;
  int* seg_offsets; int* perm; int* inv_perm; float* row_prob; long long cap;
  unsigned* bar;            // [2]: arrival count, generation (zeroed by the launcher)
  int* st;
};

// grid-wide barrier: the last CTA to arrive resets the count and bumps the
// generation; the others wait for the generation to move (bounded)
MPM_DEV bool seg_grid_sync(unsigned* bar, int* st) {
  __syncthreads();
  __shared__ int ok;
  if (threadIdx.x == 0) {
    ok = 1;
    volatile unsigned* gen = bar + 1;
    const unsigned g0 = *gen;
    __threadfence();
    if (atomicAdd(bar, 1u) == gridDim.x - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      long long n = 0;
      while (*gen == g0) {
        if (++n > (1ll << 26)) { set_status(st, MPM_ERR_DEVICE_TIMEOUT); ok = 0; break; }
        __nanosleep(32);
      }
    }
    __threadfence();
  }
  __syncthreads();
  return ok != 0;
}

__global__ void __launch_bounds__(256) seg_fused_kernel(const SegFused a) {
  extern __shared__ int sh[];                  // max(E, 8 E) ints
  const int E = a.E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // phase 0: clear the permuted buffers, per-chunk histograms
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < a.cap;
       i += (long long)gridDim.x * blockDim.x) {
    a.perm[i] = -1;
    a.row_prob[i] = 0.0f;
  }
  for (int c = blockIdx.x; c < a.nchunks; c += gridDim.x) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
    __syncthreads();
    const long long base = (long long)c * kSegChunk;
    for (int i = threadIdx.x; i < kSegChunk; i += blockDim.x) {
      const long long f = base + i;
      if (f >= a.n) break;
      const int e = a.ids[f];
      if (e >= 0 && e < E) atomicAdd(&sh[e], 1);
      else set_status(a.st, MPM_ERR_DEVICE_BOUNDS);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) a.hist[(long long)c * E + e] = sh[e];
    __syncthreads();
  }
  if (!seg_grid_sync(a.bar, a.st)) return;
  // phase 1: per-expert exclusive scan over the chunks (as seg_colscan_kernel);
  // data other CTAs wrote before a barrier is read from L2 (__ldcg)
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int per = (a.nchunks + 255) / 256;
    const int c0 = threadIdx.x * per;
    const int c1 = min(c0 + per, a.nchunks);
    int local = 0;
    for (int c = c0; c < c1; ++c) local += __ldcg(a.hist + (long long)c * E + e);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    int woff = 0;
    for (int i = 0; i < warp; ++i) woff += sh[i];
    int run = woff + incl - local;
    for (int c = c0; c < c1; ++c) {
      const int v = __ldcg(a.hist + (long long)c * E + e);
      a.base[(long long)c * E + e] = run;
      run += v;
    }
    if (threadIdx.x == 255) a.totals[e] = woff + incl;
    __syncthreads();
  }
  if (!seg_grid_sync(a.bar, a.st)) return;
  // phase 2: padded offsets, computed by every CTA from the totals (block
  // scan over E <= 1024 values: 4 per thread), written by CTA 0
  {
    int v[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = threadIdx.x * 4 + i;
      v[i] = e < E ? (__ldcg(a.totals + e) + a.pad - 1) / a.pad * a.pad : 0;
      sum += v[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    __syncthreads();
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    int woff = 0;
    for (int i = 0; i < warp; ++i) woff += sh[i];
    int run = woff + incl - sum;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = threadIdx.x * 4 + i;
      if (e < E) {
        sh[e] = run;                             // this CTA's copy of seg_offsets[e]
        if (blockIdx.x == 0) a.seg_offsets[e] = run;
      }
      run += v[i];
    }
    if (blockIdx.x == 0 && threadIdx.x == 255) a.seg_offsets[E] = run;
    __syncthreads();
  }
  // phase 3: stable scatter, one warp per chunk (as seg_scatter_kernel), the
  // warp's counters after the offsets in shared memory
  int* cnt = sh + E + warp * E;
  constexpr int kSteps = kSegChunk / 32;
  for (int c = blockIdx.x * 8 + warp; c < a.nchunks; c += gridDim.x * 8) {
    const long long c0 = (long long)c * kSegChunk;
    // the chunk's expert ids and router weights are loaded up front (all
    // in flight at once), so the ordered walk below waits on no load
    int ids_r[kSteps];
    float prob_r[kSteps];
#pragma unroll
    for (int s = 0; s < kSteps; ++s) {
      const long long f = c0 + s * 32 + lane;
      ids_r[s] = f < a.n ? a.ids[f] : -1;
      prob_r[s] = f < a.n ? a.prob[f] : 0.0f;
    }
    for (int e = lane; e < E; e += 32) cnt[e] = __ldcg(a.base + (long long)c * E + e) + sh[e];
    __syncwarp();
#pragma unroll
    for (int si = 0; si < kSteps; ++si) {
      const int s = si * 32;
      const long long f = c0 + s + lane;
      int e = -1;
      if (f < a.n) {
        e = ids_r[si];
        if (e < 0 || e >= E) e = -1;
      }
      const unsigned grp = __match_any_sync(0xFFFFFFFFu, e);
      const unsigned lt = (1u << lane) - 1u;
      const int rank = __popc(grp & lt);
      int row = -1;
      if (e >= 0) row = cnt[e] + rank;
      __syncwarp();
      if (e >= 0 && (grp >> lane) == 1u) cnt[e] += __popc(grp);
      __syncwarp();
      if (f < a.n) {
        a.inv_perm[f] = row;
        if (row >= 0) {
          a.perm[row] = (int)f;
          a.row_prob[row] = prob_r[si];
        }
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- gather
// dst[row] = src[perm[row] / k] (bf16 rows), zeros for padding rows
__global__ void __launch_bounds__(256) gather_bf16_kernel(const uint4* src, long long K8,
                                                         int k, const int* perm,
                                                         const int* seg_end, long long cap,
                                                         uint4* dst, float* amax_zero) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  long long rend = *seg_end;
  if (rend > cap) rend = cap;
  if (row >= rend) return;
  if (amax_zero && lane == 0) amax_zero[row] = 0.0f;
  const int f = perm[row];
  uint4* d = dst + row * K8;
  if (f < 0) {
    for (long long i = lane; i < K8; i += 32) d[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* s = src + (long long)(f / k) * K8;
  for (long long i = lane; i < K8; i += 32) d[i] = __ldg(s + i);
}

// NVFP4 rows: codes (K/2 bytes), 128x4-tiled scales (K/16 columns) and the
// token scale move together.  One CTA per 128 destination rows (one row of
// scale tiles): each warp copies 16 rows of codes; each 512-byte scale tile of
// the destination is assembled by 128 threads, one 4-byte word (a row's four
// scales of the tile) each, and written as one contiguous 512-byte run.
__global__ void __launch_bounds__(256) gather_nvfp4_kernel(const uint4* __restrict__ src_q,
                                                          const uint8_t* __restrict__ src_s,
                                                          const float* __restrict__ src_ts, long long K,
                                                          int k, const int* __restrict__ perm,
                                                          const int* __restrict__ seg_end, long long cap,
                                                          uint4* __restrict__ dst_q,
                                                          uint8_t* __restrict__ dst_s,
                                                          float* __restrict__ dst_ts,
                                                          float* __restrict__ amax_zero) {
  __shared__ long long tok[128];                  // source token of each row, -1 for padding
  const long long rbase = (long long)blockIdx.x * 128;
  long long rend = *seg_end;
  if (rend > cap) rend = cap;
  if (rbase >= rend) return;
  const int nrows = (int)min(128LL, rend - rbase);
  if (threadIdx.x < 128) {
    const int i = threadIdx.x;
    long long t = -1;
    if (i < nrows) {
      const int f = perm[rbase + i];
      if (f >= 0) t = f / k;
      if (amax_zero) amax_zero[rbase + i] = 0.0f;
      dst_ts[rbase + i] = t >= 0 ? src_ts[t] : 0.0f;
    }
    tok[i] = t;
  }
  __syncthreads();
  const long long q16 = K / 32;                  // uint4 chunks of packed codes per row
  const long long cpad = K / 16;                 // scale columns (K % 64 == 0: no padding)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < nrows; i += 8) {
    uint4* d = dst_q + (rbase + i) * q16;
    const long long t = tok[i];
    if (t < 0) {
#pragma unroll 4
      for (long long c = lane; c < q16; c += 32) d[c] = make_uint4(0, 0, 0, 0);
    } else {
      const uint4* sq = src_q + t * q16;
#pragma unroll 4
      for (long long c = lane; c < q16; c += 32) d[c] = __ldg(sq + c);
    }
  }
  // scale tiles: word w of a tile holds row (w % 4) * 32 + w / 4
  const long long ntiles = cpad / 4;
  const long long rt = rbase >> 7;
  const int w = threadIdx.x & 127;
  const int r = (w & 3) * 32 + (w >> 2);
  const long long t = tok[r];
#pragma unroll 4
  for (long long g = threadIdx.x >> 7; g < ntiles; g += 2) {
    if (r >= nrows) continue;
    uint32_t v = 0;
    if (t >= 0) v = *reinterpret_cast<const uint32_t*>(src_s + sf_offset(t, g * 4, cpad));
    reinterpret_cast<uint32_t*>(dst_s + (rt * ntiles + g) * 512)[w] = v;
  }
}

// ---------------------------------------------------------------- combine
// out[t] = sum_j y[inv[t*k + j]] in fp32, slot order, one rounding to bf16
__global__ void __launch_bounds__(128) combine_kernel(const uint4* y, const int* inv, long long T,
                                                     int k, long long H8, uint4* out) {
  const long long c = (long long)blockIdx.y * blockDim.x + threadIdx.x;
  const long long t = blockIdx.x;
  if (c >= H8) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int j = 0; j < k; ++j) {
    const int r = inv[t * k + j];
    if (r < 0) continue;
    const uint4 v = __ldg(y + (long long)r * H8 + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = __fadd_rn(acc[2 * i], bf16lo(w[i]));
      acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], bf16hi(w[i]));
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    o[i] = *reinterpret_cast<uint32_t*>(&b);
  }
  out[t * H8 + c] = make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------- launchers
size_t segments_ws_bytes(long long T, int k, long long E) {
  const long long n = T * k;
  const long long nchunks = (n + kSegChunk - 1) / kSegChunk;
  // histograms, chunk bases, expert totals, the fused kernel's barrier words
  return (size_t)(2 * nchunks * E + E + 2) * sizeof(int);
}

// the cooperative form; cudaErrorNotSupported when the device cannot run it
static cudaError_t launch_segments_fused(const SegFused& a, cudaStream_t s) {
  static int ctas[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorNotSupported;
  const size_t smem = (size_t)9 * 1024 * sizeof(int);     // offsets + 8 warps' counters, E <= 1024
  if (ctas[dev] == 0) {
    int sms = 0, per = 0, coop = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    err = cudaFuncSetAttribute(seg_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, seg_fused_kernel, 256, smem);
    if (err != cudaSuccess) return err;
    ctas[dev] = (coop && sms > 0 && per > 0) ? sms * (per < 2 ? per : 2) : -1;
  }
  if (ctas[dev] < 0) return cudaErrorNotSupported;
  // enough CTAs for the widest phase, no more than can be resident
  long long want = a.nchunks > a.E ? a.nchunks : a.E;
  if (want < 1) want = 1;
  const unsigned grid = (unsigned)(want < ctas[dev] ? want : ctas[dev]);
  SegFused arg = a;
  void* args[] = {&arg};
  return cudaLaunchCooperativeKernel((const void*)seg_fused_kernel, dim3(grid), dim3(256), args,
                                     smem, s);
}

cudaError_t launch_build_segments(const int* ids, const float* prob, long long T, int k,
                                  long long E, int pad, int* seg_offsets, int* perm,
                                  int* inv_perm, float* row_prob, long long cap, void* ws,
                                  int* st, cudaStream_t s) {
  const long long n = T * k;
  const int nchunks = (int)((n + kSegChunk - 1) / kSegChunk);
  int* hist = static_cast<int*>(ws);
  int* base = hist + (long long)nchunks * E;
  cudaError_t err;
  if (E <= 1024) {
    SegFused a{};
    a.ids = ids; a.prob = prob; a.n = n; a.E = (int)E; a.pad = pad; a.nchunks = nchunks;
    a.hist = hist; a.base = base; a.totals = base + (long long)nchunks * E;
    a.seg_offsets = seg_offsets; a.perm = perm; a.inv_perm = inv_perm; a.row_prob = row_prob;
    a.cap = cap;
    a.bar = reinterpret_cast<unsigned*>(a.totals + E);
    a.st = st;
    if ((err = cudaMemsetAsync(a.bar, 0, 2 * sizeof(unsigned), s)) != cudaSuccess) return err;
    err = launch_segments_fused(a, s);
    if (err != cudaErrorNotSupported) return err;
  }
  if ((err = cudaMemsetAsync(perm, 0xFF, (size_t)cap * sizeof(int), s)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(row_prob, 0, (size_t)cap * sizeof(float), s)) != cudaSuccess) return err;
  seg_hist_kernel<<<nchunks, 128, (size_t)E * sizeof(int), s>>>(ids, n, (int)E, hist, st);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  int* totals = base + (long long)nchunks * E;
  seg_colscan_kernel<<<(unsigned)E, 256, 0, s>>>(hist, nchunks, (int)E, base, totals);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  seg_offsets_kernel<<<1, 1024, 0, s>>>(totals, (int)E, pad, seg_offsets);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  seg_scatter_kernel<<<nchunks, 32, (size_t)E * sizeof(int), s>>>(ids, prob, n, (int)E, base,
                                                                  seg_offsets, perm, inv_perm,
                                                                  row_prob);
  return cudaGetLastError();
}

cudaError_t launch_gather(int what, const void* src, const uint8_t* src_s, const float* src_ts,
                          long long K, int k, const int* perm, const int* seg_end,
                          long long cap, void* dst, uint8_t* dst_s, float* dst_ts,
                          float* amax_zero, cudaStream_t s) {
  const unsigned grid = (unsigned)((cap + 7) / 8);
  if (what == MPM_GATHER_BF16) {
    gather_bf16_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(src), K / 8, k, perm,
                                            seg_end, cap, static_cast<uint4*>(dst), amax_zero);
  } else {
    gather_nvfp4_kernel<<<(unsigned)((cap + 127) / 128), 256, 0, s>>>(
        static_cast<const uint4*>(src), src_s, src_ts, K,
                                             k, perm, seg_end, cap, static_cast<uint4*>(dst),
                                             dst_s, dst_ts, amax_zero);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y, const int* inv, long long T, int k, long long H,
                           void* out, cudaStream_t s) {
  const long long H8 = H / 8;
  const dim3 grid((unsigned)T, (unsigned)((H8 + 127) / 128));
  combine_kernel<<<grid, 128, 0, s>>>(static_cast<const uint4*>(y), inv, T, k, H8,
                                      static_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace mpm
