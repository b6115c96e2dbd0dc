// Grouped block-scaled GEMM: kernel arguments and launcher.
#pragma once
#include <cuda.h>
#include "common.cuh"

namespace mpm {

struct GemmArgs {
  int group;                  // MPM_GROUP_M / MPM_GROUP_K
  int E;
  long long a_rows;           // GROUP_M: rows of A (capacity)
  long long N;                // output columns per expert
  long long K;                // reduction length (GROUP_M)
  long long M_out;            // GROUP_K: output rows per expert
  const int* seg;             // [E+1] device offsets (nullable for dense GROUP_M)
  long long b_rows_per_e;
  long long b_k_per_e;        // elements
  const uint8_t* sfa; long long sfa_cols_pad;
  const uint8_t* sfb; long long sfb_cols_pad;
  const float* alpha_a;
  const float* alpha_b;
  const float* row_prob;
  void* out; long long ldo;
  void* out2; long long ldo2;
  const void* aux; long long ld_aux;
  float* amax;
  const int* row_perm;        // nullable: rows with a negative entry are padding (small-M: not stored)
  int* status;
};

cudaError_t launch_grouped_gemm(int kind, int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                                const GemmArgs& a, dim3 grid, cudaStream_t s);
// maj: bit 0 = A MN-major, bit 1 = B MN-major (bf16 only)
// tout: the TMA-store map of the epilogue's output (bf16 / fp32 out, D, or
// dH [rows, 2N]); taux: C [rows, 2N] read by the SwiGLU-backward epilogue
cudaError_t launch_grouped_gemm_pair(int kind, int epi, int maj, const CUtensorMap& ta,
                                     const CUtensorMap& tb, const CUtensorMap& tsfa,
                                     const CUtensorMap& tsfb, const CUtensorMap& tout,
                                     const CUtensorMap& taux, const GemmArgs& a, int n_tiles,
                                     long long n_tasks, cudaStream_t s);
// small-M kernel (one CTA per 128 weight rows x 128 routed rows): n_wt
// weight tiles per chunk of 128 rows, tasks = chunks x n_wt
cudaError_t launch_grouped_gemm_small(int kind, int epi, const CUtensorMap& ta,
                                      const CUtensorMap& tb, const GemmArgs& a, int n_wt,
                                      long long n_tasks, cudaStream_t s);
// FC2 of the single-pass NVFP4 FFN (NVFP4 A quantised per 256-column tile
// against a running row amax, outer scales in a.aux [rows, a.ld_aux]):
// CTA pairs, 256 x 128 tiles, bf16 out = alpha_b[e] * sum_i gs_i * dO_i.
// tb: B map with 64-row boxes; tout: bf16 [rows, N] store map.
cudaError_t launch_fc2_online(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsfa,
                              const CUtensorMap& tsfb, const CUtensorMap& tout, const GemmArgs& a,
                              int n_tiles, long long n_tasks, cudaStream_t s);
// split-K form of the small-M kernel for one dense group of at most 128 rows:
// clusters of ks CTAs (ks divides 128, <= 8) per 128-row weight tile, fixed
// order reduction over the clusters' partials; F32 / BF16 epilogues
cudaError_t launch_gemm_splitk(int kind, int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                               const GemmArgs& a, int n_wt, int ks, cudaStream_t s);
}  // namespace mpm
