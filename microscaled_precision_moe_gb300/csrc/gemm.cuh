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
  int* status;
};

cudaError_t launch_grouped_gemm(int kind, int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                                const GemmArgs& a, dim3 grid, cudaStream_t s);
// maj: bit 0 = A MN-major, bit 1 = B MN-major (bf16 only)
cudaError_t launch_grouped_gemm_pair(int kind, int epi, int maj, const CUtensorMap& ta,
                                     const CUtensorMap& tb, const CUtensorMap& tsfa,
                                     const CUtensorMap& tsfb, const CUtensorMap& tout,
                                     const GemmArgs& a, int n_tiles, long long n_tasks,
                                     cudaStream_t s);
// small-M kernel (one CTA per 128 weight rows x 128 routed rows): n_wt
// weight tiles per chunk of 128 rows, tasks = chunks x n_wt
cudaError_t launch_grouped_gemm_small(int kind, int epi, const CUtensorMap& ta,
                                      const CUtensorMap& tb, const GemmArgs& a, int n_wt,
                                      long long n_tasks, cudaStream_t s);
}  // namespace mpm
