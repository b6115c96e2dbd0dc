/*
 * A plain C client of libmpm.  It shows that include/mpm.h compiles as C99
 * and that the library is usable without Python or PyTorch, through host-only
 * calls: the size queries, the status strings and the argument checks that
 * reject a call before anything is launched.  No call here reaches a GPU; the
 * device addresses are placeholders that the rejected calls never touch.
 * Exit status 0 when every check holds; otherwise the failing line is
 * printed.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "mpm.h"

#define CHECK(cond)                                                   \
  do {                                                                \
    if (!(cond)) {                                                    \
      fprintf(stderr, "abi_client: check failed at line %d: %s\n",    \
              __LINE__, #cond);                                       \
      return 1;                                                       \
    }                                                                 \
  } while (0)

int main(void) {
  void* dev = (void*)(uintptr_t)0x10000;   /* 16-byte aligned placeholder */
  void* odd = (void*)(uintptr_t)0x10008;   /* 8-byte aligned only */
  mpm_grouped_gemm_desc d;

  /* queries */
  CHECK(mpm_version() == 101);
  CHECK(mpm_scale_bytes(8288, 64) == (size_t)8320 * 64);
  CHECK(mpm_scale_bytes(2048, 259) == (size_t)2048 * 260);
  CHECK(mpm_scale_bytes(0, 64) == 0);
  CHECK(mpm_moe_row_capacity(32768, 8, 256, 256) == 262144 + 256 * 256);
  CHECK(mpm_moe_row_capacity(32768, 8, 256, 96) == 0);
  CHECK(mpm_nvfp4_weight_workspace_bytes(4) >= 4 * sizeof(float));
  CHECK(strcmp(mpm_status_string(MPM_OK), "MPM_OK") == 0);
  CHECK(strcmp(mpm_status_string(MPM_ERR_DEVICE_TIMEOUT), "MPM_ERR_DEVICE_TIMEOUT") == 0);
  CHECK(mpm_status_string(12345) != NULL);

  /* quantisers: a NULL input, an empty input, K not a multiple of the
     block, a misaligned input */
  CHECK(mpm_nvfp4_quantize_per_token(NULL, 4, 64, 64, NULL, dev, dev, dev, NULL, 0) ==
        MPM_ERR_NULL);
  CHECK(mpm_nvfp4_quantize_per_token(dev, 0, 64, 64, NULL, dev, dev, dev, NULL, 0) ==
        MPM_ERR_SHAPE);
  CHECK(mpm_nvfp4_quantize_per_token(dev, 4, 8256, 8256, NULL, dev, dev, dev, NULL, 0) ==
        MPM_ERR_SHAPE);
  CHECK(mpm_nvfp4_quantize_per_token(odd, 4, 64, 64, NULL, dev, dev, dev, NULL, 0) ==
        MPM_ERR_ALIGN);
  CHECK(mpm_mxfp8_quantize(dev, 4, 40, 40, MPM_ROWWISE, dev, dev, NULL, 0, NULL, NULL, 0) ==
        MPM_ERR_SHAPE);
  CHECK(mpm_mxfp8_quantize(dev, 4, 64, 64, 0u, dev, dev, dev, 16, dev, NULL, 0) ==
        MPM_ERR_SHAPE);
  /* the routed-row forms: no routing, a bad top-k, a misaligned input */
  CHECK(mpm_mxfp8_quantize_gather(dev, 4, 64, 64, NULL, 2, dev, 2, 256, MPM_ROWWISE, dev, dev,
                                  NULL, 0, NULL, 0) == MPM_ERR_NULL);
  CHECK(mpm_mxfp8_quantize_gather(dev, 4, 64, 64, dev, 0, dev, 2, 256, MPM_ROWWISE, dev, dev,
                                  NULL, 0, NULL, 0) == MPM_ERR_SHAPE);
  CHECK(mpm_mxfp8_quantize_gather(odd, 4, 64, 64, dev, 2, dev, 2, 256, MPM_ROWWISE, dev, dev,
                                  NULL, 0, NULL, 0) == MPM_ERR_ALIGN);
  CHECK(mpm_nvfp4_quantize_scatter_workspace_bytes(4, 64) == 4 * 4 + 4 * 4 + 16);
  CHECK(mpm_nvfp4_quantize_scatter(dev, 4, 64, 64, dev, 65, dev, dev, 2, 256, dev, dev, dev, NULL,
                                   dev, 48, 0) == MPM_ERR_SHAPE);

  /* segments, combine */
  CHECK(mpm_moe_build_segments(dev, dev, 0, 8, 16, 128, dev, dev, dev, dev, dev, 1u << 20, 0) ==
        MPM_ERR_SHAPE);
  CHECK(mpm_moe_combine(dev, dev, 4, 8, 12, dev, 0) == MPM_ERR_SHAPE);
  CHECK(mpm_moe_combine(odd, dev, 4, 8, 256, dev, 0) == MPM_ERR_ALIGN);

  /* grouped GEMM descriptor: no descriptor, an output width that is not a
     multiple of 256, an unknown kind */
  CHECK(mpm_moe_grouped_gemm(NULL, 0) == MPM_ERR_NULL);
  memset(&d, 0, sizeof d);
  d.kind = MPM_KIND_NVFP4;
  d.group = MPM_GROUP_M;
  d.epilogue = MPM_EPI_F32;
  d.tile_m = 128;
  d.E = 1;
  d.a_rows = 128;
  d.N = 200;
  d.K = 256;
  d.a_dev = (const uint8_t*)dev;
  d.b_dev = (const uint8_t*)dev;
  d.sfa_dev = (const uint8_t*)dev;
  d.sfb_dev = (const uint8_t*)dev;
  d.out_dev = dev;
  d.lda_bytes = d.ldb_bytes = 128;
  d.a_total_rows = d.b_total_rows = 128;
  d.sfa_cols = d.sfb_cols = 16;
  d.ldo = 256;
  CHECK(mpm_moe_grouped_gemm(&d, 0) == MPM_ERR_SHAPE);
  d.N = 256;
  d.kind = 7;
  CHECK(mpm_moe_grouped_gemm(&d, 0) == MPM_ERR_UNSUPPORTED);

  /* weight-gradient call: no descriptor; NVFP4 (wgrad is MXFP8 or BF16);
     no segment offsets; a bf16 epilogue (wgrad writes fp32).  The call sets
     the group itself, so a descriptor left at GROUP_M is taken as GROUP_K. */
  CHECK(mpm_moe_grouped_gemm_wgrad(NULL, 0) == MPM_ERR_NULL);
  d.kind = MPM_KIND_NVFP4;
  d.group = MPM_GROUP_M;
  d.N = 256;
  d.K = 0;
  d.seg_dev = (const int32_t*)dev;
  CHECK(mpm_moe_grouped_gemm_wgrad(&d, 0) == MPM_ERR_UNSUPPORTED);
  d.kind = MPM_KIND_MXFP8;
  d.seg_dev = NULL;
  CHECK(mpm_moe_grouped_gemm_wgrad(&d, 0) == MPM_ERR_NULL);
  d.seg_dev = (const int32_t*)dev;
  d.epilogue = MPM_EPI_BF16;
  CHECK(mpm_moe_grouped_gemm_wgrad(&d, 0) == MPM_ERR_UNSUPPORTED);
  d.epilogue = MPM_EPI_F32;
  d.a_rows = 200;                                   /* M_out % 128 != 0 */
  CHECK(mpm_moe_grouped_gemm_wgrad(&d, 0) == MPM_ERR_SHAPE);

  printf("abi_client: ok\n");
  return 0;
}
