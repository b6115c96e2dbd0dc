"""CPU oracle for the microscaled-precision MoE hot path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only the tests, the smoke check and the CPU-baseline leg of the benchmark
may call it. It shares no code with the CUDA path; both sides only share the
seeded input generator (``microscaled_precision_moe_gb300.synth``).

Sources (titles of the pages and the section each rule comes from):

* "Towards Blackwell-native 8-bit and 4-bit RL" (LMSYS / Miles), section
  "Format background": MXFP8 = 32 consecutive E4M3 values sharing one E8M0
  power-of-two scale, rounded up so the block max never clips; NVFP4 = E2M1
  values, one E4M3 scale per 16 values rounded to nearest, plus an FP32
  outer scale.  Section "Per-token activation scaling": the FP32 activation
  scale is computed online per token; gate and up share one FP32 weight
  scale.  Section "Recipe 1 / Training": row-wise 1x32 and column-wise 32x1
  copies are quantised independently from full precision.
* "miniTE technical report", section 2.2: decode x_hat = q * s_b * s_g.
  Section 2.3: relative L2, SNR and MAE.  Section 5.2: contiguous grouped
  buffer with expert offsets.  Section 5.3: amax computed by the producer and
  reused by the quantiser.  Section 5.4: FC1 epilogue (alpha scaling,
  gate|up, act x prob, amax of D).  Section 5.6: gs = gamax / 2688.

Modules:
  formats  - E2M1 / E4M3 / E8M0 / bf16 encode and decode
  quant    - MXFP8 row/column, NVFP4 per-token and joint-weight quantisers,
             the 128x4 scale-tile layout, dequantisation
  moe      - expert segments and permutation, fp64 grouped GEMMs, SwiGLU,
             combine, the MXFP8 and BF16 backward, the single-pass FC2 with
             online amax compensation (report section 5.6)
  metrics  - relative L2, SNR, MAE, relative Frobenius error
"""
