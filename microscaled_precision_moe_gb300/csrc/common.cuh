// Shared device helpers for libmpm (sm_103a): status word, format conversions,
// and thin inline-PTX wrappers for mbarrier, TMA, bulk copies and tcgen05.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "../../include/mpm.h"

#define MPM_DEV __device__ __forceinline__

namespace mpm {

// ---------------------------------------------------------------- status word
// One int per device (set by kernels on device-side errors, read and reset by
// mpm_get_device_status); kernels receive its address.  The first error wins.
MPM_DEV void set_status(int* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

// Bounded waits: about 2^32 cycles (~2 s at 2 GHz) before giving up.
constexpr long long kWaitLimitCycles = 1ll << 32;

// ---------------------------------------------------------------- bf16 / fp32
MPM_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
MPM_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max of |bf16| over the two halves of a word, as a 16-bit pattern pair:
// non-negative bf16 patterns order like unsigned integers.
MPM_DEV uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
  return __vmaxu2(acc, w & 0x7FFF7FFFu);
}

// two fp32 -> packed E2M1 byte (lo in the low nibble), RN, satfinite
MPM_DEV uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .b8 b;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b, %2, %1;\n\t"
      "cvt.u32.u8 %0, b;\n\t}"
      : "=r"(out) : "f"(lo), "f"(hi));
  return out;
}

// two fp32 -> packed E4M3 pair (lo in the low byte), RN, satfinite
MPM_DEV uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t out;
  asm volatile("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(out) : "f"(lo), "f"(hi));
  return out;
}

// E4M3 byte -> fp32 (exact), through the exact e4m3 -> f16 conversion
MPM_DEV float e4m3_to_f32(uint32_t code) {
  uint32_t h2;
  uint16_t in = (uint16_t)(code & 0xFF);
  asm volatile("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  __half lo = __ushort_as_half((unsigned short)(h2 & 0xFFFF));
  return __half2float(lo);
}

MPM_DEV uint32_t float_bits(float f) { return __float_as_uint(f); }

// ---------------------------------------------------------------- SwiGLU
// The activation of every FC1 epilogue and its derivative for the SwiGLU
// backward, defined once so that D (and dH) do not depend on which GEMM
// kernel produced them (the three kernels give byte-identical D).
//   silu(g) = g / (1 + e^-g)
//   D       = silu(g) * u * p
// e^-g is taken by change of base, 2^(-g log2 e): one IEEE product, then
// the hardware base-2 exponential (ex2.approx); the division is the
// hardware reciprocal (rcp.approx) of 1 + e^-g times g.  Both are a few fp32
// ulps from the correctly rounded result; every other step is one IEEE
// binary32 operation with no contraction into FMAs.  Both use their
// flush-to-zero forms.  For the exponential that changes no result: its
// argument is subnormal only for |g| below about 2^-126 (2^t is 1 either
// way), its result only for g > 87.3 (where 1 + e^-g is 1 either way).  The
// reciprocal's argument is at least 1; for g < -87.3 (1 + e^-g above 2^126)
// its result flushes to 0, so silu(g) comes out as a zero with the sign of g
// where the exact value, |g| e^g, is below 2^-119 (and reaches 0 in fp32
// only near g = -108): in a row that also holds ordinary gate values, such
// an element of D lies more than 30 orders of magnitude below the row's
// amax, and the FP4 re-quantisation codes it 0 either way.  The fast
// division this replaced returns 0 in the same range.
// Checked against CUDA's fast intrinsics (__expf, __fdividef), which this
// replaced: D of the 671B-shaped headline layer byte for byte the same, and
// that FC1 2.77 -> 2.70 ms (fewer epilogue instructions; see the last
// sentence).  The result is rounded to bf16 (8 significant
// bits) right after, so these ulps move an element of D only when its value
// lies within a few fp32 ulps of a bf16 rounding midpoint, the same order as
// the fp32 accumulation error of the GEMM itself; the FC1 parity tests
// bound D against the oracle's exact SwiGLU.  The correctly rounded forms
// (expf and IEEE division) cost 15 % of the headline FC1 on GB300 (3.21
// against 2.80 ms): every instruction the epilogue warps issue shows up in
// the MMA pace.
MPM_DEV float exp2_ftz(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}
MPM_DEV float rcp_ftz(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
// 1 / (1 + e^-g)
MPM_DEV float swiglu_sigmoid(float g) {
  return rcp_ftz(__fadd_rn(1.0f, exp2_ftz(__fmul_rn(g, -1.44269504088896341f))));
}
MPM_DEV float swiglu_silu(float g) { return __fmul_rn(g, swiglu_sigmoid(g)); }
MPM_DEV float swiglu_fwd(float g, float u, float prob) {
  return __fmul_rn(__fmul_rn(swiglu_silu(g), u), prob);
}
// Two elements of D at once: the same operations as swiglu_fwd on each
// lane, with the multiplications done as packed f32x2 IEEE products (per
// lane bit-identical to the scalar products): (acc_g, acc_u) pairs scaled by
// alpha, then silu(g) * u * p.
MPM_DEV uint64_t f32x2(float lo, float hi) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
MPM_DEV void f32x2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
MPM_DEV uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
MPM_DEV void swiglu_fwd2(uint32_t acc_g0, uint32_t acc_g1, uint32_t acc_u0, uint32_t acc_u1,
                         uint64_t alpha2, uint64_t prob2, float& d0, float& d1) {
  float g0, g1;
  f32x2_split(mul_f32x2(f32x2(__uint_as_float(acc_g0), __uint_as_float(acc_g1)), alpha2), g0, g1);
  const uint64_t u = mul_f32x2(f32x2(__uint_as_float(acc_u0), __uint_as_float(acc_u1)), alpha2);
  const uint64_t su = mul_f32x2(f32x2(swiglu_silu(g0), swiglu_silu(g1)), u);
  f32x2_split(mul_f32x2(su, prob2), d0, d1);
}
// dD -> (dg, du) for D = silu(g) * u * p with p constant:
//   dg = (dD p) u s (1 + g (1 - s)),  du = (dD p) g s,  s = 1 / (1 + e^-g)
// s is the forward's sigmoid, so for g < -87.3 it is 0 and dg, du are zeros
// where their exact values lie below 2^-119 |dD p u| (1 + |g|) and
// 2^-119 |dD p g|, as D is in the forward.
MPM_DEV void swiglu_bwd(float g, float u, float dd, float prob, float& dg, float& du) {
  const float s = swiglu_sigmoid(g);
  const float dp = __fmul_rn(dd, prob);
  const float dsilu = __fmul_rn(s, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, s))));
  dg = __fmul_rn(__fmul_rn(dp, u), dsilu);
  du = __fmul_rn(dp, __fmul_rn(g, s));
}

// ---------------------------------------------------------------- 128x4 scale tiles
// byte offset of scale entry (r, c) in a tiled [rows, cols] scale matrix whose
// padded column count is cols_pad (multiple of 4)
MPM_DEV size_t sf_offset(long long r, long long c, long long cols_pad) {
  long long rt = r >> 7, rr = r & 127, ct = c >> 2, cc = c & 3;
  return (size_t)((rt * (cols_pad >> 2) + ct) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + cc);
}

// ---------------------------------------------------------------- shared memory
MPM_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
MPM_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
MPM_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MPM_DEV void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
MPM_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
MPM_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}
MPM_DEV uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok;
}
// Bounded wait; returns false (and records MPM_ERR_DEVICE_TIMEOUT) on timeout.
MPM_DEV bool mbar_wait(uint32_t bar, uint32_t parity, int* st) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > kWaitLimitCycles) {
      set_status(st, MPM_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA / bulk copies
MPM_DEV void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar) : "memory");
}
MPM_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel in the stream finishes;
// pdl_wait returns once that kernel has completed and its writes are
// visible (at once when there is none), and pdl_launch_dependents lets the
// next such kernel start early.
MPM_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MPM_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
MPM_DEV void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}

// ---------------------------------------------------------------- clusters
MPM_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
MPM_DEV uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
MPM_DEV uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the same variable in CTA `rank` of the cluster
MPM_DEV uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
MPM_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// Arrive on an mbarrier of any CTA of the cluster (shared::cluster address).
// The release is CTA-scoped: the arrivals this is used for only count
// completed work (TMEM reads already finished by tcgen05.wait::ld) and carry
// no data to the waiter; a cluster-scoped release costs ~1.8k cycles here.
MPM_DEV void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];"
               :: "r"(cluster_addr) : "memory");
}
MPM_DEV uint32_t mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok;
}
// bounded wait with cluster-scope acquire (for barriers other CTAs arrive on)
MPM_DEV bool mbar_wait_cluster(uint32_t bar, uint32_t parity, int* st) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (clock64() - t0 > kWaitLimitCycles) {
      set_status(st, MPM_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}
// TMA load whose completion is signalled on an mbarrier that may live in the
// peer CTA of the pair (bar is a shared::cluster address)
MPM_DEV void tma_load_2d_pair(uint32_t dst, const void* tmap, int x, int y, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar_cluster) : "memory");
}
// TMA tensor store of a shared-memory box to global memory (bulk group)
MPM_DEV void tma_store_2d(const void* tmap, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
               :: "l"(tmap), "r"(x), "r"(y), "r"(src) : "memory");
}
MPM_DEV void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until this thread's bulk groups no longer read shared memory
MPM_DEV void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... all but the most recent group
MPM_DEV void bulk_wait_group_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
MPM_DEV void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
MPM_DEV void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
// named barrier among a subset of warps
MPM_DEV void named_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- tcgen05 (pair)
MPM_DEV void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
MPM_DEV void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MPM_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}
// arrive on the mbarrier at this offset in every CTA of cta_mask once all prior
// tcgen05 async ops of this thread finish
MPM_DEV void tc_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" :: "r"(bar), "h"(cta_mask) : "memory");
}
MPM_DEV void tc_cp_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;"
               :: "r"(taddr), "l"(sdesc) : "memory");
}
MPM_DEV void mma_nvf4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate),
         "r"(sfa_tmem), "r"(sfb_tmem) : "memory");
}
MPM_DEV void mma_mxf8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate),
         "r"(sfa_tmem), "r"(sfb_tmem) : "memory");
}

// bf16 x bf16 -> fp32 (kind::f16, no scale factors), M = 256 over the pair
MPM_DEV void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

// ---------------------------------------------------------------- tcgen05
MPM_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
MPM_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MPM_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}
MPM_DEV void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
MPM_DEV void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// arrive on an mbarrier once all prior tcgen05 async ops of this thread finish
MPM_DEV void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}
// copy a 32-row x 16-byte block from shared memory to TMEM, replicated into
// the four 32-lane quarters (4 columns)
MPM_DEV void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;"
               :: "r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, E2M1 x E2M1 with E4M3 scales per 16
MPM_DEV void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate),
         "r"(sfa_tmem), "r"(sfb_tmem) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 with E8M0 scales per 32
MPM_DEV void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate),
         "r"(sfa_tmem), "r"(sfb_tmem) : "memory");
}

// 32 lanes x 32 columns of 32-bit accumulator -> 32 registers per thread
MPM_DEV void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
        "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
MPM_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// one thread's four 32-bit values into four consecutive TMEM columns of its
// lane (the warp's lane quarter)
MPM_DEV void tmem_st_32x32b_x4(uint32_t taddr, const uint4& v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};"
               :: "r"(taddr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
// 32 registers per thread -> 32 lanes x 32 columns of TMEM
MPM_DEV void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
      " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
         "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
         "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
         "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
         "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
MPM_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05 format): K-major operand stored as
// rows of 128 bytes with the 128-byte swizzle, 8-row groups 1024 bytes apart.
MPM_DEV uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);          // start address
  d |= (uint64_t)1 << 16;                            // leading byte offset (unused)
  d |= (uint64_t)(1024 >> 4) << 32;                  // stride byte offset
  d |= (uint64_t)1 << 46;                            // descriptor version
  d |= (uint64_t)2 << 61;                            // 128-byte swizzle
  return d;
}
// Descriptor of an MN-major tile with the 128-byte swizzle: for each k one
// 128-byte row of the contiguous M (or N) dimension, 8-row groups 1024 bytes
// apart along K (stride byte offset), blocks of 128 bytes of M/N
// `mn_block_bytes` apart (leading byte offset).  This is the layout a TMA
// load with a 128-byte-wide box and the 128-byte swizzle writes.
MPM_DEV uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t mn_block_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((mn_block_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Descriptor of a 32-row x 16-byte block without swizzle (core matrices of
// 8 rows x 16 bytes, 128 bytes apart): the source of a scale-factor copy.
MPM_DEV uint64_t sdesc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)0 << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor of a block-scaled MMA with K-major A and B.
//   fmt: operand format code (E2M1 = 1 for mxf4nvf4, E4M3 = 0 for mxf8f6f4)
//   ue8m0: scale type (0 = UE4M3, 1 = UE8M0); sf_id: byte of the scale word
//   m: 128 (one CTA) or 256 (a CTA pair)
__host__ __device__ constexpr uint32_t idesc_block_scaled(uint32_t fmt, uint32_t n,
                                                          uint32_t ue8m0, uint32_t sf_id,
                                                          uint32_t m = 128) {
  return (sf_id << 4)            // B scale-factor id
       | (fmt << 7)              // A format
       | (fmt << 10)             // B format
       | ((n >> 3) << 17)        // N / 8
       | (ue8m0 << 23)           // scale type
       | ((m >> 4) << 24)        // M / 16
       | (sf_id << 29);          // A scale-factor id
}

// instruction descriptor of kind::f16 with bf16 A and B, fp32 D; a_mn / b_mn
// mark an operand stored MN-major (M or N contiguous) instead of K-major
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n, uint32_t m, uint32_t a_mn = 0,
                                                  uint32_t b_mn = 0) {
  return (1u << 4)               // D format fp32
       | (1u << 7)               // A format bf16
       | (1u << 10)              // B format bf16
       | (a_mn << 15)            // A major-ness
       | (b_mn << 16)            // B major-ness
       | ((n >> 3) << 17)        // N / 8
       | ((m >> 4) << 24);       // M / 16
}

}  // namespace mpm
