// Shared device helpers for the sm_103a kernels: mbarriers, bulk async copies,
// bounded waits, small numeric conversions.  Inline PTX only where CUDA C++ has
// no equivalent.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

// Make mbarrier initialisation visible to the async (bulk-copy / tensor) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Both phases complete?  The two probes are issued back to back, so their
// shared-memory round trips overlap (one barrier latency instead of two).
__device__ __forceinline__ bool mbar_try_wait2(uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p, q;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 q, [%3], %4;\n and.pred p, p, q;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(a)), "r"(pa), "r"(smem_u32(b)), "r"(pb)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase ``parity`` of ``bar`` to complete, giving up after
// ``limit_ns``.  On give-up the status word gets MOE_STATUS_WAIT_TIMEOUT and
// the function returns false; callers then stop their pipeline.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && global_ns() - t0 > limit_ns) {
      atomicOr(status, kStatusWaitTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------- bulk async copy (TMA, non-tensor)

// Global -> shared copy of ``bytes`` (multiple of 16; both addresses 16-byte
// aligned), completion counted on ``bar`` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- programmatic dependent launch

// Block until the grids this one depends on (launched before it on the
// stream) have completed and their writes are visible.  No-op for a normal launch.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next grid on the stream, if launched as a programmatic dependent,
// to start being scheduled.
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- named barriers

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- flags between CTAs of one grid

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// After relaxed loads that observed other threads' release stores: makes
// their earlier writes visible to this thread's later reads (acquire pattern).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Value that CTA ``slot`` publishes for ``token``: distinct per slot, so no
// constant fill of the flag array matches, and a bijection of the token
// (odd multiplier), so flags left by another token never match.
__device__ __forceinline__ uint32_t published_value(uint32_t token, int slot) {
  return token * 0x9E3779B1u + (uint32_t)slot;
}

// One warp waits until every flags[q], q in [lo, hi), holds
// published_value(token, q) (acquire), giving up after ``limit_ns`` like
// mbar_wait.  Every lane returns the same value.
__device__ __forceinline__ bool wait_published_range(const uint32_t* flags, int lo, int hi, uint32_t token,
                                                     uint32_t* status, uint64_t limit_ns) {
  const int lane = threadIdx.x & 31;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0;; ++i) {
    // every flag of this lane loaded at once (relaxed, independent), one
    // acquire fence once all have been seen
    bool ok = true;
    for (int q = lo + lane; q < hi; q += 32) ok &= ld_relaxed_gpu(flags + q) == published_value(token, q);
    if (__all_sync(0xffffffffu, ok)) {
      fence_acq_rel_gpu();
      return true;
    }
    const bool late = (i & 15u) == 15u && global_ns() - t0 > limit_ns;
    if (__any_sync(0xffffffffu, late)) {
      if (lane == 0) atomicOr(status, kStatusWaitTimeout);
      return false;
    }
    __nanosleep(64);
  }
}

// ---------------------------------------------------------------- checked build
//
// Compiled with -DMOE_CHECK (the checked library), the kernels pass every
// index they derive from the grouping (expert, pair, token, row, tile)
// through chk() and every E8M0 weight-scale word they read through
// chk_e8m0(): an index outside its buffer sets MOE_STATUS_BAD_INDEX and is
// replaced by 0, so the access stays in bounds; a scale byte 255 (NaN in
// E8M0) sets MOE_STATUS_NAN_SCALE.  Without the flag both compile to nothing.
#ifdef MOE_CHECK
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

__device__ __forceinline__ int chk(long long i, long long n, uint32_t* status) {
  if (kChecked && (i < 0 || i >= n)) {
    if (status) atomicOr(status, kStatusBadIndex);
    return 0;
  }
  return (int)i;
}

// ``nbytes`` (1..4) E8M0 bytes in the low bytes of ``w``.
__device__ __forceinline__ void chk_e8m0(uint32_t w, int nbytes, uint32_t* status) {
  if (kChecked) {
    bool nan = false;
    for (int b = 0; b < nbytes; ++b) nan |= ((w >> (8 * b)) & 0xFFu) == 0xFFu;
    if (nan && status) atomicOr(status, kStatusNanScale);
  }
}

// ---------------------------------------------------------------- expert ids

// Local expert id of top-k slot ``p``: ids[p], mapped through ``emap`` (G
// entries, global id -> local id or -1) when one is given; -1 when the slot
// has no expert of this GPU.
__device__ __forceinline__ int local_expert(const int32_t* ids, long long p, const int32_t* emap, int G, int E) {
  int e = ids[p];
  if (emap) e = (unsigned)e < (unsigned)G ? emap[e] : -1;
  return (unsigned)e < (unsigned)E ? e : -1;
}

// ---------------------------------------------------------------- numeric helpers

// E8M0 byte -> 2^(s-127) as float (s = 0 gives the subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_float(uint32_t s) {
  return __uint_as_float(s ? (s << 23) : 0x00400000u);
}

// 2^e as float for e in [-126, 127].
__device__ __forceinline__ float exp2_int(int e) { return __uint_as_float(uint32_t(e + 127) << 23); }

// Two packed E2M1 codes (one byte) -> two exact f16 values, low nibble in the low half.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                uint32_t& o3) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}

// Pack two floats into f16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// SiLU with the fast exponential and division (relative error a few fp32 ulp,
// far below the bf16 rounding that follows).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// D = A * B + C for one m16n8k16 tile, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// ---------------------------------------------------------------- activation quantisation
//
// The W4A4 and W4A8 schemes of vLLM PR #39136 (``w_mxfp4_a_mxfp4``,
// ``w_mxfp4_a_fp8``): each GEMM input is quantised where a kernel loads it.
// A lane holds 8 consecutive values of a row; the 4 lanes 4m .. 4m+3 hold one
// 32-value block (the MX block), so block maxima take two shuffles.

enum ActQuant : int { kActNone = 0, kActMxfp4 = 1, kActFp8 = 2 };
static_assert(kActNone == MOE_AQ_NONE && kActMxfp4 == MOE_AQ_MXFP4 && kActFp8 == MOE_AQ_FP8,
              "kernel and public activation-quantisation codes");

// OCP MX scale byte of a block with largest magnitude ``amax``:
// floor(log2 amax) - 2 + 127 (2 = E2M1's largest exponent), 0 for a block
// whose amax is below 2^-125 (zero and subnormal amax included).
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  const int eb = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  return eb > 2 ? (uint32_t)(eb - 2) : 0u;
}

// Eight floats -> eight E2M1 codes (value 2j in the low nibble of byte j),
// round to nearest even, saturating at +-6; the sign bit follows the input.
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Four floats -> four e4m3fn codes (value j in byte j), round to nearest
// even, saturating at +-448; the sign bit follows the input.
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float v0, float v1, float v2, float v3) {
  uint32_t r;
  asm("{\n .reg .b16 h0, h1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 h0, %2, %1;\n cvt.rn.satfinite.e4m3x2.f32 h1, %4, %3;\n"
      " mov.b32 %0, {h0, h1};\n}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
  return r;
}

// Four e4m3fn codes (byte j = value j) -> two f16x2 (values 0,1 and 2,3), exact.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t c, uint32_t& o0, uint32_t& o1) {
  asm("{\n .reg .b16 h0, h1;\n mov.b32 {h0, h1}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, h0;\n cvt.rn.f16x2.e4m3x2 %1, h1;\n}"
      : "=r"(o0), "=r"(o1)
      : "r"(c));
}

// The low / high f16 half of a word as float, exact.
__device__ __forceinline__ float f16_lo(uint32_t v) {
  float f;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.f32.f16 %0, l;\n}" : "=f"(f) : "r"(v));
  return f;
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
  float f;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.f32.f16 %0, h;\n}" : "=f"(f) : "r"(v));
  return f;
}

// MXFP4 quantisation of one lane's 8 values of a block (all 32 lanes call it
// together): codes, the block's scale byte, and v replaced by the dequantised
// values code * 2^(scale - 127) (exact in float).
__device__ __forceinline__ void mx_quant8(float (&v)[8], uint32_t& codes, uint32_t& sbyte) {
  float m = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(v[q]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  sbyte = mx_scale_byte(m);
  const float rcp = __uint_as_float((254u - sbyte) << 23);  // 2^(127 - scale), scale <= 252
  float r[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) r[q] = v[q] * rcp;  // exact unless far below 0.25 (rounds to 0 either way)
  codes = f32x8_to_e2m1x8(r);
  uint32_t h[4];
  e2m1x8_to_f16x8(codes, h[0], h[1], h[2], h[3]);
  const float X = e8m0_to_float(sbyte);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[2 * q] = f16_lo(h[q]) * X;
    v[2 * q + 1] = f16_hi(h[q]) * X;
  }
}

// FP8 quantisation with a static scale: codes of r = fl32(v / s) (correctly
// rounded division), and v replaced by the e4m3 values (NOT times s: the
// callers apply s to their float32 results).
//
// Without a division per value: y = v * fl32(1/s) lies within 1.5 float32
// ulps of fl32(v / s) (two roundings of 2^-24 each against the one of the
// division), so y * (1 -+ 2^-21), 3.5 ulps either side even after their own
// rounding, bracket fl32(v / s).  Rounding is monotone: where both ends give
// the same e4m3 code, so does fl32(v / s).  Where they differ (a quotient
// within a few ulps of a rounding midpoint, exact ties included) the correctly
// rounded division decides.  The bound needs 1/s and y to be normal floats:
// scales outside [2^-126, 2^126] always divide; quotients too small for the
// bound round to zero at both ends and in fact.
// The e4m3 codes of fl32(v / s) by correctly rounded division: the rare
// fallback of fp8_quant8, kept out of line so that its code does not weigh on
// the kernels that inline the quantiser (values by value, codes returned in
// registers).
struct CodePair {
  uint32_t c0, c1;
};
static __device__ __noinline__ CodePair fp8_codes_by_division(float v0, float v1, float v2, float v3, float v4, float v5,
                                                             float v6, float v7, float s) {
  return CodePair{f32x4_to_e4m3x4(__fdiv_rn(v0, s), __fdiv_rn(v1, s), __fdiv_rn(v2, s), __fdiv_rn(v3, s)),
                  f32x4_to_e4m3x4(__fdiv_rn(v4, s), __fdiv_rn(v5, s), __fdiv_rn(v6, s), __fdiv_rn(v7, s))};
}

__device__ __forceinline__ void fp8_quant8(float (&v)[8], float s, uint32_t& c0, uint32_t& c1) {
  bool exact = !(s >= 0x1p-126f && s <= 0x1p126f);
  if (!exact) {
    const float rs = __frcp_rn(s);
    float lo[8], hi[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float y = v[q] * rs;
      lo[q] = y * (1.f - 0x1p-21f);
      hi[q] = y * (1.f + 0x1p-21f);
    }
    c0 = f32x4_to_e4m3x4(lo[0], lo[1], lo[2], lo[3]);
    c1 = f32x4_to_e4m3x4(lo[4], lo[5], lo[6], lo[7]);
    // (dividing only the open values, one branch per value, measured slower
    // than dividing the whole chunk)
    exact = c0 != f32x4_to_e4m3x4(hi[0], hi[1], hi[2], hi[3]) || c1 != f32x4_to_e4m3x4(hi[4], hi[5], hi[6], hi[7]);
  }
  if (exact) {
    const CodePair c = fp8_codes_by_division(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], s);
    c0 = c.c0;
    c1 = c.c1;
  }
  uint32_t h[4];
  e4m3x4_to_f16x4(c0, h[0], h[1]);
  e4m3x4_to_f16x4(c1, h[2], h[3]);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[2 * q] = f16_lo(h[q]);
    v[2 * q + 1] = f16_hi(h[q]);
  }
}

// In-place quantise-dequantise of one lane's 8 values under ``aq``; for FP8
// the values left are the e4m3 values (the scale is the caller's).  Every
// lane of the warp must call it (block maxima use shuffles).
__device__ __forceinline__ void act_quant8(int aq, float s, float (&v)[8]) {
  uint32_t a, b;
  if (aq == kActMxfp4) mx_quant8(v, a, b);
  else if (aq == kActFp8) fp8_quant8(v, s, a, b);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

}  // namespace moe
