// mla_device.cuh -- device helpers shared by the sm_103a kernels of libmla_cache.
//
// Everything here is a thin wrapper over one PTX instruction or a short,
// documented sequence: programmatic-dependent-launch control, 16-byte global
// loads/stores, the hardware pairwise converters (bf16x2, e4m3x2, e5m2x2,
// f16x2 <- fp8x2), a warp sum, and a correctly rounded fp32 division that
// reuses one reciprocal per row.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mla {

enum Fmt : int { kBF16 = 0, kE4M3 = 1, kE5M2 = 2 };

constexpr uint32_t kErrSlotOOB = 1u;
constexpr uint32_t kErrBlockOOB = 2u;
constexpr uint32_t kErrPosOOB = 4u;
constexpr uint32_t kErrMisaligned = 8u;

// ---- programmatic dependent launch ---------------------------------------
// Wait until every grid this one depends on has completed and its memory
// operations are visible (a no-op when launched without the PDL attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid on the stream to start launching.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- global memory ----------------------------------------------------------
// Inputs are read exactly once: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  return __ldcs(reinterpret_cast<const uint2*>(p));
}
// Small tables that many rows share (weights, cos/sin, block table).
__device__ __forceinline__ uint4 ld_shared_ro16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ void st8(void* p, uint2 v) { *reinterpret_cast<uint2*>(p) = v; }

// ---- bf16 ------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> bf16x2, round to nearest even; `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- fp8 ---------------------------------------------------------------------
// Two fp32 -> fp8x2 with round-to-nearest-even and saturation of finite
// overflow to +-max (the .satfinite converters); `lo` lands in the low byte.
template <int F>
__device__ __forceinline__ uint32_t pack_fp8x2(float lo, float hi) {
  uint16_t r;
  if constexpr (F == kE4M3) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

// fp8x2 (low 16 bits of `w`) -> two exact bf16 values in one 32-bit word.
// The hardware widening to f16x2 is exact for both fp8 formats, and every
// finite f16 obtained this way is a bf16 value, so truncating the fp32 is
// exact.  A NaN becomes the quiet NaN 0x7FC0 with the fp8 code's sign.
template <int F>
__device__ __forceinline__ uint32_t fp8x2_to_bf16x2(uint32_t w) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(w);
  if constexpr (F == kE4M3) {
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  } else {
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(in));
  }
  float f0, f1;
  asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b; }"
      : "=f"(f0), "=f"(f1) : "r"(h2));
  uint32_t b0 = __float_as_uint(f0) >> 16, b1 = __float_as_uint(f1) >> 16;
  // the widening does not keep a NaN's sign: take it from the fp8 byte
  if (f0 != f0) b0 = ((in & 0x80u) << 8) | 0x7FC0u;
  if (f1 != f1) b1 = (in & 0x8000u) | 0x7FC0u;
  return b0 | (b1 << 16);
}

// ---- division ------------------------------------------------------------------
// a / b rounded to nearest even, given y = RN(1/b) with b and y normal and
// finite: q = RN(a*y) is within one ulp of a/b, the residual a - q*b is exact
// under a fused multiply-add, and one correction q + r*y lands on the
// correctly rounded quotient (Markstein, "IA-64 and elementary functions",
// 2000, the division theorem).  A zero or non-finite first quotient is already
// final (it keeps the sign of a zero numerator; an overflow saturates later).
struct ScaledDiv {
  float b, y;
  bool fast;
  __device__ __forceinline__ explicit ScaledDiv(float scale) : b(scale) {
    y = __frcp_rn(scale);
    const float ab = fabsf(scale), ay = fabsf(y);
    fast = ab >= 1.1754944e-38f && ab <= 8.5e37f && ay >= 1.1754944e-38f && ay <= 8.5e37f;
  }
  __device__ __forceinline__ float operator()(float a) const {
    if (!fast) return __fdiv_rn(a, b);
    const float q = a * y;
    if (q == 0.0f || !(fabsf(q) <= 3.4028235e38f)) return q;
    const float r = fmaf(-q, b, a);
    return fmaf(r, y, q);
  }
};

// 8 bf16 (one uint4) -> 8 fp8 (one uint2), each value divided by the scale.
template <int F>
__device__ __forceinline__ uint2 bf16x8_to_fp8x8(uint4 v, const ScaledDiv& d) {
  uint2 o;
  o.x = pack_fp8x2<F>(d(bf16lo(v.x)), d(bf16hi(v.x))) |
        (pack_fp8x2<F>(d(bf16lo(v.y)), d(bf16hi(v.y))) << 16);
  o.y = pack_fp8x2<F>(d(bf16lo(v.z)), d(bf16hi(v.z))) |
        (pack_fp8x2<F>(d(bf16lo(v.w)), d(bf16hi(v.w))) << 16);
  return o;
}

// 8 fp8 (one uint2) -> 8 bf16 (one uint4), exact.
template <int F>
__device__ __forceinline__ uint4 fp8x8_to_bf16x8(uint2 v) {
  uint4 o;
  o.x = fp8x2_to_bf16x2<F>(v.x);
  o.y = fp8x2_to_bf16x2<F>(v.x >> 16);
  o.z = fp8x2_to_bf16x2<F>(v.y);
  o.w = fp8x2_to_bf16x2<F>(v.y >> 16);
  return o;
}

// a*b - c*d accurate to two ulps even when the products cancel: the rounding
// error of c*d is recovered exactly by an FMA and added back (W. Kahan's
// algorithm; error bound by Jeannerod, Louvet and Muller, "Further analysis of
// Kahan's algorithm for the accurate computation of 2x2 determinants", Math.
// Comp. 82, 2013).
__device__ __forceinline__ float diff_of_products(float a, float b, float c, float d) {
  const float w = __fmul_rn(c, d);
  const float e = fmaf(-c, d, w);
  const float f = fmaf(a, b, -w);
  return __fadd_rn(f, e);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

}  // namespace mla
