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

enum Fmt : int { kBF16 = 0, kE4M3 = 1, kE5M2 = 2, kF16 = 3 };

// Whether a format is a 16-bit float (bf16 or fp16).
__host__ __device__ constexpr bool is16(int f) { return f == kBF16 || f == kF16; }

constexpr uint32_t kErrSlotOOB = 1u;
constexpr uint32_t kErrBlockOOB = 2u;
constexpr uint32_t kErrPosOOB = 4u;
constexpr uint32_t kErrMisaligned = 8u;
constexpr uint32_t kErrTimeout = 16u;

// ---- programmatic dependent launch ---------------------------------------
// Wait until every grid this one depends on has completed and its memory
// operations are visible (a no-op when launched without the PDL attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid on the stream to start launching.  Every kernel of this
// library calls it first: its grid never exceeds the resident CTAs, so all of
// its CTAs are running before a dependent CTA can take an SM slot, and the
// dependent's CTAs then sit resident in their own pdl_wait() until this grid
// has completed -- the next launch's latency overlaps this kernel's work.
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
// Bring the line holding p into L2 (no register result, no wait).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void st8(void* p, uint2 v) { *reinterpret_cast<uint2*>(p) = v; }

// ---- bf16 ------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---- fp16 ------------------------------------------------------------------
__device__ __forceinline__ float f16lo(uint32_t w) {
  float f;
  asm("{ .reg .b16 a, b; mov.b32 {a, b}, %1; cvt.f32.f16 %0, a; }" : "=f"(f) : "r"(w));
  return f;
}
__device__ __forceinline__ float f16hi(uint32_t w) {
  float f;
  asm("{ .reg .b16 a, b; mov.b32 {a, b}, %1; cvt.f32.f16 %0, b; }" : "=f"(f) : "r"(w));
  return f;
}
// The two 16-bit floats of a word (format IF) as exact fp32 values.
template <int IF>
__device__ __forceinline__ float x16lo(uint32_t w) {
  if constexpr (IF == kF16) return f16lo(w);
  else return __uint_as_float(w << 16);
}
template <int IF>
__device__ __forceinline__ float x16hi(uint32_t w) {
  if constexpr (IF == kF16) return f16hi(w);
  else return __uint_as_float(w & 0xFFFF0000u);
}

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

// Four fp32 -> four fp8 in one 32-bit word (a0 in the lowest byte): the two
// pairwise conversions write the two halves of the result register directly.
template <int F>
__device__ __forceinline__ uint32_t pack_fp8x4(float a0, float a1, float a2, float a3) {
  uint32_t r;
  if constexpr (F == kE4M3) {
    asm("{ .reg .b16 l, h;\n"
        "  cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n"
        "  cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n"
        "  mov.b32 %0, {l, h}; }"
        : "=r"(r) : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  } else {
    asm("{ .reg .b16 l, h;\n"
        "  cvt.rn.satfinite.e5m2x2.f32 l, %2, %1;\n"
        "  cvt.rn.satfinite.e5m2x2.f32 h, %4, %3;\n"
        "  mov.b32 %0, {l, h}; }"
        : "=r"(r) : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  }
  return r;
}

// fp8x2 (low 16 bits of `w`) -> two exact bf16 values in one 32-bit word.
// The hardware widening to f16x2 is exact for both fp8 formats, and every
// finite f16 obtained this way is a bf16 value, so truncating the fp32 is
// exact.  A NaN becomes the quiet NaN 0x7FC0 with the fp8 code's sign.
template <int F>
__device__ __forceinline__ void fp8x2_to_f32x2(uint32_t w, float& f0, float& f1) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(w);
  if constexpr (F == kE4M3) {
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  } else {
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(in));
  }
  asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b; }"
      : "=f"(f0), "=f"(f1) : "r"(h2));
}

template <int F>
__device__ __forceinline__ uint32_t fp8x2_to_bf16x2(uint32_t w) {
  const uint16_t in = static_cast<uint16_t>(w);
  float f0, f1;
  fp8x2_to_f32x2<F>(w, f0, f1);
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

// ---- packed fp32x2 arithmetic (sm_100+) --------------------------------------
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unf2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Division constants of one scale b: y = RN(1/b) (correctly rounded), and
// whether the packed fast paths below are valid for b (b and y normal).
// thr2 holds, in both 16-bit halves, 0x8000 - (T << 7), where T is the
// smallest bf16 exponent field whose values could make a*y overflow (|a| >=
// 2^(T-126) and |y| < 2^(e_y-126) give |a*y| < 2^128 only for e_a + e_y <= 380)
// -- capped at 255, so inf and NaN always count.
struct DivConst {
  float b, y;
  uint64_t y2, nb2;  // ( y,  y), (-b, -b): guarded path
  uint64_t ny2, b2;  // (-y, -y), ( b,  b): fast path
  uint32_t thr2;   // bf16 inputs
  uint32_t thr2h;  // fp16 inputs: 0x8000 - 0x7C00 (only inf / NaN are special)
                   // while |y| < 2^111 (|a| <= 65504 < 2^16 keeps a*y finite),
                   // else 0x7FFF (every nonzero value takes the guarded path)
  bool fast;
};
__device__ __forceinline__ DivConst div_const(float scale) {
  DivConst k;
  k.b = scale;
  k.y = __frcp_rn(scale);
  const float ab = fabsf(scale), ay = fabsf(k.y);
  k.fast = ab >= 1.1754944e-38f && ab <= 8.5e37f && ay >= 1.1754944e-38f && ay <= 8.5e37f;
  k.y2 = f2(k.y, k.y);
  k.nb2 = f2(-scale, -scale);
  k.ny2 = f2(-k.y, -k.y);
  k.b2 = f2(scale, scale);
  const int e_y = (int)((__float_as_uint(k.y) >> 23) & 0xFFu);
  const int t = min(381 - e_y, 255);
  const uint32_t h = 0x8000u - ((uint32_t)max(t, 1) << 7);
  k.thr2 = h | (h << 16);
  const uint32_t hh = ay < 2.5961484e33f ? 0x0400u : 0x7FFFu;  // 2^111
  k.thr2h = hh | (hh << 16);
  return k;
}

// Two correctly rounded quotients a/b at once.  GUARDED: the division theorem
// of ScaledDiv on packed fp32x2 pairs (q = a*y, r = a - q*b, q' = q + r*y),
// then per element the two special cases -- a NaN second step (the first
// quotient overflowed, or a was NaN / inf) keeps the first quotient, and a zero
// keeps the first quotient's sign.  !FAST: IEEE division (scales outside the
// range where the theorem's assumptions hold).
template <bool FAST>
__device__ __forceinline__ float2 div2(float a0, float a1, const DivConst& k) {
  if constexpr (!FAST) {
    return make_float2(__fdiv_rn(a0, k.b), __fdiv_rn(a1, k.b));
  } else {
    const uint64_t a = f2(a0, a1);
    const uint64_t q = mul2(a, k.y2);
    const uint64_t r = fma2(q, k.nb2, a);
    const float2 qq = unf2(q), c = unf2(fma2(r, k.y2, q));
    const float o0 = (c.x != c.x) ? qq.x : c.x;
    const float o1 = (c.y != c.y) ? qq.y : c.y;
    return make_float2(
        __uint_as_float((__float_as_uint(o0) & 0x7FFFFFFFu) | (__float_as_uint(qq.x) & 0x80000000u)),
        __uint_as_float((__float_as_uint(o1) & 0x7FFFFFFFu) | (__float_as_uint(qq.y) & 0x80000000u)));
  }
}

// The same two quotients of the bf16 pair in w when neither value can make
// the first quotient non-finite (see special_pairs): with the negated inputs
// -a, q = (-a)(-y), r' = q*b - a (exact), q' = q - r'*y is the correctly rounded
// a/b, and the sign of a zero input survives every step (-0 -> q = -0,
// r' = +0, q' = -0), so no per-element fix-up is needed.
template <int IF = kBF16>
__device__ __forceinline__ float2 div2_fast(uint32_t w, const DivConst& k) {
  const uint32_t nw = w ^ 0x80008000u;
  const uint64_t na = f2(x16lo<IF>(nw), x16hi<IF>(nw));
  const uint64_t q = mul2(na, k.ny2);
  const uint64_t r = fma2(q, k.b2, na);
  return unf2(fma2(r, k.ny2, q));
}

__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Whether any bf16 whose magnitude bits are folded (by max.u16x2) into m has
// an exponent field >= T: adding 0x8000 - (T << 7) to a half carries into its
// top bit exactly then (no carry crosses halves: a half is at most 0x7F80).
__device__ __forceinline__ bool special_pairs(uint32_t m, uint32_t thr2) {
  return ((m + thr2) & 0x80008000u) != 0u;
}

// 8 16-bit floats of format IF (one uint4) -> 8 fp8 (one uint2), each value
// divided by the scale; the special-value check is done once for the 8.
template <int F, int IF, bool FAST>
__device__ __forceinline__ uint2 x16x8_to_fp8x8(uint4 v, const DivConst& k) {
  uint2 o;
  if constexpr (FAST) {
    const uint32_t m = umax16x2(umax16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                umax16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    if (!special_pairs(m, IF == kF16 ? k.thr2h : k.thr2)) {
      const float2 q0 = div2_fast<IF>(v.x, k), q1 = div2_fast<IF>(v.y, k);
      const float2 q2 = div2_fast<IF>(v.z, k), q3 = div2_fast<IF>(v.w, k);
      o.x = pack_fp8x4<F>(q0.x, q0.y, q1.x, q1.y);
      o.y = pack_fp8x4<F>(q2.x, q2.y, q3.x, q3.y);
      return o;
    }
  }
  const float2 q0 = div2<FAST>(x16lo<IF>(v.x), x16hi<IF>(v.x), k);
  const float2 q1 = div2<FAST>(x16lo<IF>(v.y), x16hi<IF>(v.y), k);
  const float2 q2 = div2<FAST>(x16lo<IF>(v.z), x16hi<IF>(v.z), k);
  const float2 q3 = div2<FAST>(x16lo<IF>(v.w), x16hi<IF>(v.w), k);
  o.x = pack_fp8x4<F>(q0.x, q0.y, q1.x, q1.y);
  o.y = pack_fp8x4<F>(q2.x, q2.y, q3.x, q3.y);
  return o;
}

// Two bf16 in a 32-bit word -> two fp8 (low 16 bits), divided by the scale.
template <int F, bool FAST>
__device__ __forceinline__ uint32_t bf16x2_to_fp8x2(uint32_t w, const DivConst& k) {
  if constexpr (FAST) {
    if (!special_pairs(w & 0x7FFF7FFFu, k.thr2)) {
      const float2 q = div2_fast(w, k);
      return pack_fp8x2<F>(q.x, q.y);
    }
  }
  const float2 q = div2<FAST>(bf16lo(w), bf16hi(w), k);
  return pack_fp8x2<F>(q.x, q.y);
}

// 8 bf16 (one uint4) -> 8 fp8 (one uint2), each value divided by the scale.
template <int F, bool FAST>
__device__ __forceinline__ uint2 bf16x8_to_fp8x8(uint4 v, const DivConst& k) {
  return x16x8_to_fp8x8<F, kBF16, FAST>(v, k);
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

// fp8x2 (low 16 bits of `w`) -> two exact fp16 values (the hardware widening
// is exact for both formats); a NaN becomes the quiet NaN 0x7E00 with the fp8
// code's sign.
template <int F>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t w) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(w);
  if constexpr (F == kE4M3) {
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  } else {
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(in));
  }
  if ((h2 & 0x7FFFu) > 0x7C00u) h2 = (h2 & 0xFFFF0000u) | ((in & 0x80u) << 8) | 0x7E00u;
  if ((h2 & 0x7FFF0000u) > 0x7C000000u) h2 = (h2 & 0xFFFFu) | ((in & 0x8000u) << 16) | 0x7E000000u;
  return h2;
}

// Whether any of the 8 fp8 codes in v is a NaN (e4m3: low 7 bits 0x7F; e5m2:
// above 0x7C): adding 1 (3) to each byte's low 7 bits carries into its top
// bit exactly for those codes, and never across bytes.
template <int F>
__device__ __forceinline__ bool fp8x8_any_nan(uint2 v) {
  constexpr uint32_t kAdd = F == kE4M3 ? 0x01010101u : 0x03030303u;
  const uint32_t a = ((v.x & 0x7F7F7F7Fu) + kAdd) | ((v.y & 0x7F7F7F7Fu) + kAdd);
  return (a & 0x80808080u) != 0u;
}

// 8 fp8 (one uint2) -> 8 exact 16-bit floats of format OF (bf16 or fp16).
// Without a NaN code among the 8 the hardware widening is final (an fp8 value
// is exact in fp16, fp32 and bf16); a group holding one takes the per-element
// path, which gives each NaN the quiet NaN with its code's sign.
template <int F, int OF>
__device__ __forceinline__ uint4 fp8x8_to_x16x8(uint2 v) {
  if (!fp8x8_any_nan<F>(v)) {
    const uint32_t w[4] = {v.x, v.x >> 16, v.y, v.y >> 16};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t h2;
      const uint16_t in = static_cast<uint16_t>(w[i]);
      if constexpr (F == kE4M3) asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
      else asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(in));
      if constexpr (OF == kBF16) {
        float f0, f1;
        asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b; }"
            : "=f"(f0), "=f"(f1) : "r"(h2));
        o[i] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
      } else {
        o[i] = h2;
      }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  }
  if constexpr (OF == kBF16) {
    return fp8x8_to_bf16x8<F>(v);
  } else {
    return make_uint4(fp8x2_to_f16x2<F>(v.x), fp8x2_to_f16x2<F>(v.x >> 16),
                      fp8x2_to_f16x2<F>(v.y), fp8x2_to_f16x2<F>(v.y >> 16));
  }
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

template <int F>
__device__ __forceinline__ bool fp8_is_nan(uint32_t c) {
  return F == kE4M3 ? (c & 0x7Fu) == 0x7Fu : (c & 0x7Fu) > 0x7Cu;
}

// Eight fp8 -> bf16 dequantised by a scale (s2 = the scale in both halves):
// each element is the fp8 value (exact in f16 and in fp32) times the scale as
// one fp32 multiplication, rounded to bf16 with round to nearest even.  A NaN
// code gives the quiet NaN with the code's sign, any other NaN product the
// positive quiet NaN.  One NaN test of the sum of the eight products sends
// the rare group holding a NaN (or an inf - inf) through the per-element rule.
template <int F>
__device__ __forceinline__ uint4 fp8x8_to_bf16x8_scaled(uint2 v, uint64_t s2) {
  const uint32_t w[4] = {v.x, v.x >> 16, v.y, v.y >> 16};
  uint64_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a, b;
    fp8x2_to_f32x2<F>(w[i], a, b);
    p[i] = mul2(f2(a, b), s2);
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = unf2(p[i]);
    o[i] = pack_bf16x2(q.x, q.y);
  }
  const float2 t = unf2(add2(add2(p[0], p[1]), add2(p[2], p[3])));
  const float u = t.x + t.y;
  if (__builtin_expect(u != u, 0)) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 q = unf2(p[i]);
      const uint32_t c0 = w[i] & 0xFFu, c1 = (w[i] >> 8) & 0xFFu;
      if (q.x != q.x)
        o[i] = (o[i] & 0xFFFF0000u) | (fp8_is_nan<F>(c0) ? (c0 & 0x80u) << 8 : 0u) | 0x7FC0u;
      if (q.y != q.y)
        o[i] = (o[i] & 0xFFFFu) | (((fp8_is_nan<F>(c1) ? (c1 & 0x80u) << 8 : 0u) | 0x7FC0u) << 16);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
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

// ---- mbarrier + bulk asynchronous copies (sm_90+ PTX) ------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of `bar` with the given parity to complete, giving up
// after `limit_ns` (returns false then): no wait in this library can hang.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 255u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}
// One bulk copy global -> this CTA's shared memory, completing on `bar`
// (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds16(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds8(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

}  // namespace mla
