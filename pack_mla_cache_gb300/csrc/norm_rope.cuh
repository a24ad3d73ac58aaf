// norm_rope.cuh -- the per-lane RMSNorm and neox RoPE arithmetic of one
// [kv_c 512 | k_pe 64] bf16 row held by a warp, shared by the grouped insert
// and the standalone grouped RMSNorm + RoPE ("PR #50585 [K3 Perf] Optimize k3
// dspark fused kv", Source snippets: _precompute_fused_context_kv, a grouped
// rms_norm with one weight row per layer, then the rotation of k_pe).
//
// Row layout in a warp: lane l holds kv_c elements [8l, 8l+8) (x0) and
// [256+8l, 256+8l+8) (x1) and the rotary pair (l, l+32) of k_pe.
//   * RMSNorm: 16 squares per lane on mixed-precision FMAs (bf16 operands,
//     fp32 accumulator: no unpacking; unpacking into packed fp32x2 FMAs made
//     the grouped insert 1% slower), a 5-step xor-shuffle sum, a correctly
//     rounded reciprocal square root; y = (x * gamma, exact in fp32) * rstd,
//     one fp32 rounding, then bf16 rounding;
//   * RoPE: each rotated element is a difference of two products with an FMA
//     error correction (two-ulp accurate even when the products cancel).
#pragma once

#include "mla_device.cuh"

namespace mla {

constexpr int kNormRank = 512;  // kv_lora_rank of the rows

// Exact fp32 value of a*b + c for bf16 a, b (mixed-precision FMA, sm_100+).
__device__ __forceinline__ float fma_bf16lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;\n"
      "  fma.rn.f32.bf16 %0, al, bl, %3; }" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_bf16hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;\n"
      "  fma.rn.f32.bf16 %0, ah, bh, %3; }" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

// ---- the sum of squares of a row ---------------------------------------------
// One summation tree for both layouts (one row per warp, or per half warp), so
// that every kernel normalises a row to the same bits whichever layout the
// call size picks: the 512 elements are 64 units of 8 (16 bytes, unit u =
// elements [8u, 8u + 8)); S(u) sums a unit's squares in two chains (low and
// high halves of its 4 words, in word order) added at the end; position
// p < 16 combines units p, p + 16, p + 32, p + 48 as
// (S(p) + S(p + 16)) + (S(p + 32) + S(p + 48)); the 16 positions are then
// added by an xor butterfly (offsets 8, 4, 2, 1).

// S(u) of one unit.
__device__ __forceinline__ float unit_sq(const uint4& x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  float lo = 0.f, hi = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    lo = fma_bf16lo(w[i], w[i], lo);
    hi = fma_bf16hi(w[i], w[i], hi);
  }
  return lo + hi;
}

// The row's sum of squares in the one-row-per-warp layout: lane l holds
// units l (x0) and 32 + l (x1).  Lanes l and l ^ 16 together hold position
// l % 16's four units, so each completes the position's sum with the other's
// two; both halves then run the same butterfly.
__device__ __forceinline__ float row_sum_sq(const uint4& x0, const uint4& x1, int lane) {
  const float a = unit_sq(x0), b = unit_sq(x1);
  const float pa = __shfl_xor_sync(0xFFFFFFFFu, a, 16), pb = __shfl_xor_sync(0xFFFFFFFFu, b, 16);
  // lane < 16: a = S(p), b = S(p + 32), pa = S(p + 16), pb = S(p + 48)
  float v = lane < 16 ? (a + pa) + (b + pb) : (pa + a) + (pb + b);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// y = x * gamma * rstd for this lane's 16 elements (x * gamma is exact in
// fp32), rounded to bf16.  NEG gives -y instead (the same roundings, since
// round-to-nearest-even is symmetric) for consumers that start from -y.
template <bool NEG = false>
__device__ __forceinline__ void scale16(const uint4& x0, const uint4& x1, const uint4& g0,
                                        const uint4& g1, float rstd, uint4& y0, uint4& y1) {
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  const uint64_t rstd2 = NEG ? f2(-rstd, -rstd) : f2(rstd, rstd);
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t xg = f2(fma_bf16lo(w[i], gw[i], -0.0f), fma_bf16hi(w[i], gw[i], -0.0f));
    const float2 y = unf2(mul2(xg, rstd2));
    o[i] = pack_bf16x2(y.x, y.y);
  }
  y0 = make_uint4(o[0], o[1], o[2], o[3]);
  y1 = make_uint4(o[4], o[5], o[6], o[7]);
}

// RMSNorm of this lane's 16 kv_c elements (words x0 / x1) with the row's
// gamma words g0 / g1: returns the bf16-rounded results in y0 / y1.
__device__ __forceinline__ void rms_norm16(const uint4& x0, const uint4& x1, const uint4& g0,
                                           const uint4& g1, float eps, uint4& y0, uint4& y1,
                                           int lane) {
  const float ss = row_sum_sq(x0, x1, lane);
  // mean over 512 (exact power-of-two scaling) + eps, one rounding
  scale16(x0, x1, g0, g1, __frsqrt_rn(fmaf(ss, 1.0f / kNormRank, eps)), y0, y1);
}

// The neox rotation of this lane's k_pe pair (element lane in the low half,
// lane+32 in the high half) by (cos, sin).
__device__ __forceinline__ uint32_t rope_pair(uint32_t pe, float2 cs) {
  const float u = bf16lo(pe), v = bf16hi(pe);
  return pack_bf16x2(diff_of_products(u, cs.x, v, cs.y), diff_of_products(v, cs.x, -u, cs.y));
}

// ---- rows held by a half warp ----------------------------------------------
// Half-warp layout (16 lanes per row, two rows per warp): lane hl = lane & 15
// of a half holds kv_c elements [8 hl + 128 c, 8 hl + 128 c + 8) for c = 0..3
// (x[c], the 16-byte unit at byte 16 hl + 256 c of the bf16 row), and the k_pe
// elements 2 hl, 2 hl + 1 (word lo) and 2 hl + 32, 2 hl + 33 (word hi), i.e.
// the neox pairs (2 hl, 2 hl + 32) and (2 hl + 1, 2 hl + 33).  The row-uniform
// work (the reduction, the reciprocal square root, the row's slot) is then
// shared by the two rows a warp instruction serves.

// This lane's position sum in the half-warp layout (units hl + 16 c in x[c]):
// the tree above.
__device__ __forceinline__ float sum_sq32(const uint4 (&x)[4]) {
  return (unit_sq(x[0]) + unit_sq(x[1])) + (unit_sq(x[2]) + unit_sq(x[3]));
}

// Sum over the 16 lanes of a half warp (xor offsets stay inside the half).
__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// y = x * gamma * rstd for this lane's 32 elements, in place, as scale16 (NEG:
// -y).
template <bool NEG = false>
__device__ __forceinline__ void scale32(uint4 (&x)[4], const uint4 (&g)[4], float rstd) {
  const uint64_t rstd2 = NEG ? f2(-rstd, -rstd) : f2(rstd, rstd);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w[4] = {x[c].x, x[c].y, x[c].z, x[c].w};
    const uint32_t gw[4] = {g[c].x, g[c].y, g[c].z, g[c].w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t xg = f2(fma_bf16lo(w[i], gw[i], -0.0f), fma_bf16hi(w[i], gw[i], -0.0f));
      const float2 y = unf2(mul2(xg, rstd2));
      o[i] = pack_bf16x2(y.x, y.y);
    }
    x[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// RMSNorm of this lane's 32 kv_c elements in place (gamma words g).
template <bool NEG = false>
__device__ __forceinline__ void rms_norm32(uint4 (&x)[4], const uint4 (&g)[4], float eps) {
  const float ss = half_sum(sum_sq32(x));
  // mean over 512 (exact power-of-two scaling) + eps, one rounding
  scale32<NEG>(x, g, __frsqrt_rn(fmaf(ss, 1.0f / kNormRank, eps)));
}

// The same with gamma read from `gr` (this lane's first unit of the row's
// weights; unit c at gr + 256 c) one unit at a time where it is used, which
// keeps 12 fewer registers live than holding all four.
template <bool NEG = false>
__device__ __forceinline__ void rms_norm32_g(uint4 (&x)[4], const uint8_t* gr, float eps) {
  const float ss = half_sum(sum_sq32(x));
  const float rstd = __frsqrt_rn(fmaf(ss, 1.0f / kNormRank, eps));
  const uint64_t rstd2 = NEG ? f2(-rstd, -rstd) : f2(rstd, rstd);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(gr + 256 * c));
    const uint32_t w[4] = {x[c].x, x[c].y, x[c].z, x[c].w};
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t xg = f2(fma_bf16lo(w[i], gw[i], -0.0f), fma_bf16hi(w[i], gw[i], -0.0f));
      const float2 y = unf2(mul2(xg, rstd2));
      o[i] = pack_bf16x2(y.x, y.y);
    }
    x[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The neox rotation of this lane's two k_pe pairs in place: lo holds elements
// (2 hl, 2 hl + 1), hi (2 hl + 32, 2 hl + 33); cs = (cos(2 hl), cos(2 hl + 1),
// sin(2 hl), sin(2 hl + 1)).
__device__ __forceinline__ void rope_pairs2(uint32_t& lo, uint32_t& hi, float4 cs) {
  const uint32_t p0 = __byte_perm(lo, hi, 0x5410);  // (2 hl, 2 hl + 32)
  const uint32_t p1 = __byte_perm(lo, hi, 0x7632);  // (2 hl + 1, 2 hl + 33)
  const uint32_t r0 = rope_pair(p0, make_float2(cs.x, cs.z));
  const uint32_t r1 = rope_pair(p1, make_float2(cs.y, cs.w));
  lo = __byte_perm(r0, r1, 0x5410);
  hi = __byte_perm(r0, r1, 0x7632);
}

// (cos, cos, sin, sin) of this lane's pairs from a table row (cos of the 32
// pairs, then their sin).
__device__ __forceinline__ float4 load_cs2(const float* row, int hl) {
  const float2 c = __ldg(reinterpret_cast<const float2*>(row + 2 * hl));
  const float2 s = __ldg(reinterpret_cast<const float2*>(row + 32 + 2 * hl));
  return make_float4(c.x, c.y, s.x, s.y);
}

// ---- rows held by a quarter warp ----------------------------------------------
// Quarter-warp layout (8 lanes per row, four rows per warp): lane ql = lane & 7
// of a quarter holds positions ql and ql + 8 of the tree above: x[c] is unit
// ql + 16 c and x[4 + c] unit ql + 8 + 16 c (bytes 16 ql + 256 c and 16 ql +
// 128 + 256 c of the bf16 row); its k_pe elements are 4 ql .. 4 ql + 3 (lo)
// and 4 ql + 32 .. 4 ql + 35 (hi), the neox pairs (4 ql + j, 4 ql + 32 + j).
// The row-uniform work is shared by the four rows a warp instruction serves.

// This lane's sum of its two positions: the butterfly's offset-8 step taken
// inside the lane (position ql first, as in the half-warp layout's lane ql).
__device__ __forceinline__ float sum_sq64(const uint4 (&x)[8]) {
  const float a = (unit_sq(x[0]) + unit_sq(x[1])) + (unit_sq(x[2]) + unit_sq(x[3]));
  const float b = (unit_sq(x[4]) + unit_sq(x[5])) + (unit_sq(x[6]) + unit_sq(x[7]));
  return a + b;
}

// The rest of the butterfly (offsets 4, 2, 1) over the 8 lanes of a quarter.
__device__ __forceinline__ float quarter_sum(float v) {
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// RMSNorm of this lane's 64 kv_c elements in place, gamma read unit by unit
// from `gr` (this lane's unit ql of the row's weights) where it is used.
template <bool NEG = false>
__device__ __forceinline__ void rms_norm64_g(uint4 (&x)[8], const uint8_t* gr, float eps) {
  const float ss = quarter_sum(sum_sq64(x));
  const float rstd = __frsqrt_rn(fmaf(ss, 1.0f / kNormRank, eps));
  const uint64_t rstd2 = NEG ? f2(-rstd, -rstd) : f2(rstd, rstd);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(gr + 256 * (c & 3) + 128 * (c >> 2)));
    const uint32_t w[4] = {x[c].x, x[c].y, x[c].z, x[c].w};
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t xg = f2(fma_bf16lo(w[i], gw[i], -0.0f), fma_bf16hi(w[i], gw[i], -0.0f));
      const float2 y = unf2(mul2(xg, rstd2));
      o[i] = pack_bf16x2(y.x, y.y);
    }
    x[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The neox rotation of this lane's four k_pe pairs in place; c = cos of
// elements 4 ql .. 4 ql + 3, sn = their sin.
__device__ __forceinline__ void rope_pairs4(uint2& lo, uint2& hi, float4 c, float4 sn) {
  rope_pairs2(lo.x, hi.x, make_float4(c.x, c.y, sn.x, sn.y));
  rope_pairs2(lo.y, hi.y, make_float4(c.z, c.w, sn.z, sn.w));
}

}  // namespace mla
