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

// This lane's part of a row's sum of squares (16 kv_c elements in x0 / x1).
__device__ __forceinline__ float sum_sq16(const uint4& x0, const uint4& x1) {
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a0 = fma_bf16lo(w[i], w[i], a0);
    a1 = fma_bf16hi(w[i], w[i], a1);
  }
  return a0 + a1;
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
                                           const uint4& g1, float eps, uint4& y0, uint4& y1) {
  const float ss = warp_sum(sum_sq16(x0, x1));
  // mean over 512 (exact power-of-two scaling) + eps, one rounding
  scale16(x0, x1, g0, g1, __frsqrt_rn(fmaf(ss, 1.0f / kNormRank, eps)), y0, y1);
}

// The neox rotation of this lane's k_pe pair (element lane in the low half,
// lane+32 in the high half) by (cos, sin).
__device__ __forceinline__ uint32_t rope_pair(uint32_t pe, float2 cs) {
  const float u = bf16lo(pe), v = bf16hi(pe);
  return pack_bf16x2(diff_of_products(u, cs.x, v, cs.y), diff_of_products(v, cs.x, -u, cs.y));
}

}  // namespace mla
