// pack.cu -- chunked-context K/V pack for sm_103a.
//
// What it computes: the contiguous full key [k_nope | k_pe] (k_pe broadcast to
// every head) and the contiguous V from the strided kv_b_proj output and a
// k_pe that may still be fp8 from the cache, in bf16 or fp8 ("PR #51772
// [Attention][MLA] Fuse Kimi-K3 chunked-context K/V packing", Implementation
// item 1 and Source snippets: fused_mla_kv_concat /
// fused_mla_kv_concat_quant_fp8).
//
// Design:
//   * one warp per token, grid capped at the resident-CTA count, grid-stride
//     loop over tokens (long contexts never grow the grid);
//   * the unit of work is 8 elements = one 16-byte bf16 load; a token's 16
//     heads x (16 k_nope + 16 v) units are 8 + 8 loads per lane, all issued
//     before the first store (8 KB in flight per warp).  Each warp load covers
//     two whole 256-byte head rows, so the 64-element row padding of the
//     kv_b_proj output is never touched;
//   * k_pe: lane l only ever writes part (l % 8) of the rope slice, so it loads
//     that 8-element part once and writes it to its four heads;
//   * outputs are written as 8-byte (fp8) or 16-byte (bf16) vectors, 16 lanes
//     covering a head's k_nope slice, so every warp store is whole sectors;
//   * fp8: correctly rounded division by the scale, hardware .satfinite
//     converters; an fp8 k_pe is copied byte for byte; an fp8 k_pe into a bf16
//     key goes through the exact hardware widening;
//   * output format, k_pe format and the head count (16, or any at runtime) are
//     template parameters.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kNope = 128, kRope = 64, kV = 128, kKey = kNope + kRope;

template <int OF, int KF, int HC>
__global__ void __launch_bounds__(kThreads) pack_kernel(const PackArgs a) {
  pdl_wait();
  constexpr int OE = (OF == kBF16) ? 2 : 1;  // output bytes per element
  const int lane = threadIdx.x & 31;
  const int H = HC ? HC : a.num_heads;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const bool has_v = a.vout != nullptr;
  float scale = 1.0f;
  if constexpr (OF != kBF16) {
    if (a.out_scale) scale = *a.out_scale;
  }
  const ScaledDiv d(scale);
  const int nope_units = H * (kNope / 8);  // 8-element units; v has as many
  const int pe_units = H * (kRope / 8);
  const int part_pe = lane & 7;

  for (int64_t t = warp; t < a.num_tokens; t += nwarps) {
    const uint8_t* kn = a.k_nope + t * a.kn_ts;
    const uint8_t* vv = a.v + t * a.v_ts;
    uint8_t* key = a.key + t * (int64_t)H * kKey * OE;
    uint8_t* vo = has_v ? a.vout + t * (int64_t)H * kV * OE : nullptr;

    // k_pe part of this lane, converted once
    uint4 pe16 = make_uint4(0, 0, 0, 0);
    uint2 pe8 = make_uint2(0, 0);
    {
      const uint8_t* pe = a.k_pe + t * a.kpe_ts;
      if constexpr (KF == kBF16) {
        const uint4 x = ld_stream16(pe + part_pe * 16);
        if constexpr (OF == kBF16) pe16 = x;
        else pe8 = bf16x8_to_fp8x8<OF>(x, d);
      } else {
        const uint2 x = ld_stream8(pe + part_pe * 8);
        if constexpr (OF == kBF16) pe16 = fp8x8_to_bf16x8<KF>(x);
        else pe8 = x;  // same fp8 format: raw bytes
      }
    }

    for (int ub = 0; ub < nope_units; ub += 8 * 32) {
      uint4 kr[8], vr[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int u = ub + i * 32 + lane;
        kr[i] = vr[i] = make_uint4(0, 0, 0, 0);
        if (HC == 16 || u < nope_units) {
          const int h = u >> 4, part = u & 15;
          kr[i] = ld_stream16(kn + h * a.kn_hs + part * 16);
          if (has_v) vr[i] = ld_stream16(vv + h * a.v_hs + part * 16);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int u = ub + i * 32 + lane;
        if (HC == 16 || u < nope_units) {
          const int h = u >> 4, part = u & 15;
          uint8_t* kd = key + (h * kKey + part * 8) * OE;
          if constexpr (OF == kBF16) st16(kd, kr[i]);
          else st8(kd, bf16x8_to_fp8x8<OF>(kr[i], d));
          if (has_v) {
            uint8_t* vd = vo + (h * kV + part * 8) * OE;
            if constexpr (OF == kBF16) st16(vd, vr[i]);
            else st8(vd, bf16x8_to_fp8x8<OF>(vr[i], d));
          }
        }
      }
    }
    // rope slice of every head: unit u = (head u/8, part u%8 == lane%8)
    for (int u = lane; u < pe_units; u += 32) {
      uint8_t* kd = key + ((u >> 3) * kKey + kNope + part_pe * 8) * OE;
      if constexpr (OF == kBF16) st16(kd, pe16);
      else st8(kd, pe8);
    }
  }
  pdl_trigger();
}

template <int OF, int KF, int HC>
cudaError_t launch_t(const PackArgs& a, const LaunchCfg& cfg) {
  auto kern = pack_kernel<OF, KF, HC>;
  const int64_t ctas = ((int64_t)a.num_tokens + kThreads / 32 - 1) / (kThreads / 32);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(capped_grid(reinterpret_cast<const void*>(kern), kThreads, ctas));
  lc.blockDim = dim3(kThreads);
  lc.stream = cfg.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = cfg.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, kern, a);
}

template <int OF, int KF>
cudaError_t launch_heads(const PackArgs& a, const LaunchCfg& cfg) {
  if (a.num_heads == 16) return launch_t<OF, KF, 16>(a, cfg);
  return launch_t<OF, KF, 0>(a, cfg);
}

template <int OF>
cudaError_t launch_kpe(const PackArgs& a, int kpe_fmt, const LaunchCfg& cfg) {
  if (kpe_fmt == kBF16) return launch_heads<OF, kBF16>(a, cfg);
  if constexpr (OF == kBF16 || OF == kE4M3) {
    if (kpe_fmt == kE4M3) return launch_heads<OF, kE4M3>(a, cfg);
  }
  if constexpr (OF == kBF16 || OF == kE5M2) {
    if (kpe_fmt == kE5M2) return launch_heads<OF, kE5M2>(a, cfg);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_pack(const PackArgs& a, int out_fmt, int kpe_fmt, const LaunchCfg& cfg) {
  switch (out_fmt) {
    case kBF16: return launch_kpe<kBF16>(a, kpe_fmt, cfg);
    case kE4M3: return launch_kpe<kE4M3>(a, kpe_fmt, cfg);
    case kE5M2: return launch_kpe<kE5M2>(a, kpe_fmt, cfg);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
