// norm_rope.cu -- standalone grouped RMSNorm + RoPE for sm_103a.
//
// What it computes: for every (token, layer) row of a [kv_c 512 | k_pe 64]
// bf16 input (any token / layer strides, e.g. the [T, L, 576] DSpark context
// projection read in place), kv_c RMS-normalised with layer l's weight row and
// k_pe rotated (neox) with the token's position -- the same position for every
// layer -- each rounded to bf16 and written to caller-strided outputs (e.g.
// the layer-major [L, T, 512] and [L, T, 64] the insert consumes) ("PR #50585
// [K3 Perf] Optimize k3 dspark fused kv", Implementation item 3 and Source
// snippets: _precompute_fused_context_kv, which makes both parts layer-major
// with permute().contiguous(), then runs the grouped rms_norm and the
// rotation as separate passes).  Here the layout change, the norm and the
// rotation are one pass: each row is read once and written once.
//
// Design: rows in token-major order, normalised and rotated with the
// insert's arithmetic (norm_rope.cuh).  Small and large calls take one row per
// warp (two 512-byte kv_c warp loads and the k_pe pair; 115.4 us for 65536
// tokens x 5 layers, 6.7 TB/s, against 139.7 us with 4 rows a warp in
// lockstep); mid-size calls take two rows per warp, 16 lanes each (half the
// row-uniform work per row).  The grid is capped at the resident CTAs and
// loops over the rows.
#include "mla_device.cuh"
#include "mla_internal.h"
#include "norm_rope.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 1;  // rows per warp per iteration (more warps beat more rows a warp)
constexpr int kP = 64;

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) {
  return __ldcs(reinterpret_cast<const unsigned short*>(p));
}
__device__ __forceinline__ void st_u16(uint8_t* p, uint32_t v) {
  *reinterpret_cast<unsigned short*>(p) = static_cast<unsigned short>(v);
}

template <bool NORM, bool ROPE, bool PAIRS>
__global__ void __launch_bounds__(kThreads) norm_rope_kernel(const NormRopeArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const uint32_t L = (uint32_t)a.num_layers;
  uint32_t errbits = 0;
  if constexpr (PAIRS) {
    // Two rows per warp, 16 lanes each (the half-warp layout of norm_rope.cuh;
    // the grouped insert's arithmetic in either layout, so the results equal a
    // bf16 insert's): rows 2w + half, 2w + half + 2 nwarps, ...
    const int hl = lane & 15, half = lane >> 4;
    for (int64_t r0 = 2 * warp; r0 < a.num_rows; r0 += 2 * nwarps) {
      const int64_t r = r0 + half;
      const bool have = r < a.num_rows;
      uint32_t t = 0, l = 0;
      uint4 x[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                    make_uint4(0, 0, 0, 0)};
      uint32_t lo = 0, hi = 0;
      int64_t pos = 0;
      if (have) {
        t = (uint32_t)r / L;  // rows < 2^32
        l = (uint32_t)r - t * L;
        const uint8_t* src = a.kv_c + (int64_t)t * a.kvc_ts + (int64_t)l * a.kvc_ls + hl * 16;
#pragma unroll
        for (int c = 0; c < 4; ++c) x[c] = ld_stream16(src + 256 * c);
        const uint8_t* p = a.k_pe + (int64_t)t * a.kpe_ts + (int64_t)l * a.kpe_ls + hl * 4;
        lo = __ldcs(reinterpret_cast<const uint32_t*>(p));
        hi = __ldcs(reinterpret_cast<const uint32_t*>(p + kP));
        if constexpr (ROPE) pos = __ldg(a.positions + t);
      }
      bool ok = have;
      float4 cs = make_float4(1.f, 1.f, 0.f, 0.f);
      if (ROPE && have) {
        if (pos < 0 || pos >= a.max_position) {
          errbits |= kErrPosOOB;
          ok = false;
        } else {
          cs = load_cs2(a.cos_sin + pos * kP, hl);
        }
      }
      if constexpr (NORM) {
        uint4 g[4];
        const uint8_t* gr = a.gamma + (int64_t)l * a.gamma_ls + hl * 16;
#pragma unroll
        for (int c = 0; c < 4; ++c) g[c] = ld_shared_ro16(gr + 256 * c);
        rms_norm32(x, g, a.eps);  // every lane: the shuffles span the warp
      }
      if constexpr (ROPE) rope_pairs2(lo, hi, cs);
      if (ok) {
        uint8_t* dc = a.out_c + (int64_t)t * a.oc_ts + (int64_t)l * a.oc_ls + hl * 16;
#pragma unroll
        for (int c = 0; c < 4; ++c) st16(dc + 256 * c, x[c]);
        uint8_t* dp = a.out_p + (int64_t)t * a.op_ts + (int64_t)l * a.op_ls + hl * 4;
        *reinterpret_cast<uint32_t*>(dp) = lo;
        *reinterpret_cast<uint32_t*>(dp + kP) = hi;
      }
    }
    errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
    if (errbits && lane == 0 && a.err) atomicOr(a.err, errbits);
  } else {
  // one row per warp
  for (int64_t r0 = warp * kRows; r0 < a.num_rows; r0 += nwarps * kRows) {
    uint4 x0[kRows], x1[kRows];
    uint32_t pe[kRows];
    int64_t pos[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      x0[k] = x1[k] = make_uint4(0, 0, 0, 0);
      pe[k] = 0;
      pos[k] = 0;
      const int64_t r = r0 + k;
      if (r >= a.num_rows) continue;
      const uint32_t t = (uint32_t)r / L, l = (uint32_t)r - t * L;  // rows < 2^32
      const uint8_t* src = a.kv_c + (int64_t)t * a.kvc_ts + (int64_t)l * a.kvc_ls;
      x0[k] = ld_stream16(src + lane * 16);
      x1[k] = ld_stream16(src + 512 + lane * 16);
      const uint8_t* p = a.k_pe + (int64_t)t * a.kpe_ts + (int64_t)l * a.kpe_ls;
      pe[k] = ld_u16(p + lane * 2) | (ld_u16(p + kP + lane * 2) << 16);
      if constexpr (ROPE) pos[k] = __ldg(a.positions + t);
    }
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      const int64_t r = r0 + k;
      if (r >= a.num_rows) continue;
      const uint32_t t = (uint32_t)r / L, l = (uint32_t)r - t * L;
      float2 cs = make_float2(1.f, 0.f);
      if constexpr (ROPE) {
        if (pos[k] < 0 || pos[k] >= a.max_position) {  // uniform across the warp
          errbits |= kErrPosOOB;
          continue;
        }
        const float* row = a.cos_sin + pos[k] * kP;
        cs = make_float2(__ldg(row + lane), __ldg(row + kP / 2 + lane));
      }
      uint4 y0 = x0[k], y1 = x1[k];
      if constexpr (NORM) {
        const uint8_t* g = a.gamma + (int64_t)l * a.gamma_ls;
        rms_norm16(x0[k], x1[k], ld_shared_ro16(g + lane * 16),
                   ld_shared_ro16(g + 512 + lane * 16), a.eps, y0, y1, lane);
      }
      uint32_t p = pe[k];
      if constexpr (ROPE) p = rope_pair(pe[k], cs);
      uint8_t* dc = a.out_c + (int64_t)t * a.oc_ts + (int64_t)l * a.oc_ls;
      st16(dc + lane * 16, y0);
      st16(dc + 512 + lane * 16, y1);
      uint8_t* dp = a.out_p + (int64_t)t * a.op_ts + (int64_t)l * a.op_ls;
      st_u16(dp + lane * 2, p);
      st_u16(dp + kP + lane * 2, p >> 16);
    }
  }
  if (errbits && lane == 0 && a.err) atomicOr(a.err, errbits);
  }
}

// With RMSNorm or RoPE, calls of 8192 to 131071 rows take two rows per warp:
// 20480 rows (4096 tokens x 5 layers) 6.55 vs 7.4 us, while 327680 rows ran
// 117.7 vs 115.4 us (HBM-bound either way) and one-wave calls are latency-bound.
constexpr int64_t kPairsMinRows = 8192, kPairsMaxRows = 131072;

template <bool NORM, bool ROPE>
cudaError_t launch_t(const NormRopeArgs& a, const LaunchCfg& cfg) {
  const bool pairs =
      (NORM || ROPE) && a.num_rows >= kPairsMinRows && a.num_rows < kPairsMaxRows;
  auto kern = pairs ? norm_rope_kernel<NORM, ROPE, NORM || ROPE>
                    : norm_rope_kernel<NORM, ROPE, false>;
  const int64_t warps = pairs ? (a.num_rows + 1) / 2 : (a.num_rows + kRows - 1) / kRows;
  const int64_t ctas = (warps + kThreads / 32 - 1) / (kThreads / 32);
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

}  // namespace

cudaError_t launch_norm_rope(const NormRopeArgs& a, bool norm, bool rope, const LaunchCfg& cfg) {
  if (norm) return rope ? launch_t<true, true>(a, cfg) : launch_t<true, false>(a, cfg);
  return rope ? launch_t<false, true>(a, cfg) : launch_t<false, false>(a, cfg);
}

}  // namespace mla
