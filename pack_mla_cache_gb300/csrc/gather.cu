// gather.cu -- context gather from the paged latent cache for sm_103a.
//
// What it computes: output row i of sequence s is the cache row of context
// position chunk_starts[s] + (i - cu_chunk_lens[s]), found through the block
// table, copied raw or widened fp8 -> bf16 / fp16 ("PR #51772 [Attention][MLA] Fuse
// Kimi-K3 chunked-context K/V packing", Implementation item 2:
// _gather_context_latent, and item 5: the conditional cast to the kv_b_proj
// input dtype, fused here into the gather).  The widening is exact, or
// dequantising: the fp8 value times k_scale as one fp32 product, rounded to
// bf16 (for caches written with a k_scale other than 1, "PR #55356 [Kimi Perf]
// Group fp8 mla cache insertion", Source snippets: scaled_convert).
//
// Design: one warp per output row (kRows per iteration, loads issued before
// stores); the row lookup (paged.cuh) costs a ballot and one block-table load.
// A chunk of 8192 rows is latency-bound (sequence table -> block table -> row),
// so as many warps as rows wins: 3.6 us per 8192-row chunk against 4.9 us with
// 4 rows per warp; at 262144 rows both run at ~5.9 TB/s.  When the caller
// declares its tables complete before the call, a warp's first lookup is done
// before the programmatic-launch wait, so only the cache row load follows the
// previous kernel.
#include "mla_device.cuh"
#include "mla_internal.h"
#include "paged.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 1;   // rows per warp per iteration (more warps beat more rows a warp)
constexpr int kMaxChunks = 3;        // up to 96 x 16 B = 1536-byte rows

// MODE 0: raw copy; kE4M3 / kE5M2: widen that fp8 format to OUT (bf16 or
// fp16; bf16 times the dequantisation scale when SCALED).
template <int MODE, int OUT, bool SCALED>
__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherArgs a) {
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  uint32_t errbits = 0;
  // The first rows' lookups read only the sequence and block tables.  When the
  // caller has declared them complete before the call (early_tables), they
  // run before the wait on the previous grid, so two of the three dependent
  // loads of a row overlap its tail; otherwise after it (plain stream order;
  // the second wait below is then a no-op).  Each later lookup is done at the
  // end of the previous iteration (the loop is rotated), which keeps the
  // register count of the plain loop.
  if (!a.early_tables) pdl_wait();
  const SeqLanes sl = load_seq_lanes(a.src, lane);
  const uint8_t* src[kRows];
#pragma unroll
  for (int k = 0; k < kRows; ++k) {
    const int64_t r = warp * kRows + k;
    src[k] = r < a.num_tokens ? paged_row(a.src, sl, lane, r, errbits) : nullptr;
  }
  pdl_wait();
  uint64_t s2 = 0;
  if constexpr (SCALED) {
    const float sc = *a.dequant_scale;
    s2 = f2(sc, sc);
  }

  for (int64_t r0 = warp * kRows; r0 < a.num_tokens;) {
    uint4 v[kRows][kMaxChunks];
#pragma unroll
    for (int k = 0; k < kRows; ++k)
#pragma unroll
      for (int c = 0; c < kMaxChunks; ++c) {
        const int ch = lane + 32 * c;
        v[k][c] = make_uint4(0, 0, 0, 0);
        if (src[k] && ch < a.row_chunks) v[k][c] = ld_stream16(src[k] + ch * 16);
      }

#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      if (!src[k]) continue;
      uint8_t* dst = a.out + (r0 + k) * a.out_rs;
#pragma unroll
      for (int c = 0; c < kMaxChunks; ++c) {
        const int ch = lane + 32 * c;
        if (ch >= a.row_chunks) continue;
        if constexpr (MODE == 0) {
          st16(dst + ch * 16, v[k][c]);
        } else if constexpr (SCALED) {
          st16(dst + ch * 32, fp8x8_to_bf16x8_scaled<MODE>(make_uint2(v[k][c].x, v[k][c].y), s2));
          st16(dst + ch * 32 + 16,
               fp8x8_to_bf16x8_scaled<MODE>(make_uint2(v[k][c].z, v[k][c].w), s2));
        } else {
          st16(dst + ch * 32, fp8x8_to_x16x8<MODE, OUT>(make_uint2(v[k][c].x, v[k][c].y)));
          st16(dst + ch * 32 + 16, fp8x8_to_x16x8<MODE, OUT>(make_uint2(v[k][c].z, v[k][c].w)));
        }
      }
    }
    r0 += nwarps * kRows;
#pragma unroll
    for (int k = 0; k < kRows; ++k)
      src[k] = r0 + k < a.num_tokens ? paged_row(a.src, sl, lane, r0 + k, errbits) : nullptr;
  }
  errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
  if (errbits && lane == 0 && a.err) atomicOr(a.err, errbits);
}

template <int MODE, int OUT, bool SCALED>
cudaError_t launch_t(const GatherArgs& a, const LaunchCfg& cfg) {
  auto kern = gather_kernel<MODE, OUT, SCALED>;
  const int64_t warps = ((int64_t)a.num_tokens + kRows - 1) / kRows;
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

template <int MODE>
cudaError_t launch_widen(const GatherArgs& a, int out_fmt, const LaunchCfg& cfg) {
  if (a.dequant_scale)
    return out_fmt == kBF16 ? launch_t<MODE, kBF16, true>(a, cfg) : cudaErrorInvalidValue;
  if (out_fmt == kBF16) return launch_t<MODE, kBF16, false>(a, cfg);
  if (out_fmt == kF16) return launch_t<MODE, kF16, false>(a, cfg);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gather(const GatherArgs& a, int mode, int out_fmt, const LaunchCfg& cfg) {
  switch (mode) {
    case 0: return launch_t<0, kBF16, false>(a, cfg);
    case kE4M3: return launch_widen<kE4M3>(a, out_fmt, cfg);
    case kE5M2: return launch_widen<kE5M2>(a, out_fmt, cfg);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
