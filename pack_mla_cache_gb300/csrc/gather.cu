// gather.cu -- context gather from the paged latent cache for sm_103a: the
// kernel instances and their launch (what a row holds and the per-warp row
// loop: gather_rows.cuh).  The grid is capped at the resident CTAs and loops
// over the rows.  When the caller declares its tables complete before the
// call, a warp's first lookup is done before the programmatic-launch wait, so
// only the cache row load follows the previous kernel.
#include "mla_device.cuh"
#include "mla_internal.h"
#include "gather_rows.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;

template <int MODE, int OUT, bool SCALED>
__device__ __forceinline__ void gather_body(const GatherArgs& a) {
  const int lane = threadIdx.x & 31;
  uint32_t errbits = 0;
  gather_rows<MODE, OUT, SCALED>(a, ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5,
                                 ((int64_t)gridDim.x * kThreads) >> 5, lane, errbits);
  errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
  if (errbits && lane == 0 && a.err) atomicOr(a.err, errbits);
}

// The copy and the exact widening fit in 32 registers, so 8 CTAs (64 warps,
// one row in flight each) run per SM: 131072 rows widened to bf16 in 41.8 us
// against 45.0 us at 37 registers (6 CTAs).
template <int MODE, int OUT>
__global__ void __launch_bounds__(kThreads, 8) gather_kernel(const GatherArgs a) {
  pdl_trigger();
  gather_body<MODE, OUT, false>(a);
}

// The dequantising widening keeps its 40 registers (6 CTAs per SM): held to
// 32 it spills and ran 47.9 against 45.4 us for 131072 rows.
template <int MODE>
__global__ void __launch_bounds__(kThreads) gather_scaled_kernel(const GatherArgs a) {
  pdl_trigger();
  gather_body<MODE, kBF16, true>(a);
}

template <int MODE, int OUT, bool SCALED>
cudaError_t launch_t(const GatherArgs& a, const LaunchCfg& cfg) {
  void (*kern)(const GatherArgs);
  if constexpr (SCALED) kern = gather_scaled_kernel<MODE>;
  else kern = gather_kernel<MODE, OUT>;
  const int64_t warps = ((int64_t)a.num_tokens + kGatherRows - 1) / kGatherRows;
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
