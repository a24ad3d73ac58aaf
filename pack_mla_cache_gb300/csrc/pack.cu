// pack.cu -- chunked-context K/V pack for sm_103a: the bf16-input instances
// and the dispatch on the input format (kernel design: pack_kernel.cuh).
#include "pack_kernel.cuh"

namespace mla {

cudaError_t launch_pack_f16(const PackArgs& a, int out_fmt, int kpe_fmt, bool paged,
                            const GatherArgs* next_gather, int gather_mode,
                            const LaunchCfg& cfg);

cudaError_t launch_pack(const PackArgs& a, int in_fmt, int out_fmt, int kpe_fmt, bool paged,
                        const LaunchCfg& cfg, const GatherArgs* next_gather, int gather_mode) {
  if (in_fmt == kF16)
    return launch_pack_f16(a, out_fmt, kpe_fmt, paged, next_gather, gather_mode, cfg);
  if (in_fmt == kBF16)
    return launch_pack_in<kBF16>(a, out_fmt, kpe_fmt, paged, next_gather, gather_mode, cfg);
  return cudaErrorInvalidValue;
}

}  // namespace mla
