// pack_f16.cu -- chunked-context K/V pack for sm_103a: the fp16-input
// instances ("PR #51772 [Attention][MLA] Fuse Kimi-K3 chunked-context K/V
// packing", Review: the fused kernel is tested with bf16 and fp16 inputs).
#include "pack_kernel.cuh"

namespace mla {

cudaError_t launch_pack_f16(const PackArgs& a, int out_fmt, int kpe_fmt, bool paged,
                            const GatherArgs* next_gather, int gather_mode,
                            const LaunchCfg& cfg) {
  return launch_pack_in<kF16>(a, out_fmt, kpe_fmt, paged, next_gather, gather_mode, cfg);
}

}  // namespace mla
