// rope_table.cu -- the rotary cos/sin table read by the insert's RoPE step.
//
// Row p holds cos(p * f_i) for i < rot/2, then sin(p * f_i), with
// f_i = base^(-2i/rot) -- the cached cos/sin of the rotary embedding that
// rotates k_pe ("PR #50585 [K3 Perf] Optimize k3 dspark fused kv", Source
// snippets: the RoPE of k_pe with positions repeated per layer).  Angles and
// their cos/sin are evaluated in double precision and rounded once to fp32, so
// positions up to 32768 (angles of ~3e4 rad) keep full fp32 accuracy.  Built
// once per model; not on the per-step path.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

__global__ void rope_table_kernel(float* __restrict__ out, int64_t max_position, int32_t rot_dim,
                                  double base) {
  pdl_trigger();
  pdl_wait();
  const int32_t half = rot_dim / 2;
  const int64_t n = max_position * half;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n;
       k += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = k / half;
    const int32_t i = (int32_t)(k - p * half);
    const double inv_freq = pow(base, -2.0 * (double)i / (double)rot_dim);
    const double theta = (double)p * inv_freq;
    double s, c;
    sincos(theta, &s, &c);
    out[p * rot_dim + i] = (float)c;
    out[p * rot_dim + half + i] = (float)s;
  }
}

}  // namespace

cudaError_t launch_rope_table(float* out, int64_t max_position, int32_t rot_dim, double base,
                              const LaunchCfg& cfg) {
  const int threads = 256;
  const int64_t work = (max_position * (rot_dim / 2) + threads - 1) / threads;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(capped_grid(reinterpret_cast<const void*>(rope_table_kernel), threads, work));
  lc.blockDim = dim3(threads);
  lc.stream = cfg.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = cfg.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, rope_table_kernel, out, max_position, rot_dim, base);
}

}  // namespace mla
