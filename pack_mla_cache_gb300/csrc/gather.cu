// gather.cu -- context gather from the paged latent cache for sm_103a.
//
// What it computes: output row i of sequence s is the cache row of context
// position chunk_starts[s] + (i - cu_chunk_lens[s]), found through the block
// table, copied raw or widened exactly fp8 -> bf16 ("PR #51772
// [Attention][MLA] Fuse Kimi-K3 chunked-context K/V packing", Implementation
// item 2: _gather_context_latent, and item 5: the conditional cast to the
// kv_b_proj input dtype, fused here into the gather).
//
// Design: one warp per output row, 4 rows per warp per iteration with all
// their 16-byte loads issued before any store; the per-sequence prefix sums
// and chunk starts are staged once per CTA in shared memory (binary search
// there), so a row costs one block-table load and its cache row.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;
constexpr int kMaxChunks = 3;        // up to 96 x 16 B = 1536-byte rows
constexpr int kSmemSeqs = 1024;      // sequences staged in shared memory

// Largest s with cu[s] <= i, searched in cu[0..n]; -1 if none.
__device__ __forceinline__ int find_seq(const int32_t* cu, int n, int64_t i) {
  int lo = 0, hi = n + 1;  // invariant: cu[lo-1] <= i < cu[hi] (virtual ends)
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)cu[mid] <= i) lo = mid + 1;
    else hi = mid;
  }
  return lo - 1;
}

template <int MODE>  // 0: raw copy; kE4M3 / kE5M2: widen that fp8 format to bf16
__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherArgs a) {
  __shared__ int32_t s_cu[kSmemSeqs + 1];
  __shared__ int32_t s_st[kSmemSeqs];
  pdl_wait();
  const bool staged = a.num_seqs <= kSmemSeqs;
  if (staged) {
    for (int i = threadIdx.x; i <= a.num_seqs; i += kThreads) s_cu[i] = a.cu[i];
    for (int i = threadIdx.x; i < a.num_seqs; i += kThreads) s_st[i] = a.starts[i];
    __syncthreads();
  }
  const int32_t* cu = staged ? s_cu : a.cu;
  const int32_t* st = staged ? s_st : a.starts;

  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  uint32_t errbits = 0;

  for (int64_t r0 = warp * kRows; r0 < a.num_tokens; r0 += nwarps * kRows) {
    const uint8_t* src[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      src[k] = nullptr;
      const int64_t i = r0 + k;
      if (i >= a.num_tokens) continue;
      const int s = find_seq(cu, a.num_seqs, i);
      if (s < 0 || s >= a.num_seqs || i >= (int64_t)cu[s + 1]) continue;  // owned by no sequence
      const int64_t p = (int64_t)st[s] + (i - cu[s]);
      const int64_t kb = p >= 0 ? (a.bs_shift >= 0 ? (p >> a.bs_shift) : p / a.block_size) : -1;
      if (kb < 0 || kb >= a.bt_stride) {
        errbits |= kErrBlockOOB;
        continue;
      }
      const int32_t blk = a.block_table[(int64_t)s * a.bt_stride + kb];
      if (blk < 0 || (int64_t)blk >= a.num_blocks) {
        errbits |= kErrBlockOOB;
        continue;
      }
      const int64_t off = p - kb * a.block_size;
      src[k] = a.cache + (int64_t)blk * a.block_stride + off * a.entry_stride;
    }

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
        } else {
          st16(dst + ch * 32, fp8x8_to_bf16x8<MODE>(make_uint2(v[k][c].x, v[k][c].y)));
          st16(dst + ch * 32 + 16, fp8x8_to_bf16x8<MODE>(make_uint2(v[k][c].z, v[k][c].w)));
        }
      }
    }
  }
  errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
  if (errbits && lane == 0 && a.err) atomicOr(a.err, errbits);
  pdl_trigger();
}

template <int MODE>
cudaError_t launch_t(const GatherArgs& a, const LaunchCfg& cfg) {
  auto kern = gather_kernel<MODE>;
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

}  // namespace

cudaError_t launch_gather(const GatherArgs& a, int mode, const LaunchCfg& cfg) {
  switch (mode) {
    case 0: return launch_t<0>(a, cfg);
    case kE4M3: return launch_t<kE4M3>(a, cfg);
    case kE5M2: return launch_t<kE5M2>(a, cfg);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
