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
// their 16-byte loads issued before any store.  With fewer than 32 sequences
// each warp keeps the prefix sums and chunk starts in its lanes and finds a
// row's sequence with one ballot, so a row costs one block-table load and its
// cache row; more sequences use a binary search in global memory.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;
constexpr int kMaxChunks = 3;        // up to 96 x 16 B = 1536-byte rows

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
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  // Up to 31 sequences: lane l holds cu[l] and starts[l], and a row's sequence
  // is found with one ballot (no shared-memory staging, no block barrier).
  const bool few = a.num_seqs < 32;
  int32_t my_cu = 0, my_st = 0;
  if (few) {
    if (lane <= a.num_seqs) my_cu = a.cu[lane];
    if (lane < a.num_seqs) my_st = a.starts[lane];
  }
  uint32_t errbits = 0;

  for (int64_t r0 = warp * kRows; r0 < a.num_tokens; r0 += nwarps * kRows) {
    const uint8_t* src[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      src[k] = nullptr;
      const int64_t i = r0 + k;
      if (i >= a.num_tokens) continue;
      int s;
      int64_t c0, c1, st;
      if (few) {
        const unsigned m = __ballot_sync(0xFFFFFFFFu, lane <= a.num_seqs && (int64_t)my_cu <= i);
        s = __popc(m) - 1;  // the largest s with cu[s] <= i (cu non-decreasing)
        c0 = __shfl_sync(0xFFFFFFFFu, my_cu, s < 0 ? 0 : s);
        c1 = __shfl_sync(0xFFFFFFFFu, my_cu, s + 1 > 31 ? 31 : s + 1);
        st = __shfl_sync(0xFFFFFFFFu, my_st, s < 0 ? 0 : s);
      } else {
        s = find_seq(a.cu, a.num_seqs, i);
        c0 = s >= 0 ? a.cu[s] : 0;
        c1 = (s >= 0 && s < a.num_seqs) ? a.cu[s + 1] : 0;
        st = (s >= 0 && s < a.num_seqs) ? a.starts[s] : 0;
      }
      if (s < 0 || s >= a.num_seqs || i >= c1) continue;  // owned by no sequence
      const int64_t p = st + (i - c0);
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
