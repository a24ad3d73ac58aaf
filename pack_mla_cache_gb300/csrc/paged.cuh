// paged.cuh -- finding a chunk token's row in the paged latent cache, shared by
// the context gather and the pack that reads k_pe from the cache.
//
// Chunk token i belongs to the sequence s with cu[s] <= i < cu[s+1] (cu
// non-decreasing); its context position is starts[s] + i - cu[s], held at
// offset position % block_size of block block_table[s][position / block_size]
// ("PR #51772 [Attention][MLA] Fuse Kimi-K3 chunked-context K/V packing",
// Implementation item 2: _gather_context_latent over the block table).
//
// With fewer than 32 sequences each warp keeps cu and starts in its lanes and
// finds a token's sequence with one ballot, so a row costs one block-table
// load; more sequences use a binary search in global memory.
#pragma once

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

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

// Per-warp copy of the sequence table (used when num_seqs < 32).
struct SeqLanes {
  bool few;
  int32_t cu, st;  // lane l: cu[l] (l <= num_seqs) and starts[l] (l < num_seqs)
};

__device__ __forceinline__ SeqLanes load_seq_lanes(const PagedSrc& p, int lane) {
  SeqLanes sl{p.num_seqs < 32, 0, 0};
  if (sl.few) {
    if (lane <= p.num_seqs) sl.cu = p.cu[lane];
    if (lane < p.num_seqs) sl.st = p.starts[lane];
  }
  return sl;
}

// Start of chunk token i's cache row, or nullptr when no sequence owns i or
// its block index / block id is out of range (the latter ORs kErrBlockOOB
// into errbits).  All 32 lanes must call it together with the same i.
__device__ __forceinline__ const uint8_t* paged_row(const PagedSrc& p, const SeqLanes& sl,
                                                    int lane, int64_t i, uint32_t& errbits) {
  int s;
  int64_t c0, c1, st;
  if (sl.few) {
    const unsigned m = __ballot_sync(0xFFFFFFFFu, lane <= p.num_seqs && (int64_t)sl.cu <= i);
    s = __popc(m) - 1;  // the largest s with cu[s] <= i
    c0 = __shfl_sync(0xFFFFFFFFu, sl.cu, s < 0 ? 0 : s);
    c1 = __shfl_sync(0xFFFFFFFFu, sl.cu, s + 1 > 31 ? 31 : s + 1);
    st = __shfl_sync(0xFFFFFFFFu, sl.st, s < 0 ? 0 : s);
  } else {
    s = find_seq(p.cu, p.num_seqs, i);
    c0 = s >= 0 ? p.cu[s] : 0;
    c1 = (s >= 0 && s < p.num_seqs) ? p.cu[s + 1] : 0;
    st = (s >= 0 && s < p.num_seqs) ? p.starts[s] : 0;
  }
  if (s < 0 || s >= p.num_seqs || i >= c1) return nullptr;  // owned by no sequence
  const int64_t pos = st + (i - c0);
  const int64_t kb = pos >= 0 ? (p.bs_shift >= 0 ? (pos >> p.bs_shift) : pos / p.block_size) : -1;
  if (kb < 0 || kb >= p.bt_stride) {
    errbits |= kErrBlockOOB;
    return nullptr;
  }
  const int32_t blk = p.block_table[(int64_t)s * p.bt_stride + kb];
  if (blk < 0 || (int64_t)blk >= p.num_blocks) {
    errbits |= kErrBlockOOB;
    return nullptr;
  }
  return p.cache + (int64_t)blk * p.block_stride + (pos - kb * p.block_size) * p.entry_stride;
}

}  // namespace mla
