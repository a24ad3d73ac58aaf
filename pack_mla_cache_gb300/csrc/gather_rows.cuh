// gather_rows.cuh -- the context gather's per-warp row loop, shared by the
// gather kernel (gather.cu) and the pack launch that also gathers the next
// chunk's latent rows (pack_kernel.cuh).
//
// What it computes: output row i of sequence s is the cache row of context
// position chunk_starts[s] + (i - cu_chunk_lens[s]), found through the block
// table, copied raw or widened fp8 -> bf16 / fp16 ("PR #51772 [Attention][MLA]
// Fuse Kimi-K3 chunked-context K/V packing", Implementation item 2:
// _gather_context_latent, and item 5: the conditional cast to the kv_b_proj
// input dtype, fused here into the gather).  The widening is exact, or
// dequantising: the fp8 value times k_scale as one fp32 product, rounded to
// bf16 (for caches written with a k_scale other than 1, "PR #55356 [Kimi Perf]
// Group fp8 mla cache insertion", Source snippets: scaled_convert).
//
// Design: one warp per output row (rows warp, warp + nwarps, ...), loads
// issued before stores; the row lookup (paged.cuh) costs a ballot and one
// block-table load.  A chunk of 8192 rows is latency-bound (sequence table ->
// block table -> row), so as many warps as rows wins: 3.6 us per 8192-row
// chunk against 4.9 us with 4 rows per warp; at 262144 rows both run at
// ~5.9 TB/s.  The widening forms read 8-byte units of the fp8 row, so each
// lane's 16-byte output lands next to its neighbours' and a warp store writes
// 512 contiguous bytes (16-byte units made two stores of 16 bytes at a 32-byte
// stride: 131072 rows widened to bf16 58.3 vs 63.9 us, dequantised 45.4 vs
// 50.7 us).
#pragma once

#include "mla_device.cuh"
#include "mla_internal.h"
#include "paged.cuh"

namespace mla {

constexpr int kGatherRows = 1;       // rows per warp per iteration
constexpr int kGatherMaxChunks = 3;  // up to 96 x 16 B = 1536-byte rows

// The rows of one warp.  MODE 0: raw copy; kE4M3 / kE5M2: widen that fp8
// format to OUT (bf16 or fp16; bf16 times the dequantisation scale when
// SCALED).  Waits for the previous grid (programmatic dependent launch) itself;
// ORs skipped rows' error bits into errbits.  All 32 lanes call it together.
template <int MODE, int OUT, bool SCALED>
__device__ __forceinline__ void gather_rows(const GatherArgs& a, int64_t warp, int64_t nwarps,
                                            int lane, uint32_t& errbits) {
  // The first row's lookup reads only the sequence and block tables.  When the
  // caller has declared them complete before the call (early_tables), it runs
  // before the wait on the previous grid, so two of the three dependent loads
  // of a row overlap that grid's tail; otherwise after it (plain stream order;
  // the second wait below is then a no-op).  Each later lookup is done at the
  // end of the previous iteration (the loop is rotated), which keeps the
  // register count of the plain loop.
  if (!a.early_tables) pdl_wait();
  const SeqLanes sl = load_seq_lanes(a.src, lane);
  int64_t r = warp;
  const uint8_t* src = r < a.num_tokens ? paged_row(a.src, sl, lane, r, errbits) : nullptr;
  pdl_wait();
  uint64_t s2 = 0;
  if constexpr (SCALED) {
    const float sc = *a.dequant_scale;
    s2 = f2(sc, sc);
  }
  if constexpr (MODE != 0) {
    // widening: 8-byte input units (up to 192 per row)
    constexpr int kU = 2 * kGatherMaxChunks;
    const int units = 2 * a.row_chunks;
    while (r < a.num_tokens) {
      uint2 v[kU];
#pragma unroll
      for (int c = 0; c < kU; ++c) {
        const int ch = lane + 32 * c;
        v[c] = make_uint2(0, 0);
        if (src && ch < units) v[c] = ld_stream8(src + ch * 8);
      }
      if (src) {
        uint8_t* dst = a.out + r * a.out_rs;
#pragma unroll
        for (int c = 0; c < kU; ++c) {
          const int ch = lane + 32 * c;
          if (ch >= units) continue;
          if constexpr (SCALED) st16(dst + ch * 16, fp8x8_to_bf16x8_scaled<MODE>(v[c], s2));
          else st16(dst + ch * 16, fp8x8_to_x16x8<MODE, OUT>(v[c]));
        }
      }
      r += nwarps;
      src = r < a.num_tokens ? paged_row(a.src, sl, lane, r, errbits) : nullptr;
    }
  } else {
    // raw copy: 16-byte units (up to 96 per row)
    while (r < a.num_tokens) {
      uint4 v[kGatherMaxChunks];
#pragma unroll
      for (int c = 0; c < kGatherMaxChunks; ++c) {
        const int ch = lane + 32 * c;
        v[c] = make_uint4(0, 0, 0, 0);
        if (src && ch < a.row_chunks) v[c] = ld_stream16(src + ch * 16);
      }
      if (src) {
        uint8_t* dst = a.out + r * a.out_rs;
#pragma unroll
        for (int c = 0; c < kGatherMaxChunks; ++c) {
          const int ch = lane + 32 * c;
          if (ch < a.row_chunks) st16(dst + ch * 16, v[c]);
        }
      }
      r += nwarps;
      src = r < a.num_tokens ? paged_row(a.src, sl, lane, r, errbits) : nullptr;
    }
  }
}

}  // namespace mla
