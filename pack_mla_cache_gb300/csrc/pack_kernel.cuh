// pack_kernel.cuh -- the chunked-context K/V pack kernel templates, included by
// one translation unit per 16-bit input format (pack.cu: bf16, pack_f16.cu:
// fp16) so the instances compile in parallel.
//
// What it computes: the contiguous full key [k_nope | k_pe] (k_pe broadcast to
// every head) and the contiguous V from the strided kv_b_proj output and a
// k_pe that may still be fp8 from the cache, in the input's 16-bit format (bf16
// or fp16) or fp8 ("PR #51772
// [Attention][MLA] Fuse Kimi-K3 chunked-context K/V packing", Implementation
// item 1 and Source snippets: fused_mla_kv_concat /
// fused_mla_kv_concat_quant_fp8).
//
// Design: a work item is one token's group of up to 4 heads (2 KB of k_nope +
// v), so a 16-head token is four items; one warp per item, its 4 16-byte loads
// per lane issued before the first store.  Smaller items mean fewer registers,
// more resident warps and a shorter tail: 19.7 vs 20.2 us per 8192-token chunk
// in the benchmark's step with 8-head items, 22.1 us with 2-head items;
// staging the items through shared memory with bulk copies measured slower
// still (19.8 vs 17.6 us per chunk against the 8-head plain kernel).  The grid
// is capped at the resident CTAs and loops over items (long contexts never
// grow the grid); lanes 0-15 write a head's
// k_nope slice and lanes 16-31 its V slice, 8 elements each, so every warp
// store is whole sectors; k_pe part (lane % 8) is loaded and converted once
// per item; fp8 output uses the exact division by the scale (fast path chosen
// once per launch) and the hardware .satfinite converters; an fp8 k_pe is
// copied byte for byte; an fp8 k_pe into a 16-bit key goes through the exact
// widening.  Any strides, no-V packs and any head count take the same kernel.
//
// The paged form reads each token's k_pe straight from the paged cache (the
// row the context gather would fetch, paged.cuh), so the gather workspace only
// needs the kv_c columns; a token whose row is not found keeps its key's rope
// slice and, for a bad block index or id, sets MLA_ERRBIT_BLOCK_OOB.
#pragma once

#include <algorithm>

#include "mla_device.cuh"
#include "mla_internal.h"
#include "gather_rows.cuh"
#include "paged.cuh"

namespace mla {
namespace {

constexpr int kNope = 128, kRope = 64, kV = 128, kKey = kNope + kRope;
// Heads per work item: 4 for the plain pack; 8 for the paged one, whose
// per-item row lookup is then shared by twice as many heads (76.5 vs 70.3 us
// for 32768 tokens under the profiler with 4- and 8-head items).
template <bool PAGED>
constexpr int group_of() { return PAGED ? 8 : 4; }

struct Item {
  int64_t t;
  int h0, nh;  // first head and head count of the item
};

// Item j -> (token, head group).  Item counts stay below 2^32 (checked by the
// host), so 32-bit division suffices; a power-of-two group count (gshift >= 0,
// e.g. 4 groups of 16 heads) is a shift.
template <int kGroup>
__device__ __forceinline__ Item item_of(int64_t j, int groups, int gshift, int H) {
  Item it;
  const uint32_t ju = (uint32_t)j;
  it.t = gshift >= 0 ? (int64_t)(ju >> gshift) : (int64_t)(ju / (uint32_t)groups);
  const int g = (int)(ju - (uint32_t)it.t * (uint32_t)groups);
  it.h0 = g * kGroup;
  it.nh = min(kGroup, H - it.h0);
  return it;
}

// The k_pe part of this lane (elements 8*(lane%8) .. +8) in the output format.
// A 16-bit k_pe has the input format IF.
template <int OF, int KF, int IF, bool FAST>
__device__ __forceinline__ void pe_part(const uint4& x16, const uint2& x8, const DivConst& k,
                                        uint4& o16, uint2& o8) {
  if constexpr (is16(KF)) {
    if constexpr (is16(OF)) o16 = x16;
    else o8 = x16x8_to_fp8x8<OF, IF, FAST>(x16, k);
  } else {
    if constexpr (is16(OF)) o16 = fp8x8_to_x16x8<KF, OF>(x8);
    else o8 = x8;  // same fp8 format: raw bytes
  }
}

// One head row (lane < 16: k_nope part `lane`; lane >= 16: v part lane-16).
template <int OF, int IF, bool FAST>
__device__ __forceinline__ void put_unit(uint8_t* dst, const uint4& x, const DivConst& k) {
  if constexpr (is16(OF)) st16(dst, x);
  else st8(dst, x16x8_to_fp8x8<OF, IF, FAST>(x, k));
}

template <int OF>
__device__ __forceinline__ void put_pe(uint8_t* dst, const uint4& o16, const uint2& o8) {
  if constexpr (is16(OF)) st16(dst, o16);
  else st8(dst, o8);
}

// ---- plain vectorised variant -------------------------------------------------
constexpr int kThreads = 256;

// The items of one warp: warp0, warp0 + nwarps, ...
template <int OF, int KF, int IF, bool FAST, bool PAGED>
__device__ __forceinline__ void pack_plain_items(const PackArgs& a, const DivConst& k,
                                                 int64_t warp0, int64_t nwarps) {
  constexpr int OE = is16(OF) ? 2 : 1;
  constexpr int kGroup = group_of<PAGED>();
  const int lane = threadIdx.x & 31, H = a.num_heads;
  const int groups = (H + kGroup - 1) / kGroup;
  const int gshift = (groups & (groups - 1)) ? -1 : __ffs(groups) - 1;
  const int64_t n_items = (int64_t)a.num_tokens * groups;
  const bool has_v = a.vout != nullptr;
  const int part_pe = lane & 7;
  const int half = lane >> 4, part = lane & 15;  // v half (lanes 16-31) / unit in the half
  SeqLanes sl{};
  if constexpr (PAGED) sl = load_seq_lanes(a.paged, lane);
  uint32_t errbits = 0;
  for (int64_t j = warp0; j < n_items; j += nwarps) {
    const Item it = item_of<kGroup>(j, groups, gshift, H);
    const uint8_t* pe;
    if constexpr (PAGED) {
      pe = paged_row(a.paged, sl, lane, it.t, errbits);
      if (pe) pe += a.pe_off;
    } else {
      pe = a.k_pe + it.t * a.kpe_ts;
    }
    const uint8_t* src = (half ? a.v + it.t * a.v_ts : a.k_nope + it.t * a.kn_ts) + part * 16;
    const int64_t hs = half ? a.v_hs : a.kn_hs;
    uint4 x[kGroup];
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      x[i] = make_uint4(0, 0, 0, 0);
      if (i < it.nh && (!half || has_v)) x[i] = ld_stream16(src + (int64_t)(it.h0 + i) * hs);
    }
    uint4 p16 = make_uint4(0, 0, 0, 0);
    uint2 p8 = make_uint2(0, 0);
    if (!PAGED || pe) {
      uint4 x16 = make_uint4(0, 0, 0, 0);
      uint2 x8 = make_uint2(0, 0);
      if constexpr (is16(KF)) x16 = ld_stream16(pe + part_pe * 16);
      else x8 = ld_stream8(pe + part_pe * 8);
      pe_part<OF, KF, IF, FAST>(x16, x8, k, p16, p8);
    }
    uint8_t* key = a.key + (it.t * H + it.h0) * (int64_t)kKey * OE;
    uint8_t* dst = half ? a.vout + (it.t * H + it.h0) * (int64_t)kV * OE + part * 8 * OE
                        : key + part * 8 * OE;
    const int dstride = (half ? kV : kKey) * OE;
#pragma unroll
    for (int i = 0; i < kGroup; ++i)
      if (i < it.nh && (!half || has_v)) put_unit<OF, IF, FAST>(dst + i * dstride, x[i], k);
    if (!PAGED || pe)
      for (int u = lane; u < it.nh * 8; u += 32)
        put_pe<OF>(key + ((u >> 3) * kKey + kNope + part_pe * 8) * OE, p16, p8);
  }
  if constexpr (PAGED) {
    errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
    if (errbits && lane == 0 && a.err) atomicOr(a.err, errbits);
  }
}

// The pack's part of a launch: its warps are warp0, warp0 + nwarps, ...
// PREFETCH: first ask L2 for the warp's first item, whose loads are issued only
// after the scale has been read and the division form chosen, one memory
// latency later (in the launch that also gathers: 21.30 -> 21.12 us per chunk;
// the pack alone measured 19.36 -> 19.45 us, so it does not prefetch).
template <int OF, int KF, int IF, bool PAGED, bool PREFETCH = false>
__device__ __forceinline__ void pack_part(const PackArgs& a, int64_t warp0, int64_t nwarps) {
  pdl_wait();
  if constexpr (!PAGED && PREFETCH) {
    constexpr int kGroup = group_of<false>();
    const int groups = (a.num_heads + kGroup - 1) / kGroup;
    if (warp0 < (int64_t)a.num_tokens * groups) {
      const int lane = threadIdx.x & 31, half = lane >> 4, part = lane & 15;
      const int gshift = (groups & (groups - 1)) ? -1 : __ffs(groups) - 1;
      const Item it = item_of<kGroup>(warp0, groups, gshift, a.num_heads);
      const uint8_t* src =
          (half ? a.v + it.t * a.v_ts : a.k_nope + it.t * a.kn_ts) + part * 16;
      const int64_t hs = half ? a.v_hs : a.kn_hs;
      if (!half || a.vout) {
#pragma unroll
        for (int i = 0; i < kGroup; ++i)
          if (i < it.nh) prefetch_l2(src + (int64_t)(it.h0 + i) * hs);
      }
    }
  }
  float scale = 1.0f;
  if constexpr (!is16(OF)) {
    if (a.out_scale) scale = *a.out_scale;
  }
  const DivConst k = div_const(scale);
  if constexpr (is16(OF)) {
    pack_plain_items<OF, KF, IF, true, PAGED>(a, k, warp0, nwarps);
  } else {
    if (k.fast) pack_plain_items<OF, KF, IF, true, PAGED>(a, k, warp0, nwarps);
    else pack_plain_items<OF, KF, IF, false, PAGED>(a, k, warp0, nwarps);
  }
}

template <int OF, int KF, int IF, bool PAGED>
__global__ void __launch_bounds__(kThreads) pack_kernel(const PackArgs a) {
  pdl_trigger();
  pack_part<OF, KF, IF, PAGED>(a, ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5,
                               ((int64_t)gridDim.x * kThreads) >> 5);
}

// ---- the pack of one chunk and the gather of the next, one launch -------------
// In the chunk loop (gather chunk c -> kv_b_proj -> pack chunk c), the gather
// of chunk c + 1 depends only on the cache and its tables, so it can run in
// chunk c's pack launch (into the other of two workspaces): one launch per
// chunk instead of two.  Measured on the benchmark's chunks, each launch costs
// a fixed ~2.4 us (pack) or ~1.5 us (gather) on top of its bytes at 6.4 TB/s
// (ramp-up and drain around the programmatic-launch handoff); the gather's
// dependent row lookups also hide under the pack's streaming here.  The first
// gather_ctas CTAs gather (one row per warp per iteration, gather_rows.cuh),
// the others pack; gmode is 0 (raw copy) or the cache's fp8 format widened to
// the pack's 16-bit input format IF.
template <int OF, int KF, int IF>
__global__ void __launch_bounds__(kThreads) pack_gather_kernel(const PackArgs a,
                                                               const GatherArgs g,
                                                               int gather_ctas, int gmode) {
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  constexpr int kWarps = kThreads / 32;
  if ((int)blockIdx.x < gather_ctas) {
    uint32_t errbits = 0;
    const int64_t w = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gather_ctas * kWarps;
    if (gmode == kE4M3) gather_rows<kE4M3, IF, false>(g, w, nw, lane, errbits);
    else if (gmode == kE5M2) gather_rows<kE5M2, IF, false>(g, w, nw, lane, errbits);
    else gather_rows<0, IF, false>(g, w, nw, lane, errbits);
    errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
    if (errbits && lane == 0 && g.err) atomicOr(g.err, errbits);
    return;
  }
  pack_part<OF, KF, IF, false, true>(
      a, (int64_t)(blockIdx.x - gather_ctas) * kWarps + (threadIdx.x >> 5),
      (int64_t)(gridDim.x - gather_ctas) * kWarps);
}

// The split of a capped grid: the gather moves far fewer bytes but its rows
// are a chain of dependent loads, so it needs at least a seventh of the CTAs
// (an eighth made it the longer half: 22.3 against 21.0 us per chunk); the
// pack takes the rest, cut to the fewest warps that keep its items per warp
// (so its last round of items is full), the gather the CTAs that frees:
// 32768 items of an 8192-token chunk on 608 CTAs give 512 pack CTAs of 8
// items per warp and 96 gather CTAs (21.12 -> 20.86 us per chunk against a
// sixth of the grid, whose 507 pack CTAs left a last round 8% full).
constexpr int kGatherMinShareDiv = 7;

cudaLaunchConfig_t base_cfg(const LaunchCfg& cfg, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t lc = {};
  lc.stream = cfg.stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = cfg.pdl ? 1 : 0;
  return lc;
}

template <int OF, int KF, int IF, bool PAGED>
cudaError_t launch_plain_t(const PackArgs& a, const LaunchCfg& cfg) {
  auto kern = pack_kernel<OF, KF, IF, PAGED>;
  constexpr int kGroup = group_of<PAGED>();
  const int64_t items = (int64_t)a.num_tokens * ((a.num_heads + kGroup - 1) / kGroup);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = base_cfg(cfg, attr);
  lc.gridDim = dim3(capped_grid(reinterpret_cast<const void*>(kern), kThreads,
                                (items + kThreads / 32 - 1) / (kThreads / 32)));
  lc.blockDim = dim3(kThreads);
  return cudaLaunchKernelEx(&lc, kern, a);
}

template <int OF, int KF, int IF>
cudaError_t launch_pack_gather_t(const PackArgs& a, const GatherArgs& g, int gmode,
                                 const LaunchCfg& cfg) {
  auto kern = pack_gather_kernel<OF, KF, IF>;
  constexpr int kGroup = group_of<false>();
  constexpr int kWarps = kThreads / 32;
  const int64_t items = (int64_t)a.num_tokens * ((a.num_heads + kGroup - 1) / kGroup);
  const int64_t pack_ctas = (items + kWarps - 1) / kWarps;
  const int64_t gather_ctas = ((int64_t)g.num_tokens + kWarps - 1) / kWarps;
  const int resident = capped_grid(reinterpret_cast<const void*>(kern), kThreads,
                                   int64_t(1) << 30);
  int grid, gctas;
  if (pack_ctas + gather_ctas <= resident) {  // one wave: a warp per row and per item
    grid = (int)(pack_ctas + gather_ctas);
    gctas = (int)gather_ctas;
  } else {
    grid = resident;
    const int gmin = std::max(1, resident / kGatherMinShareDiv);
    const int64_t pmax = (int64_t)(resident - gmin) * kWarps;  // most pack warps
    const int64_t rounds = (items + pmax - 1) / pmax;           // items per pack warp
    const int64_t pwarps = (items + rounds - 1) / rounds;       // fewest warps for that
    const int pctas = (int)((pwarps + kWarps - 1) / kWarps);
    gctas = (int)std::min<int64_t>(gather_ctas, resident - pctas);
    if (pack_ctas < grid - gctas) grid = gctas + (int)pack_ctas;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = base_cfg(cfg, attr);
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(kThreads);
  return cudaLaunchKernelEx(&lc, kern, a, g, gctas, gmode);
}

// The leaf of the dispatch: the plain or paged pack, or (next_gather set; not
// paged) the pack with the next chunk's gather in the same launch.
template <int OF, int KF, int IF>
cudaError_t launch_variant(const PackArgs& a, bool paged, const GatherArgs* next_gather,
                           int gmode, const LaunchCfg& cfg) {
  if (next_gather) {
    if (paged) return cudaErrorInvalidValue;
    return launch_pack_gather_t<OF, KF, IF>(a, *next_gather, gmode, cfg);
  }
  return paged ? launch_plain_t<OF, KF, IF, true>(a, cfg)
               : launch_plain_t<OF, KF, IF, false>(a, cfg);
}

// Output OF of input IF: a 16-bit k_pe must have the input's format; an fp8
// k_pe is copied raw into an fp8 key of its own format or widened into a
// 16-bit key.
template <int OF, int IF>
cudaError_t launch_kpe(const PackArgs& a, int kpe_fmt, bool paged, const GatherArgs* ng,
                       int gmode, const LaunchCfg& cfg) {
  if (kpe_fmt == IF) return launch_variant<OF, IF, IF>(a, paged, ng, gmode, cfg);
  if constexpr (is16(OF) || OF == kE4M3) {
    if (kpe_fmt == kE4M3) return launch_variant<OF, kE4M3, IF>(a, paged, ng, gmode, cfg);
  }
  if constexpr (is16(OF) || OF == kE5M2) {
    if (kpe_fmt == kE5M2) return launch_variant<OF, kE5M2, IF>(a, paged, ng, gmode, cfg);
  }
  return cudaErrorInvalidValue;
}

// Every output format for one input format IF (a 16-bit output has IF's
// format).
template <int IF>
cudaError_t launch_pack_in(const PackArgs& a, int out_fmt, int kpe_fmt, bool paged,
                           const GatherArgs* ng, int gmode, const LaunchCfg& cfg) {
  switch (out_fmt) {
    case IF: return launch_kpe<IF, IF>(a, kpe_fmt, paged, ng, gmode, cfg);
    case kE4M3: return launch_kpe<kE4M3, IF>(a, kpe_fmt, paged, ng, gmode, cfg);
    case kE5M2: return launch_kpe<kE5M2, IF>(a, kpe_fmt, paged, ng, gmode, cfg);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace mla
