// pack.cu -- chunked-context K/V pack for sm_103a.
//
// What it computes: the contiguous full key [k_nope | k_pe] (k_pe broadcast to
// every head) and the contiguous V from the strided kv_b_proj output and a
// k_pe that may still be fp8 from the cache, in bf16 or fp8 ("PR #51772
// [Attention][MLA] Fuse Kimi-K3 chunked-context K/V packing", Implementation
// item 1 and Source snippets: fused_mla_kv_concat /
// fused_mla_kv_concat_quant_fp8).
//
// Work item: one token's group of up to 8 heads (4 KB of k_nope + v), so a
// 16-head token is two items.  Two variants compute identical results:
//
//   * pack_tma_kernel (the layout the kv_b_proj GEMM produces: each token's
//     heads' [k_nope | v] rows back to back) -- a producer warp streams each
//     item's contiguous block and the token's k_pe row into a ring of 32
//     shared-memory stages with cp.async.bulk (completion counted in bytes on a
//     per-stage mbarrier; each of its lanes fills its own stage, since one
//     issuing lane cannot keep a ring of 4 KB copies busy); 16 consumer warps
//     convert from shared memory and store.  Memory-level parallelism is set by the ring (32 stages of 4 KB per
//     SM), not by registers, so the conversion work of 16 warps overlaps the
//     copies of the following items.
//   * pack_kernel (any strides, no V, more than 16 heads) -- one warp per item,
//     its 8 16-byte loads per lane issued before the first store.
//
// Both: the grid is capped at the resident CTAs and loops over items (long
// contexts never grow the grid); lanes 0-15 write a head's k_nope slice and
// lanes 16-31 its V slice, 8 elements each, so every warp store is whole
// sectors; k_pe part (lane % 8) is loaded and converted once per item; fp8
// output uses the exact division by the scale (fast path chosen once per
// launch) and the hardware .satfinite converters; an fp8 k_pe is copied byte
// for byte; an fp8 k_pe into a bf16 key goes through the exact widening.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kNope = 128, kRope = 64, kV = 128, kKey = kNope + kRope;
constexpr int kGroup = 8;  // heads per work item

struct Item {
  int64_t t;
  int h0, nh;  // first head and head count of the item
};

__device__ __forceinline__ Item item_of(int64_t j, int groups, int H) {
  Item it;
  it.t = j / groups;
  const int g = (int)(j - it.t * groups);
  it.h0 = g * kGroup;
  it.nh = min(kGroup, H - it.h0);
  return it;
}

// The k_pe part of this lane (elements 8*(lane%8) .. +8) in the output format.
template <int OF, int KF, bool FAST>
__device__ __forceinline__ void pe_part(const uint4& x16, const uint2& x8, const DivConst& k,
                                        uint4& o16, uint2& o8) {
  if constexpr (KF == kBF16) {
    if constexpr (OF == kBF16) o16 = x16;
    else o8 = bf16x8_to_fp8x8<OF, FAST>(x16, k);
  } else {
    if constexpr (OF == kBF16) o16 = fp8x8_to_bf16x8<KF>(x8);
    else o8 = x8;  // same fp8 format: raw bytes
  }
}

// One head row (lane < 16: k_nope part `lane`; lane >= 16: v part lane-16).
template <int OF, bool FAST>
__device__ __forceinline__ void put_unit(uint8_t* dst, const uint4& x, const DivConst& k) {
  if constexpr (OF == kBF16) st16(dst, x);
  else st8(dst, bf16x8_to_fp8x8<OF, FAST>(x, k));
}

template <int OF>
__device__ __forceinline__ void put_pe(uint8_t* dst, const uint4& o16, const uint2& o8) {
  if constexpr (OF == kBF16) st16(dst, o16);
  else st8(dst, o8);
}

// ---- plain vectorised variant -------------------------------------------------
constexpr int kThreads = 256;

template <int OF, int KF, bool FAST>
__device__ __forceinline__ void pack_plain_items(const PackArgs& a, const DivConst& k) {
  constexpr int OE = (OF == kBF16) ? 2 : 1;
  const int lane = threadIdx.x & 31, H = a.num_heads;
  const int groups = (H + kGroup - 1) / kGroup;
  const int64_t n_items = (int64_t)a.num_tokens * groups;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const bool has_v = a.vout != nullptr;
  const int part_pe = lane & 7;
  const int half = lane >> 4, part = lane & 15;  // v half (lanes 16-31) / unit in the half
  for (int64_t j = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5; j < n_items; j += nwarps) {
    const Item it = item_of(j, groups, H);
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
    {
      const uint8_t* pe = a.k_pe + it.t * a.kpe_ts;
      uint4 x16 = make_uint4(0, 0, 0, 0);
      uint2 x8 = make_uint2(0, 0);
      if constexpr (KF == kBF16) x16 = ld_stream16(pe + part_pe * 16);
      else x8 = ld_stream8(pe + part_pe * 8);
      pe_part<OF, KF, FAST>(x16, x8, k, p16, p8);
    }
    uint8_t* key = a.key + (it.t * H + it.h0) * (int64_t)kKey * OE;
    uint8_t* dst = half ? a.vout + (it.t * H + it.h0) * (int64_t)kV * OE + part * 8 * OE
                        : key + part * 8 * OE;
    const int dstride = (half ? kV : kKey) * OE;
#pragma unroll
    for (int i = 0; i < kGroup; ++i)
      if (i < it.nh && (!half || has_v)) put_unit<OF, FAST>(dst + i * dstride, x[i], k);
    for (int u = lane; u < it.nh * 8; u += 32)
      put_pe<OF>(key + ((u >> 3) * kKey + kNope + part_pe * 8) * OE, p16, p8);
  }
}

template <int OF, int KF>
__global__ void __launch_bounds__(kThreads) pack_kernel(const PackArgs a) {
  pdl_trigger();
  pdl_wait();
  float scale = 1.0f;
  if constexpr (OF != kBF16) {
    if (a.out_scale) scale = *a.out_scale;
  }
  const DivConst k = div_const(scale);
  if constexpr (OF == kBF16) {
    pack_plain_items<OF, KF, true>(a, k);
  } else {
    if (k.fast) pack_plain_items<OF, KF, true>(a, k);
    else pack_plain_items<OF, KF, false>(a, k);
  }
}

// ---- bulk-copy pipeline variant ----------------------------------------------
// Each consumer warp owns the stages s == warp (mod kConsumers) and takes their
// fills in order, so a warp never waits on a stage more than one phase ahead
// of the fill it needs (an mbarrier parity wait cannot tell phases n and n+2
// apart).  Item i of a CTA goes to stage i % kStages and consumer i % kConsumers.
constexpr int kConsumers = 16;
constexpr int kStagesPerConsumer = 2;
constexpr int kStages = kConsumers * kStagesPerConsumer;
static_assert(kStages == 32, "producer lane s owns stage s");
constexpr int kTmaThreads = (kConsumers + 1) * 32;
constexpr int kStageBytes = kGroup * 512 + 128;  // 8 heads of [k_nope | v] + the k_pe row
constexpr int kTmaSmem = kStages * kStageBytes + 2 * kStages * 8 + 16;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: a wait that long means a fault

template <int OF, int KF, bool FAST>
__device__ __forceinline__ void pack_tma_consume(const PackArgs& a, const DivConst& k,
                                                 uint32_t stage0, uint32_t full0, uint32_t empty0,
                                                 int64_t n_local, int64_t G, volatile int* abort_flag) {
  constexpr int OE = (OF == kBF16) ? 2 : 1;
  constexpr uint32_t pe_off = kGroup * 512;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, H = a.num_heads;
  const int groups = (H + kGroup - 1) / kGroup;
  const int part_pe = lane & 7;
  const int half = lane >> 4, part = lane & 15;
  const int dstride = (half ? kV : kKey) * OE;
  for (int64_t i = warp; i < n_local; i += kConsumers) {
    const int s = (int)(i % kStages);
    if (!mbar_wait(full0 + 8 * s, (uint32_t)((i / kStages) & 1), kWaitLimitNs)) {
      *abort_flag = 1;
      break;
    }
    const Item it = item_of(blockIdx.x + G * i, groups, H);
    const uint32_t src = stage0 + (uint32_t)(s * kStageBytes);
    uint8_t* key = a.key + (it.t * H + it.h0) * (int64_t)kKey * OE;
    uint8_t* dst = half ? a.vout + (it.t * H + it.h0) * (int64_t)kV * OE + part * 8 * OE
                        : key + part * 8 * OE;
    if (it.nh == kGroup) {
#pragma unroll 4
      for (int j = 0; j < kGroup; ++j)
        put_unit<OF, FAST>(dst + j * dstride, lds16(src + j * 512 + lane * 16), k);
    } else {
      for (int j = 0; j < it.nh; ++j)
        put_unit<OF, FAST>(dst + j * dstride, lds16(src + j * 512 + lane * 16), k);
    }
    uint4 p16 = make_uint4(0, 0, 0, 0);
    uint2 p8 = make_uint2(0, 0);
    {
      uint4 x16 = make_uint4(0, 0, 0, 0);
      uint2 x8 = make_uint2(0, 0);
      if constexpr (KF == kBF16) x16 = lds16(src + pe_off + part_pe * 16);
      else x8 = lds8(src + pe_off + part_pe * 8);
      pe_part<OF, KF, FAST>(x16, x8, k, p16, p8);
    }
    for (int u = lane; u < it.nh * 8; u += 32)
      put_pe<OF>(key + ((u >> 3) * kKey + kNope + part_pe * 8) * OE, p16, p8);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
}

template <int OF, int KF>
__global__ void __launch_bounds__(kTmaThreads, 1) pack_tma_kernel(const PackArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr uint32_t pe_bytes = (KF == kBF16) ? 128u : 64u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kStages * kStageBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages);
  const uint32_t stage0 = smem_addr(smem);
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, H = a.num_heads;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  const int groups = (H + kGroup - 1) / kGroup;
  const int64_t n_items = (int64_t)a.num_tokens * groups;
  const int64_t G = gridDim.x, b = blockIdx.x;
  const int64_t n_local = n_items > b ? (n_items - 1 - b) / G + 1 : 0;
  int64_t fills = 0;  // producer lane: fills issued to its stage

  if (warp == kConsumers) {
    // ---------------- producer: lane s fills stage s -----------------------------
    // (one issuing lane sustains only about one bulk copy per ~270 cycles, so
    // all 32 lanes issue, each for its own stage)
    const int s = lane;
    for (int64_t i = lane; i < n_local; i += kStages) {
      const int64_t n = i / kStages;
      if (n > 0 && !mbar_wait(empty0 + 8 * s, (uint32_t)((n - 1) & 1), kWaitLimitNs)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      const Item it = item_of(b + G * i, groups, H);
      const uint32_t dst = stage0 + (uint32_t)(s * kStageBytes);
      const uint32_t block = (uint32_t)it.nh * 512u;
      mbar_arrive_expect_tx(full0 + 8 * s, block + pe_bytes);
      bulk_g2s(dst, a.k_nope + it.t * a.kn_ts + (int64_t)it.h0 * 512, block, full0 + 8 * s);
      bulk_g2s(dst + kGroup * 512, a.k_pe + it.t * a.kpe_ts, pe_bytes, full0 + 8 * s);
      fills = n + 1;
    }
  } else {
    // ---------------- consumers --------------------------------------------------
    float scale = 1.0f;
    if constexpr (OF != kBF16) {
      if (a.out_scale) scale = *a.out_scale;
    }
    const DivConst k = div_const(scale);
    if constexpr (OF == kBF16) {
      pack_tma_consume<OF, KF, true>(a, k, stage0, full0, empty0, n_local, G, abort_flag);
    } else {
      if (k.fast)
        pack_tma_consume<OF, KF, true>(a, k, stage0, full0, empty0, n_local, G, abort_flag);
      else
        pack_tma_consume<OF, KF, false>(a, k, stage0, full0, empty0, n_local, G, abort_flag);
    }
  }
  __syncthreads();
  if (*abort_flag) {
    // Let every copy this CTA issued land before its shared memory is released
    // (a stage's phases complete in order, so its last fill is enough).
    if (warp == kConsumers && fills > 0)
      (void)mbar_wait(full0 + 8 * lane, (uint32_t)((fills - 1) & 1), kWaitLimitNs / 8);
    if (threadIdx.x == 0 && a.err) atomicOr(a.err, kErrTimeout);
  }
}

cudaLaunchConfig_t base_cfg(const LaunchCfg& cfg, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t lc = {};
  lc.stream = cfg.stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = cfg.pdl ? 1 : 0;
  return lc;
}

template <int OF, int KF>
cudaError_t launch_tma_t(const PackArgs& a, const LaunchCfg& cfg) {
  auto kern = pack_tma_kernel<OF, KF>;
  static bool configured = false;  // per instance
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t items = (int64_t)a.num_tokens * ((a.num_heads + kGroup - 1) / kGroup);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = base_cfg(cfg, attr);
  lc.gridDim = dim3(capped_grid(reinterpret_cast<const void*>(kern), kTmaThreads,
                                (items + kConsumers - 1) / kConsumers, kTmaSmem));
  lc.blockDim = dim3(kTmaThreads);
  lc.dynamicSmemBytes = kTmaSmem;
  return cudaLaunchKernelEx(&lc, kern, a);
}

template <int OF, int KF>
cudaError_t launch_plain_t(const PackArgs& a, const LaunchCfg& cfg) {
  auto kern = pack_kernel<OF, KF>;
  const int64_t items = (int64_t)a.num_tokens * ((a.num_heads + kGroup - 1) / kGroup);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = base_cfg(cfg, attr);
  lc.gridDim = dim3(capped_grid(reinterpret_cast<const void*>(kern), kThreads,
                                (items + kThreads / 32 - 1) / (kThreads / 32)));
  lc.blockDim = dim3(kThreads);
  return cudaLaunchKernelEx(&lc, kern, a);
}

// The bulk-copy variant needs the interleaved [k_nope | v] head rows, a V
// output and 16-byte aligned k_pe rows (bulk copies move 16-byte multiples
// between 16-byte aligned addresses).
bool tma_layout(const PackArgs& a) {
  return a.vout != nullptr && a.v == a.k_nope + 256 && a.kn_hs == 512 && a.v_hs == 512 &&
         a.v_ts == a.kn_ts && (reinterpret_cast<uintptr_t>(a.k_pe) & 15) == 0 &&
         (a.kpe_ts & 15) == 0;
}

template <int OF, int KF>
cudaError_t launch_variant(const PackArgs& a, const LaunchCfg& cfg) {
  if (a.use_tma && tma_layout(a)) return launch_tma_t<OF, KF>(a, cfg);
  return launch_plain_t<OF, KF>(a, cfg);
}

template <int OF>
cudaError_t launch_kpe(const PackArgs& a, int kpe_fmt, const LaunchCfg& cfg) {
  if (kpe_fmt == kBF16) return launch_variant<OF, kBF16>(a, cfg);
  if constexpr (OF == kBF16 || OF == kE4M3) {
    if (kpe_fmt == kE4M3) return launch_variant<OF, kE4M3>(a, cfg);
  }
  if constexpr (OF == kBF16 || OF == kE5M2) {
    if (kpe_fmt == kE5M2) return launch_variant<OF, kE5M2>(a, cfg);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_pack(const PackArgs& a, int out_fmt, int kpe_fmt, const LaunchCfg& cfg) {
  switch (out_fmt) {
    case kBF16: return launch_kpe<kBF16>(a, kpe_fmt, cfg);
    case kE4M3: return launch_kpe<kE4M3>(a, kpe_fmt, cfg);
    case kE5M2: return launch_kpe<kE5M2>(a, kpe_fmt, cfg);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
