// insert.cu -- grouped multi-layer MLA cache insert for sm_103a.
//
// What it computes: for every (token, layer) row, [kv_c | k_pe] (bf16),
// optionally RMSNorm-ed / RoPE-rotated, is written raw (bf16 cache) or as
// fp8(value / k_scale[layer]) into the paged cache of its layer at the row
// named by slot_mapping -- all layers in one launch ("PR #55356 [Kimi Perf]
// Group fp8 mla cache insertion", Source snippets: the grouped kernel; the
// norm and rotation are those of "PR #50585 [K3 Perf] Optimize k3 dspark fused
// kv", Source snippets: _precompute_fused_context_kv).
//
// Design (not the pages' one-CTA-per-(token, layer) scalar loop):
//   * one warp per row.  kv_c: lane l holds elements [8l, 8l+8) and
//     [256+8l, 256+8l+8) -- two fully coalesced 512-byte warp loads; the fp8
//     stores are two 256-byte warp stores, the bf16 stores two 512-byte ones.
//     k_pe: lane l holds the neox pair (l, l+32), so the rotation needs no
//     shuffle and every lane does one pair;
//   * RMSNorm: 16 squares per lane on mixed-precision bf16 x bf16 + fp32 FMAs,
//     a 5-step xor-shuffle sum, a correctly rounded reciprocal square root
//     (norm_rope.cuh);
//   * RoPE: each rotated element is a difference of two products with an FMA
//     error correction (two-ulp accurate even when the products cancel);
//   * fp8: a correctly rounded division per element on packed fp32x2 pairs
//     (one reciprocal per row), then the hardware .satfinite pairwise
//     converter;
//   * two launch shapes: one warp per (token, layer) row, rows in token-major
//     order, for any strides (e.g. the [T, L, 576] projection read in place)
//     and for small batches; from 40960 rows with RMSNorm (131072 without),
//     dense layer-major rows run the bulk-copy pipeline (below), which only
//     pays once its ring is full for long (RMSNorm + RoPE, 5 layers, ring vs
//     rows: 8192 tokens 16.8 vs 19.1 us, 16384 35.6 vs 36.3, 24576 49.9 vs
//     53.6; raw: 8192 12.7 vs 14.5, 16384 28.6 vs 26.0, 24576 39.7 vs 41.5);
//     both loop over a grid capped at the resident-CTA count;
//   * dtype, norm and rope are template parameters: no runtime format branches
//     in the hot loop.
#include <atomic>

#include "mla_device.cuh"
#include "mla_internal.h"
#include "norm_rope.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kR = 512;  // kv_lora_rank
constexpr int kP = 64;   // pe_dim

constexpr int kMaxLayers = 128;

struct RowIn {
  uint4 x0, x1;     // kv_c elements [8l, 8l+8) and [256+8l, 256+8l+8)
  uint32_t pe;      // k_pe elements l (low half) and l+32 (high half)
  int64_t slot;
};

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) {
  return __ldcs(reinterpret_cast<const unsigned short*>(p));
}
__device__ __forceinline__ void st_u16(uint8_t* p, uint32_t v) {
  *reinterpret_cast<unsigned short*>(p) = static_cast<unsigned short>(v);
}
__device__ __forceinline__ void st_u8(uint8_t* p, uint32_t v) { *p = static_cast<uint8_t>(v); }

template <int F, bool ROPE>
__device__ __forceinline__ void load_row(const InsertArgs& a, int64_t t, int l, int lane,
                                         RowIn& r) {
  const uint8_t* src = a.kv_c + t * a.kvc_ts + (int64_t)l * a.kvc_ls;
  r.x0 = ld_stream16(src + lane * 16);
  r.x1 = ld_stream16(src + 512 + lane * 16);
  const uint8_t* pe = a.k_pe + t * a.kpe_ts + (int64_t)l * a.kpe_ls;
  r.pe = ld_u16(pe + lane * 2) | (ld_u16(pe + 64 + lane * 2) << 16);
  r.slot = a.slots[(int64_t)l * a.slot_ls + t];
}

// Store one finished row: bf16 words y0 / y1 (kv_c) and p (k_pe pair), raw
// into a bf16 cache or divided by `scale` and converted into an fp8 cache.
template <int F, bool FAST>
__device__ __forceinline__ void write_row_k(uint8_t* dst, int lane, const uint4& y0,
                                            const uint4& y1, uint32_t p, const DivConst& k) {
  if constexpr (F == kBF16) {
    st16(dst + lane * 16, y0);
    st16(dst + 512 + lane * 16, y1);
    st_u16(dst + 2 * kR + lane * 2, p);
    st_u16(dst + 2 * kR + kP + lane * 2, p >> 16);
  } else {
    st8(dst + lane * 8, bf16x8_to_fp8x8<F, FAST>(y0, k));
    st8(dst + 256 + lane * 8, bf16x8_to_fp8x8<F, FAST>(y1, k));
    const uint32_t q = bf16x2_to_fp8x2<F, FAST>(p, k);
    st_u8(dst + kR + lane, q);
    st_u8(dst + kR + kP / 2 + lane, q >> 8);
  }
}

// write_row_k for normalised kv_c words that hold -y (scale16<true>): the
// exact division's fast path starts from the negated input (div2_fast), so the
// per-pair negation is skipped; rows with special values take the guarded
// path on the restored words.  1.3% faster insert with RMSNorm (130.0 vs
// 131.7 us for 65536 tokens x 5 layers).
//
// CHECK false: the caller knows no value can make the first quotient overflow
// (normalised rows of a layer whose bound allows it, see layer_needs_check), so
// the special-value test of each 8 values is skipped (5 of 119 us for 65536
// tokens x 5 layers); a zero or NaN still takes the fast path correctly.
template <int F, bool CHECK = true>
__device__ __forceinline__ uint2 neg_bf16x8_to_fp8x8(uint4 v, const DivConst& k) {
  bool fast = true;
  if constexpr (CHECK) {
    const uint32_t m = umax16x2(umax16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                umax16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    fast = !special_pairs(m, k.thr2);
  }
  if (fast) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float2 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t na = f2(bf16lo(w[i]), bf16hi(w[i]));
      const uint64_t q0 = mul2(na, k.ny2);
      q[i] = unf2(fma2(fma2(q0, k.b2, na), k.ny2, q0));
    }
    return make_uint2(pack_fp8x4<F>(q[0].x, q[0].y, q[1].x, q[1].y),
                      pack_fp8x4<F>(q[2].x, q[2].y, q[3].x, q[3].y));
  }
  const uint32_t s = 0x80008000u;
  return bf16x8_to_fp8x8<F, true>(make_uint4(v.x ^ s, v.y ^ s, v.z ^ s, v.w ^ s), k);
}

// The kv_c part of a row (words holding -y) into an fp8 cache.
template <int F, bool CHECK>
__device__ __forceinline__ void write_kv_neg(uint8_t* dst, int lane, const uint4& ny0,
                                             const uint4& ny1, const DivConst& k) {
  st8(dst + lane * 8, neg_bf16x8_to_fp8x8<F, CHECK>(ny0, k));
  st8(dst + 256 + lane * 8, neg_bf16x8_to_fp8x8<F, CHECK>(ny1, k));
}

// The kv_c part of a row into a bf16 or fp8 cache.
template <int F, bool FAST>
__device__ __forceinline__ void write_kv_k(uint8_t* dst, int lane, const uint4& y0,
                                           const uint4& y1, const DivConst& k) {
  if constexpr (F == kBF16) {
    st16(dst + lane * 16, y0);
    st16(dst + 512 + lane * 16, y1);
  } else {
    st8(dst + lane * 8, bf16x8_to_fp8x8<F, FAST>(y0, k));
    st8(dst + 256 + lane * 8, bf16x8_to_fp8x8<F, FAST>(y1, k));
  }
}

// The k_pe pair (lane, lane + 32) of a row into a bf16 or fp8 cache.
template <int F, bool FAST>
__device__ __forceinline__ void write_pe_k(uint8_t* dst, int lane, uint32_t p, const DivConst& k) {
  if constexpr (F == kBF16) {
    st_u16(dst + 2 * kR + lane * 2, p);
    st_u16(dst + 2 * kR + kP + lane * 2, p >> 16);
  } else {
    const uint32_t q = bf16x2_to_fp8x2<F, FAST>(p, k);
    st_u8(dst + kR + lane, q);
    st_u8(dst + kR + kP / 2 + lane, q >> 8);
  }
}

template <int F>
__device__ __forceinline__ void write_row_dc(uint8_t* dst, int lane, const uint4& y0,
                                             const uint4& y1, uint32_t p, const DivConst& k) {
  if (F == kBF16 || k.fast) write_row_k<F, true>(dst, lane, y0, y1, p, k);
  else write_row_k<F, false>(dst, lane, y0, y1, p, k);
}

// Start of the cache row of a valid slot s (0 <= s < capacity) in the cache
// at cptr: block s / block_size, offset s % block_size.
__device__ __forceinline__ uint8_t* slot_dst(const InsertArgs& a, int64_t s, int64_t cptr) {
  int64_t blk, off;
  if (a.bs_shift >= 0) {
    blk = s >> a.bs_shift;
    off = s & (a.block_size - 1);
  } else {
    blk = s / a.block_size;
    off = s - blk * a.block_size;
  }
  return reinterpret_cast<uint8_t*>(cptr) + blk * a.block_stride + off * a.entry_stride;
}

// Half-warp rows (16 lanes per row, norm_rope.cuh): the kv_c part of a row
// held as x[4] into a bf16 or fp8 cache (fp8: NEG = the words hold -y).
template <int F, bool FAST, bool NEG, bool CHECK>
__device__ __forceinline__ void write_kv32(uint8_t* dst, int hl, const uint4 (&x)[4],
                                           const DivConst& k) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if constexpr (F == kBF16) st16(dst + hl * 16 + 256 * c, x[c]);
    else if constexpr (NEG) st8(dst + hl * 8 + 128 * c, neg_bf16x8_to_fp8x8<F, CHECK>(x[c], k));
    else st8(dst + hl * 8 + 128 * c, bf16x8_to_fp8x8<F, FAST>(x[c], k));
  }
}

// Quarter-warp rows (8 lanes per row, norm_rope.cuh): the kv_c part of a row
// held as x[8] (units ql + 16 c and ql + 8 + 16 c).
template <int F, bool FAST, bool NEG, bool CHECK>
__device__ __forceinline__ void write_kv64(uint8_t* dst, int ql, const uint4 (&x)[8],
                                           const DivConst& k) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int u = ql + 16 * (c & 3) + 8 * (c >> 2);
    if constexpr (F == kBF16) st16(dst + u * 16, x[c]);
    else if constexpr (NEG) st8(dst + u * 8, neg_bf16x8_to_fp8x8<F, CHECK>(x[c], k));
    else st8(dst + u * 8, bf16x8_to_fp8x8<F, FAST>(x[c], k));
  }
}

// The k_pe elements 4 ql .. 4 ql + 3 (lo) and 4 ql + 32 .. 4 ql + 35 (hi) of a
// row held by a quarter warp.
template <int F, bool FAST>
__device__ __forceinline__ void write_pe64(uint8_t* dst, int ql, uint2 lo, uint2 hi,
                                           const DivConst& k) {
  if constexpr (F == kBF16) {
    st8(dst + 2 * kR + ql * 8, lo);
    st8(dst + 2 * kR + kP + ql * 8, hi);
  } else {
    const uint32_t a = (bf16x2_to_fp8x2<F, FAST>(lo.x, k) & 0xFFFFu) |
                       (bf16x2_to_fp8x2<F, FAST>(lo.y, k) << 16);
    const uint32_t b = (bf16x2_to_fp8x2<F, FAST>(hi.x, k) & 0xFFFFu) |
                       (bf16x2_to_fp8x2<F, FAST>(hi.y, k) << 16);
    *reinterpret_cast<uint32_t*>(dst + kR + ql * 4) = a;
    *reinterpret_cast<uint32_t*>(dst + kR + kP / 2 + ql * 4) = b;
  }
}

// The k_pe words lo (elements 2 hl, 2 hl + 1) and hi (2 hl + 32, 2 hl + 33)
// of a row held by a half warp.
template <int F, bool FAST>
__device__ __forceinline__ void write_pe32(uint8_t* dst, int hl, uint32_t lo, uint32_t hi,
                                           const DivConst& k) {
  if constexpr (F == kBF16) {
    *reinterpret_cast<uint32_t*>(dst + 2 * kR + hl * 4) = lo;
    *reinterpret_cast<uint32_t*>(dst + 2 * kR + kP + hl * 4) = hi;
  } else {
    st_u16(dst + kR + hl * 2, bf16x2_to_fp8x2<F, FAST>(lo, k));
    st_u16(dst + kR + kP / 2 + hl * 2, bf16x2_to_fp8x2<F, FAST>(hi, k));
  }
}

// Normalise / rotate / convert one loaded row and store it into the cache at
// `cptr` (its layer's base; `k` its layer's division constants).  `cs` =
// (cos, sin) of this lane's rotary pair.  Returns the error bits of a skipped
// row.
template <int F, bool NORM, bool ROPE>
__device__ __forceinline__ uint32_t store_row(const InsertArgs& a, int l, int lane, const RowIn& r,
                                              bool pos_ok, float2 cs, int64_t cptr,
                                              const DivConst& k) {
  const int64_t s = r.slot;
  if (s < 0) return 0;  // padding slot (uniform across the warp)
  if (s >= a.capacity) return kErrSlotOOB;
  if (ROPE && !pos_ok) return kErrPosOOB;
  if (cptr == 0 || (cptr & 15)) return kErrMisaligned;
  int64_t blk, off;
  if (a.bs_shift >= 0) {
    blk = s >> a.bs_shift;
    off = s & (a.block_size - 1);
  } else {
    blk = s / a.block_size;
    off = s - blk * a.block_size;
  }
  uint8_t* dst = reinterpret_cast<uint8_t*>(cptr) + blk * a.block_stride + off * a.entry_stride;

  // kv_c (optionally RMSNorm-ed) as bf16 words
  uint4 y0 = r.x0, y1 = r.x1;
  if constexpr (NORM) {
    const uint8_t* g = a.gamma + (int64_t)l * a.gamma_ls;
    rms_norm16(r.x0, r.x1, ld_shared_ro16(g + lane * 16), ld_shared_ro16(g + 512 + lane * 16),
               a.eps, y0, y1, lane);
  }
  // k_pe pair (l, l+32), optionally rotated
  uint32_t p = r.pe;
  if constexpr (ROPE) p = rope_pair(r.pe, cs);

  write_row_dc<F>(dst, lane, y0, y1, p, k);
  return 0;
}

template <bool ROPE>
__device__ __forceinline__ bool load_rope(const InsertArgs& a, int64_t t, int lane, float2& cs) {
  cs = make_float2(1.f, 0.f);
  if constexpr (!ROPE) return true;
  const int64_t pos = a.positions[t];
  if (pos < 0 || pos >= a.max_position) return false;
  const float* row = a.cos_sin + pos * kP;
  cs = make_float2(__ldg(row + lane), __ldg(row + kP / 2 + lane));
  return true;
}

// Whether normalised kv_c values of a layer can make the exact division's
// first quotient overflow, so each group of 8 needs the special-value test.
// A normalised element is x_i * gamma_i * rstd with x_i^2 <= sum(x^2): when
// the row's sum of squares is finite, |y_i| <= sqrt(512) |gamma_i| (1 + 2^-7)
// < 23 gmax, and x_i * gamma_i cannot overflow while gmax < 2^64 (|x_i| <
// 2^64 then); when it is infinite or NaN, rstd is 0 or NaN and every y_i is
// +-0 or NaN, which the fast path also handles.  So the test can be skipped
// when 23 gmax stays below the first value the test would flag, 2^(T - 127)
// with T the threshold exponent field of thr2.  gmax: the layer's largest
// |gamma| (inf / NaN: the test stays).
__device__ __forceinline__ bool layer_needs_check(const DivConst& k, uint32_t gmax_bits) {
  if (!k.fast) return true;
  const uint32_t h = k.thr2 & 0xFFFFu;           // 0x8000 - (T << 7)
  const int T = (int)((0x8000u - h) >> 7);
  const float lim = ldexpf(1.0f, T - 127);       // inf for T = 255
  const float g = __uint_as_float(gmax_bits << 16);
  return !(g < 1.8446744e19f && 23.0f * g < lim);
}

// The largest |gamma| of layer l as bf16 bits (a NaN's bits exceed every
// finite one's), over the whole warp; all 32 lanes call it together.
__device__ __forceinline__ uint32_t layer_gmax(const InsertArgs& a, int l, int lane) {
  const uint8_t* g = a.gamma + (int64_t)l * a.gamma_ls;
  const uint4 g0 = ld_shared_ro16(g + lane * 16), g1 = ld_shared_ro16(g + 512 + lane * 16);
  const uint32_t m = umax16x2(umax16x2(umax16x2(g0.x & 0x7FFF7FFFu, g0.y & 0x7FFF7FFFu),
                                       umax16x2(g0.z & 0x7FFF7FFFu, g0.w & 0x7FFF7FFFu)),
                              umax16x2(umax16x2(g1.x & 0x7FFF7FFFu, g1.y & 0x7FFF7FFFu),
                                       umax16x2(g1.z & 0x7FFF7FFFu, g1.w & 0x7FFF7FFFu)));
  return __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
}

// Shape 1: one warp per (token, layer) row, rows in token-major order.  For
// more than a few rows per warp each CTA first puts the layers' cache bases
// and division constants in shared memory; tiny calls (decode) skip that step,
// which would sit on their critical path, and load them per row.
constexpr int64_t kRowPreloadMinRows = 2048;

// TRIM (normalised fp8 rows two per warp, per-layer tables built before the
// launch wait): the rows are computed negated (the exact division then skips
// its negation) and, per layer, without the special-value test when the gamma
// bound allows it, as in the bulk-copy shape (4096 tokens x 5 layers back to
// back: 10.37 -> 10.07 us).  Only with early tables: after the wait the gamma
// loads and reduction cost more than the test they save (2048 tokens x 5
// layers 7.43 vs 7.24 us), and the negated form with the test kept is slower
// than the plain one (11.30 vs 10.95 us).
template <int F, bool NORM, bool ROPE, bool PAIRS, bool TRIM = false>
__global__ void __launch_bounds__(kThreads) insert_row_kernel(const InsertArgs a) {
  static_assert(!TRIM || (PAIRS && NORM && F != kBF16), "TRIM: normalised fp8 pairs");
  constexpr bool kTrim = TRIM;
  __shared__ int64_t s_cptr[kMaxLayers];
  __shared__ DivConst s_k[F == kBF16 ? 1 : kMaxLayers];
  __shared__ uint8_t s_check[kTrim ? kMaxLayers : 1];
  pdl_trigger();
  // The per-layer table (cache bases, division constants) reads only
  // cache_ptrs and scales.  When the caller has declared them complete before
  // the call (early_tables), it is built before the wait on the previous grid,
  // so its load latency overlaps that grid's tail (4096 tokens x 5 layers:
  // 10.99 -> 10.37 us back to back); otherwise after it (plain stream order;
  // the second wait is then a no-op).
  if (!a.early_tables) pdl_wait();
  const bool pre = a.num_rows >= kRowPreloadMinRows;  // uniform across the grid
  if (pre) {
    for (int l = threadIdx.x; l < a.num_layers; l += kThreads) {
      s_cptr[l] = a.cache_ptrs[l];
      if constexpr (F != kBF16) s_k[l] = div_const(a.scales[l]);
    }
    if constexpr (kTrim) {  // the gamma bound, one warp per layer
      for (int l = threadIdx.x >> 5; l < a.num_layers; l += kThreads / 32) {
        const bool check = layer_needs_check(div_const(a.scales[l]),
                                             layer_gmax(a, l, threadIdx.x & 31));
        if ((threadIdx.x & 31) == 0) s_check[l] = check ? 1 : 0;
      }
    }
    __syncthreads();
  }
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const bool rows32 = a.num_rows < (int64_t(1) << 32);
  auto split = [&](int64_t r, int64_t& t, int& l) {
    if (rows32) {
      const uint32_t tu = (uint32_t)r / (uint32_t)a.num_layers;
      t = tu;
      l = (int)((uint32_t)r - tu * (uint32_t)a.num_layers);
    } else {
      t = r / a.num_layers;
      l = (int)(r - t * a.num_layers);
    }
  };
  uint32_t errbits = 0;
  if constexpr (PAIRS) {
    // Two rows per warp, 16 lanes each (the half-warp layout of norm_rope.cuh):
    // the rows 2w + half, 2w + half + 2 nwarps, ...
    const int hl = lane & 15, half = lane >> 4;
    for (int64_t r0 = 2 * warp; r0 < a.num_rows; r0 += 2 * nwarps) {
      const int64_t r = r0 + half;
      const bool have = r < a.num_rows;
      int64_t t = 0;
      int l = 0;
      uint4 x[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                    make_uint4(0, 0, 0, 0)};
      uint32_t lo = 0, hi = 0;
      int64_t slot = -1, pos = 0;
      if (have) {
        split(r, t, l);
        const uint8_t* src = a.kv_c + t * a.kvc_ts + (int64_t)l * a.kvc_ls + hl * 16;
#pragma unroll
        for (int c = 0; c < 4; ++c) x[c] = ld_stream16(src + 256 * c);
        const uint8_t* pe = a.k_pe + t * a.kpe_ts + (int64_t)l * a.kpe_ls + hl * 4;
        lo = __ldcs(reinterpret_cast<const uint32_t*>(pe));
        hi = __ldcs(reinterpret_cast<const uint32_t*>(pe + kP));
        slot = __ldg(a.slots + (int64_t)l * a.slot_ls + t);
        if (ROPE) pos = __ldg(a.positions + t);
      }
      DivConst k{};
      int64_t cptr = 0;
      float4 cs = make_float4(1.f, 1.f, 0.f, 0.f);
      const uint8_t* gr = a.gamma;
      bool ok = false;
      uint8_t* dst = nullptr;
      if (have) {
        if constexpr (F != kBF16) k = pre ? s_k[l] : div_const(a.scales[l]);
        cptr = pre ? s_cptr[l] : a.cache_ptrs[l];
        if (slot < 0) {
        } else if (slot >= a.capacity) {
          errbits |= kErrSlotOOB;
        } else if (ROPE && (pos < 0 || pos >= a.max_position)) {
          errbits |= kErrPosOOB;
        } else if (cptr == 0 || (cptr & 15)) {
          errbits |= kErrMisaligned;
        } else {
          ok = true;
          dst = slot_dst(a, slot, cptr);
        }
        if (ROPE && ok) cs = load_cs2(a.cos_sin + pos * kP, hl);
        if constexpr (NORM) gr = a.gamma + (int64_t)l * a.gamma_ls + hl * 16;
      }
      // every lane: the shuffles span the warp (a lane without a row reads
      // layer 0's weights)
      if constexpr (NORM) rms_norm32_g<kTrim>(x, have ? gr : a.gamma + hl * 16, a.eps);
      if constexpr (ROPE) rope_pairs2(lo, hi, cs);
      if (ok) {
        if (F == kBF16 || k.fast) {
          if constexpr (kTrim) {
            if (s_check[l]) write_kv32<F, true, true, true>(dst, hl, x, k);
            else write_kv32<F, true, true, false>(dst, hl, x, k);
          } else {
            write_kv32<F, true, false, true>(dst, hl, x, k);
          }
          write_pe32<F, true>(dst, hl, lo, hi, k);
        } else {
          if constexpr (kTrim) {  // undo the negation (exact: a sign flip)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              x[c] = make_uint4(x[c].x ^ 0x80008000u, x[c].y ^ 0x80008000u,
                                x[c].z ^ 0x80008000u, x[c].w ^ 0x80008000u);
          }
          write_kv32<F, false, false, true>(dst, hl, x, k);
          write_pe32<F, false>(dst, hl, lo, hi, k);
        }
      }
    }
    errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
  } else {
    for (int64_t r = warp; r < a.num_rows; r += nwarps) {
      int64_t t;
      int l;
      split(r, t, l);
      RowIn in;
      load_row<F, ROPE>(a, t, l, lane, in);
      float2 cs;
      const bool pos_ok = load_rope<ROPE>(a, t, lane, cs);
      DivConst k{};
      if constexpr (F != kBF16) k = pre ? s_k[l] : div_const(a.scales[l]);
      const int64_t cptr = pre ? s_cptr[l] : a.cache_ptrs[l];
      errbits |= store_row<F, NORM, ROPE>(a, l, lane, in, pos_ok, cs, cptr, k);
    }
  }
  if (errbits && lane == 0 && a.err) atomicOr(a.err, errbits);
}

// Shape 1, four rows per warp (8 lanes each, the quarter-warp layout of
// norm_rope.cuh), for calls with RMSNorm or RoPE that it covers in one round
// where two rows per warp would take two (see launch_t): at 80 registers (3
// CTAs per SM) a round takes 14592 rows against 9728.  The same arithmetic,
// hence the same bits, as the other layouts; TRIM as in insert_row_kernel.
template <int F, bool NORM, bool ROPE, bool TRIM>
__global__ void __launch_bounds__(kThreads, 3) insert_quad_kernel(const InsertArgs a) {
  static_assert(NORM || ROPE, "the quad layout serves RMSNorm / RoPE rows");
  static_assert(!TRIM || (NORM && F != kBF16), "TRIM: normalised fp8 rows");
  __shared__ int64_t s_cptr[kMaxLayers];
  __shared__ DivConst s_k[F == kBF16 ? 1 : kMaxLayers];
  __shared__ uint8_t s_check[TRIM ? kMaxLayers : 1];
  pdl_trigger();
  if (!a.early_tables) pdl_wait();
  for (int l = threadIdx.x; l < a.num_layers; l += kThreads) {
    s_cptr[l] = a.cache_ptrs[l];
    if constexpr (F != kBF16) s_k[l] = div_const(a.scales[l]);
  }
  if constexpr (TRIM) {  // the gamma bound, one warp per layer
    for (int l = threadIdx.x >> 5; l < a.num_layers; l += kThreads / 32) {
      const bool check = layer_needs_check(div_const(a.scales[l]),
                                           layer_gmax(a, l, threadIdx.x & 31));
      if ((threadIdx.x & 31) == 0) s_check[l] = check ? 1 : 0;
    }
  }
  __syncthreads();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int ql = lane & 7, quad = lane >> 3;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  uint32_t errbits = 0;
  const bool rows32 = a.num_rows < (int64_t(1) << 32);
  // the rows 4w + quad, 4w + quad + 4 nwarps, ...
  for (int64_t r0 = 4 * warp; r0 < a.num_rows; r0 += 4 * nwarps) {
    const int64_t r = r0 + quad;
    const bool have = r < a.num_rows;
    int64_t t = 0;
    int l = 0;
    uint4 x[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = make_uint4(0, 0, 0, 0);
    uint2 lo = make_uint2(0, 0), hi = make_uint2(0, 0);
    int64_t slot = -1, pos = 0;
    if (have) {
      if (rows32) {
        const uint32_t tu = (uint32_t)r / (uint32_t)a.num_layers;
        t = tu;
        l = (int)((uint32_t)r - tu * (uint32_t)a.num_layers);
      } else {
        t = r / a.num_layers;
        l = (int)(r - t * a.num_layers);
      }
      const uint8_t* src = a.kv_c + t * a.kvc_ts + (int64_t)l * a.kvc_ls + ql * 16;
#pragma unroll
      for (int c = 0; c < 8; ++c) x[c] = ld_stream16(src + 256 * (c & 3) + 128 * (c >> 2));
      const uint8_t* pe = a.k_pe + t * a.kpe_ts + (int64_t)l * a.kpe_ls + ql * 8;
      lo = ld_stream8(pe);
      hi = ld_stream8(pe + kP);
      slot = __ldg(a.slots + (int64_t)l * a.slot_ls + t);
      if (ROPE) pos = __ldg(a.positions + t);
    }
    DivConst k{};
    float4 cc = make_float4(1.f, 1.f, 1.f, 1.f), sn = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint8_t* gr = a.gamma + ql * 16;
    bool ok = false;
    uint8_t* dst = nullptr;
    if (have) {
      if constexpr (F != kBF16) k = s_k[l];
      const int64_t cptr = s_cptr[l];
      if (slot < 0) {
      } else if (slot >= a.capacity) {
        errbits |= kErrSlotOOB;
      } else if (ROPE && (pos < 0 || pos >= a.max_position)) {
        errbits |= kErrPosOOB;
      } else if (cptr == 0 || (cptr & 15)) {
        errbits |= kErrMisaligned;
      } else {
        ok = true;
        dst = slot_dst(a, slot, cptr);
      }
      if (ROPE && ok) {
        const float* row = a.cos_sin + pos * kP;
        cc = __ldg(reinterpret_cast<const float4*>(row + 4 * ql));
        sn = __ldg(reinterpret_cast<const float4*>(row + 32 + 4 * ql));
      }
      if constexpr (NORM) gr = a.gamma + (int64_t)l * a.gamma_ls + ql * 16;
    }
    // every lane: the shuffles span the warp (a lane without a row reads
    // layer 0's weights)
    if constexpr (NORM) rms_norm64_g<TRIM>(x, gr, a.eps);
    if constexpr (ROPE) rope_pairs4(lo, hi, cc, sn);
    if (ok) {
      if (F == kBF16 || k.fast) {
        if constexpr (TRIM) {
          if (s_check[l]) write_kv64<F, true, true, true>(dst, ql, x, k);
          else write_kv64<F, true, true, false>(dst, ql, x, k);
        } else {
          write_kv64<F, true, false, true>(dst, ql, x, k);
        }
        write_pe64<F, true>(dst, ql, lo, hi, k);
      } else {
        if constexpr (TRIM) {  // undo the negation (exact: a sign flip)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            x[c] = make_uint4(x[c].x ^ 0x80008000u, x[c].y ^ 0x80008000u,
                              x[c].z ^ 0x80008000u, x[c].w ^ 0x80008000u);
        }
        write_kv64<F, false, false, true>(dst, ql, x, k);
        write_pe64<F, false>(dst, ql, lo, hi, k);
      }
    }
  }
  errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
  if (errbits && lane == 0 && a.err) atomicOr(a.err, errbits);
}

// Shape 2 (bulk-copy pipeline): for dense per-layer rows (kv_c token stride
// 512, k_pe token stride 64 -- the layer-major [L, T, .] buffers), one layer's
// run of kRun consecutive tokens is contiguous.  A work item is such a run: a
// producer warp streams its kv_c rows into a ring of 46 shared-memory stages
// (Ring below) with one cp.async.bulk per item (byte-counted on a per-stage
// mbarrier; lane s of the producer fills stages s and s + 32), and 23 consumer
// warps process the rows from shared memory (the item's slots, positions and
// k_pe words are loaded from global memory while the consumer waits for its
// stage -- with RMSNorm + RoPE the k_pe words only after the wait, see below
// -- the rotary cos/sin of the item's rows together, the layer's gamma once
// per item).  Each consumer owns the stages s == warp (mod kIConsumers) and
// takes their fills in order, so no parity wait can alias an older phase.
// A consumer hands the stage back as soon as the item's last row is in
// registers (before that row is computed), so the producer refills it
// meanwhile.
constexpr int kRun = 4;
constexpr int kIConsumers = 23;
constexpr int kIThreads = (kIConsumers + 1) * 32;
// A stage holds an item's kv_c rows only.  Each lane reads its few k_pe
// bytes from global memory instead: staging them as a second bulk copy per
// item cost more (65536 tokens x 5 layers: RMSNorm + RoPE 100.7 vs 98.6 us,
// RMSNorm alone 97.1 vs 94.5, RoPE alone 95.4 vs 93.0, raw 94.6 vs 94.3).
constexpr int kIStageBytes = kRun * 2 * kR;  // 4096
// The ring: 2 stages per consumer, 46 in all (producer lanes 0-13 own two).
// 23 consumers of one row at a time (72 registers: 6 warps per SM
// sub-partition) beat 16 consumers of two rows in lockstep (91 registers):
// 130.5 vs 137 us with RMSNorm + RoPE and 99.5 vs 101 us raw (65536 tokens x
// 5 layers); one stage per consumer starves them (174-182 us), and 24
// consumers with 48 stages (the most that fit) ran 139 vs 131.5 us.
template <bool NORM>
struct Ring {
  static constexpr int kStages = kIConsumers * 2;
  static constexpr int kOffBars = kStages * kIStageBytes;
  static constexpr int kOffLayers = kOffBars + 2 * kStages * 8 + 16;
  // per layer: cache base (8 B), scale (4 B), needs-check flag (1 B)
  static constexpr int kSmem = kOffLayers + kMaxLayers * (8 + 4 + 1);
  static_assert(kStages <= 64, "a producer lane owns at most two stages");
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

constexpr int kILP = 1;  // rows of an item processed in lockstep (full-warp form)

// One item (a layer's run of up to kRun tokens) from its shared-memory stage,
// one row at a time by the whole warp (the raw insert: without RMSNorm and
// RoPE the half-warp form below saves little and ran 98.4 vs 94.5 us for 65536
// tokens x 5 layers).  The k_pe pairs are stored after the last row.
template <int F, bool NORM, bool ROPE, bool FAST, bool CHECK>
__device__ __forceinline__ uint32_t insert_consume_rows(
    const InsertArgs& a, uint32_t src, int l, int lane, int64_t cptr, const DivConst& k,
    uint32_t empty_bar, const int64_t* slot, const int64_t* pos, const uint32_t* pe_in) {
  uint32_t err = 0;
  // the fp8 fast path takes the normalised rows negated (write_kv_neg)
  constexpr bool kNeg = NORM && F != kBF16 && FAST;
  // validity and destination of every row (uniform across the warp)
  uint8_t* dst[kRun];
  bool ok[kRun];
#pragma unroll
  for (int r = 0; r < kRun; ++r) {
    const int64_t s = slot[r];
    ok[r] = false;
    dst[r] = nullptr;
    if (s < 0) continue;  // padding slot or past the tail
    if (s >= a.capacity) { err |= kErrSlotOOB; continue; }
    if (ROPE && (pos[r] < 0 || pos[r] >= a.max_position)) { err |= kErrPosOOB; continue; }
    if (cptr == 0 || (cptr & 15)) { err |= kErrMisaligned; continue; }
    int64_t blk, off;
    if (a.bs_shift >= 0) {
      blk = s >> a.bs_shift;
      off = s & (a.block_size - 1);
    } else {
      blk = s / a.block_size;
      off = s - blk * a.block_size;
    }
    ok[r] = true;
    dst[r] = reinterpret_cast<uint8_t*>(cptr) + blk * a.block_stride + off * a.entry_stride;
  }
  float2 cs[kRun];
#pragma unroll
  for (int r = 0; r < kRun; ++r) {
    cs[r] = make_float2(1.f, 0.f);
    if (ROPE && ok[r]) {
      const float* row = a.cos_sin + pos[r] * kP;
      cs[r] = make_float2(__ldg(row + lane), __ldg(row + kP / 2 + lane));
    }
  }
  uint4 g0 = make_uint4(0, 0, 0, 0), g1 = g0;
  if constexpr (NORM) {
    const uint8_t* g = a.gamma + (int64_t)l * a.gamma_ls;
    g0 = ld_shared_ro16(g + lane * 16);
    g1 = ld_shared_ro16(g + 512 + lane * 16);
  }
  uint32_t pe[kRun];
#pragma unroll
  for (int h = 0; h < kRun; h += kILP) {
    uint4 x0[kILP], x1[kILP], y0[kILP], y1[kILP];
#pragma unroll
    for (int i = 0; i < kILP; ++i) {
      const uint32_t row = src + (h + i) * 2 * kR;
      x0[i] = y0[i] = lds16(row + lane * 16);
      x1[i] = y1[i] = lds16(row + 512 + lane * 16);
      pe[h + i] = pe_in[h + i];
    }
    if (h + kILP >= kRun) {
      // every read of the stage is done: hand it back to the producer before
      // the last rows are computed
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    }
    if constexpr (NORM) {
      float ss[kILP];
#pragma unroll
      for (int i = 0; i < kILP; ++i) ss[i] = row_sum_sq(x0[i], x1[i], lane);
#pragma unroll
      for (int i = 0; i < kILP; ++i) {
        // mean over 512 (exact power-of-two scaling) + eps, one rounding
        const float rstd = __frsqrt_rn(fmaf(ss[i], 1.0f / kR, a.eps));
        scale16<kNeg>(x0[i], x1[i], g0, g1, rstd, y0[i], y1[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < kILP; ++i) {
      if (ok[h + i]) {
        if constexpr (kNeg) write_kv_neg<F, CHECK>(dst[h + i], lane, y0[i], y1[i], k);
        else write_kv_k<F, FAST>(dst[h + i], lane, y0[i], y1[i], k);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kRun; ++r) {
    if (!ok[r]) continue;
    const uint32_t p = ROPE ? rope_pair(pe[r], cs[r]) : pe[r];
    write_pe_k<F, FAST || F == kBF16>(dst[r], lane, p, k);
  }
  return err;
}

// One item (a layer's run of up to kRun tokens) from its shared-memory stage,
// two rows at a time (with RMSNorm or RoPE: 102.3 vs 113.0 us with RMSNorm +
// RoPE for 65536 tokens x 5 layers, one row per warp instruction before):
// lanes 0-15 take rows 0 and 2 of the item, lanes 16-31
// rows 1 and 3 (this lane's rows: slot[p] / pos[p] of row 2p + half).  The
// rows' kv_c are normalised, converted and stored one pair of rows after the
// other; the k_pe pairs are rotated and stored after the last, so the
// cos/sin loads issued first have the whole item to arrive.  The k_pe words
// (lo / hi: elements 2 hl, 2 hl + 1 and 32 + 2 hl, 33 + 2 hl of the lane's
// rows) come loaded before the stage wait, or, with RMSNorm + RoPE (kLatePe),
// are loaded here from global memory: held across the wait they crowd the
// 80 registers of that form (100.9 vs 98.6 us).  Returns this lane's error
// bits.
template <int F, bool NORM, bool ROPE, bool FAST, bool CHECK>
__device__ __forceinline__ uint32_t insert_consume_pairs(
    const InsertArgs& a, uint32_t src, int l, int lane, int64_t cptr, const DivConst& k,
    uint32_t empty_bar, const int64_t (&slot)[2], const int64_t (&pos)[2],
    const uint32_t (&lo_in)[2], const uint32_t (&hi_in)[2], int64_t t0, int nt) {
  constexpr bool kLatePe = NORM && ROPE;
  const int hl = lane & 15, half = lane >> 4;
  uint32_t err = 0;
  // the fp8 fast path takes the normalised rows negated (write_kv32<.., NEG>)
  constexpr bool kNeg = NORM && F != kBF16 && FAST;
  // validity and destination of this lane's rows (uniform across its half)
  uint8_t* dst[2];
  bool ok[2];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int64_t s = slot[p];
    ok[p] = false;
    dst[p] = nullptr;
    if (s < 0) continue;  // padding slot or past the tail
    if (s >= a.capacity) { err |= kErrSlotOOB; continue; }
    if (ROPE && (pos[p] < 0 || pos[p] >= a.max_position)) { err |= kErrPosOOB; continue; }
    if (cptr == 0 || (cptr & 15)) { err |= kErrMisaligned; continue; }
    ok[p] = true;
    dst[p] = slot_dst(a, s, cptr);
  }
  float4 cs[2];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    cs[p] = make_float4(1.f, 1.f, 0.f, 0.f);
    if (ROPE && ok[p]) cs[p] = load_cs2(a.cos_sin + pos[p] * kP, hl);
  }
  // The layer's gamma: held in registers for both row pairs, or, with RoPE
  // (whose cos/sin must be held from the start of the item), read again at
  // each use from L1 (65536 tokens x 5 layers: 102.3 -> 100.7 us with RMSNorm
  // + RoPE; RMSNorm alone 97.1 vs 98.2 us with the gamma held, so it keeps it).
  const uint8_t* gr = a.gamma + (int64_t)l * a.gamma_ls + hl * 16;
  uint4 g[4];
  if constexpr (NORM && !ROPE) {
#pragma unroll
    for (int c = 0; c < 4; ++c) g[c] = ld_shared_ro16(gr + 256 * c);
  }
  uint32_t lo[2], hi[2];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    lo[p] = lo_in[p];
    hi[p] = hi_in[p];
    if constexpr (kLatePe) {
      lo[p] = hi[p] = 0;
      if (2 * p + half < nt) {
        const uint8_t* pe = a.k_pe + (t0 + 2 * p + half) * a.kpe_ts + (int64_t)l * a.kpe_ls + hl * 4;
        lo[p] = __ldcs(reinterpret_cast<const uint32_t*>(pe));
        hi[p] = __ldcs(reinterpret_cast<const uint32_t*>(pe + kP));
      }
    }
  }
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const uint32_t row = src + (2 * p + half) * 2 * kR + hl * 16;
    uint4 x[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) x[c] = lds16(row + 256 * c);
    if (p == 1) {
      // every read of the stage is done: hand it back to the producer before
      // the last rows are computed
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    }
    if constexpr (NORM && ROPE) rms_norm32_g<kNeg>(x, gr, a.eps);
    else if constexpr (NORM) rms_norm32<kNeg>(x, g, a.eps);
    if (ok[p]) write_kv32<F, FAST, kNeg, CHECK>(dst[p], hl, x, k);
  }
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    if (!ok[p]) continue;
    if constexpr (ROPE) rope_pairs2(lo[p], hi[p], cs[p]);
    write_pe32<F, FAST || F == kBF16>(dst[p], hl, lo[p], hi[p], k);
  }
  return err;
}

template <int F, bool NORM, bool ROPE>
__global__ void __launch_bounds__(kIThreads, 1) insert_tma_kernel(const InsertArgs a) {
  constexpr int kIStages = Ring<NORM>::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ring<NORM>::kOffBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kIStages);
  int64_t* s_cptr = reinterpret_cast<int64_t*>(smem + Ring<NORM>::kOffLayers);
  float* s_scale = reinterpret_cast<float*>(s_cptr + kMaxLayers);
  uint8_t* s_check = reinterpret_cast<uint8_t*>(s_scale + kMaxLayers);
  const uint32_t stage0 = smem_addr(smem);
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kIStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kIStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  // No early trigger of the next launch: in a step of chunk launches after the
  // insert, a trigger at the start cost ~80 us (506.7 vs 588 us per step) and
  // one after each CTA's last copy ~60 us (0.464 vs 0.524 ms): the launch
  // follows the last CTA's exit.
  // With early_tables (cache_ptrs, scales and gamma declared complete before
  // the call) the consumers build the per-layer table before the wait on the
  // previous grid (8192 tokens x 5 layers back to back: 17.39 -> 17.19 us);
  // the producer, which reads kv_c, always waits first.
  if (!a.early_tables) pdl_wait();
  __syncthreads();  // the barriers are initialised
  if (warp == kIConsumers) pdl_wait();
  // The producer starts copying at once; the consumers first fill the
  // per-layer table (one warp per layer: cache base, scale, and whether
  // normalised rows need the special-value test) and sync among themselves.
  if (warp < kIConsumers) {
    for (int l = warp; l < a.num_layers; l += kIConsumers) {
      float sc = 1.0f;
      if constexpr (F != kBF16) sc = a.scales[l];
      bool check = true;
      if constexpr (NORM && F != kBF16) {
        const uint8_t* g = a.gamma + (int64_t)l * a.gamma_ls;
        const uint4 g0 = ld_shared_ro16(g + lane * 16), g1 = ld_shared_ro16(g + 512 + lane * 16);
        const uint32_t m = umax16x2(umax16x2(umax16x2(g0.x & 0x7FFF7FFFu, g0.y & 0x7FFF7FFFu),
                                             umax16x2(g0.z & 0x7FFF7FFFu, g0.w & 0x7FFF7FFFu)),
                                    umax16x2(umax16x2(g1.x & 0x7FFF7FFFu, g1.y & 0x7FFF7FFFu),
                                             umax16x2(g1.z & 0x7FFF7FFFu, g1.w & 0x7FFF7FFFu)));
        const uint32_t gmax = __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
        check = layer_needs_check(div_const(sc), gmax);
      }
      if (lane == 0) {
        s_cptr[l] = a.cache_ptrs[l];
        s_scale[l] = sc;
        s_check[l] = check ? 1 : 0;
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kIConsumers * 32) : "memory");
    pdl_wait();  // (a no-op without early_tables)
  }

  const int L = a.num_layers;
  const int64_t runs = ((int64_t)a.num_tokens + kRun - 1) / kRun;
  const int64_t n_items = runs * L;
  const int64_t G = gridDim.x, b = blockIdx.x;
  const int64_t n_local = n_items > b ? (n_items - 1 - b) / G + 1 : 0;
  int64_t fills0 = 0, fills1 = 0;  // producer lane: fills issued to its stages lane, lane + 32
  uint32_t errbits = 0;

  if (warp == kIConsumers) {
    // ---------------- producer: lane s fills stages s and s + 32 -----------------
    // (one issuing lane sustains only about one bulk copy per ~270 cycles, so
    // all 32 lanes issue, each for its own stages).  A lane takes its items in
    // order: item i goes to stage i % kIStages (items per CTA < 2^32).
    for (int64_t i = lane; lane < kIStages && i < n_local;) {
      const int s = (int)((uint32_t)i % (uint32_t)kIStages);
      const int64_t n = (int64_t)((uint32_t)i / (uint32_t)kIStages);
      if (n > 0 && !mbar_wait(empty0 + 8 * s, (uint32_t)((n - 1) & 1), a.wait_limit_ns)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      const int64_t j = b + G * i;
      const int64_t run = (int64_t)((uint32_t)j / (uint32_t)L);
      const int l = (int)((uint32_t)j - (uint32_t)run * (uint32_t)L);
      const int64_t t0 = run * kRun;
      const int nt = (int)min((int64_t)kRun, (int64_t)a.num_tokens - t0);
      const uint32_t dst = stage0 + (uint32_t)(s * kIStageBytes);
      if (b != 0 || i != a.skip_item) {  // (the test hook issues nothing for one item)
        mbar_arrive_expect_tx(full0 + 8 * s, (uint32_t)nt * (2 * kR));
        bulk_g2s(dst, a.kv_c + t0 * a.kvc_ts + (int64_t)l * a.kvc_ls, (uint32_t)nt * 2 * kR,
                 full0 + 8 * s);
        if (kIStages <= 32 || s < 32) fills0 = n + 1;
        else fills1 = n + 1;
      }
      // next item of this lane: its second stage in this round, else its first
      // stage in the next round
      if constexpr (kIStages <= 32) i += kIStages;
      else i += (s == lane && lane + 32 < kIStages) ? 32 : kIStages - (s - lane);
    }
  } else {
    // ---------------- consumers --------------------------------------------------
    for (int64_t i = warp; i < n_local && !*abort_flag; i += kIConsumers) {
      const int s = (int)((uint32_t)i % (uint32_t)kIStages);
      const int64_t j = b + G * i;
      const int64_t run = (int64_t)((uint32_t)j / (uint32_t)L);
      const int l = (int)((uint32_t)j - (uint32_t)run * (uint32_t)L);
      const int64_t t0 = run * kRun;
      const int nt = (int)min((int64_t)kRun, (int64_t)a.num_tokens - t0);
      // The item's slots, positions and (but with RMSNorm + RoPE) k_pe words
      // are read from global memory before the wait on its stage, so their
      // latency overlaps it; bulk-copying slots and positions too doubled the
      // copies per item, and the copy rate, not the bytes, then held the
      // consumers back (129.6 vs 118.9 us for 65536 tokens x 5 layers).
      // half-warp form: this lane's rows 2p + (lane >> 4); full-warp form: all
      // kRun rows
      constexpr bool kPairs = NORM || ROPE;
      constexpr int kSlots = kPairs ? 2 : kRun;
      int64_t slot[kSlots], pos[kSlots];
      uint32_t pe_lo[kSlots], pe_hi[kSlots];
#pragma unroll
      for (int p = 0; p < kSlots; ++p) {
        const int r = kPairs ? 2 * p + (lane >> 4) : p;
        slot[p] = -1;
        pos[p] = 0;
        pe_lo[p] = pe_hi[p] = 0;
        if (r < nt) {
          slot[p] = __ldg(a.slots + (int64_t)l * a.slot_ls + t0 + r);
          if (ROPE) pos[p] = __ldg(a.positions + t0 + r);
          const uint8_t* pe = a.k_pe + (t0 + r) * a.kpe_ts + (int64_t)l * a.kpe_ls;
          if constexpr (!kPairs) {
            // this lane's pair (lane, lane + 32) of the row
            const uint32_t lo = __ldcs(reinterpret_cast<const uint16_t*>(pe + lane * 2));
            const uint32_t hi = __ldcs(reinterpret_cast<const uint16_t*>(pe + kP + lane * 2));
            pe_lo[p] = lo | (hi << 16);
          } else if constexpr (!(NORM && ROPE)) {
            pe_lo[p] = __ldcs(reinterpret_cast<const uint32_t*>(pe + (lane & 15) * 4));
            pe_hi[p] = __ldcs(reinterpret_cast<const uint32_t*>(pe + kP + (lane & 15) * 4));
          }
        }
      }
      if (!mbar_wait(full0 + 8 * s, ((uint32_t)i / (uint32_t)kIStages) & 1u, a.wait_limit_ns)) {
        *abort_flag = 1;
        break;
      }
      const uint32_t src = stage0 + (uint32_t)(s * kIStageBytes);
      const DivConst k = div_const(s_scale[l]);
      const int64_t cptr = s_cptr[l];
      const uint32_t eb = empty0 + 8 * s;
      if constexpr (kPairs) {
        if (F != kBF16 && !k.fast)
          errbits |= insert_consume_pairs<F, NORM, ROPE, false, true>(
              a, src, l, lane, cptr, k, eb, slot, pos, pe_lo, pe_hi, t0, nt);
        else if (NORM && F != kBF16 && !s_check[l])
          errbits |= insert_consume_pairs<F, NORM, ROPE, true, false>(
              a, src, l, lane, cptr, k, eb, slot, pos, pe_lo, pe_hi, t0, nt);
        else
          errbits |= insert_consume_pairs<F, NORM, ROPE, true, true>(
              a, src, l, lane, cptr, k, eb, slot, pos, pe_lo, pe_hi, t0, nt);
      } else {
        if (F != kBF16 && !k.fast)
          errbits |= insert_consume_rows<F, NORM, ROPE, false, true>(a, src, l, lane, cptr, k,
                                                                     eb, slot, pos, pe_lo);
        else
          errbits |= insert_consume_rows<F, NORM, ROPE, true, true>(a, src, l, lane, cptr, k,
                                                                    eb, slot, pos, pe_lo);
      }
    }
  }
  __syncthreads();
  if (*abort_flag) {
    // Let every copy this CTA issued land before its shared memory is released:
    // a stage holds at most one fill in flight (the next one waits for the
    // stage's release), so waiting for each stage's last issued fill suffices.
    // A copy of a few KB from valid memory completes in microseconds; the wait
    // is bounded all the same.
    if (warp == kIConsumers) {
      if (fills0 > 0)
        (void)mbar_wait(full0 + 8 * lane, (uint32_t)((fills0 - 1) & 1), a.wait_limit_ns);
      if (kIStages > 32 && fills1 > 0)
        (void)mbar_wait(full0 + 8 * (lane + 32), (uint32_t)((fills1 - 1) & 1), a.wait_limit_ns);
    }
    errbits |= kErrTimeout;
  }
  errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);  // the two halves' rows differ
  if (errbits && lane == 0 && a.err) atomicOr(a.err, errbits);
}

// The bulk-copy shape needs dense per-layer token rows.
bool insert_tma_layout(const InsertArgs& a) {
  return a.kvc_ts == 2 * kR && a.kpe_ts == 2 * kP && a.num_layers <= kMaxLayers;
}

// From this many rows the bulk-copy shape runs by default (the RMSNorm
// variant's heavier rows keep its ring full from a smaller batch).
constexpr int64_t kBulkMinRows = 131072;
constexpr int64_t kBulkMinRowsNorm = 40960;

template <int F, bool NORM, bool ROPE>
cudaError_t launch_tma(const InsertArgs& a, const LaunchCfg& cfg) {
  auto kern = insert_tma_kernel<F, NORM, ROPE>;
  // the shared-memory opt-in is a per-device attribute: set once per device
  // (devices 0-63; others set it on every launch)
  static std::atomic<uint64_t> configured{0};  // per instance
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const uint64_t bit = dev < 64 ? uint64_t(1) << dev : 0;
  if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Ring<NORM>::kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  const int64_t items = ((int64_t)a.num_tokens + kRun - 1) / kRun * a.num_layers;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(capped_grid(reinterpret_cast<const void*>(kern), kIThreads,
                                (items + kIConsumers - 1) / kIConsumers, Ring<NORM>::kSmem));
  lc.blockDim = dim3(kIThreads);
  lc.dynamicSmemBytes = Ring<NORM>::kSmem;
  lc.stream = cfg.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = cfg.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, kern, a);
}

template <int F, bool NORM, bool ROPE>
cudaError_t launch_t(const InsertArgs& a, const LaunchCfg& cfg) {
  const int64_t min_rows = NORM ? kBulkMinRowsNorm : kBulkMinRows;
  const bool bulk = a.bulk_mode == 2 || (a.bulk_mode == 1 && a.num_rows >= min_rows);
  if (bulk && insert_tma_layout(a)) return launch_tma<F, NORM, ROPE>(a, cfg);
  // With RMSNorm or RoPE the row shape takes one, two or four rows per warp
  // (the same bits in every layout).  Two rows per warp once one row per warp
  // would take a second round (its
  // 48 registers allow 5 CTAs per SM: 6080 rows a round on 152 SMs); within
  // one round one row per warp is faster (1024 tokens x 5 layers: 4.57 vs 5.37
  // us).  1400 tokens x 5 layers: 5.33 -> 4.87 us, 1638: 6.57 -> 5.08.
  bool pairs = false;
  if constexpr (NORM || ROPE) {
    if (a.num_rows >= kRowPreloadMinRows) {  // (small calls skip the occupancy lookup)
      const int64_t one_rows = (int64_t)capped_grid(
          reinterpret_cast<const void*>(insert_row_kernel<F, NORM, ROPE, false>), kThreads,
          int64_t(1) << 30) * (kThreads / 32);
      pairs = a.num_rows > one_rows;
    }
  }
  auto kern = pairs ? insert_row_kernel<F, NORM, ROPE, NORM || ROPE>
                    : insert_row_kernel<F, NORM, ROPE, false>;
  if constexpr (NORM && F != kBF16)
    if (pairs && a.early_tables) kern = insert_row_kernel<F, NORM, ROPE, true, true>;
  // Four rows per warp where that takes one round and two rows per warp would
  // take two: a round of either shape costs about the same per row, but a
  // second, partly filled round of the two-row shape costs a whole round's
  // latency (1800 tokens x 5 layers: 5.24 vs 6.14 us; 2048: 6.51 vs 6.32;
  // 2400: 7.25 vs 6.57; 2800: 8.27 vs 6.88; 3200: 8.41 vs 8.98).
  bool quads = false;
  if constexpr (NORM || ROPE) {
    if (pairs) {
      auto qkern = insert_quad_kernel<F, NORM, ROPE, false>;
      const int64_t pair_rows = (int64_t)capped_grid(reinterpret_cast<const void*>(kern), kThreads,
                                                     int64_t(1) << 30) * (kThreads / 32) * 2;
      const int64_t quad_rows = (int64_t)capped_grid(reinterpret_cast<const void*>(qkern), kThreads,
                                                     int64_t(1) << 30) * (kThreads / 32) * 4;
      quads = a.num_rows > pair_rows && a.num_rows <= quad_rows;
      if (quads) kern = insert_quad_kernel<F, NORM, ROPE, false>;
      if constexpr (NORM && F != kBF16)
        if (quads && a.early_tables) kern = insert_quad_kernel<F, NORM, ROPE, true>;
    }
  }
  const int64_t rows_per_warp = quads ? 4 : pairs ? 2 : 1;
  const int64_t warps = (a.num_rows + rows_per_warp - 1) / rows_per_warp;
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

template <int F>
cudaError_t launch_fmt(const InsertArgs& a, bool norm, bool rope, const LaunchCfg& cfg) {
  if (norm && rope) return launch_t<F, true, true>(a, cfg);
  if (norm) return launch_t<F, true, false>(a, cfg);
  if (rope) return launch_t<F, false, true>(a, cfg);
  return launch_t<F, false, false>(a, cfg);
}

}  // namespace

cudaError_t launch_insert(const InsertArgs& a, int cache_fmt, bool norm, bool rope,
                          const LaunchCfg& cfg) {
  switch (cache_fmt) {
    case kBF16: return launch_fmt<kBF16>(a, norm, rope, cfg);
    case kE4M3: return launch_fmt<kE4M3>(a, norm, rope, cfg);
    case kE5M2: return launch_fmt<kE5M2>(a, norm, rope, cfg);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
