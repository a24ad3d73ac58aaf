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
//   * one warp per row, ROWS rows per warp per iteration, rows in token-major
//     order (a warp's rows share a token's slot / position / cos-sin), and a
//     grid-stride loop over a grid capped at the resident-CTA count;
//   * every global load of the ROWS rows is issued before the first row is
//     processed (memory-level parallelism: 1152 B per row in flight);
//   * kv_c: lane l holds elements [8l, 8l+8) and [256+8l, 256+8l+8) -- two
//     fully coalesced 512-byte warp loads; the fp8 stores are two 256-byte
//     warp stores, the bf16 stores two 512-byte ones (576 / 1152-byte cache
//     rows are whole 32-byte sectors);
//   * k_pe with RoPE: lanes 0-3 hold the neox pairs (8l+i, 32+8l+i), so the
//     rotation needs no shuffle; each rotated element is a difference of two
//     products evaluated with an FMA error correction (two-ulp accurate even
//     when the products cancel);
//   * RMSNorm: 16 squares per lane, a 5-step xor-shuffle sum, a correctly
//     rounded reciprocal square root;
//   * fp8: one correctly rounded division per element (ScaledDiv, one
//     reciprocal per row) then the hardware .satfinite pairwise converter;
//   * dtype, norm, rope and ROWS are template parameters: the hot loop has no
//     runtime format branches.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kR = 512;  // kv_lora_rank
constexpr int kP = 64;   // pe_dim

template <int F, bool NORM, bool ROPE, int ROWS>
__global__ void __launch_bounds__(kThreads) insert_kernel(const InsertArgs a) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  uint32_t errbits = 0;

  for (int64_t r0 = warp * ROWS; r0 < a.num_rows; r0 += nwarps * ROWS) {
    int32_t tok[ROWS], lay[ROWS];
    bool live[ROWS];
    {
      int32_t t = (int32_t)(r0 / a.num_layers);
      int32_t l = (int32_t)(r0 - (int64_t)t * a.num_layers);
#pragma unroll
      for (int k = 0; k < ROWS; ++k) {
        tok[k] = t;
        lay[k] = l;
        live[k] = (r0 + k) < a.num_rows;
        if (++l == a.num_layers) {
          l = 0;
          ++t;
        }
      }
    }

    // ---- issue all loads of the ROWS rows --------------------------------
    uint4 x0[ROWS], x1[ROWS], p0[ROWS], p1[ROWS];
    int64_t slot[ROWS], cptr[ROWS], pos[ROWS];
    float scale[ROWS];
#pragma unroll
    for (int k = 0; k < ROWS; ++k) {
      slot[k] = -1;
      cptr[k] = 0;
      pos[k] = 0;
      scale[k] = 1.0f;
      p0[k] = make_uint4(0, 0, 0, 0);
      p1[k] = make_uint4(0, 0, 0, 0);
      if (live[k]) {
        const uint8_t* src = a.kv_c + (int64_t)tok[k] * a.kvc_ts + (int64_t)lay[k] * a.kvc_ls;
        x0[k] = ld_stream16(src + lane * 16);
        x1[k] = ld_stream16(src + 512 + lane * 16);
        const uint8_t* pe = a.k_pe + (int64_t)tok[k] * a.kpe_ts + (int64_t)lay[k] * a.kpe_ls;
        if constexpr (ROPE) {
          if (lane < 4) {
            p0[k] = ld_stream16(pe + lane * 16);       // x_i,      i in [8l, 8l+8)
            p1[k] = ld_stream16(pe + 64 + lane * 16);  // x_{i+32}
          }
          pos[k] = a.positions[tok[k]];
        } else if (lane < 8) {
          p0[k] = ld_stream16(pe + lane * 16);
        }
        slot[k] = a.slots[(int64_t)lay[k] * a.slot_ls + tok[k]];
        cptr[k] = a.cache_ptrs[lay[k]];
        if constexpr (F != kBF16) scale[k] = a.scales[lay[k]];
      } else {
        x0[k] = make_uint4(0, 0, 0, 0);
        x1[k] = make_uint4(0, 0, 0, 0);
      }
    }

    // cos / sin of each row's position (a small L2-resident table)
    float4 c0[ROWS], c1[ROWS], s0[ROWS], s1[ROWS];
    if constexpr (ROPE) {
#pragma unroll
      for (int k = 0; k < ROWS; ++k) {
        c0[k] = c1[k] = s0[k] = s1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane < 4 && slot[k] >= 0 && pos[k] >= 0 && pos[k] < a.max_position) {
          const float* cs = a.cos_sin + pos[k] * kP + lane * 8;
          c0[k] = __ldg(reinterpret_cast<const float4*>(cs));
          c1[k] = __ldg(reinterpret_cast<const float4*>(cs + 4));
          s0[k] = __ldg(reinterpret_cast<const float4*>(cs + 32));
          s1[k] = __ldg(reinterpret_cast<const float4*>(cs + 36));
        }
      }
    }

    // ---- process and store -------------------------------------------------
#pragma unroll
    for (int k = 0; k < ROWS; ++k) {
      const int64_t s = slot[k];
      if (s < 0) continue;  // padding slot (uniform across the warp)
      if (s >= a.capacity) {
        errbits |= kErrSlotOOB;
        continue;
      }
      if constexpr (ROPE) {
        if (pos[k] < 0 || pos[k] >= a.max_position) {
          errbits |= kErrPosOOB;
          continue;
        }
      }
      if (cptr[k] & 15) {
        errbits |= kErrMisaligned;
        continue;
      }
      int64_t blk, off;
      if (a.bs_shift >= 0) {
        blk = s >> a.bs_shift;
        off = s & (a.block_size - 1);
      } else {
        blk = s / a.block_size;
        off = s - blk * a.block_size;
      }
      uint8_t* dst = reinterpret_cast<uint8_t*>(cptr[k]) + blk * a.block_stride + off * a.entry_stride;

      // kv_c (optionally RMSNorm-ed) as bf16 words
      uint4 y0 = x0[k], y1 = x1[k];
      if constexpr (NORM) {
        const uint32_t w[8] = {x0[k].x, x0[k].y, x0[k].z, x0[k].w,
                               x1[k].x, x1[k].y, x1[k].z, x1[k].w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[2 * i] = bf16lo(w[i]);
          v[2 * i + 1] = bf16hi(w[i]);
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) ss = fmaf(v[i], v[i], ss);
        ss = warp_sum(ss);
        // mean over 512 (exact power-of-two scaling) + eps, one rounding
        const float rstd = __frsqrt_rn(fmaf(ss, 1.0f / kR, a.eps));
        const uint8_t* g = a.gamma + (int64_t)lay[k] * a.gamma_ls;
        const uint4 g0 = ld_shared_ro16(g + lane * 16);
        const uint4 g1 = ld_shared_ro16(g + 512 + lane * 16);
        const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          o[i] = pack_bf16x2((v[2 * i] * rstd) * bf16lo(gw[i]),
                             (v[2 * i + 1] * rstd) * bf16hi(gw[i]));
        y0 = make_uint4(o[0], o[1], o[2], o[3]);
        y1 = make_uint4(o[4], o[5], o[6], o[7]);
      }

      // k_pe (optionally rotated) as bf16 words: q0 first half, q1 second half
      uint4 q0 = p0[k], q1 = p1[k];
      if constexpr (ROPE) {
        if (lane < 4) {
          const uint32_t a1[4] = {p0[k].x, p0[k].y, p0[k].z, p0[k].w};
          const uint32_t a2[4] = {p1[k].x, p1[k].y, p1[k].z, p1[k].w};
          const float c[8] = {c0[k].x, c0[k].y, c0[k].z, c0[k].w, c1[k].x, c1[k].y, c1[k].z, c1[k].w};
          const float sn[8] = {s0[k].x, s0[k].y, s0[k].z, s0[k].w, s1[k].x, s1[k].y, s1[k].z, s1[k].w};
          uint32_t o1[4], o2[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float u0 = bf16lo(a1[i]), u1 = bf16hi(a1[i]);
            const float w0 = bf16lo(a2[i]), w1 = bf16hi(a2[i]);
            const float cA = c[2 * i], cB = c[2 * i + 1], sA = sn[2 * i], sB = sn[2 * i + 1];
            o1[i] = pack_bf16x2(diff_of_products(u0, cA, w0, sA),
                                diff_of_products(u1, cB, w1, sB));
            o2[i] = pack_bf16x2(diff_of_products(w0, cA, -u0, sA),
                                diff_of_products(w1, cB, -u1, sB));
          }
          q0 = make_uint4(o1[0], o1[1], o1[2], o1[3]);
          q1 = make_uint4(o2[0], o2[1], o2[2], o2[3]);
        }
      }

      if constexpr (F == kBF16) {
        st16(dst + lane * 16, y0);
        st16(dst + 512 + lane * 16, y1);
        if constexpr (ROPE) {
          if (lane < 4) {
            st16(dst + 2 * kR + lane * 16, q0);
            st16(dst + 2 * kR + 64 + lane * 16, q1);
          }
        } else if (lane < 8) {
          st16(dst + 2 * kR + lane * 16, q0);
        }
      } else {
        const ScaledDiv d(scale[k]);
        st8(dst + lane * 8, bf16x8_to_fp8x8<F>(y0, d));
        st8(dst + 256 + lane * 8, bf16x8_to_fp8x8<F>(y1, d));
        if constexpr (ROPE) {
          if (lane < 4) {
            st8(dst + kR + lane * 8, bf16x8_to_fp8x8<F>(q0, d));
            st8(dst + kR + 32 + lane * 8, bf16x8_to_fp8x8<F>(q1, d));
          }
        } else if (lane < 8) {
          st8(dst + kR + lane * 8, bf16x8_to_fp8x8<F>(q0, d));
        }
      }
    }
  }
  if (errbits && lane == 0 && a.err) atomicOr(a.err, errbits);
  pdl_trigger();
}

template <int F, bool NORM, bool ROPE, int ROWS>
cudaError_t launch_t(const InsertArgs& a, const LaunchCfg& cfg) {
  auto kern = insert_kernel<F, NORM, ROPE, ROWS>;
  const int64_t warps = (a.num_rows + ROWS - 1) / ROWS;
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

template <int F, bool NORM, bool ROPE>
cudaError_t launch_rows(const InsertArgs& a, const LaunchCfg& cfg) {
  // Few rows: one row per warp spreads them over the most SMs (latency);
  // many rows: several rows per warp keep more bytes in flight per SM.
  if (a.num_rows >= (int64_t)1 << 15) return launch_t<F, NORM, ROPE, (NORM || ROPE) ? 2 : 4>(a, cfg);
  return launch_t<F, NORM, ROPE, 1>(a, cfg);
}

template <int F>
cudaError_t launch_fmt(const InsertArgs& a, bool norm, bool rope, const LaunchCfg& cfg) {
  if (norm && rope) return launch_rows<F, true, true>(a, cfg);
  if (norm) return launch_rows<F, true, false>(a, cfg);
  if (rope) return launch_rows<F, false, true>(a, cfg);
  return launch_rows<F, false, false>(a, cfg);
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
