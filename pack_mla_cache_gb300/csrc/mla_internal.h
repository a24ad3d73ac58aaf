// mla_internal.h -- launch descriptors shared by the C-ABI layer (abi.cu) and
// the kernel translation units.  All strides here are in BYTES; the ABI layer
// converts the element strides of the public header.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mla {

struct InsertArgs {
  const uint8_t* kv_c;
  int64_t kvc_ts, kvc_ls;  // token / layer strides
  const uint8_t* k_pe;
  int64_t kpe_ts, kpe_ls;
  int64_t num_rows;  // num_tokens * num_layers
  int32_t num_tokens, num_layers;
  const int64_t* slots;
  int64_t slot_ls;  // elements (0 = shared)
  const int64_t* cache_ptrs;
  const float* scales;
  int64_t capacity;  // num_blocks * block_size
  int32_t block_size;
  int32_t bs_shift;  // log2(block_size) if a power of two, else -1
  int64_t block_stride, entry_stride;
  const uint8_t* gamma;
  int64_t gamma_ls;
  float eps;
  const int64_t* positions;
  const float* cos_sin;
  int64_t max_position;
  uint32_t* err;
  int bulk_mode;  // bulk-copy pipeline shape: 0 never, 1 large calls, 2 always
  // bulk-copy shape only: how long a pipeline wait may last before the
  // kernel gives up (MLA_ERRBIT_TIMEOUT), and a test hook: CTA 0's producer
  // issues no copies for its local item `skip_item` (-1: none), so the
  // consumer waiting for that item runs out of time.
  uint64_t wait_limit_ns;
  int64_t skip_item;
  // cache_ptrs, scales (and, in the bulk-copy shape, gamma) may be read into
  // the per-layer table before the wait on the previous grid (the caller
  // declared them complete)
  bool early_tables;
};

// A paged cache and the chunk's sequences: chunk token i of sequence s
// (cu[s] <= i < cu[s+1]) is context position starts[s] + i - cu[s], held in
// block block_table[s * bt_stride + position / block_size].
struct PagedSrc {
  const uint8_t* cache;
  int64_t block_stride, entry_stride;
  int64_t num_blocks;
  int32_t block_size, bs_shift;  // bs_shift = log2(block_size) or -1
  const int32_t* block_table;
  int64_t bt_stride;  // elements
  const int32_t* cu;
  const int32_t* starts;
  int32_t num_seqs;
};

struct GatherArgs {
  PagedSrc src;
  int32_t row_chunks;  // 16-byte chunks of the copied part of a cache row
  int32_t num_tokens;
  uint8_t* out;
  int64_t out_rs;
  const float* dequant_scale;  // scaled widening only
  uint32_t* err;
  // read the sequence and block tables before waiting for the previous grid
  // (programmatic dependent launch); only for callers whose tables are
  // complete before the call is enqueued
  bool early_tables;
};

struct PackArgs {
  const uint8_t* k_nope;
  int64_t kn_ts, kn_hs;
  const uint8_t* v;
  int64_t v_ts, v_hs;
  const uint8_t* k_pe;
  int64_t kpe_ts;
  int32_t num_tokens, num_heads;
  uint8_t* key;
  uint8_t* vout;  // may be null
  const float* out_scale;  // may be null (1.0)
  uint32_t* err;  // may be null; only the paged pack sets bits
  PagedSrc paged;  // paged pack: k_pe = the cache row of each token, at pe_off
  int64_t pe_off;  // bytes
};

// Standalone grouped RMSNorm + RoPE: row (t, l) of kv_c / k_pe to the
// outputs at t * token stride + l * layer stride (bytes).
struct NormRopeArgs {
  const uint8_t* kv_c;
  int64_t kvc_ts, kvc_ls;
  const uint8_t* k_pe;
  int64_t kpe_ts, kpe_ls;
  int64_t num_rows;  // num_tokens * num_layers, < 2^32
  int32_t num_tokens, num_layers;
  const uint8_t* gamma;
  int64_t gamma_ls;
  float eps;
  const int64_t* positions;
  const float* cos_sin;
  int64_t max_position;
  uint8_t* out_c;
  int64_t oc_ts, oc_ls;
  uint8_t* out_p;
  int64_t op_ts, op_ls;
  uint32_t* err;
};

struct LaunchCfg {
  cudaStream_t stream;
  bool pdl;
};

// Each returns cudaSuccess or the launch error.  cache_fmt / out_fmt / kpe_fmt
// take the values of mla::Fmt.
cudaError_t launch_insert(const InsertArgs& a, int cache_fmt, bool norm, bool rope,
                          const LaunchCfg& cfg);
// mode: 0 raw copy, else the fp8 format widened to out_fmt (bf16 or fp16;
// bf16 times the scale when a.dequant_scale is set).
cudaError_t launch_gather(const GatherArgs& a, int mode, int out_fmt, const LaunchCfg& cfg);
// in_fmt: kBF16 or kF16 (k_nope / v); paged: k_pe from a.paged (kpe_fmt = the
// cache's format) instead of a.k_pe.  next_gather (not paged): the same launch
// also runs that gather (gather_mode 0: raw copy, or the cache's fp8 format
// widened to in_fmt; its num_tokens > 0).
cudaError_t launch_pack(const PackArgs& a, int in_fmt, int out_fmt, int kpe_fmt, bool paged,
                        const LaunchCfg& cfg, const GatherArgs* next_gather = nullptr,
                        int gather_mode = 0);
cudaError_t launch_norm_rope(const NormRopeArgs& a, bool norm, bool rope, const LaunchCfg& cfg);
cudaError_t launch_rope_table(float* out, int64_t max_position, int32_t rot_dim, double base,
                              const LaunchCfg& cfg);

// Grid size for a grid-stride kernel: enough CTAs to cover `work_ctas`, capped
// at the number that can be resident at once on the current device.
int capped_grid(const void* kernel, int threads, int64_t work_ctas, int dyn_smem = 0);

}  // namespace mla
