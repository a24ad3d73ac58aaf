// abi.cu -- the extern "C" entry points of libmla_cache (include/mla_cache.h):
// argument validation, conversion of element strides to byte strides, and
// dispatch to the template instance of each kernel.
//
// Validation follows the host checks of the grouped insert ("PR #55356 [Kimi
// Perf] Group fp8 mla cache insertion", Source snippets: the dtype whitelist,
// "FP8 ... requires kv_scales", "BF16 ... does not use kv_scales", scales on
// the same CUDA device) and adds the alignment and layout checks that the
// vectorised kernels need.  Every check that needs no CUDA call runs first, so
// an invalid call is rejected identically on a machine without a GPU.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "mla_cache.h"
#include "mla_device.cuh"
#include "mla_internal.h"

namespace {

thread_local std::string g_err;
std::atomic<int> g_pdl{1};
std::atomic<int> g_bulk{1};
std::atomic<int> g_ptr_checks{1};
std::atomic<int> g_gather_early{0};
std::atomic<int> g_insert_early{0};
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s: a wait that long means a fault
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int64_t> g_skip_item{-1};

mla_status_t fail(mla_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

inline bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool m16(int64_t bytes) { return (bytes & 15) == 0; }
inline bool valid_dtype(int d) {
  return d == MLA_BF16 || d == MLA_FP8_E4M3 || d == MLA_FP8_E5M2 || d == MLA_FP16;
}
inline bool is16(int d) { return d == MLA_BF16 || d == MLA_FP16; }
inline int elt_size(int d) { return is16(d) ? 2 : 1; }
inline int log2_exact(int64_t v) {
  if (v <= 0 || (v & (v - 1))) return -1;
  int s = 0;
  while ((int64_t(1) << s) < v) ++s;
  return s;
}

// The pointer must be device (or managed) memory of the current device
// (skipped while the caller has switched the checks off).
mla_status_t check_device_ptr(const void* p, const char* name) {
  if (!g_ptr_checks.load(std::memory_order_relaxed)) return MLA_OK;
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(MLA_ERR_CUDA, "%s: cudaPointerGetAttributes failed: %s", name,
                cudaGetErrorString(e));
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(MLA_ERR_INVALID_ARG, "%s must be device memory on the same CUDA device", name);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(MLA_ERR_CUDA, "cudaGetDevice failed");
  }
  if (attr.device != dev)
    return fail(MLA_ERR_INVALID_ARG,
                "%s must be on the same CUDA device as the launch (it is on device %d, the "
                "current device is %d)",
                name, attr.device, dev);
  return MLA_OK;
}

mla_status_t launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(MLA_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  }
  return MLA_OK;
}

mla::LaunchCfg cfg_for(mla_stream_t stream) {
  return mla::LaunchCfg{reinterpret_cast<cudaStream_t>(stream), g_pdl.load() != 0};
}

#define MLA_TRY(expr)                  \
  do {                                 \
    mla_status_t st_ = (expr);         \
    if (st_ != MLA_OK) return st_;     \
  } while (0)

// Checks of a paged cache and its chunk's sequence description, shared by the
// gathers and the paged pack; no CUDA call.  Each cache row is read from
// element row_off for row_len elements of size ce.
mla_status_t check_paged(const void* kv_cache, int64_t num_blocks, int32_t block_size,
                         int64_t block_stride, int64_t entry_stride, int64_t row_off,
                         int64_t row_len, int ce, const int32_t* block_table,
                         int64_t block_table_stride, const int32_t* cu, const int32_t* starts,
                         int32_t num_seqs) {
  if (num_seqs <= 0) return fail(MLA_ERR_INVALID_ARG, "num_seqs must be >= 1");
  if (block_size <= 0 || num_blocks <= 0 || block_table_stride <= 0)
    return fail(MLA_ERR_INVALID_ARG, "block_size, num_blocks and block_table_stride must be >= 1");
  if (row_off < 0 || row_len <= 0 || row_off + row_len > entry_stride)
    return fail(MLA_ERR_INVALID_ARG, "the row part read must lie in [0, entry_stride)");
  if (block_stride < (int64_t)(block_size - 1) * entry_stride + row_off + row_len)
    return fail(MLA_ERR_INVALID_ARG, "block_stride is too small for block_size entries");
  if (!a16(kv_cache) || !m16(block_stride * ce) || !m16(entry_stride * ce))
    return fail(MLA_ERR_MISALIGNED, "cache rows must start on 16-byte boundaries");
  if ((reinterpret_cast<uintptr_t>(block_table) | reinterpret_cast<uintptr_t>(cu) |
       reinterpret_cast<uintptr_t>(starts)) & 3)
    return fail(MLA_ERR_MISALIGNED, "int32 index arrays must be 4-byte aligned");
  return MLA_OK;
}

// The optional RMSNorm / RoPE description (no CUDA call): what it asks for
// and its layout checks.
mla_status_t check_norm_rope(const mla_norm_rope_t* nr, bool& norm, bool& rope) {
  norm = rope = false;
  if (!nr) return MLA_OK;
  norm = nr->gamma != nullptr;
  rope = nr->positions != nullptr;
  if (norm) {
    if (!a16(nr->gamma) || !m16(nr->gamma_layer_stride * 2))
      return fail(MLA_ERR_MISALIGNED, "gamma rows must start on 16-byte boundaries");
    if (!(nr->eps >= 0.0f) || !(nr->eps < 3.0e38f))
      return fail(MLA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  }
  if (rope) {
    if (!nr->cos_sin_cache || nr->max_position <= 0)
      return fail(MLA_ERR_INVALID_ARG, "RoPE needs cos_sin_cache and max_position >= 1");
    if (!a16(nr->cos_sin_cache))
      return fail(MLA_ERR_MISALIGNED, "cos_sin_cache must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(nr->positions) & 7)
      return fail(MLA_ERR_MISALIGNED, "positions must be 8-byte aligned");
  }
  return MLA_OK;
}

mla_status_t check_norm_rope_ptrs(const mla_norm_rope_t* nr, bool norm, bool rope) {
  if (norm) MLA_TRY(check_device_ptr(nr->gamma, "gamma"));
  if (rope) {
    MLA_TRY(check_device_ptr(nr->positions, "positions"));
    MLA_TRY(check_device_ptr(nr->cos_sin_cache, "cos_sin_cache"));
  }
  return MLA_OK;
}

mla::PagedSrc paged_src(const void* kv_cache, int64_t num_blocks, int32_t block_size,
                        int64_t block_stride, int64_t entry_stride, int ce,
                        const int32_t* block_table, int64_t block_table_stride,
                        const int32_t* cu, const int32_t* starts, int32_t num_seqs) {
  mla::PagedSrc p{};
  p.cache = static_cast<const uint8_t*>(kv_cache);
  p.block_stride = block_stride * ce;
  p.entry_stride = entry_stride * ce;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.bs_shift = log2_exact(block_size);
  p.block_table = block_table;
  p.bt_stride = block_table_stride;
  p.cu = cu;
  p.starts = starts;
  p.num_seqs = num_seqs;
  return p;
}

mla_status_t check_paged_ptrs(const int32_t* block_table, const int32_t* cu,
                              const int32_t* starts) {
  MLA_TRY(check_device_ptr(block_table, "block_table"));
  MLA_TRY(check_device_ptr(cu, "cu_chunk_lens"));
  return check_device_ptr(starts, "chunk_starts");
}

}  // namespace

namespace mla {

int capped_grid(const void* kernel, int threads, int64_t work_ctas, int dyn_smem) {
  struct Entry {
    int dev;
    const void* kernel;
    int threads;
    int smem;
    int resident;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  (void)cudaGetDevice(&dev);
  int resident = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry& e : cache)
      if (e.dev == dev && e.kernel == kernel && e.threads == threads && e.smem == dyn_smem)
        resident = e.resident;
    if (resident == 0) {
      int sms = 0, occ = 0;
      (void)cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      (void)cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, dyn_smem);
      (void)cudaGetLastError();
      resident = (sms > 0 ? sms : 1) * (occ > 0 ? occ : 1);
      cache.push_back(Entry{dev, kernel, threads, dyn_smem, resident});
    }
  }
  if (work_ctas < 1) work_ctas = 1;
  return static_cast<int>(work_ctas < resident ? work_ctas : resident);
}

}  // namespace mla

extern "C" {

int mla_dtype_from_string(const char* s) {
  if (!s) return -1;
  if (!strcmp(s, "auto") || !strcmp(s, "bfloat16")) return MLA_BF16;
  if (!strcmp(s, "fp8") || !strcmp(s, "fp8_e4m3")) return MLA_FP8_E4M3;
  if (!strcmp(s, "fp8_e5m2")) return MLA_FP8_E5M2;
  return -1;
}

const char* mla_last_error(void) { return g_err.c_str(); }

const char* mla_version(void) { return "mla_cache 1.0 sm_103a"; }

int mla_set_pdl(int enable) { return g_pdl.exchange(enable ? 1 : 0); }

int mla_set_bulk_copy(int mode) { return g_bulk.exchange(mode >= 0 && mode <= 2 ? mode : 1); }

int mla_set_pointer_checks(int enable) { return g_ptr_checks.exchange(enable ? 1 : 0); }

int mla_set_gather_early_tables(int enable) { return g_gather_early.exchange(enable ? 1 : 0); }

int mla_set_insert_early_tables(int enable) { return g_insert_early.exchange(enable ? 1 : 0); }

int mla_test_insert_timeout(uint64_t wait_limit_ns, int64_t skip_item) {
  if (wait_limit_ns == 0) wait_limit_ns = kDefaultWaitNs;
  g_wait_ns.store(wait_limit_ns);
  g_skip_item.store(skip_item < 0 ? -1 : skip_item);
  return 0;
}

mla_status_t mla_cache_insert_grouped(
    const void* kv_c, int64_t kvc_token_stride, int64_t kvc_layer_stride, const void* k_pe,
    int64_t kpe_token_stride, int64_t kpe_layer_stride, int32_t num_tokens, int32_t num_layers,
    int32_t kv_lora_rank, int32_t pe_dim, const int64_t* slot_mapping, int64_t slot_layer_stride,
    const int64_t* kv_cache_ptrs, const float* kv_scales, mla_dtype_t cache_dtype,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride,
    const mla_norm_rope_t* norm_rope, uint32_t* err_word, mla_stream_t stream) {
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens must be >= 0");
  if (num_layers <= 0) return fail(MLA_ERR_INVALID_ARG, "num_layers must be >= 1");
  if (num_layers > 128) return fail(MLA_ERR_UNSUPPORTED, "at most 128 layers per call are built");
  if (cache_dtype != MLA_BF16 && cache_dtype != MLA_FP8_E4M3 && cache_dtype != MLA_FP8_E5M2)
    return fail(MLA_ERR_INVALID_ARG,
                "cache_dtype must be MLA_BF16, MLA_FP8_E4M3 or MLA_FP8_E5M2; got %d",
                (int)cache_dtype);
  if (kv_lora_rank != 512 || pe_dim != 64)
    return fail(MLA_ERR_UNSUPPORTED,
                "only kv_lora_rank 512 and pe_dim 64 are built (got %d, %d)", kv_lora_rank,
                pe_dim);
  const bool fp8 = cache_dtype != MLA_BF16;
  if (fp8 && !kv_scales) return fail(MLA_ERR_INVALID_ARG, "FP8 grouped cache insert requires kv_scales");
  if (!fp8 && kv_scales)
    return fail(MLA_ERR_INVALID_ARG, "BF16 grouped cache insert does not use kv_scales");
  if (slot_layer_stride < 0) return fail(MLA_ERR_INVALID_ARG, "slot_layer_stride must be >= 0");
  if (block_size <= 0 || num_blocks <= 0)
    return fail(MLA_ERR_INVALID_ARG, "block_size and num_blocks must be >= 1");
  if (num_blocks > INT64_MAX / block_size)
    return fail(MLA_ERR_INVALID_ARG, "num_blocks * block_size overflows int64");
  if (entry_stride < kv_lora_rank + pe_dim)
    return fail(MLA_ERR_INVALID_ARG, "entry_stride must be >= kv_lora_rank + pe_dim");
  if (block_stride < (int64_t)(block_size - 1) * entry_stride + kv_lora_rank + pe_dim)
    return fail(MLA_ERR_INVALID_ARG, "block_stride is too small for block_size entries");
  const int ce = elt_size(cache_dtype);
  if (!a16(kv_c) || !m16(kvc_token_stride * 2) || !m16(kvc_layer_stride * 2))
    return fail(MLA_ERR_MISALIGNED, "kv_c rows must start on 16-byte boundaries");
  if (!a16(k_pe) || !m16(kpe_token_stride * 2) || !m16(kpe_layer_stride * 2))
    return fail(MLA_ERR_MISALIGNED, "k_pe rows must start on 16-byte boundaries");
  if (!m16(block_stride * ce) || !m16(entry_stride * ce))
    return fail(MLA_ERR_MISALIGNED, "cache block_stride / entry_stride must be multiples of 16 bytes");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7) || (reinterpret_cast<uintptr_t>(kv_cache_ptrs) & 7))
    return fail(MLA_ERR_MISALIGNED, "slot_mapping and kv_cache_ptrs must be 8-byte aligned");
  if (err_word && (reinterpret_cast<uintptr_t>(err_word) & 3))
    return fail(MLA_ERR_MISALIGNED, "err_word must be 4-byte aligned");
  bool norm = false, rope = false;
  MLA_TRY(check_norm_rope(norm_rope, norm, rope));
  if ((int64_t)((num_tokens + 3) / 4) * num_layers >= (int64_t(1) << 32))
    return fail(MLA_ERR_UNSUPPORTED, "num_tokens * num_layers is too large for one call");
  if (num_tokens == 0) return MLA_OK;  // empty inputs may have null data pointers
  if (!kv_c || !k_pe || !slot_mapping || !kv_cache_ptrs)
    return fail(MLA_ERR_INVALID_ARG, "kv_c, k_pe, slot_mapping and kv_cache_ptrs must be non-null");

  MLA_TRY(check_device_ptr(kv_c, "kv_c"));
  MLA_TRY(check_device_ptr(k_pe, "k_pe"));
  MLA_TRY(check_device_ptr(slot_mapping, "slot_mapping"));
  MLA_TRY(check_device_ptr(kv_cache_ptrs, "kv_cache_ptrs"));
  if (fp8) MLA_TRY(check_device_ptr(kv_scales, "kv_scales"));
  MLA_TRY(check_norm_rope_ptrs(norm_rope, norm, rope));

  mla::InsertArgs a{};
  a.kv_c = static_cast<const uint8_t*>(kv_c);
  a.kvc_ts = kvc_token_stride * 2;
  a.kvc_ls = kvc_layer_stride * 2;
  a.k_pe = static_cast<const uint8_t*>(k_pe);
  a.kpe_ts = kpe_token_stride * 2;
  a.kpe_ls = kpe_layer_stride * 2;
  a.num_rows = (int64_t)num_tokens * num_layers;
  a.num_tokens = num_tokens;
  a.num_layers = num_layers;
  a.slots = slot_mapping;
  a.slot_ls = slot_layer_stride;
  a.cache_ptrs = kv_cache_ptrs;
  a.scales = kv_scales;
  a.capacity = num_blocks * block_size;
  a.block_size = block_size;
  a.bs_shift = log2_exact(block_size);
  a.block_stride = block_stride * ce;
  a.entry_stride = entry_stride * ce;
  if (norm) {
    a.gamma = static_cast<const uint8_t*>(norm_rope->gamma);
    a.gamma_ls = norm_rope->gamma_layer_stride * 2;
    a.eps = norm_rope->eps;
  }
  if (rope) {
    a.positions = norm_rope->positions;
    a.cos_sin = norm_rope->cos_sin_cache;
    a.max_position = norm_rope->max_position;
  }
  a.err = err_word;
  a.bulk_mode = g_bulk.load();
  a.wait_limit_ns = g_wait_ns.load();
  a.skip_item = g_skip_item.load();
  a.early_tables = g_insert_early.load() != 0;
  return launched(mla::launch_insert(a, (int)cache_dtype, norm, rope, cfg_for(stream)),
                  "mla_cache_insert_grouped");
}

}  // extern "C"

namespace {

// The gathers: out_dtype == cache_dtype (raw) or MLA_BF16 from an fp8 cache
// (widened exactly, or times *dequant_scale when it is set).
// Validates a gather and fills its launch arguments (a.num_tokens == 0: valid,
// nothing to launch); *mode is 0 (raw copy) or the widened fp8 cache format.
mla_status_t gather_prep(const void* kv_cache, mla_dtype_t cache_dtype, int64_t num_blocks,
                         int32_t block_size, int64_t block_stride, int64_t entry_stride,
                         int32_t entry_dim, const int32_t* block_table,
                         int64_t block_table_stride, const int32_t* cu_chunk_lens,
                         const int32_t* chunk_starts, int32_t num_seqs, int32_t num_tokens,
                         void* out, int64_t out_row_stride, mla_dtype_t out_dtype,
                         const float* dequant_scale, uint32_t* err_word, mla::GatherArgs& a,
                         int* mode) {
  a = mla::GatherArgs{};
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens must be >= 0");
  if (!valid_dtype(cache_dtype) || !valid_dtype(out_dtype))
    return fail(MLA_ERR_INVALID_ARG, "cache_dtype / out_dtype must be an mla_dtype_t value");
  if (out_dtype != cache_dtype && !(!is16(cache_dtype) && is16(out_dtype)))
    return fail(MLA_ERR_UNSUPPORTED,
                "out_dtype must equal cache_dtype (raw) or be MLA_BF16 / MLA_FP16 from an fp8 "
                "cache");
  const int ce = elt_size(cache_dtype), oe = elt_size(out_dtype);
  MLA_TRY(check_paged(kv_cache, num_blocks, block_size, block_stride, entry_stride, 0, entry_dim,
                      ce, block_table, block_table_stride, cu_chunk_lens, chunk_starts,
                      num_seqs));
  if (out_row_stride < entry_dim) return fail(MLA_ERR_INVALID_ARG, "out_row_stride must be >= entry_dim");
  if (!m16((int64_t)entry_dim * ce))
    return fail(MLA_ERR_MISALIGNED, "entry_dim must span a multiple of 16 bytes");
  if ((int64_t)entry_dim * ce > 1536)
    return fail(MLA_ERR_UNSUPPORTED, "rows longer than 1536 bytes are not built");
  if (!a16(out) || !m16(out_row_stride * oe))
    return fail(MLA_ERR_MISALIGNED, "out rows must start on 16-byte boundaries");
  if (dequant_scale && (reinterpret_cast<uintptr_t>(dequant_scale) & 3))
    return fail(MLA_ERR_MISALIGNED, "k_scale must be 4-byte aligned");
  if (err_word && (reinterpret_cast<uintptr_t>(err_word) & 3))
    return fail(MLA_ERR_MISALIGNED, "err_word must be 4-byte aligned");
  *mode = (out_dtype == cache_dtype) ? 0 : (int)cache_dtype;
  a.num_tokens = num_tokens;
  if (num_tokens == 0) return MLA_OK;  // empty inputs may have null data pointers
  if (!kv_cache || !block_table || !cu_chunk_lens || !chunk_starts || !out)
    return fail(MLA_ERR_INVALID_ARG, "kv_cache, block_table, cu_chunk_lens, chunk_starts and out must be non-null");

  a.src = paged_src(kv_cache, num_blocks, block_size, block_stride, entry_stride, ce, block_table,
                    block_table_stride, cu_chunk_lens, chunk_starts, num_seqs);
  a.row_chunks = (int32_t)((int64_t)entry_dim * ce / 16);
  a.out = static_cast<uint8_t*>(out);
  a.out_rs = out_row_stride * oe;
  a.dequant_scale = dequant_scale;
  a.err = err_word;
  a.early_tables = g_gather_early.load() != 0;
  return MLA_OK;
}

// The device-pointer checks of a gather that gather_prep accepted with rows.
mla_status_t gather_ptr_checks(const void* kv_cache, const void* out, const int32_t* block_table,
                               const int32_t* cu_chunk_lens, const int32_t* chunk_starts,
                               const float* dequant_scale) {
  MLA_TRY(check_device_ptr(kv_cache, "kv_cache"));
  MLA_TRY(check_device_ptr(out, "out"));
  MLA_TRY(check_paged_ptrs(block_table, cu_chunk_lens, chunk_starts));
  if (dequant_scale) MLA_TRY(check_device_ptr(dequant_scale, "k_scale"));
  return MLA_OK;
}

mla_status_t gather_impl(const void* kv_cache, mla_dtype_t cache_dtype, int64_t num_blocks,
                         int32_t block_size, int64_t block_stride, int64_t entry_stride,
                         int32_t entry_dim, const int32_t* block_table,
                         int64_t block_table_stride, const int32_t* cu_chunk_lens,
                         const int32_t* chunk_starts, int32_t num_seqs, int32_t num_tokens,
                         void* out, int64_t out_row_stride, mla_dtype_t out_dtype,
                         const float* dequant_scale, uint32_t* err_word, mla_stream_t stream,
                         const char* what) {
  mla::GatherArgs a;
  int mode = 0;
  MLA_TRY(gather_prep(kv_cache, cache_dtype, num_blocks, block_size, block_stride, entry_stride,
                      entry_dim, block_table, block_table_stride, cu_chunk_lens, chunk_starts,
                      num_seqs, num_tokens, out, out_row_stride, out_dtype, dequant_scale,
                      err_word, a, &mode));
  if (num_tokens == 0) return MLA_OK;
  MLA_TRY(gather_ptr_checks(kv_cache, out, block_table, cu_chunk_lens, chunk_starts,
                            dequant_scale));
  return launched(mla::launch_gather(a, mode, (int)out_dtype, cfg_for(stream)), what);
}

// The packs: k_pe given as rows (paged == nullptr) or read from the paged
// cache at element rope_offset of each token's row (kpe_dtype = the cache's).
struct PagedKpe {
  const void* kv_cache;
  int64_t num_blocks;
  int32_t block_size;
  int64_t block_stride, entry_stride, rope_offset;
  const int32_t* block_table;
  int64_t block_table_stride;
  const int32_t* cu;
  const int32_t* starts;
  int32_t num_seqs;
};

// Validates a pack and fills its launch arguments (a.num_tokens == 0: valid,
// nothing to launch).
mla_status_t pack_prep(const void* k_nope, int64_t kn_token_stride, int64_t kn_head_stride,
                       const void* v, int64_t v_token_stride, int64_t v_head_stride,
                       mla_dtype_t in_dtype, const void* k_pe, int64_t kpe_token_stride, mla_dtype_t kpe_dtype,
                       const PagedKpe* paged, int32_t num_tokens, int32_t num_heads,
                       int32_t nope_dim, int32_t rope_dim, int32_t v_dim, void* key_out,
                       void* v_out, mla_dtype_t out_dtype, const float* out_scale,
                       uint32_t* err_word, mla::PackArgs& a) {
  a = mla::PackArgs{};
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens must be >= 0");
  if (num_heads <= 0) return fail(MLA_ERR_INVALID_ARG, "num_heads must be >= 1");
  if ((int64_t)num_tokens * ((num_heads + 3) / 4) >= (int64_t(1) << 32))
    return fail(MLA_ERR_UNSUPPORTED, "num_tokens * ceil(num_heads / 4) must be below 2^32");
  if (!valid_dtype(out_dtype) || !valid_dtype(kpe_dtype) || !valid_dtype(in_dtype))
    return fail(MLA_ERR_INVALID_ARG, "in_dtype / out_dtype / %s must be an mla_dtype_t value",
                paged ? "cache_dtype" : "kpe_dtype");
  if (!is16(in_dtype))
    return fail(MLA_ERR_UNSUPPORTED, "k_nope and v must be MLA_BF16 or MLA_FP16 (in_dtype)");
  if (nope_dim != 128 || rope_dim != 64 || v_dim != 128)
    return fail(MLA_ERR_UNSUPPORTED, "only nope 128, rope 64, v 128 are built (got %d, %d, %d)",
                nope_dim, rope_dim, v_dim);
  if (is16(out_dtype) && out_dtype != in_dtype)
    return fail(MLA_ERR_UNSUPPORTED, "a 16-bit output has the input's type (in_dtype)");
  if (is16(kpe_dtype) && kpe_dtype != in_dtype)
    return fail(MLA_ERR_UNSUPPORTED, "a 16-bit k_pe must have k_nope's type (in_dtype)");
  if (!is16(out_dtype) && !is16(kpe_dtype) && kpe_dtype != out_dtype)
    return fail(MLA_ERR_UNSUPPORTED,
                "an fp8 k_pe is copied raw, so it must have the fp8 output's format");
  if (is16(out_dtype) && out_scale)
    return fail(MLA_ERR_INVALID_ARG, "a 16-bit pack does not use out_scale");
  if (!a16(k_nope) || !m16(kn_token_stride * 2) || !m16(kn_head_stride * 2))
    return fail(MLA_ERR_MISALIGNED, "k_nope rows must start on 16-byte boundaries");
  if (v_out && (!a16(v) || !m16(v_token_stride * 2) || !m16(v_head_stride * 2)))
    return fail(MLA_ERR_MISALIGNED, "v rows must start on 16-byte boundaries");
  const int ke = elt_size(kpe_dtype);
  const int kpe_align = ke == 2 ? 15 : 7;
  if (paged) {
    MLA_TRY(check_paged(paged->kv_cache, paged->num_blocks, paged->block_size,
                        paged->block_stride, paged->entry_stride, paged->rope_offset, rope_dim,
                        ke, paged->block_table, paged->block_table_stride, paged->cu,
                        paged->starts, paged->num_seqs));
    if ((paged->rope_offset * ke) & kpe_align)
      return fail(MLA_ERR_MISALIGNED, "rope_offset must start k_pe on a %d-byte boundary",
                  kpe_align + 1);
  } else if ((reinterpret_cast<uintptr_t>(k_pe) & kpe_align) ||
             ((kpe_token_stride * ke) & kpe_align)) {
    return fail(MLA_ERR_MISALIGNED, "k_pe rows must start on %d-byte boundaries", kpe_align + 1);
  }
  if (!a16(key_out) || (v_out && !a16(v_out)))
    return fail(MLA_ERR_MISALIGNED, "key_out and v_out must be 16-byte aligned");
  if (out_scale && (reinterpret_cast<uintptr_t>(out_scale) & 3))
    return fail(MLA_ERR_MISALIGNED, "out_scale must be 4-byte aligned");
  if (err_word && (reinterpret_cast<uintptr_t>(err_word) & 3))
    return fail(MLA_ERR_MISALIGNED, "err_word must be 4-byte aligned");
  a.num_tokens = num_tokens;
  if (num_tokens == 0) return MLA_OK;  // empty inputs may have null data pointers
  if (!k_nope || !key_out || (v_out && !v))
    return fail(MLA_ERR_INVALID_ARG, "k_nope, key_out (and v when v_out is set) must be non-null");
  if (paged ? (!paged->kv_cache || !paged->block_table || !paged->cu || !paged->starts) : !k_pe)
    return fail(MLA_ERR_INVALID_ARG,
                paged ? "kv_cache, block_table, cu_chunk_lens and chunk_starts must be non-null"
                      : "k_pe must be non-null");

  a.k_nope = static_cast<const uint8_t*>(k_nope);
  a.kn_ts = kn_token_stride * 2;
  a.kn_hs = kn_head_stride * 2;
  a.v = static_cast<const uint8_t*>(v);
  a.v_ts = v_token_stride * 2;
  a.v_hs = v_head_stride * 2;
  a.k_pe = static_cast<const uint8_t*>(k_pe);
  a.kpe_ts = kpe_token_stride * ke;
  a.num_tokens = num_tokens;
  a.num_heads = num_heads;
  a.key = static_cast<uint8_t*>(key_out);
  a.vout = static_cast<uint8_t*>(v_out);
  a.out_scale = out_scale;
  a.err = err_word;
  if (paged) {
    a.paged = paged_src(paged->kv_cache, paged->num_blocks, paged->block_size,
                        paged->block_stride, paged->entry_stride, ke, paged->block_table,
                        paged->block_table_stride, paged->cu, paged->starts, paged->num_seqs);
    a.pe_off = paged->rope_offset * ke;
  }
  return MLA_OK;
}

// The device-pointer checks of a pack that pack_prep accepted with tokens.
mla_status_t pack_ptr_checks(const void* k_nope, const void* v, const void* k_pe,
                             const PagedKpe* paged, const void* key_out, const void* v_out,
                             const float* out_scale) {
  MLA_TRY(check_device_ptr(k_nope, "k_nope"));
  if (v_out) {
    MLA_TRY(check_device_ptr(v, "v"));
    MLA_TRY(check_device_ptr(v_out, "v_out"));
  }
  MLA_TRY(check_device_ptr(key_out, "key_out"));
  if (out_scale) MLA_TRY(check_device_ptr(out_scale, "out_scale"));
  if (paged) {
    MLA_TRY(check_device_ptr(paged->kv_cache, "kv_cache"));
    return check_paged_ptrs(paged->block_table, paged->cu, paged->starts);
  }
  return check_device_ptr(k_pe, "k_pe");
}

mla_status_t pack_impl(const void* k_nope, int64_t kn_token_stride, int64_t kn_head_stride,
                       const void* v, int64_t v_token_stride, int64_t v_head_stride,
                       mla_dtype_t in_dtype, const void* k_pe, int64_t kpe_token_stride, mla_dtype_t kpe_dtype,
                       const PagedKpe* paged, int32_t num_tokens, int32_t num_heads,
                       int32_t nope_dim, int32_t rope_dim, int32_t v_dim, void* key_out,
                       void* v_out, mla_dtype_t out_dtype, const float* out_scale,
                       uint32_t* err_word, mla_stream_t stream, const char* what) {
  mla::PackArgs a;
  MLA_TRY(pack_prep(k_nope, kn_token_stride, kn_head_stride, v, v_token_stride, v_head_stride,
                    in_dtype, k_pe, kpe_token_stride, kpe_dtype, paged, num_tokens, num_heads,
                    nope_dim, rope_dim, v_dim, key_out, v_out, out_dtype, out_scale, err_word, a));
  if (num_tokens == 0) return MLA_OK;
  MLA_TRY(pack_ptr_checks(k_nope, v, k_pe, paged, key_out, v_out, out_scale));
  return launched(mla::launch_pack(a, (int)in_dtype, (int)out_dtype, (int)kpe_dtype,
                                   paged != nullptr, cfg_for(stream)),
                  what);
}

// [lo, hi) byte span of rows of `row_bytes` at `rows` row starts `stride` apart
// (plus an inner head dimension), for the fused call's overlap check.
struct Span {
  uintptr_t lo, hi;
};
Span span_of(const void* base, int64_t rows, int64_t row_stride_b, int64_t heads,
             int64_t head_stride_b, int64_t row_bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(base);
  if (!base || rows <= 0) return Span{lo, lo};
  const int64_t last = (rows - 1) * row_stride_b + (heads - 1) * head_stride_b + row_bytes;
  return Span{lo, lo + (uintptr_t)last};
}
bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

}  // namespace

extern "C" {

mla_status_t mla_context_gather(const void* kv_cache, mla_dtype_t cache_dtype, int64_t num_blocks,
                                int32_t block_size, int64_t block_stride, int64_t entry_stride,
                                int32_t entry_dim, const int32_t* block_table,
                                int64_t block_table_stride, const int32_t* cu_chunk_lens,
                                const int32_t* chunk_starts, int32_t num_seqs, int32_t num_tokens,
                                void* out, int64_t out_row_stride, mla_dtype_t out_dtype,
                                uint32_t* err_word, mla_stream_t stream) {
  return gather_impl(kv_cache, cache_dtype, num_blocks, block_size, block_stride, entry_stride,
                     entry_dim, block_table, block_table_stride, cu_chunk_lens, chunk_starts,
                     num_seqs, num_tokens, out, out_row_stride, out_dtype, nullptr, err_word,
                     stream, "mla_context_gather");
}

mla_status_t mla_context_gather_scaled(const void* kv_cache, mla_dtype_t cache_dtype,
                                       int64_t num_blocks, int32_t block_size,
                                       int64_t block_stride, int64_t entry_stride,
                                       int32_t entry_dim, const int32_t* block_table,
                                       int64_t block_table_stride, const int32_t* cu_chunk_lens,
                                       const int32_t* chunk_starts, int32_t num_seqs,
                                       int32_t num_tokens, void* out, int64_t out_row_stride,
                                       const float* k_scale, uint32_t* err_word,
                                       mla_stream_t stream) {
  if (cache_dtype != MLA_FP8_E4M3 && cache_dtype != MLA_FP8_E5M2)
    return fail(valid_dtype(cache_dtype) ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG,
                "the scaled gather dequantises an fp8 cache (cache_dtype must be fp8)");
  if (!k_scale) return fail(MLA_ERR_INVALID_ARG, "k_scale must be non-null");
  return gather_impl(kv_cache, cache_dtype, num_blocks, block_size, block_stride, entry_stride,
                     entry_dim, block_table, block_table_stride, cu_chunk_lens, chunk_starts,
                     num_seqs, num_tokens, out, out_row_stride, MLA_BF16, k_scale, err_word,
                     stream, "mla_context_gather_scaled");
}

mla_status_t mla_context_kv_pack(const void* k_nope, int64_t kn_token_stride,
                                 int64_t kn_head_stride, const void* v, int64_t v_token_stride,
                                 int64_t v_head_stride, mla_dtype_t in_dtype, const void* k_pe,
                                 int64_t kpe_token_stride, mla_dtype_t kpe_dtype,
                                 int32_t num_tokens, int32_t num_heads, int32_t nope_dim,
                                 int32_t rope_dim, int32_t v_dim, void* key_out, void* v_out,
                                 mla_dtype_t out_dtype, const float* out_scale,
                                 uint32_t* err_word, mla_stream_t stream) {
  return pack_impl(k_nope, kn_token_stride, kn_head_stride, v, v_token_stride, v_head_stride,
                   in_dtype, k_pe, kpe_token_stride, kpe_dtype, nullptr, num_tokens, num_heads, nope_dim,
                   rope_dim, v_dim, key_out, v_out, out_dtype, out_scale, err_word, stream,
                   "mla_context_kv_pack");
}

mla_status_t mla_context_kv_pack_paged(
    const void* k_nope, int64_t kn_token_stride, int64_t kn_head_stride, const void* v,
    int64_t v_token_stride, int64_t v_head_stride, mla_dtype_t in_dtype, const void* kv_cache,
    mla_dtype_t cache_dtype, int64_t num_blocks, int32_t block_size, int64_t block_stride,
    int64_t entry_stride, int64_t rope_offset, const int32_t* block_table,
    int64_t block_table_stride, const int32_t* cu_chunk_lens, const int32_t* chunk_starts,
    int32_t num_seqs, int32_t num_tokens, int32_t num_heads, int32_t nope_dim, int32_t rope_dim,
    int32_t v_dim, void* key_out, void* v_out, mla_dtype_t out_dtype, const float* out_scale,
    uint32_t* err_word, mla_stream_t stream) {
  const PagedKpe pk{kv_cache,      num_blocks,   block_size,  block_stride,
                    entry_stride,  rope_offset,  block_table, block_table_stride,
                    cu_chunk_lens, chunk_starts, num_seqs};
  return pack_impl(k_nope, kn_token_stride, kn_head_stride, v, v_token_stride, v_head_stride,
                   in_dtype, nullptr, 0, cache_dtype, &pk, num_tokens, num_heads, nope_dim, rope_dim,
                   v_dim, key_out, v_out, out_dtype, out_scale, err_word, stream,
                   "mla_context_kv_pack_paged");
}

mla_status_t mla_norm_rope_grouped(const void* kv_c, int64_t kvc_token_stride,
                                   int64_t kvc_layer_stride, const void* k_pe,
                                   int64_t kpe_token_stride, int64_t kpe_layer_stride,
                                   int32_t num_tokens, int32_t num_layers, int32_t kv_lora_rank,
                                   int32_t pe_dim, const mla_norm_rope_t* norm_rope,
                                   void* kv_c_out, int64_t out_c_token_stride,
                                   int64_t out_c_layer_stride, void* k_pe_out,
                                   int64_t out_pe_token_stride, int64_t out_pe_layer_stride,
                                   uint32_t* err_word, mla_stream_t stream) {
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARG, "num_tokens must be >= 0");
  if (num_layers <= 0) return fail(MLA_ERR_INVALID_ARG, "num_layers must be >= 1");
  if (kv_lora_rank != 512 || pe_dim != 64)
    return fail(MLA_ERR_UNSUPPORTED,
                "only kv_lora_rank 512 and pe_dim 64 are built (got %d, %d)", kv_lora_rank,
                pe_dim);
  if (!a16(kv_c) || !m16(kvc_token_stride * 2) || !m16(kvc_layer_stride * 2))
    return fail(MLA_ERR_MISALIGNED, "kv_c rows must start on 16-byte boundaries");
  if (!a16(k_pe) || !m16(kpe_token_stride * 2) || !m16(kpe_layer_stride * 2))
    return fail(MLA_ERR_MISALIGNED, "k_pe rows must start on 16-byte boundaries");
  if (!a16(kv_c_out) || !m16(out_c_token_stride * 2) || !m16(out_c_layer_stride * 2))
    return fail(MLA_ERR_MISALIGNED, "kv_c_out rows must start on 16-byte boundaries");
  if (!a16(k_pe_out) || !m16(out_pe_token_stride * 2) || !m16(out_pe_layer_stride * 2))
    return fail(MLA_ERR_MISALIGNED, "k_pe_out rows must start on 16-byte boundaries");
  if (err_word && (reinterpret_cast<uintptr_t>(err_word) & 3))
    return fail(MLA_ERR_MISALIGNED, "err_word must be 4-byte aligned");
  bool norm = false, rope = false;
  MLA_TRY(check_norm_rope(norm_rope, norm, rope));
  if ((int64_t)num_tokens * num_layers + 3 >= (int64_t(1) << 32))
    return fail(MLA_ERR_UNSUPPORTED, "num_tokens * num_layers is too large for one call");
  if (num_tokens == 0) return MLA_OK;  // empty inputs may have null data pointers
  if (!kv_c || !k_pe || !kv_c_out || !k_pe_out)
    return fail(MLA_ERR_INVALID_ARG, "kv_c, k_pe, kv_c_out and k_pe_out must be non-null");
  MLA_TRY(check_device_ptr(kv_c, "kv_c"));
  MLA_TRY(check_device_ptr(k_pe, "k_pe"));
  MLA_TRY(check_device_ptr(kv_c_out, "kv_c_out"));
  MLA_TRY(check_device_ptr(k_pe_out, "k_pe_out"));
  MLA_TRY(check_norm_rope_ptrs(norm_rope, norm, rope));

  mla::NormRopeArgs a{};
  a.kv_c = static_cast<const uint8_t*>(kv_c);
  a.kvc_ts = kvc_token_stride * 2;
  a.kvc_ls = kvc_layer_stride * 2;
  a.k_pe = static_cast<const uint8_t*>(k_pe);
  a.kpe_ts = kpe_token_stride * 2;
  a.kpe_ls = kpe_layer_stride * 2;
  a.num_rows = (int64_t)num_tokens * num_layers;
  a.num_tokens = num_tokens;
  a.num_layers = num_layers;
  if (norm) {
    a.gamma = static_cast<const uint8_t*>(norm_rope->gamma);
    a.gamma_ls = norm_rope->gamma_layer_stride * 2;
    a.eps = norm_rope->eps;
  }
  if (rope) {
    a.positions = norm_rope->positions;
    a.cos_sin = norm_rope->cos_sin_cache;
    a.max_position = norm_rope->max_position;
  }
  a.out_c = static_cast<uint8_t*>(kv_c_out);
  a.oc_ts = out_c_token_stride * 2;
  a.oc_ls = out_c_layer_stride * 2;
  a.out_p = static_cast<uint8_t*>(k_pe_out);
  a.op_ts = out_pe_token_stride * 2;
  a.op_ls = out_pe_layer_stride * 2;
  a.err = err_word;
  return launched(mla::launch_norm_rope(a, norm, rope, cfg_for(stream)), "mla_norm_rope_grouped");
}

mla_status_t mla_context_kv_pack_gather(const mla_kv_pack_t* pack,
                                        const mla_context_gather_t* next_gather,
                                        uint32_t* gather_err_word, mla_stream_t stream) {
  if (!pack || !next_gather)
    return fail(MLA_ERR_INVALID_ARG, "pack and next_gather must be non-null");
  const mla_kv_pack_t& p = *pack;
  const mla_context_gather_t& g = *next_gather;
  if (!is16(p.in_dtype))
    return fail(valid_dtype(p.in_dtype) ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG,
                "k_nope and v must be MLA_BF16 or MLA_FP16 (in_dtype)");
  if (g.out_dtype != g.cache_dtype && g.out_dtype != p.in_dtype)
    return fail(MLA_ERR_UNSUPPORTED,
                "the gather's out_dtype must equal its cache_dtype (raw) or the pack's in_dtype "
                "(widened from an fp8 cache)");
  mla::PackArgs pa;
  MLA_TRY(pack_prep(p.k_nope, p.kn_token_stride, p.kn_head_stride, p.v, p.v_token_stride,
                    p.v_head_stride, p.in_dtype, p.k_pe, p.kpe_token_stride, p.kpe_dtype, nullptr,
                    p.num_tokens, p.num_heads, p.nope_dim, p.rope_dim, p.v_dim, p.key_out,
                    p.v_out, p.out_dtype, p.out_scale, nullptr, pa));
  mla::GatherArgs ga;
  int gmode = 0;
  MLA_TRY(gather_prep(g.kv_cache, g.cache_dtype, g.num_blocks, g.block_size, g.block_stride,
                      g.entry_stride, g.entry_dim, g.block_table, g.block_table_stride,
                      g.cu_chunk_lens, g.chunk_starts, g.num_seqs, g.num_tokens, g.out,
                      g.out_row_stride, g.out_dtype, nullptr, gather_err_word, ga, &gmode));
  if (p.num_tokens > 0 && g.num_tokens > 0) {
    // the gather writes nothing the pack reads or writes
    const int ie = 2, oe = elt_size(p.out_dtype), ke = elt_size(p.kpe_dtype);
    const Span out = span_of(g.out, g.num_tokens, g.out_row_stride * elt_size(g.out_dtype), 1, 0,
                             (int64_t)g.entry_dim * elt_size(g.out_dtype));
    const Span ins[] = {
        span_of(p.k_nope, p.num_tokens, p.kn_token_stride * ie, p.num_heads, p.kn_head_stride * ie,
                (int64_t)p.nope_dim * ie),
        p.v_out ? span_of(p.v, p.num_tokens, p.v_token_stride * ie, p.num_heads,
                          p.v_head_stride * ie, (int64_t)p.v_dim * ie)
                : Span{0, 0},
        span_of(p.k_pe, p.num_tokens, p.kpe_token_stride * ke, 1, 0, (int64_t)p.rope_dim * ke),
        span_of(p.key_out, p.num_tokens, (int64_t)p.num_heads * (p.nope_dim + p.rope_dim) * oe, 1,
                0, (int64_t)p.num_heads * (p.nope_dim + p.rope_dim) * oe),
        p.v_out ? span_of(p.v_out, p.num_tokens, (int64_t)p.num_heads * p.v_dim * oe, 1, 0,
                          (int64_t)p.num_heads * p.v_dim * oe)
                : Span{0, 0}};
    for (const Span& sp : ins)
      if (overlaps(out, sp))
        return fail(MLA_ERR_INVALID_ARG,
                    "the gather's output overlaps a buffer of the pack (use a second workspace)");
  }
  if (p.num_tokens > 0)
    MLA_TRY(pack_ptr_checks(p.k_nope, p.v, p.k_pe, nullptr, p.key_out, p.v_out, p.out_scale));
  if (g.num_tokens > 0)
    MLA_TRY(gather_ptr_checks(g.kv_cache, g.out, g.block_table, g.cu_chunk_lens, g.chunk_starts,
                              nullptr));
  if (p.num_tokens == 0 && g.num_tokens == 0) return MLA_OK;
  if (p.num_tokens == 0)
    return launched(mla::launch_gather(ga, gmode, (int)g.out_dtype, cfg_for(stream)),
                    "mla_context_kv_pack_gather");
  if (g.num_tokens == 0)
    return launched(mla::launch_pack(pa, (int)p.in_dtype, (int)p.out_dtype, (int)p.kpe_dtype,
                                     false, cfg_for(stream)),
                    "mla_context_kv_pack_gather");
  return launched(mla::launch_pack(pa, (int)p.in_dtype, (int)p.out_dtype, (int)p.kpe_dtype, false,
                                   cfg_for(stream), &ga, gmode),
                  "mla_context_kv_pack_gather");
}

mla_status_t mla_rope_cos_sin_cache(float* out, int64_t max_position, int32_t rot_dim,
                                    double base, mla_stream_t stream) {
  if (!out) return fail(MLA_ERR_INVALID_ARG, "out must be non-null");
  if (max_position <= 0 || rot_dim <= 0 || (rot_dim & 1))
    return fail(MLA_ERR_INVALID_ARG, "max_position must be >= 1 and rot_dim even and >= 2");
  if (!(base > 1.0) || !(base < 1e300)) return fail(MLA_ERR_INVALID_ARG, "base must be > 1");
  if (!a16(out)) return fail(MLA_ERR_MISALIGNED, "out must be 16-byte aligned");
  MLA_TRY(check_device_ptr(out, "out"));
  return launched(mla::launch_rope_table(out, max_position, rot_dim, base, cfg_for(stream)),
                  "mla_rope_cos_sin_cache");
}

}  // extern "C"
