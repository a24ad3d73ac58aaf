/*
 * mla_cache.h -- C ABI of libmla_cache, the GB300 (sm_103a) library for the
 * MLA latent-KV data-movement path:
 *
 *   1. the grouped multi-layer cache insert ("PR #55356 [Kimi Perf] Group fp8
 *      mla cache insertion", Implementation items 2-3 and Source snippets:
 *      concat_and_cache_mla_grouped), optionally preceded by the per-layer
 *      RMSNorm of kv_c and the RoPE rotation of k_pe that the DSpark drafter
 *      applies before it ("PR #50585 [K3 Perf] Optimize k3 dspark fused kv",
 *      Source snippets: _precompute_fused_context_kv);
 *   2. the chunked-context K/V pack: gather of latent rows from the paged cache
 *      with the conditional dtype cast, then the fused [k_nope | k_pe] key and V
 *      pack ("PR #51772 [Attention][MLA] Fuse Kimi-K3 chunked-context K/V
 *      packing", Implementation items 1-2 and Source snippets:
 *      fused_mla_kv_concat / fused_mla_kv_concat_quant_fp8).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Ownership: the caller owns every buffer.  The library allocates no memory,
 *   never synchronises the host with the device, and launches its kernels on
 *   the stream it is given (NULL = the legacy default stream).  Every call
 *   returns as soon as its launch is queued.
 * - Pointers: every data pointer is a DEVICE pointer on the current CUDA
 *   device unless the comment says otherwise.  Every pointer argument a kernel
 *   dereferences (inputs, outputs, per-layer cache pointer array, slot
 *   mapping, scales, positions, tables) is checked with
 *   cudaPointerGetAttributes; a host pointer, or device memory of another
 *   device, is rejected with MLA_ERR_INVALID_ARG before any launch.  These
 *   checks cost host time on every call (about one CUDA runtime query per
 *   pointer); a caller that guarantees its pointers can switch them off with
 *   mla_set_pointer_checks(0).  The per-layer cache bases inside
 *   kv_cache_ptrs live in device memory and are checked by the kernel only
 *   for null and alignment (MLA_ERRBIT_MISALIGNED).
 * - Strides and sizes are in ELEMENTS of the named tensor's element type.
 * - Alignment: every row that is read or written must start on a 16-byte
 *   boundary (base pointer and strides), else MLA_ERR_MISALIGNED.  There is no
 *   unaligned fallback.
 * - Outputs never alias inputs.
 * - Errors: arguments are validated synchronously, before any launch, and the
 *   call returns a status; the message of the last failure on the calling
 *   thread is returned by mla_last_error().  A failed launch returns
 *   MLA_ERR_CUDA.  Bad DATA found by a kernel (a slot or block id out of
 *   range, a position outside the rotary table, a misaligned per-layer cache
 *   pointer) never traps: the affected row is skipped (left untouched) and the
 *   matching MLA_ERRBIT_* is OR-ed into *err_word when err_word is not NULL.
 * - num_tokens == 0 returns MLA_OK and launches nothing.
 * - Kernels are launched with programmatic dependent launch enabled (each
 *   kernel waits for the previous grid on the stream before touching any
 *   memory), so back-to-back calls overlap launch latency while plain stream
 *   order holds for every argument; see mla_set_pdl().  A caller whose
 *   context-gather tables, or whose insert's per-layer cache pointers and
 *   scales, are complete before the call is enqueued may let the kernel read
 *   them before that wait (mla_set_gather_early_tables,
 *   mla_set_insert_early_tables).
 */
#ifndef MLA_CACHE_H
#define MLA_CACHE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t. */
typedef struct CUstream_st* mla_stream_t;

/* Element formats of caches, inputs and outputs.  The vLLM cache-dtype strings
 * map as "auto"/"bfloat16" -> MLA_BF16, "fp8"/"fp8_e4m3" -> MLA_FP8_E4M3,
 * "fp8_e5m2" -> MLA_FP8_E5M2 ("PR #55356", Source snippets: the host dtype
 * whitelist and the three template instances).  MLA_FP16 (IEEE binary16) is
 * an input / output format of the chunked-context path only: an fp16
 * kv_b_proj output into the pack, and the gather's widening for an fp16
 * kv_b_proj input ("PR #51772", Review: bf16 and fp16 inputs); the grouped
 * insert takes bf16 input and bf16 / fp8 caches only. */
typedef enum { MLA_BF16 = 0, MLA_FP8_E4M3 = 1, MLA_FP8_E5M2 = 2, MLA_FP16 = 3 } mla_dtype_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* a null / inconsistent / host-side argument */
  MLA_ERR_UNSUPPORTED = 2, /* a valid request the library does not implement */
  MLA_ERR_MISALIGNED = 3,  /* a row would not start on a 16-byte boundary */
  MLA_ERR_CUDA = 4         /* the CUDA runtime reported an error */
} mla_status_t;

/* Bits a kernel ORs into *err_word for data it skipped. */
enum {
  MLA_ERRBIT_SLOT_OOB = 1u,   /* slot >= num_blocks * block_size */
  MLA_ERRBIT_BLOCK_OOB = 2u,  /* block table index or block id out of range */
  MLA_ERRBIT_POS_OOB = 4u,    /* position outside [0, max_position) */
  MLA_ERRBIT_MISALIGNED = 8u, /* a per-layer cache base null or not 16-byte aligned */
  MLA_ERRBIT_TIMEOUT = 16u     /* a pipeline wait of the grouped insert gave up (see
                                  mla_cache_insert_grouped) */
};

/* Map a vLLM kv-cache-dtype string to mla_dtype_t; -1 if it is not one of
 * the five accepted strings.  Host only. */
int mla_dtype_from_string(const char* kv_cache_dtype);

/* Message of the last failed call on this thread ("" if none).  The pointer
 * stays valid until the next call on the same thread. */
const char* mla_last_error(void);

/* Library version string, e.g. "mla_cache 1.0 sm_103a". */
const char* mla_version(void);

/* Enable (1, the default) or disable (0) programmatic dependent launch for
 * every later launch from this process.  Returns the previous setting. */
int mla_set_pdl(int enable);

/* When the grouped insert uses its bulk-copy pipeline shape (shared-memory
 * staging by cp.async.bulk) for every later launch from this process:
 * 1 (the default) for calls of 131072 rows (tokens x layers) or more, or
 * 40960 rows or more with RMSNorm, 2 for every call, 0 never.  A call whose layout does not qualify, and every call
 * the mode leaves out, runs the row-per-warp shape.  Both shapes compute
 * identical results.  Returns the previous mode (other values set 1). */
int mla_set_bulk_copy(int mode);

/* Enable (1, the default) or disable (0), for every later call from this
 * process, the cudaPointerGetAttributes checks of pointer arguments (see the
 * conventions above).  With the checks off a host pointer is not caught
 * before the launch, and the kernel that dereferences it faults; every other
 * argument check still runs.  Returns the previous setting. */
int mla_set_pointer_checks(int enable);

/* Let the context gathers (mla_context_gather, mla_context_gather_scaled)
 * read block_table, cu_chunk_lens and chunk_starts BEFORE they wait for the
 * previous grid on the stream (1), or keep plain stream order (0, the
 * default), for every later call from this process.  With 1 and PDL on, those
 * three arrays must be complete before the call is enqueued, or be written by
 * stream work that does not trigger its dependents early (a copy, a host
 * write or an ordinary kernel is fine; a kernel that executes
 * griddepcontrol.launch_dependents before it has written them is not): the
 * gather's first table lookups then overlap the previous kernel's tail.
 * Returns the previous setting. */
int mla_set_gather_early_tables(int enable);

/* Let the grouped insert (mla_cache_insert_grouped) read kv_cache_ptrs,
 * kv_scales and the RMSNorm gamma BEFORE it waits for the previous grid on
 * the stream (1), or keep plain stream order (0, the default), for every
 * later call from this process.  The same contract as
 * mla_set_gather_early_tables: with 1 and PDL on, those arrays must be
 * complete before the call is enqueued, or be written by stream work that
 * does not trigger its dependents early.  The per-layer table (cache bases,
 * division constants; in the bulk-copy shape also whether a layer's gamma
 * bound lets normalised rows skip the special-value test) is then built while
 * the previous kernel finishes: row-per-warp calls of 2048 rows (tokens x
 * layers) or more (4096 tokens x 5 layers back to back: 10.4 vs 11.0 us) and
 * bulk-copy calls (8192 tokens x 5 layers: 17.2 vs 17.4 us); smaller calls
 * read them after the wait either way.  Results are identical.  Returns the
 * previous setting. */
int mla_set_insert_early_tables(int enable);

/* TESTING HOOK for the grouped insert's bulk-copy pipeline, applied to every
 * later call from this process (not for production use).  wait_limit_ns: how
 * long a pipeline wait may last before the kernel gives up (0 restores the
 * default of 2 s).  skip_item >= 0: the producer of the pipeline's first CTA
 * issues no copies for its local work item skip_item (a run of up to 4 tokens
 * of one layer), so the consumer waiting for it runs out of time; -1 (the
 * default) skips nothing.  A kernel that gives up sets MLA_ERRBIT_TIMEOUT,
 * stops issuing work, waits (bounded by the same limit) for the copies it has
 * issued, and returns; the rows it had not written are left untouched.
 * Returns 0. */
int mla_test_insert_timeout(uint64_t wait_limit_ns, int64_t skip_item);

/*
 * Optional pre-processing of the grouped insert ("PR #50585", Source snippets:
 * ops.rms_norm with a [L, kv_lora_rank] weight, then the rotary embedding with
 * the token positions repeated for every layer).  Pass NULL for a raw insert.
 *
 *   gamma               bf16 [L, kv_lora_rank], layer l's row at
 *                       l * gamma_layer_stride; NULL = no RMSNorm.
 *                       y = x / sqrt(mean(x^2) + eps) * gamma[l], in fp32,
 *                       rounded to bf16 (round to nearest even).
 *   eps                 RMSNorm epsilon (>= 0).
 *   positions           int64 [num_tokens], the same for every layer;
 *                       NULL = no RoPE.
 *   cos_sin_cache       fp32 [max_position, pe_dim]; row p = cos(p f_i) for
 *                       i < pe_dim/2 then sin(p f_i) (see
 *                       mla_rope_cos_sin_cache).  Neox pairing: element i
 *                       rotates with element i + pe_dim/2; the result is
 *                       rounded to bf16.
 *   max_position        rows of cos_sin_cache; a position outside
 *                       [0, max_position) skips the row (MLA_ERRBIT_POS_OOB).
 * The rounded bf16 values are what the fp8 conversion then divides by k_scale.
 */
typedef struct {
  const void* gamma;
  int64_t gamma_layer_stride;
  float eps;
  const int64_t* positions;
  const float* cos_sin_cache;
  int64_t max_position;
} mla_norm_rope_t;

/*
 * Grouped multi-layer MLA cache insert, all layers in ONE launch
 * ("PR #55356 [Kimi Perf] Group fp8 mla cache insertion", Source snippets:
 * concat_and_cache_mla_grouped_kernel and its host function; the result must
 * equal one single-layer insert per layer, test_concat_and_cache_mla_grouped).
 *
 * For every layer l < num_layers and token t < num_tokens:
 *   s = slot_mapping[l * slot_layer_stride + t]      (slot_layer_stride 0 =
 *       one mapping shared by all layers); s < 0 is padding and is skipped;
 *   row = [kv_c[l, t, 0:kv_lora_rank] | k_pe[l, t, 0:pe_dim]]   (bf16),
 *       after the optional RMSNorm / RoPE of norm_rope;
 *   cache_l = (element type*) kv_cache_ptrs[l];
 *   cache_l[(s / block_size) * block_stride + (s % block_size) * entry_stride
 *           + i] = row[i]                 for a bf16 cache (the bf16 bits), or
 *           = fp8(float(row[i]) / kv_scales[l])  for an fp8 cache, with
 *           round-to-nearest-even and saturation to +-max (448 for e4m3, 57344
 *           for e5m2), the quotient an IEEE fp32 division.
 *
 *   kv_c, k_pe          bf16; element (l, t, i) at l * layer_stride +
 *                       t * token_stride + i.  Both [L, T, .] layer-major
 *                       buffers and the DSpark projection output [T, L, 576]
 *                       (kv_c = base, k_pe = base + 512) are accepted as is.
 *   kv_lora_rank, pe_dim  must be 512 and 64 (else MLA_ERR_UNSUPPORTED).
 *   slot_mapping        int64 device array.
 *   kv_cache_ptrs       int64 device array [num_layers] of cache base
 *                       addresses (each 16-byte aligned).
 *   kv_scales           fp32 device array [num_layers]: required for an fp8
 *                       cache, must be NULL for a bf16 cache.
 *   num_blocks, block_size, block_stride, entry_stride
 *                       the paged layout shared by every layer's cache
 *                       (elements of the cache type).
 *   norm_rope           NULL, or the optional RMSNorm / RoPE (above).
 *   err_word            NULL, or a device uint32 that receives MLA_ERRBIT_*.
 * num_layers must be at most 128 (else MLA_ERR_UNSUPPORTED).
 * Valid slots must be distinct within a layer (else the row written last is
 * unspecified).
 * For 131072 or more rows (40960 with RMSNorm) with dense layer-major inputs
 * (token strides 512 and 64), the bulk-copy pipeline shape runs (see
 * mla_set_bulk_copy).  Its waits between the copy-issuing warp and the
 * computing warps are bounded by wall-clock time (2 s); one that runs out
 * (which means a fault, or a CTA stalled for seconds, e.g. by a debugger or a
 * time-sliced GPU) makes the kernel stop, and the rows it had not yet written
 * are left untouched.  err_word then receives MLA_ERRBIT_TIMEOUT: it is the
 * only signal of those dropped rows, so pass one when that matters.
 */
mla_status_t mla_cache_insert_grouped(
    const void* kv_c, int64_t kvc_token_stride, int64_t kvc_layer_stride,
    const void* k_pe, int64_t kpe_token_stride, int64_t kpe_layer_stride,
    int32_t num_tokens, int32_t num_layers, int32_t kv_lora_rank, int32_t pe_dim,
    const int64_t* slot_mapping, int64_t slot_layer_stride, const int64_t* kv_cache_ptrs,
    const float* kv_scales, mla_dtype_t cache_dtype, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, const mla_norm_rope_t* norm_rope,
    uint32_t* err_word, mla_stream_t stream);

/*
 * Gather latent rows of context chunks from a paged cache, with the optional
 * exact widening fp8 -> bf16 or fp16 ("PR #51772", Implementation item 2:
 * _gather_context_latent, then the conditional .to() of item 5; no scale is
 * applied, a plain fp8 gather returns fp8).
 *
 * Sequence s < num_seqs owns output rows [cu_chunk_lens[s], cu_chunk_lens[s+1]);
 * output row i of sequence s holds context position
 *   p = chunk_starts[s] + (i - cu_chunk_lens[s]),
 * stored in block blk = block_table[s * block_table_stride + p / block_size]
 * at offset p % block_size:
 *   out[i * out_row_stride + e] = cache[blk * block_stride +
 *                                       (p % block_size) * entry_stride + e],
 * for e < entry_dim, copied raw (out_dtype == cache_dtype) or widened exactly
 * (cache fp8, out_dtype MLA_BF16 or MLA_FP16: the kv_b_proj input's type; a
 * NaN code gives that format's quiet NaN with the code's sign).
 *
 *   block_table         int32 device [num_seqs, block_table_stride]; the row
 *                       width is block_table_stride.  A table index outside
 *                       the row or a block id outside [0, num_blocks) skips the
 *                       output row (MLA_ERRBIT_BLOCK_OOB).
 *   cu_chunk_lens       int32 device [num_seqs + 1], non-decreasing.
 *   chunk_starts        int32 device [num_seqs].
 *   num_tokens          output rows; rows owned by no sequence are untouched.
 * See mla_set_gather_early_tables for when the tables are read.
 */
mla_status_t mla_context_gather(
    const void* kv_cache, mla_dtype_t cache_dtype, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, int32_t entry_dim, const int32_t* block_table,
    int64_t block_table_stride, const int32_t* cu_chunk_lens, const int32_t* chunk_starts,
    int32_t num_seqs, int32_t num_tokens, void* out, int64_t out_row_stride,
    mla_dtype_t out_dtype, uint32_t* err_word, mla_stream_t stream);

/*
 * The gather of mla_context_gather from an fp8 cache into bf16, dequantised:
 *   out[i * out_row_stride + e] = bf16(fp32(value(code) * *k_scale))
 * the exact value of the fp8 code times the scale as ONE fp32 multiplication
 * (round to nearest even), then rounded to bf16 (round to nearest even).  A NaN
 * code gives the quiet NaN with the code's sign (0x7FC0 | sign); any other NaN
 * product (an infinity times zero, a NaN scale) gives 0x7FC0.
 *
 * For caches written with a k_scale other than 1: the insert stores
 * value / k_scale ("PR #55356", Source snippets: scaled_convert with the
 * layer's scale), and the chunked-context path casts the gathered latent to a
 * bf16 kv_b_proj input ("PR #51772", Implementation items 2 and 5, where the
 * cast is a plain .to()); this is that cast with the scale applied.
 *
 *   cache_dtype   MLA_FP8_E4M3 or MLA_FP8_E5M2 (else UNSUPPORTED).
 *   out           bf16 rows, 16-byte aligned row starts.
 *   k_scale       device fp32 scalar (required).
 * Every other argument, the row rules and the error bits are those of
 * mla_context_gather.
 */
mla_status_t mla_context_gather_scaled(
    const void* kv_cache, mla_dtype_t cache_dtype, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, int32_t entry_dim, const int32_t* block_table,
    int64_t block_table_stride, const int32_t* cu_chunk_lens, const int32_t* chunk_starts,
    int32_t num_seqs, int32_t num_tokens, void* out, int64_t out_row_stride,
    const float* k_scale, uint32_t* err_word, mla_stream_t stream);

/*
 * Chunked-context K/V pack: one launch writes the contiguous full key
 * [k_nope | k_pe] and V from the strided kv_b_proj output and a k_pe that may
 * still be in the fp8 cache layout ("PR #51772", Source snippets:
 * fused_mla_kv_concat and fused_mla_kv_concat_quant_fp8; Implementation item 1:
 * strided inputs, k_pe broadcast over heads, fp8 cast by the native pairwise
 * converters, capped grid with a grid-stride loop).
 *
 *   key_out[t, h, i]          = conv(k_nope[t, h, i])        i < nope_dim
 *   key_out[t, h, nope_dim+j] = kpe(k_pe[t, j])               j < rope_dim
 *   v_out[t, h, i]            = conv(v[t, h, i])              i < v_dim
 * with conv = identity for a 16-bit output (of the input's type) and
 * fp8(float(e) / *out_scale) (round to nearest even, saturating) for fp8
 * output; kpe = conv for a 16-bit k_pe, the raw byte for an fp8 k_pe into an
 * fp8 key of the same format (no rescale), and the exact unscaled widening for
 * an fp8 k_pe into a 16-bit key.
 *
 *   k_nope, v           element (t, h, i) at t * token_stride +
 *                       h * head_stride + i (e.g. the two halves of a
 *                       [T, H, nope + v] kv_b_proj output, row stride 4160).
 *   in_dtype            their type: MLA_BF16 or MLA_FP16 ("PR #51772",
 *                       Review: bf16 and fp16 inputs).
 *   k_pe                [T, rope_dim] with row stride kpe_token_stride, of type
 *                       kpe_dtype (in_dtype, or the cache's fp8).
 *   nope_dim, rope_dim, v_dim  must be 128, 64, 128 (else UNSUPPORTED).
 *   num_heads           any >= 1, with num_tokens * ceil(num_heads / 4) < 2^32.
 *   out_dtype           in_dtype, MLA_FP8_E4M3 or MLA_FP8_E5M2.
 *   key_out             contiguous [T, H, nope_dim + rope_dim] of out_dtype.
 *   v_out               contiguous [T, H, v_dim] of out_dtype, or NULL = no V.
 *   out_scale           device fp32 scalar for fp8 output (NULL = 1.0); must be
 *                       NULL for a 16-bit output.
 *   err_word            NULL, or a device uint32 for MLA_ERRBIT_* (this pack
 *                       reads no indices, so no condition sets a bit; the paged
 *                       pack below sets MLA_ERRBIT_BLOCK_OOB).
 */
mla_status_t mla_context_kv_pack(
    const void* k_nope, int64_t kn_token_stride, int64_t kn_head_stride, const void* v,
    int64_t v_token_stride, int64_t v_head_stride, mla_dtype_t in_dtype, const void* k_pe,
    int64_t kpe_token_stride,
    mla_dtype_t kpe_dtype, int32_t num_tokens, int32_t num_heads, int32_t nope_dim,
    int32_t rope_dim, int32_t v_dim, void* key_out, void* v_out, mla_dtype_t out_dtype,
    const float* out_scale, uint32_t* err_word, mla_stream_t stream);

/*
 * The pack of mla_context_kv_pack with k_pe read straight from the paged cache
 * instead of a gathered workspace ("PR #51772", Implementation item 1: the
 * kernel consumes a k_pe still in the fp8 cache layout; here that layout is
 * the cache itself, so the gather before it only needs the kv_c columns).
 *
 * Token t's k_pe is the rope_dim elements at rope_offset of the cache row that
 * mla_context_gather would copy into output row t (same sequence, position and
 * block-table rules), of the cache's element type:
 *   key_out[t, h, nope_dim + j] = kpe(row_t[rope_offset + j])
 * with kpe as in mla_context_kv_pack for kpe_dtype = cache_dtype (raw bytes for
 * an fp8 cache into an fp8 key of its format, the exact widening into a 16-bit
 * key, the output conversion for a 16-bit cache of in_dtype's type).  k_nope and V are packed as in
 * mla_context_kv_pack for every token.  A token whose row is not found keeps
 * the rope slice of its key untouched: silently when no sequence owns it, and
 * with MLA_ERRBIT_BLOCK_OOB when its block index or block id is out of range.
 *
 *   kv_cache ... chunk_starts   the paged cache and the chunk's sequences, as
 *                               in mla_context_gather; cache rows must start
 *                               on 16-byte boundaries.
 *   rope_offset                 element offset of k_pe in a cache row
 *                               (kv_lora_rank, 512); rope_offset * element size
 *                               a multiple of 16 (bf16) or 8 (fp8) bytes.
 *   num_tokens                  the chunk's tokens (kv_b_proj output rows).
 * Every other argument is that of mla_context_kv_pack.
 */
mla_status_t mla_context_kv_pack_paged(
    const void* k_nope, int64_t kn_token_stride, int64_t kn_head_stride, const void* v,
    int64_t v_token_stride, int64_t v_head_stride, mla_dtype_t in_dtype, const void* kv_cache,
    mla_dtype_t cache_dtype,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride,
    int64_t rope_offset, const int32_t* block_table, int64_t block_table_stride,
    const int32_t* cu_chunk_lens, const int32_t* chunk_starts, int32_t num_seqs,
    int32_t num_tokens, int32_t num_heads, int32_t nope_dim, int32_t rope_dim, int32_t v_dim,
    void* key_out, void* v_out, mla_dtype_t out_dtype, const float* out_scale,
    uint32_t* err_word, mla_stream_t stream);

/*
 * The arguments of mla_context_kv_pack (non-paged) and of mla_context_gather
 * as structs, for mla_context_kv_pack_gather below.  Each field has the
 * meaning, layout and rules of the same-named argument there.
 */
typedef struct {
  const void* k_nope;
  int64_t kn_token_stride, kn_head_stride;
  const void* v;
  int64_t v_token_stride, v_head_stride;
  mla_dtype_t in_dtype;
  const void* k_pe;
  int64_t kpe_token_stride;
  mla_dtype_t kpe_dtype;
  int32_t num_tokens, num_heads, nope_dim, rope_dim, v_dim;
  void* key_out;
  void* v_out;
  mla_dtype_t out_dtype;
  const float* out_scale;
} mla_kv_pack_t;

typedef struct {
  const void* kv_cache;
  mla_dtype_t cache_dtype;
  int64_t num_blocks;
  int32_t block_size;
  int64_t block_stride, entry_stride;
  int32_t entry_dim;
  const int32_t* block_table;
  int64_t block_table_stride;
  const int32_t* cu_chunk_lens;
  const int32_t* chunk_starts;
  int32_t num_seqs, num_tokens;
  void* out;
  int64_t out_row_stride;
  mla_dtype_t out_dtype;
} mla_context_gather_t;

/*
 * The pack of one context chunk and the gather of the NEXT chunk's latent
 * rows in one launch: the result equals mla_context_kv_pack(*pack) followed by
 * mla_context_gather(*next_gather) (gather errors into gather_err_word).
 *
 * In the chunked-context loop ("PR #51772 [Attention][MLA] Fuse Kimi-K3
 * chunked-context K/V packing", Implementation items 1-2: per chunk, gather
 * the latent rows, run kv_b_proj on them, then pack the key and V), chunk
 * c + 1's gather depends only on the cache and its tables, so with two gather
 * workspaces it can run inside chunk c's pack launch:
 *     gather(0); for c: kv_b_proj(c); pack(c) + gather(c + 1) in one call
 * -- one launch per chunk instead of two, with the gather's dependent row
 * lookups overlapping the pack's streaming.
 *
 * Rules: those of the two calls, plus:
 *   - the gather's out_dtype is its cache_dtype (raw copy) or the pack's
 *     in_dtype (an fp8 cache widened exactly); no scaled dequantisation;
 *   - the gather's output rows must not overlap any buffer of the pack
 *     (k_nope, v, k_pe, key_out, v_out; checked: MLA_ERR_INVALID_ARG) -- in
 *     particular the pack's k_pe must come from the OTHER workspace;
 *   - key_out and v_out must not overlap the gather's cache or tables (not
 *     checked; the two halves run concurrently, so such an overlap would not
 *     give the result of the two calls in sequence);
 *   - either num_tokens may be 0 (that half is skipped).
 * With mla_set_gather_early_tables(1) the gather's tables are read before the
 * launch waits for the previous grid, as for mla_context_gather.
 */
mla_status_t mla_context_kv_pack_gather(const mla_kv_pack_t* pack,
                                        const mla_context_gather_t* next_gather,
                                        uint32_t* gather_err_word, mla_stream_t stream);

/*
 * Grouped RMSNorm + RoPE on its own, for when the grouped insert is not the
 * consumer ("PR #50585 [K3 Perf] Optimize k3 dspark fused kv", Implementation
 * item 3 and Source snippets: _precompute_fused_context_kv splits the
 * [num_ctx, L, 576] context projection into kv_c and k_pe, makes both
 * layer-major, normalises kv_c with one weight row per layer and rotates k_pe
 * with the token positions repeated for every layer).  One pass: for every
 * layer l < num_layers and token t < num_tokens,
 *   kv_c_out[t, l, :] = rmsnorm(kv_c[t, l, :], gamma[l])   (a copy without gamma)
 *   k_pe_out[t, l, :] = rope(k_pe[t, l, :], positions[t])  (a copy without positions)
 * with the arithmetic, rounding and table of mla_norm_rope_t (the same as the
 * grouped insert's, so its bf16 results are identical).  A position outside
 * [0, max_position) skips the row in both outputs (MLA_ERRBIT_POS_OOB).
 *
 *   kv_c, k_pe          bf16 inputs, element (t, l, i) at t * token_stride +
 *                       l * layer_stride + i; for the [T, L, 576] projection
 *                       read in place: kv_c = base, k_pe = base + 512, token
 *                       stride L * 576, layer stride 576.  Rows start on
 *                       16-byte boundaries.
 *   kv_lora_rank, pe_dim  must be 512 and 64 (else UNSUPPORTED).
 *   norm_rope           as for the grouped insert; NULL = the plain layout
 *                       change.
 *   kv_c_out, k_pe_out  bf16 outputs addressed the same way with their own
 *                       strides (layer-major [L, T, 512] / [L, T, 64]: token
 *                       stride 512 / 64, layer stride T * 512 / T * 64); they
 *                       must not overlap the inputs.  Rows start on 16-byte
 *                       boundaries.
 *   num_tokens * num_layers < 2^32.
 */
mla_status_t mla_norm_rope_grouped(
    const void* kv_c, int64_t kvc_token_stride, int64_t kvc_layer_stride, const void* k_pe,
    int64_t kpe_token_stride, int64_t kpe_layer_stride, int32_t num_tokens, int32_t num_layers,
    int32_t kv_lora_rank, int32_t pe_dim, const mla_norm_rope_t* norm_rope, void* kv_c_out,
    int64_t out_c_token_stride, int64_t out_c_layer_stride, void* k_pe_out,
    int64_t out_pe_token_stride, int64_t out_pe_layer_stride, uint32_t* err_word,
    mla_stream_t stream);

/*
 * Fill the rotary cos/sin table the insert's RoPE reads ("PR #50585", Source
 * snippets: the k_pe rotation; the table is the rotary embedding's cached
 * cos/sin): out[p * rot_dim + i] = cos(p * base^(-2i/rot_dim)) and
 * out[p * rot_dim + rot_dim/2 + i] = sin(same), for p < max_position and
 * i < rot_dim/2, evaluated in double precision and rounded to fp32.
 *   out  fp32 device [max_position, rot_dim], 16-byte aligned; rot_dim even.
 */
mla_status_t mla_rope_cos_sin_cache(float* out, int64_t max_position, int32_t rot_dim,
                                    double base, mla_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MLA_CACHE_H */
