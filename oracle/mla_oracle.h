/*
 * mla_oracle.h -- plain, slow, single-threaded CPU oracle for the MLA latent-KV
 * data-movement path (grouped multi-layer cache insert, context gather,
 * chunked-context K/V pack).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library under pack_mla_cache_gb300/) shares no code with it and never
 * calls it.
 *
 * Sources the oracle follows (each function below names its passage):
 *   [P1] "PR #51772 [Attention][MLA] Fuse Kimi-K3 chunked-context K/V packing"
 *        -- Implementation items 1-2, Source snippets (fused_mla_kv_concat,
 *        fused_mla_kv_concat_quant_fp8), Review.
 *   [P2] "PR #50585 [K3 Perf] Optimize k3 dspark fused kv" -- Source snippets
 *        (_precompute_fused_context_kv: grouped RMSNorm, RoPE with positions
 *        repeated per layer).
 *   [P3] "PR #55356 [Kimi Perf] Group fp8 mla cache insertion" -- Implementation
 *        items 2-3, Source snippets (concat_and_cache_mla_grouped_kernel and its
 *        host function), test_concat_and_cache_mla_grouped.
 *   [OFP8] OCP 8-bit Floating Point Specification (OFP8), rev. 1.0: the E4M3
 *        (no infinities, single NaN mantissa pattern) and E5M2 (IEEE-like)
 *        encodings.
 *   [IEEE] IEEE 754-2008 binary16 (fp16): 1 sign, 5 exponent (bias 15), 10
 *        mantissa bits, subnormals, infinities and NaNs.
 *
 * All floating point arithmetic that produces a rounded result is done in
 * double precision and rounded ONCE to the target format with round-to-nearest,
 * ties-to-even.  The one exception is the fp8 cache conversion, whose operand
 * the pages fix as an fp32 value: float(bf16 value) / k_scale is an IEEE fp32
 * division (the file is compiled with -ffp-contract=off), and that exact fp32
 * value is then rounded to fp8.
 *
 * Status: every function here is pinned by tests/test_oracle_*.py against
 * format definitions, library routines, closed forms and brute force; none is
 * "parity unpinned".
 */
#ifndef MLA_ORACLE_H
#define MLA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Cache / tensor element formats.  Numbering matches the product's public
 * enum by convention only; the oracle defines its own. */
enum { ORC_BF16 = 0, ORC_FP8_E4M3 = 1, ORC_FP8_E5M2 = 2, ORC_F16 = 3 };

/* Error bits returned by the row-skipping functions. */
enum { ORC_ERR_SLOT_OOB = 1u, ORC_ERR_BLOCK_OOB = 2u, ORC_ERR_POS_OOB = 4u };

/* ---- scalar codecs ------------------------------------------------------ */
uint16_t orc_bf16_from_f64(double x);
uint16_t orc_bf16_from_f32(float x);
double orc_bf16_to_f64(uint16_t b);
uint8_t orc_fp8_from_f32(float x, int fmt);
double orc_fp8_to_f64(uint8_t c, int fmt);
uint16_t orc_bf16_from_fp8(uint8_t c, int fmt);
uint16_t orc_f16_from_f64(double x);
double orc_f16_to_f64(uint16_t h);
uint16_t orc_f16_from_fp8(uint8_t c, int fmt);

/* ---- array forms of the codecs (for exhaustive tests) ------------------- */
void orc_fp8_encode_f32_array(const float* x, int64_t n, int fmt, uint8_t* out);
void orc_fp8_decode_array(const uint8_t* c, int64_t n, int fmt, double* out);
void orc_bf16_from_f64_array(const double* x, int64_t n, uint16_t* out);
void orc_bf16_from_f32_array(const float* x, int64_t n, uint16_t* out);

/* ---- RMSNorm and RoPE on one row ---------------------------------------- */
void orc_rope_cos_sin_cache(int64_t max_position, int32_t rot_dim, double base, float* out);
void orc_rms_norm_row(const uint16_t* x, const uint16_t* gamma, int32_t n, float eps,
                      uint16_t* y);
void orc_rope_neox_row(const uint16_t* x, const float* cos_sin_row, int32_t rot_dim,
                       uint16_t* y);

/* ---- grouped multi-layer cache insert ----------------------------------- */
uint32_t orc_insert_layer(const uint16_t* kv_c, int64_t kvc_token_stride,
                          const uint16_t* k_pe, int64_t kpe_token_stride, int32_t num_tokens,
                          int32_t kv_lora_rank, int32_t pe_dim, const int64_t* slot_mapping,
                          void* cache, int32_t cache_dtype, int64_t num_blocks,
                          int32_t block_size, int64_t block_stride, int64_t entry_stride,
                          float k_scale, const uint16_t* gamma, float eps,
                          const int64_t* positions, const float* cos_sin_cache,
                          int64_t max_position);

uint32_t orc_insert_grouped(const uint16_t* kv_c, int64_t kvc_token_stride,
                            int64_t kvc_layer_stride, const uint16_t* k_pe,
                            int64_t kpe_token_stride, int64_t kpe_layer_stride,
                            int32_t num_tokens, int32_t num_layers, int32_t kv_lora_rank,
                            int32_t pe_dim, const int64_t* slot_mapping,
                            int64_t slot_layer_stride, void* const* caches,
                            const float* k_scales, int32_t cache_dtype, int64_t num_blocks,
                            int32_t block_size, int64_t block_stride, int64_t entry_stride,
                            const uint16_t* gamma, int64_t gamma_layer_stride, float eps,
                            const int64_t* positions, const float* cos_sin_cache,
                            int64_t max_position);

uint32_t orc_norm_rope_grouped(const uint16_t* kv_c, int64_t kvc_token_stride,
                               int64_t kvc_layer_stride, const uint16_t* k_pe,
                               int64_t kpe_token_stride, int64_t kpe_layer_stride,
                               int32_t num_tokens, int32_t num_layers, int32_t kv_lora_rank,
                               int32_t pe_dim, const uint16_t* gamma, int64_t gamma_layer_stride,
                               float eps, const int64_t* positions, const float* cos_sin_cache,
                               int64_t max_position, uint16_t* kv_c_out, int64_t oc_token_stride,
                               int64_t oc_layer_stride, uint16_t* k_pe_out,
                               int64_t op_token_stride, int64_t op_layer_stride);

/* ---- context gather and element cast ------------------------------------ */
uint32_t orc_context_gather(const void* cache, int32_t cache_dtype, int64_t num_blocks,
                            int32_t block_size, int64_t block_stride, int64_t entry_stride,
                            int32_t entry_dim, const int32_t* block_table,
                            int64_t block_table_stride, const int32_t* cu_chunk_lens,
                            const int32_t* chunk_starts, int32_t num_seqs, int32_t num_tokens,
                            void* out, int64_t out_row_stride, int32_t out_dtype);

void orc_cast_rows(const void* src, int32_t src_dtype, int64_t src_row_stride, int64_t rows,
                   int64_t cols, void* dst, int32_t dst_dtype, int64_t dst_row_stride);

uint16_t orc_bf16_from_fp8_scaled(uint8_t c, int fmt, float scale);

uint32_t orc_context_gather_scaled(const void* cache, int32_t cache_dtype, int64_t num_blocks,
                                   int32_t block_size, int64_t block_stride, int64_t entry_stride,
                                   int32_t entry_dim, const int32_t* block_table,
                                   int64_t block_table_stride, const int32_t* cu_chunk_lens,
                                   const int32_t* chunk_starts, int32_t num_seqs,
                                   int32_t num_tokens, uint16_t* out, int64_t out_row_stride,
                                   float dequant_scale);

/* ---- chunked-context K/V pack ------------------------------------------- */
void orc_concat_key(const uint16_t* k_nope, int64_t kn_token_stride, int64_t kn_head_stride,
                    const uint16_t* k_pe, int64_t kpe_token_stride, int32_t num_tokens,
                    int32_t num_heads, int32_t nope_dim, int32_t rope_dim, uint16_t* key);

void orc_context_kv_pack(const uint16_t* k_nope, int64_t kn_token_stride,
                         int64_t kn_head_stride, const uint16_t* v, int64_t v_token_stride,
                         int64_t v_head_stride, const void* k_pe, int64_t kpe_token_stride,
                         int32_t kpe_dtype, int32_t num_tokens, int32_t num_heads,
                         int32_t nope_dim, int32_t rope_dim, int32_t v_dim, void* key_out,
                         void* v_out, int32_t out_dtype, float out_scale, int32_t in_dtype);

uint32_t orc_context_kv_pack_paged(
    const uint16_t* k_nope, int64_t kn_token_stride, int64_t kn_head_stride, const uint16_t* v,
    int64_t v_token_stride, int64_t v_head_stride, const void* cache, int32_t cache_dtype,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride,
    int32_t rope_offset, const int32_t* block_table, int64_t block_table_stride,
    const int32_t* cu_chunk_lens, const int32_t* chunk_starts, int32_t num_seqs,
    int32_t num_tokens, int32_t num_heads, int32_t nope_dim, int32_t rope_dim, int32_t v_dim,
    void* key_out, void* v_out, int32_t out_dtype, float out_scale, int32_t in_dtype);

/* ---- the row loops above split over host threads (mla_oracle_split.c) ---
 * For the multi-core CPU baseline only: each cuts its rows into `threads`
 * contiguous ranges and runs the unchanged function above on each range in its
 * own thread; the output is byte-identical to the single-threaded call. */
uint32_t orc_split_insert_grouped(
    int32_t threads, const uint16_t* kv_c, int64_t kvc_token_stride, int64_t kvc_layer_stride,
    const uint16_t* k_pe, int64_t kpe_token_stride, int64_t kpe_layer_stride,
    int32_t num_tokens, int32_t num_layers, int32_t kv_lora_rank, int32_t pe_dim,
    const int64_t* slot_mapping, int64_t slot_layer_stride, void* const* caches,
    const float* k_scales, int32_t cache_dtype, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, const uint16_t* gamma,
    int64_t gamma_layer_stride, float eps, const int64_t* positions,
    const float* cos_sin_cache, int64_t max_position);

uint32_t orc_split_context_gather(int32_t threads, const void* cache, int32_t cache_dtype,
                                  int64_t num_blocks, int32_t block_size, int64_t block_stride,
                                  int64_t entry_stride, int32_t entry_dim,
                                  const int32_t* block_table, int64_t block_table_stride,
                                  const int32_t* cu_chunk_lens, const int32_t* chunk_starts,
                                  int32_t num_seqs, int32_t num_tokens, void* out,
                                  int64_t out_row_stride, int32_t out_dtype);

void orc_split_context_kv_pack(int32_t threads, const uint16_t* k_nope, int64_t kn_token_stride,
                               int64_t kn_head_stride, const uint16_t* v, int64_t v_token_stride,
                               int64_t v_head_stride, const void* k_pe, int64_t kpe_token_stride,
                               int32_t kpe_dtype, int32_t num_tokens, int32_t num_heads,
                               int32_t nope_dim, int32_t rope_dim, int32_t v_dim, void* key_out,
                               void* v_out, int32_t out_dtype, float out_scale,
                               int32_t in_dtype);

#ifdef __cplusplus
}
#endif
#endif /* MLA_ORACLE_H */
