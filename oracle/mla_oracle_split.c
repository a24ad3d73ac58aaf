/*
 * mla_oracle_split.c -- the oracle's row loops split over host threads, for the
 * multi-core CPU baseline.
 *
 * TEST / BENCHMARK INFRASTRUCTURE ONLY, like the rest of oracle/.  Nothing here
 * does arithmetic: each function cuts its problem into `threads` contiguous
 * ranges of independent rows and runs the UNCHANGED single-threaded oracle
 * function (mla_oracle.c) on each range in its own POSIX thread.  The rows of
 * every function are independent in the pages' definitions (an insert row
 * writes the cache row its slot names, and valid slots are distinct within a
 * layer; a gather row and a pack token write only their own output rows), so
 * the output is byte-identical to the single-threaded call for every split;
 * tests/test_oracle_split.py checks that.
 *
 * Splits:
 *   insert   tokens [t0, t1) of every layer: kv_c, k_pe, slot_mapping and
 *            positions advanced by t0 tokens;
 *   gather   output rows [r0, r1): the sequence table rebased to the range
 *            (cu' = clamp(cu - r0, 0, r1 - r0), and a sequence that began
 *            before r0 starts r0 - cu[s] positions later);
 *   pack     tokens [t0, t1): inputs and outputs advanced by t0 tokens.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#include "mla_oracle.h"

#define ORC_SPLIT_MAX_THREADS 512

static int clamp_threads(int threads, int64_t rows) {
  if (threads < 1) threads = 1;
  if (threads > ORC_SPLIT_MAX_THREADS) threads = ORC_SPLIT_MAX_THREADS;
  if ((int64_t)threads > rows) threads = rows > 0 ? (int)rows : 1;
  return threads;
}

/* Range i of `threads` near-equal contiguous ranges of [0, n). */
static void range_of(int64_t n, int threads, int i, int64_t* lo, int64_t* hi) {
  *lo = n * i / threads;
  *hi = n * (i + 1) / threads;
}

/* ---------------------------------------------------------------- insert */
typedef struct {
  const uint16_t* kv_c;
  int64_t kvc_ts, kvc_ls;
  const uint16_t* k_pe;
  int64_t kpe_ts, kpe_ls;
  int32_t num_tokens, num_layers, kv_lora_rank, pe_dim;
  const int64_t* slot_mapping;
  int64_t slot_ls;
  void* const* caches;
  const float* k_scales;
  int32_t cache_dtype;
  int64_t num_blocks;
  int32_t block_size;
  int64_t block_stride, entry_stride;
  const uint16_t* gamma;
  int64_t gamma_ls;
  float eps;
  const int64_t* positions;
  const float* cos_sin_cache;
  int64_t max_position;
  uint32_t err;
} InsertJob;

static void* insert_worker(void* p) {
  InsertJob* j = (InsertJob*)p;
  j->err = orc_insert_grouped(j->kv_c, j->kvc_ts, j->kvc_ls, j->k_pe, j->kpe_ts, j->kpe_ls,
                              j->num_tokens, j->num_layers, j->kv_lora_rank, j->pe_dim,
                              j->slot_mapping, j->slot_ls, j->caches, j->k_scales,
                              j->cache_dtype, j->num_blocks, j->block_size, j->block_stride,
                              j->entry_stride, j->gamma, j->gamma_ls, j->eps, j->positions,
                              j->cos_sin_cache, j->max_position);
  return NULL;
}

uint32_t orc_split_insert_grouped(
    int32_t threads, const uint16_t* kv_c, int64_t kvc_token_stride, int64_t kvc_layer_stride,
    const uint16_t* k_pe, int64_t kpe_token_stride, int64_t kpe_layer_stride,
    int32_t num_tokens, int32_t num_layers, int32_t kv_lora_rank, int32_t pe_dim,
    const int64_t* slot_mapping, int64_t slot_layer_stride, void* const* caches,
    const float* k_scales, int32_t cache_dtype, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, const uint16_t* gamma,
    int64_t gamma_layer_stride, float eps, const int64_t* positions,
    const float* cos_sin_cache, int64_t max_position) {
  const int n = clamp_threads(threads, num_tokens);
  InsertJob jobs[ORC_SPLIT_MAX_THREADS];
  pthread_t tid[ORC_SPLIT_MAX_THREADS];
  int started[ORC_SPLIT_MAX_THREADS];
  for (int i = 0; i < n; ++i) {
    int64_t t0, t1;
    range_of(num_tokens, n, i, &t0, &t1);
    InsertJob* j = &jobs[i];
    j->kv_c = kv_c + t0 * kvc_token_stride;
    j->kvc_ts = kvc_token_stride;
    j->kvc_ls = kvc_layer_stride;
    j->k_pe = k_pe + t0 * kpe_token_stride;
    j->kpe_ts = kpe_token_stride;
    j->kpe_ls = kpe_layer_stride;
    j->num_tokens = (int32_t)(t1 - t0);
    j->num_layers = num_layers;
    j->kv_lora_rank = kv_lora_rank;
    j->pe_dim = pe_dim;
    j->slot_mapping = slot_mapping + t0;
    j->slot_ls = slot_layer_stride;
    j->caches = caches;
    j->k_scales = k_scales;
    j->cache_dtype = cache_dtype;
    j->num_blocks = num_blocks;
    j->block_size = block_size;
    j->block_stride = block_stride;
    j->entry_stride = entry_stride;
    j->gamma = gamma;
    j->gamma_ls = gamma_layer_stride;
    j->eps = eps;
    j->positions = positions ? positions + t0 : NULL;
    j->cos_sin_cache = cos_sin_cache;
    j->max_position = max_position;
    j->err = 0;
  }
  for (int i = 1; i < n; ++i) started[i] = pthread_create(&tid[i], NULL, insert_worker, &jobs[i]) == 0;
  insert_worker(&jobs[0]);
  uint32_t err = jobs[0].err;
  for (int i = 1; i < n; ++i) {
    if (started[i]) pthread_join(tid[i], NULL);
    else insert_worker(&jobs[i]);
    err |= jobs[i].err;
  }
  return err;
}

/* ---------------------------------------------------------------- gather */
typedef struct {
  const void* cache;
  int32_t cache_dtype;
  int64_t num_blocks;
  int32_t block_size;
  int64_t block_stride, entry_stride;
  int32_t entry_dim;
  const int32_t* block_table;
  int64_t bt_stride;
  int32_t* cu;      /* rebased copy, [num_seqs + 1] */
  int32_t* starts;  /* rebased copy, [num_seqs] */
  int32_t num_seqs, num_tokens;
  void* out;
  int64_t out_row_stride;
  int32_t out_dtype;
  uint32_t err;
} GatherJob;

static void* gather_worker(void* p) {
  GatherJob* j = (GatherJob*)p;
  j->err = orc_context_gather(j->cache, j->cache_dtype, j->num_blocks, j->block_size,
                              j->block_stride, j->entry_stride, j->entry_dim, j->block_table,
                              j->bt_stride, j->cu, j->starts, j->num_seqs, j->num_tokens, j->out,
                              j->out_row_stride, j->out_dtype);
  return NULL;
}

static int elt_bytes(int32_t fmt) { return (fmt == ORC_BF16 || fmt == ORC_F16) ? 2 : 1; }

uint32_t orc_split_context_gather(int32_t threads, const void* cache, int32_t cache_dtype,
                                  int64_t num_blocks, int32_t block_size, int64_t block_stride,
                                  int64_t entry_stride, int32_t entry_dim,
                                  const int32_t* block_table, int64_t block_table_stride,
                                  const int32_t* cu_chunk_lens, const int32_t* chunk_starts,
                                  int32_t num_seqs, int32_t num_tokens, void* out,
                                  int64_t out_row_stride, int32_t out_dtype) {
  int n = clamp_threads(threads, num_tokens);
  /* a rebased start must stay an int32; otherwise run unsplit */
  for (int32_t s = 0; s < num_seqs && n > 1; ++s) {
    const int64_t shifted = (int64_t)chunk_starts[s] + (int64_t)num_tokens - cu_chunk_lens[s];
    if (shifted > INT32_MAX || (int64_t)chunk_starts[s] - cu_chunk_lens[s] < INT32_MIN) n = 1;
  }
  if (n == 1)
    return orc_context_gather(cache, cache_dtype, num_blocks, block_size, block_stride,
                              entry_stride, entry_dim, block_table, block_table_stride,
                              cu_chunk_lens, chunk_starts, num_seqs, num_tokens, out,
                              out_row_stride, out_dtype);
  GatherJob jobs[ORC_SPLIT_MAX_THREADS];
  pthread_t tid[ORC_SPLIT_MAX_THREADS];
  int started[ORC_SPLIT_MAX_THREADS];
  int32_t* tables = (int32_t*)malloc(sizeof(int32_t) * (size_t)n * (2 * (size_t)num_seqs + 1));
  if (!tables)
    return orc_context_gather(cache, cache_dtype, num_blocks, block_size, block_stride,
                              entry_stride, entry_dim, block_table, block_table_stride,
                              cu_chunk_lens, chunk_starts, num_seqs, num_tokens, out,
                              out_row_stride, out_dtype);
  const int ob = elt_bytes(out_dtype);
  for (int i = 0; i < n; ++i) {
    int64_t r0, r1;
    range_of(num_tokens, n, i, &r0, &r1);
    const int64_t len = r1 - r0;
    GatherJob* j = &jobs[i];
    j->cu = tables + (size_t)i * (2 * (size_t)num_seqs + 1);
    j->starts = j->cu + num_seqs + 1;
    for (int32_t s = 0; s <= num_seqs; ++s) {
      int64_t c = (int64_t)cu_chunk_lens[s] - r0;
      j->cu[s] = (int32_t)(c < 0 ? 0 : (c > len ? len : c));
    }
    for (int32_t s = 0; s < num_seqs; ++s) {
      const int64_t before = r0 - (int64_t)cu_chunk_lens[s];  /* rows of s before the range */
      j->starts[s] = (int32_t)((int64_t)chunk_starts[s] + (before > 0 ? before : 0));
    }
    j->cache = cache;
    j->cache_dtype = cache_dtype;
    j->num_blocks = num_blocks;
    j->block_size = block_size;
    j->block_stride = block_stride;
    j->entry_stride = entry_stride;
    j->entry_dim = entry_dim;
    j->block_table = block_table;
    j->bt_stride = block_table_stride;
    j->num_seqs = num_seqs;
    j->num_tokens = (int32_t)len;
    j->out = (uint8_t*)out + r0 * out_row_stride * ob;
    j->out_row_stride = out_row_stride;
    j->out_dtype = out_dtype;
    j->err = 0;
  }
  for (int i = 1; i < n; ++i) started[i] = pthread_create(&tid[i], NULL, gather_worker, &jobs[i]) == 0;
  gather_worker(&jobs[0]);
  uint32_t err = jobs[0].err;
  for (int i = 1; i < n; ++i) {
    if (started[i]) pthread_join(tid[i], NULL);
    else gather_worker(&jobs[i]);
    err |= jobs[i].err;
  }
  free(tables);
  return err;
}

/* ------------------------------------------------------------------ pack */
typedef struct {
  const uint16_t* k_nope;
  int64_t kn_ts, kn_hs;
  const uint16_t* v;
  int64_t v_ts, v_hs;
  const void* k_pe;
  int64_t kpe_ts;
  int32_t kpe_dtype, num_tokens, num_heads, nope_dim, rope_dim, v_dim;
  void* key_out;
  void* v_out;
  int32_t out_dtype;
  float out_scale;
  int32_t in_dtype;
} PackJob;

static void* pack_worker(void* p) {
  PackJob* j = (PackJob*)p;
  orc_context_kv_pack(j->k_nope, j->kn_ts, j->kn_hs, j->v, j->v_ts, j->v_hs, j->k_pe, j->kpe_ts,
                      j->kpe_dtype, j->num_tokens, j->num_heads, j->nope_dim, j->rope_dim,
                      j->v_dim, j->key_out, j->v_out, j->out_dtype, j->out_scale, j->in_dtype);
  return NULL;
}

void orc_split_context_kv_pack(int32_t threads, const uint16_t* k_nope, int64_t kn_token_stride,
                               int64_t kn_head_stride, const uint16_t* v, int64_t v_token_stride,
                               int64_t v_head_stride, const void* k_pe, int64_t kpe_token_stride,
                               int32_t kpe_dtype, int32_t num_tokens, int32_t num_heads,
                               int32_t nope_dim, int32_t rope_dim, int32_t v_dim, void* key_out,
                               void* v_out, int32_t out_dtype, float out_scale,
                               int32_t in_dtype) {
  const int n = clamp_threads(threads, num_tokens);
  PackJob jobs[ORC_SPLIT_MAX_THREADS];
  pthread_t tid[ORC_SPLIT_MAX_THREADS];
  int started[ORC_SPLIT_MAX_THREADS];
  const int ob = elt_bytes(out_dtype), kb = elt_bytes(kpe_dtype);
  const int64_t key_tok = (int64_t)num_heads * (nope_dim + rope_dim) * ob;
  const int64_t v_tok = (int64_t)num_heads * v_dim * ob;
  for (int i = 0; i < n; ++i) {
    int64_t t0, t1;
    range_of(num_tokens, n, i, &t0, &t1);
    PackJob* j = &jobs[i];
    j->k_nope = k_nope + t0 * kn_token_stride;
    j->kn_ts = kn_token_stride;
    j->kn_hs = kn_head_stride;
    j->v = v ? v + t0 * v_token_stride : NULL;
    j->v_ts = v_token_stride;
    j->v_hs = v_head_stride;
    j->k_pe = (const uint8_t*)k_pe + t0 * kpe_token_stride * kb;
    j->kpe_ts = kpe_token_stride;
    j->kpe_dtype = kpe_dtype;
    j->num_tokens = (int32_t)(t1 - t0);
    j->num_heads = num_heads;
    j->nope_dim = nope_dim;
    j->rope_dim = rope_dim;
    j->v_dim = v_dim;
    j->key_out = (uint8_t*)key_out + t0 * key_tok;
    j->v_out = v_out ? (uint8_t*)v_out + t0 * v_tok : NULL;
    j->out_dtype = out_dtype;
    j->out_scale = out_scale;
    j->in_dtype = in_dtype;
  }
  for (int i = 1; i < n; ++i) started[i] = pthread_create(&tid[i], NULL, pack_worker, &jobs[i]) == 0;
  pack_worker(&jobs[0]);
  for (int i = 1; i < n; ++i) {
    if (started[i]) pthread_join(tid[i], NULL);
    else pack_worker(&jobs[i]);
  }
}
