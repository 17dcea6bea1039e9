/*
 * libpagedattn — attention over a paged (block-table) bf16 KV cache, GB300 (sm_103a).
 *
 * The cache of one layer is two tensors (K and V), each laid out
 *     [num_blocks][block_size][num_kv_heads][head_dim]   bf16, row-major,
 * the per-layer view of the cache described in "手搓 vLLM 推理引擎"
 * (LLM-101-CN nano-vllm walkthrough), Step 5, "KV Cache 的内存布局".  A token's
 * slot is block_id * block_size + offset_in_block; row `slot` of the cache holds
 * its num_kv_heads*head_dim values.
 *
 * Three device operations, always in this order within one attention layer
 * (same page, Step 4, Attention.forward): store the new tokens' K/V, then run
 * prefill or decode attention.  All of them only enqueue work on `stream`: no
 * host synchronisation, no allocation, no device-to-host reads.  Every buffer
 * is owned by the caller.
 *
 * Host-side metadata (cu_seqlens, block tables, slot mapping, work lists) is
 * packed on the CPU into ONE caller-provided buffer by pa_pack_prefill /
 * pa_pack_decode and uploaded with one asynchronous copy (pa_upload or the
 * caller's own cudaMemcpyAsync); the library never reads device metadata on
 * the host ("面试问答准备: nano-vLLM 推理引擎优化", Q1, item 2: scheduling
 * metadata is computed on the CPU so that no .item() sync is needed).
 *
 * Error behaviour: every entry point validates its arguments on the host
 * before any launch and returns a PA_ERR_* code with no device side effect on
 * failure.  PA_ERR_CUDA means a CUDA call failed; pa_last_error_string()
 * gives the text (thread-local).
 *
 * Supported: head_dim 64 or 128; num_heads % num_kv_heads == 0 with group
 * size num_heads/num_kv_heads <= 16; block_size a power of two in [16, 1024];
 * bf16 data.  Device pointers must be 16-byte aligned.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *pa_stream_t;

enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* malformed sizes, pointers or metadata */
    PA_ERR_UNSUPPORTED = 2, /* head_dim, group size or block_size outside the supported set */
    PA_ERR_WORKSPACE = 3,   /* caller buffer (metadata image or decode workspace) too small */
    PA_ERR_CUDA = 4         /* a CUDA runtime/driver call failed; see pa_last_error_string() */
};

/* Shapes of one layer's cache and attention heads.  Passed by pointer to every call. */
typedef struct pa_dims {
    int32_t num_blocks;   /* physical blocks in the pool */
    int32_t block_size;   /* tokens per block */
    int32_t num_heads;    /* query heads Hq */
    int32_t num_kv_heads; /* KV heads Hkv; query head h reads KV head h / (Hq/Hkv) */
    int32_t head_dim;     /* D */
} pa_dims;

/*
 * Packed prefill metadata: host scalars plus byte offsets of each int32 array
 * inside the metadata image written by pa_pack_prefill.  After the image is
 * copied to device memory at `dev`, array X lives at dev + off_X.
 */
typedef struct pa_prefill_meta {
    int32_t num_seqs;
    int32_t total_q;            /* sum of query lengths = rows of q/out */
    int32_t max_seqlen_q;
    int32_t max_seqlen_k;
    int32_t max_blocks_per_seq; /* row pitch of block_tables */
    int32_t num_tiles;          /* work items = CTAs of the prefill launch */
    int32_t rows_per_tile;      /* query positions per query tile (128 / group, floored);
                                   a work item covers two query tiles */
    int32_t prefix_aligned;     /* 1 if the cached prefix (seq_len - query_len) of every
                                   sequence with new tokens is a multiple of
                                   min(block_size, 128) (then no key box of the fused
                                   launch needs its new rows patched in); informational:
                                   pa_prefill_varlen_fused runs as one launch either way */
    uint64_t off_cu_seqlens_q;  /* int32 [num_seqs+1] */
    uint64_t off_cu_seqlens_k;  /* int32 [num_seqs+1] */
    uint64_t off_block_tables;  /* int32 [num_seqs][max_blocks_per_seq], -1 padded */
    uint64_t off_slot_mapping;  /* int32 [total_q] */
    uint64_t off_tiles;         /* int32 [num_tiles][8] work list, longest first: sequence,
                                   first query row, KV head, key tiles, first packed
                                   query row of the sequence, query length, key length,
                                   physical block holding key 0 */
    uint64_t total_bytes;       /* size of the image */
    uint64_t off_scratch_tables; /* int32 [num_seqs][scratch_pitch], -1 padded: the blocks
                                   of sequence b in the INT8 prefill's bf16 scratch cache
                                   (ceil(seq_len / 128) consecutive 128-token blocks for
                                   each sequence with new tokens, none for the others) */
    uint64_t off_scratch_items; /* int32 [scratch_blocks][8] per scratch block: sequence b, its
                                   first key (128 x block index within b), key count
                                   seq_len, cached prefix seq_len - query_len, packed
                                   row of b's new keys minus the prefix
                                   (cu_seqlens_q[b] - prefix), 0, 0, 0 */
    uint64_t workspace_bytes;   /* device workspace pa_prefill_varlen_int8(_fused) needs:
                                   the scratch cache, K then V, bf16
                                   [scratch_blocks * 128][num_kv_heads][head_dim] each */
    int32_t scratch_blocks;     /* 128-token blocks of the scratch cache */
    int32_t scratch_pitch;      /* row pitch of the scratch tables (>= 1) */
} pa_prefill_meta;

/* Packed decode metadata (one query token per sequence). */
typedef struct pa_decode_meta {
    int32_t num_seqs;
    int32_t max_blocks_per_seq;
    int32_t num_items;          /* (sequence, key split) work items */
    int32_t split_tokens;       /* keys per split (multiple of 64) */
    int32_t max_splits;         /* largest split count of any sequence */
    int32_t num_partials;       /* partial results in the workspace (sequences with > 1 split) */
    uint64_t off_context_lens;  /* int32 [num_seqs] */
    uint64_t off_block_tables;  /* int32 [num_seqs][max_blocks_per_seq], -1 padded */
    uint64_t off_slot_mapping;  /* int32 [num_seqs] */
    uint64_t off_items;         /* int32 [num_items][4] work list, longest first */
    uint64_t off_seq_items;     /* int32 [num_seqs+1] first work item of each sequence */
    uint64_t total_bytes;
    uint64_t workspace_bytes;   /* device workspace pa_decode needs */
} pa_decode_meta;

/* ------------------------------------------------------------------ host packing */

/*
 * pa_pack_prefill — build the metadata of a prefill batch on the CPU.
 * Source: "手搓 vLLM 推理引擎", Step 5, prepare_prefill(): sequence b has
 * seq_lens[b] tokens of which the first seq_lens[b]-query_lens[b] are already
 * cached (prefix-cache hit); cu_seqlens_q/k are prefix sums of the query and
 * key lengths; the new tokens are positions [cached, len) and their slots are
 * block_table[pos / block_size]*block_size + pos % block_size.
 *   seq_lens, query_lens: host int32 [num_seqs], 0 <= query_lens[b] <= seq_lens[b]
 *   block_offsets:        host int32 [num_seqs+1]; sequence b's physical blocks
 *                         are block_ids[block_offsets[b] .. block_offsets[b+1])
 *                         and must number at least ceil(seq_lens[b]/block_size)
 *   host_buf:             caller memory (pinned for an asynchronous upload) of
 *                         host_buf_bytes; NULL to only compute meta->total_bytes
 * Returns PA_ERR_WORKSPACE (with meta->total_bytes set) when the buffer is too small.
 */
int pa_pack_prefill(const pa_dims *dims, int32_t num_seqs, const int32_t *seq_lens,
                    const int32_t *query_lens, const int32_t *block_offsets,
                    const int32_t *block_ids, void *host_buf, size_t host_buf_bytes,
                    pa_prefill_meta *meta);

/*
 * pa_pack_decode — build the metadata of a decode batch (one new token per
 * sequence) on the CPU.  Source: same page, Step 5, prepare_decode():
 * context_lens[b] = len(seq) includes the token being decoded; its slot is
 * block_table[-1]*block_size + last_block_num_tokens - 1.
 * The context of each sequence is cut into splits of `split_tokens` keys
 * (a multiple of 64; 0 = choose from the current device's SM count) whose
 * partial results are merged by log-sum-exp ("面试问答准备", the Split-K entry:
 * each segment yields a local max, normaliser and fp32 accumulator, a second
 * kernel merges them).
 */
int pa_pack_decode(const pa_dims *dims, int32_t num_seqs, const int32_t *context_lens,
                   const int32_t *block_offsets, const int32_t *block_ids, int32_t split_tokens,
                   void *host_buf, size_t host_buf_bytes, pa_decode_meta *meta);

/* One asynchronous host-to-device copy of a packed metadata image. */
int pa_upload(void *dev_dst, const void *host_src, size_t bytes, pa_stream_t stream);

/* ------------------------------------------------------------------ device operations */

/*
 * pa_store_kvcache — KV scatter.  Source: "手搓 vLLM 推理引擎", Step 4,
 * "Triton Kernel：写入 KV Cache": token t with slot s = slot_mapping[t] copies
 * its K and V rows (num_kv_heads*head_dim bf16 each) to cache row s; s == -1
 * (padding) is skipped.  Bit-exact copy.
 *   k, v:          device bf16 [num_tokens][num_kv_heads][head_dim]
 *   k_cache/v_cache: device bf16 [num_blocks][block_size][num_kv_heads][head_dim]
 *   slot_mapping:  device int32 [num_tokens], each -1 or in [0, num_blocks*block_size)
 * Slots must be unique (duplicates race).  num_tokens == 0 launches nothing.
 */
int pa_store_kvcache(const pa_dims *dims, const void *k, const void *v, void *k_cache,
                     void *v_cache, const int32_t *slot_mapping, int32_t num_tokens,
                     pa_stream_t stream);

/*
 * pa_prefill_varlen — causal variable-length prefill over the paged cache.
 * Source: "手搓 vLLM 推理引擎", Step 4 (flash_attn_varlen_func with
 * cu_seqlens_q/k and block_table; prefix-cache hits have cu_seqlens_k >
 * cu_seqlens_q) and "推理系统" (KV-cache toy: new token i of T sees the first
 * S-T+i+1 keys).  For sequence b, query row i (0 <= i < Lq) at absolute
 * position Lk-Lq+i, head h:
 *   out = softmax(scale * q . K^T over keys j <= Lk-Lq+i) V,  K/V of key j at
 *   slot block_tables[b][j/block_size]*block_size + j%block_size, KV head h/G.
 * The K/V of every key (including the new tokens) must already be stored.
 *   q, out:  device bf16 [meta->total_q][num_heads][head_dim]
 *   cu_seqlens_q, cu_seqlens_k, block_tables, tiles: device copies of the
 *            arrays pa_pack_prefill wrote (dev + meta->off_*)
 * bf16 in, fp32 accumulation and softmax, bf16 out (round to nearest even).
 * scale must be finite and > 0 (PA_ERR_INVALID_ARG otherwise).  PA_ERR_UNSUPPORTED,
 * before any launch, if the library's prefill kernel was compiled with other
 * than 168 registers per thread (its warps re-divide exactly that many).
 * Every hand-off inside the kernel waits with a time limit (2 s); a wait that
 * runs out sets bit 1 of the device error word and the kernel returns early,
 * so `out` is undefined whenever pa_read_device_error reports bit 1 (the same
 * holds for pa_prefill_varlen_fused and pa_prefill_varlen_int8).
 */
int pa_prefill_varlen(const pa_dims *dims, const void *q, const void *k_cache,
                      const void *v_cache, const int32_t *cu_seqlens_q,
                      const int32_t *cu_seqlens_k, const int32_t *block_tables, float scale,
                      void *out, const pa_prefill_meta *meta, const int32_t *tiles,
                      pa_stream_t stream);

/*
 * pa_prefill_varlen_fused — pa_store_kvcache of the new tokens followed by
 * pa_prefill_varlen, with the same result, in one launch.  Source: "手搓 vLLM
 * 推理引擎", Step 4 (store_kvcache, then attention over the cache); "面试问答准备:
 * nano-vLLM 推理引擎优化", Q1 (chunked prefill resumes at any token count, so a
 * cached prefix need not end on a block boundary).  The prefill reads the new
 * tokens' keys and values from k and v themselves (the same bf16 values the
 * store writes) and the cached prefix from the cache; a key box that starts in
 * the prefix and ends among the new keys is read from the cache and its new
 * rows are replaced from k and v before use.  Meanwhile one warp of each CTA
 * copies the rows of its work item's query positions into their slots (each
 * (token, KV head) row by exactly one item).
 *   k, v:          device bf16 [meta->total_q][num_kv_heads][head_dim], row t
 *                  the key/value of packed query row t
 *   slot_mapping:  device int32 [meta->total_q] (dev + meta->off_slot_mapping);
 *                  -1 skips the row, a slot outside [-1, num_blocks*block_size)
 *                  is skipped and flagged (pa_read_device_error bit 0)
 * The new tokens' slots must not hold keys that a sequence of the call reads
 * from the cache (true of any slot mapping a block allocator produces).
 * Other arguments, errors and numerics as pa_prefill_varlen.
 */
int pa_prefill_varlen_fused(const pa_dims *dims, const void *q, const void *k, const void *v, void *k_cache,
                            void *v_cache, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            const int32_t *block_tables, const int32_t *slot_mapping, float scale, void *out,
                            const pa_prefill_meta *meta, const int32_t *tiles, pa_stream_t stream);

/*
 * pa_decode — batched single-token GQA decode over the paged cache.
 * Source: "手搓 vLLM 推理引擎", Step 4 (flash_attn_with_kvcache with
 * cache_seqlens and block_table) and "推理系统" (decode reads the whole cache
 * and is bandwidth bound).  For sequence b and query head h, the single query
 * sees all context_lens[b] keys:
 *   out[b][h] = softmax(scale * q[b][h] . K^T) V.
 * Long contexts are split per the packed plan; partial (max, sum, fp32
 * accumulator) triples go to `workspace` and a combine kernel merges them by
 * log-sum-exp.
 *   q, out:     device bf16 [num_seqs][num_heads][head_dim]
 *   workspace:  device memory of at least meta->workspace_bytes (may be NULL
 *               when that is 0), 256-byte aligned
 * scale must be finite and > 0 (PA_ERR_INVALID_ARG otherwise).
 */
int pa_decode(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *context_lens, const int32_t *block_tables, float scale, void *out,
              const pa_decode_meta *meta, const int32_t *items, const int32_t *seq_items,
              void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_pack_decode_fixed — a decode plan whose shapes do not depend on the
 * contexts, for replaying captured launches (CUDA graphs) across steps.
 * Source: "手搓 vLLM 推理引擎", Step 5 (ModelRunner): decode runs as a
 * CUDA graph captured once per batch-size bucket, and at replay the rows a
 * batch does not use get slot -1 (the store skips it) and context length 0.
 * Every sequence gets
 * ceil(max_context / split) key ranges of split_tokens keys (0: one range of
 * max_context keys), empty ones included, and the block-table rows are
 * ceil(max_context / block_size) wide; so meta's sizes, offsets, item count
 * and workspace_bytes depend only on (dims, num_seqs, max_context,
 * split_tokens).  Re-packing new contexts into the same host buffer,
 * uploading it to the same device buffer and replaying launches captured
 * with that meta is valid.  Padding entries: context_lens[b] = 0 (slot -1,
 * output rows of zeros).  Requires num_seqs >= 1, 1 <= max_context, every
 * context in [0, max_context], split_tokens 0 or a positive multiple of 64.
 * Same buffer and error rules as pa_pack_decode.
 */
int pa_pack_decode_fixed(const pa_dims *dims, int32_t num_seqs, const int32_t *context_lens,
                         const int32_t *block_offsets, const int32_t *block_ids, int32_t max_context,
                         int32_t split_tokens, void *host_buf, size_t host_buf_bytes, pa_decode_meta *meta);

/*
 * pa_decode_fused — store + decode in one launch: writes k[b], v[b] (bf16
 * [num_seqs][num_kv_heads][head_dim], the new token of each sequence) into
 * cache row slot_mapping[b] and returns what pa_store_kvcache followed by
 * pa_decode returns.  Source: "手搓 vLLM 推理引擎", Step 4 (Attention.forward
 * stores the new K/V, then attends over the cache including them); fusing
 * the two removes one launch and the ordering between them.  The work item
 * that ends at the last key takes that key from k/v and writes the row; the
 * other items read the cache.  slot_mapping is the plan's (meta
 * off_slot_mapping); slot -1 writes nothing, other out-of-range slots are
 * skipped and flagged (pa_read_device_error bit 0).  Same plan, workspace and
 * error rules as pa_decode.
 */
int pa_decode_fused(const pa_dims *dims, const void *q, const void *k, const void *v, void *k_cache, void *v_cache,
                    const int32_t *slot_mapping, const int32_t *context_lens, const int32_t *block_tables,
                    float scale, void *out, const pa_decode_meta *meta, const int32_t *items,
                    const int32_t *seq_items, void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_copy_blocks — copy-on-write of shared cache blocks.  Source: "vLLM /
 * SGLang 面试源码深挖", section 4 (KV block fork): when an append would land in
 * a shared, still-mutable block, the child gets a new block and the valid KV
 * is copied into it; "推理系统", PagedAttention paragraph (copy on write).
 *   triples: device int32 [num_triples][3] = (src block, dst block, n valid
 *            tokens); rows src*bs + i are copied to dst*bs + i for i < n, in
 *            both K and V, bit for bit.
 * dst blocks must be distinct and must not be the src of another triple
 * (otherwise the result depends on order).  A triple with a block id outside
 * [0, num_blocks) or n outside [0, block_size] is skipped and flagged in the
 * device error word (pa_read_device_error bit 2).  num_triples == 0 launches
 * nothing.
 */
int pa_copy_blocks(const pa_dims *dims, void *k_cache, void *v_cache, const int32_t *triples,
                   int32_t num_triples, pa_stream_t stream);

/* ------------------------------------------------------------------ INT8 KV cache */

/*
 * INT8 cache variant.  Source: "面试问答准备: nano-vLLM 推理引擎优化", Q3
 * (KV cache quantisation): each token's K (and V) vector of one KV head is
 * stored as int8 codes with one scale, scale = max|x| / 127, code =
 * round(x / scale); the attention kernel dequantises (code * scale) as it
 * loads, so decode reads half the bytes of the bf16 cache.  The pages fix no
 * rounding rule or scale type; this library reads them as: fp32 arithmetic
 * with IEEE division, scale floored at 1e-8 (an all-zero vector), rounding
 * half away from zero, scale stored as fp16 (round to nearest even) and the
 * dequantised value being code * (fp16 scale).
 *
 * Layout (per layer; both owned by the caller):
 *   k_cache, v_cache: int8  [num_blocks][block_size][num_kv_heads][head_dim]
 *                     (the bf16 layout with 1-byte elements)
 *   k_scale, v_scale: fp16  [num_blocks][num_kv_heads][block_size]
 *                     (head-major inside a block: one head's scales for a
 *                     run of tokens are contiguous)
 * All four pointers must be 16-byte aligned.
 */

/*
 * pa_store_kvcache_int8 — quantising scatter: for each token t with
 * slot_mapping[t] != -1, quantise k[t][g][:] and v[t][g][:] (bf16) for every
 * KV head g into the codes of row slot and the scales at
 * [slot / block_size][g][slot % block_size].  Codes and scales are
 * deterministic (bit-identical on every run).  Slots outside [-1, num_slots)
 * are skipped and flagged (pa_read_device_error bit 0).
 */
int pa_store_kvcache_int8(const pa_dims *dims, const void *k, const void *v, void *k_cache, void *v_cache,
                          void *k_scale, void *v_scale, const int32_t *slot_mapping, int32_t num_tokens,
                          pa_stream_t stream);

/*
 * pa_decode_int8 — pa_decode over an INT8 cache: the same plan
 * (pa_pack_decode), arguments, workspace and result, with the cached K and V
 * read as code * scale.  Internally the codes (exact in fp16) and q (rounded
 * to fp16; exact for bf16 magnitudes in [2^-14, 65504], clamped to +-65504)
 * feed fp16 tensor-core products with fp32 accumulation; the V scale is
 * applied to the softmax weights before the P.V product.  Its staged loads
 * are waited for with a time limit (2 s); a wait that runs out sets bit 3 of
 * the device error word and the kernel returns early, so `out` is undefined
 * whenever pa_read_device_error reports bit 3 (also for pa_decode_int8_fused).
 */
int pa_decode_int8(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                   const void *k_scale, const void *v_scale, const int32_t *context_lens,
                   const int32_t *block_tables, float scale, void *out, const pa_decode_meta *meta,
                   const int32_t *items, const int32_t *seq_items, void *workspace, size_t workspace_bytes,
                   pa_stream_t stream);

/*
 * pa_prefill_varlen_int8 — pa_prefill_varlen over an INT8 cache: the same
 * plan (pa_pack_prefill), arguments and result, with the cached K and V read
 * as code * scale.  Source: "面试问答准备: nano-vLLM 推理引擎优化", Q3, the
 * prefill's dequantisation path: the keys and values the block table
 * references are read as code * token scale in fp32 and rounded to the model's
 * dtype (bf16, round to nearest even; code * fp16 scale is exact in fp32, so
 * this is one rounding of the exact value), then the bf16 attention runs over
 * them.  Two launches on `stream`: a gather kernel writes every key and value
 * of each sequence with new tokens, dequantised, into a bf16 scratch cache in
 * `workspace` (128-token blocks, the plan's scratch tables), and the
 * pa_prefill_varlen kernel attends over it.
 *   scratch_tables: device int32 [num_seqs][meta->scratch_pitch]
 *                   (dev + meta->off_scratch_tables)
 *   scratch_items:  device int32 [meta->scratch_blocks][8] (dev + meta->off_scratch_items)
 *   workspace:      device memory of at least meta->workspace_bytes, 16-byte
 *                   aligned, owned by the caller; overwritten by the call
 *                   (two calls in flight at once need separate workspaces)
 * PA_ERR_WORKSPACE if workspace_bytes < meta->workspace_bytes; other errors as
 * pa_prefill_varlen.
 */
int pa_prefill_varlen_int8(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                           const void *k_scale, const void *v_scale, const int32_t *cu_seqlens_q,
                           const int32_t *cu_seqlens_k, const int32_t *block_tables,
                           const int32_t *scratch_tables, const int32_t *scratch_items, float scale, void *out,
                           const pa_prefill_meta *meta, const int32_t *tiles, void *workspace,
                           size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_prefill_varlen_int8_fused — pa_store_kvcache_int8 of the new tokens
 * followed by pa_prefill_varlen_int8, with the same codes, scales and output
 * bit for bit, in two launches instead of three.  Source: "面试问答准备:
 * nano-vLLM 推理引擎优化", Q3 (the INT8 cache's prefill cost comes from work
 * outside the attention kernel) and "手搓 vLLM 推理引擎", Step 4
 * (store_kvcache, then attention over the cache).  The gather launch quantises
 * each new (token, KV head) row into the cache (as pa_store_kvcache_int8
 * does) and writes its scratch row from those codes and the stored fp16
 * scale; the cached prefix is dequantised from the cache; then the bf16
 * attention runs over the scratch cache.
 *   k, v:          device bf16 [meta->total_q][num_kv_heads][head_dim], row t
 *                  the key/value of packed query row t
 *   slot_mapping:  device int32 [meta->total_q] (dev + meta->off_slot_mapping);
 *                  -1 skips the row's store, a slot outside
 *                  [-1, num_blocks*block_size) is skipped and flagged
 *                  (pa_read_device_error bit 0); the attention sees every new
 *                  row as the store writes it either way
 * Other arguments, errors and numerics as pa_prefill_varlen_int8 and
 * pa_store_kvcache_int8; the new tokens' slots must not hold keys that a
 * sequence of the call reads from the cache.
 */
int pa_prefill_varlen_int8_fused(const pa_dims *dims, const void *q, const void *k, const void *v,
                                 void *k_cache, void *v_cache, void *k_scale, void *v_scale,
                                 const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                 const int32_t *block_tables, const int32_t *slot_mapping,
                                 const int32_t *scratch_tables, const int32_t *scratch_items, float scale,
                                 void *out, const pa_prefill_meta *meta, const int32_t *tiles,
                                 void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_int8_fused — pa_store_kvcache_int8 followed by pa_decode_int8 in
 * one launch: quantises k[b], v[b] (bf16 [num_seqs][num_kv_heads][head_dim],
 * the new token of each sequence) into cache row slot_mapping[b] (codes and
 * scales, bit-identical to pa_store_kvcache_int8) and decodes over the cache
 * including it.  The work item that ends at the last key does the store and
 * takes that key's dequantised values from its registers.  Same plan,
 * workspace and error rules as pa_decode_int8; slot -1 writes nothing, other
 * out-of-range slots are skipped and flagged (bit 0).
 */
int pa_decode_int8_fused(const pa_dims *dims, const void *q, const void *k, const void *v, void *k_cache,
                         void *v_cache, void *k_scale, void *v_scale, const int32_t *slot_mapping,
                         const int32_t *context_lens, const int32_t *block_tables, float scale, void *out,
                         const pa_decode_meta *meta, const int32_t *items, const int32_t *seq_items,
                         void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_copy_blocks_int8 — pa_copy_blocks on an INT8 cache: for each (src, dst, n)
 * triple the codes of rows src*bs + i go to dst*bs + i and, for every KV head
 * g, the scales [src][g][i] to [dst][g][i], i < n, bit for bit (the
 * copy-on-write fork of "vLLM / SGLang 面试源码深挖", section 4, on the cache
 * of "面试问答准备: nano-vLLM 推理引擎优化", Q3).  Same triple rules and error
 * flag (bit 2) as pa_copy_blocks.
 */
int pa_copy_blocks_int8(const pa_dims *dims, void *k_cache, void *v_cache, void *k_scale, void *v_scale,
                        const int32_t *triples, int32_t num_triples, pa_stream_t stream);

/*
 * pa_decode_static — pa_decode for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point: it exists for callers
 * that have no way to obtain a decode workspace, e.g. code that runs while a
 * stream is being captured into a CUDA graph (cudaMalloc is not allowed
 * during capture in the default mode) or runtimes that only hand out fixed,
 * pre-planned buffers.  It computes exactly what pa_decode computes, with the
 * same arguments minus the workspace.
 *
 * Scratch: instead of a caller workspace it uses one array inside the library,
 * PA_DECODE_STATIC_SCRATCH_BYTES (16 MiB) of device memory that every GPU
 * which loads the library keeps until the process exits.  It calls no
 * cudaMalloc/cudaFree and no allocating library routine.
 *  - Limit: a plan whose meta->workspace_bytes exceeds the array is rejected
 *    with PA_ERR_WORKSPACE before any launch (use pa_decode, or a larger
 *    split_tokens when packing, for such batches).
 *  - Set-up: the first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress, with that device current); make that first
 *    call before any stream capture.  Later calls do no set-up and reuse that
 *    address for the life of the process: after cudaDeviceReset (or anything
 *    else that destroys the device's primary context) the library's module is
 *    loaded again at another address, so do not call pa_decode_static on that
 *    device again in this process.
 *  - Sharing: every call on a device uses the same array and it keeps the
 *    last call's contents.  Nothing in it needs to start at zero: each call
 *    writes every partial it reads.  Calls whose work overlaps on the GPU
 *    (different streams, not ordered) race on the array; order them.
 * The call works on the current device.
 */
#define PA_DECODE_STATIC_SCRATCH_BYTES (16u << 20)
int pa_decode_static(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *context_lens, const int32_t *block_tables, float scale, void *out,
                     const pa_decode_meta *meta, const int32_t *items, const int32_t *seq_items,
                     pa_stream_t stream);

/* ------------------------------------------------------------------ diagnostics */

/* Text of the last error on this thread ("" if none). */
const char *pa_last_error_string(void);

/*
 * Reads and clears the device-side error word (0 = none).  Bits: 0 a store
 * met a slot outside [-1, num_slots); 1 a bounded wait in the prefill kernel
 * timed out; 2 a block-copy triple was out of range; 3 a bounded wait in the
 * INT8 decode kernel timed out; 4 the wait of pa_selftest_bounded_wait timed
 * out.  Synchronises `stream`: for tests and debugging, never on the hot path.
 */
int pa_read_device_error(uint32_t *code, pa_stream_t stream);

/*
 * pa_selftest_bounded_wait — diagnostic of the library's failure path.  Every
 * kernel hand-off waits on an mbarrier with a time limit; on expiry the kernel
 * records the fact in the device error word and returns instead of hanging.
 * This launches one warp that runs that same bounded wait on a barrier
 * nothing completes (arrive_first == 0: bit 4 is set after about timeout_us
 * microseconds) or one it completes itself first (arrive_first != 0: no
 * error).  timeout_us in [1, 10^7], else PA_ERR_INVALID_ARG.  The GPU context
 * stays usable either way.
 */
int pa_selftest_bounded_wait(uint32_t timeout_us, int arrive_first, pa_stream_t stream);

/*
 * pa_stream_read — measurement helper, not part of the attention path.  Reads
 * every 16-byte vector of the device buffer src[0 .. bytes) once with
 * streaming (non-caching) loads and XOR-folds the words into *sink (device,
 * 4 bytes, caller-owned; its value is meaningless, it only keeps the loads
 * live).  It is the read-only memory bandwidth that bounds the decode kernels
 * (they read the whole cache and write little), so timing it beside them gives
 * the ceiling they are measured against; the pages' "decode time = bytes /
 * bandwidth" ("推理系统", 瓶颈不是算力，是带宽) states the bound.  src and sink
 * 16- and 4-byte aligned, bytes a multiple of 16, else PA_ERR_INVALID_ARG;
 * bytes == 0 launches nothing.  Asynchronous on `stream`.
 */
int pa_stream_read(const void *src, size_t bytes, uint32_t *sink, pa_stream_t stream);

/* Library version, e.g. 0x000500 for 0.5.0.  0.2.0 added pa_prefill_varlen_fused
 * and gave pa_prefill_meta's spare field its meaning (prefix_aligned); 0.3.0
 * made pa_prefill_varlen_fused one launch for any cached prefix and added
 * pa_stream_read; 0.4.0 added pa_prefill_varlen_int8_fused; 0.5.0 made the
 * INT8 prefill a bf16 gather into caller workspace followed by the bf16 kernel
 * (pa_prefill_varlen_int8 and pa_prefill_varlen_int8_fused take the scratch
 * tables, the scratch items and the workspace) and replaced pa_prefill_meta's
 * barrier words with the scratch fields (after total_bytes: the earlier fields
 * keep their offsets). */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
