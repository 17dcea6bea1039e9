// C ABI of libpagedattn: argument validation on the host, then kernel launches.
// No entry point allocates, synchronises or reads device memory on the host
// (except pa_read_device_error, a debugging aid).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <cuda_runtime.h>

#include "internal.h"

namespace pa {

static thread_local char g_err[512] = "";

void set_error(const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int check_dims(const pa_dims *dims)
{
    if (!dims)
        return fail(PA_ERR_INVALID_ARG, "dims is NULL");
    const pa_dims &d = *dims;
    if (d.num_blocks < 0 || d.block_size <= 0 || d.num_heads <= 0 || d.num_kv_heads <= 0 || d.head_dim <= 0)
        return fail(PA_ERR_INVALID_ARG, "dims must be positive (num_blocks may be 0)");
    if (d.num_heads % d.num_kv_heads != 0)
        return fail(PA_ERR_UNSUPPORTED, "num_heads (%d) is not a multiple of num_kv_heads (%d)", d.num_heads,
                    d.num_kv_heads);
    if (d.num_heads / d.num_kv_heads > kMaxGroup)
        return fail(PA_ERR_UNSUPPORTED, "group size %d > %d", d.num_heads / d.num_kv_heads, kMaxGroup);
    if (d.head_dim != 64 && d.head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d not in {64, 128}", d.head_dim);
    if (d.block_size < 16 || d.block_size > 1024 || (d.block_size & (d.block_size - 1)))
        return fail(PA_ERR_UNSUPPORTED, "block_size %d is not a power of two in [16, 1024]", d.block_size);
    if ((int64_t)d.num_blocks * d.block_size > INT32_MAX)
        return fail(PA_ERR_UNSUPPORTED, "num_blocks*block_size exceeds int32");
    return PA_OK;
}

static bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

} // namespace pa

using namespace pa;

extern "C" const char *pa_last_error_string(void) { return g_err; }

extern "C" int pa_version(void) { return 0x000500; }

extern "C" int pa_upload(void *dev_dst, const void *host_src, size_t bytes, pa_stream_t stream)
{
    if (bytes == 0)
        return PA_OK;
    if (!dev_dst || !host_src)
        return fail(PA_ERR_INVALID_ARG, "pa_upload: NULL pointer");
    cudaError_t e = cudaMemcpyAsync(dev_dst, host_src, bytes, cudaMemcpyHostToDevice, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "cudaMemcpyAsync: %s", cudaGetErrorString(e));
    return PA_OK;
}

extern "C" int pa_store_kvcache(const pa_dims *dims, const void *k, const void *v, void *k_cache, void *v_cache,
                                const int32_t *slot_mapping, int32_t num_tokens, pa_stream_t stream)
{
    int rc = check_dims(dims);
    if (rc != PA_OK)
        return rc;
    if (num_tokens < 0)
        return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0)
        return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "pa_store_kvcache: NULL pointer");
    if (misaligned(k) || misaligned(v) || misaligned(k_cache) || misaligned(v_cache))
        return fail(PA_ERR_INVALID_ARG, "pa_store_kvcache: tensors must be 16-byte aligned");
    return launch_store_kvcache(*dims, k, v, k_cache, v_cache, slot_mapping, num_tokens, stream);
}

// Host-side checks shared by pa_prefill_varlen and pa_prefill_varlen_int8;
// fills `a`.  Sets *nothing when the plan has no work (then no launch happens).
static int prepare_prefill(const char *fn, const pa_dims *dims, const void *q, const void *k_cache,
                           const void *v_cache, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                           const int32_t *block_tables, float scale, void *out, const pa_prefill_meta *meta,
                           const int32_t *tiles, PrefillArgs *a, bool *nothing)
{
    *nothing = false;
    int rc = check_dims(dims);
    if (rc != PA_OK)
        return rc;
    if (!meta)
        return fail(PA_ERR_INVALID_ARG, "meta is NULL");
    if (meta->num_tiles < 0 || meta->total_q < 0 || meta->num_seqs < 0 || meta->max_blocks_per_seq < 1)
        return fail(PA_ERR_INVALID_ARG, "malformed prefill meta");
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(PA_ERR_INVALID_ARG, "scale must be finite and > 0");
    const int group = dims->num_heads / dims->num_kv_heads;
    if (meta->rows_per_tile != (kPrefillRows / group > 0 ? kPrefillRows / group : 1))
        return fail(PA_ERR_INVALID_ARG, "prefill meta was packed for other dims");
    if (meta->num_tiles == 0 || meta->total_q == 0) {
        *nothing = true;
        return PA_OK;
    }
    if (!q || !k_cache || !v_cache || !cu_seqlens_q || !cu_seqlens_k || !block_tables || !out || !tiles)
        return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    if (misaligned(q) || misaligned(k_cache) || misaligned(v_cache) || misaligned(out))
        return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", fn);
    if (dims->num_blocks == 0)
        return fail(PA_ERR_INVALID_ARG, "empty KV pool");
    *a = PrefillArgs{};
    a->dims = *dims;
    a->q = q;
    a->k_cache = k_cache;
    a->v_cache = v_cache;
    a->cu_seqlens_q = cu_seqlens_q;
    a->cu_seqlens_k = cu_seqlens_k;
    a->block_tables = block_tables;
    a->tiles = tiles;
    a->out = out;
    a->scale = scale;
    a->num_tiles = meta->num_tiles;
    a->total_q = meta->total_q;
    a->max_blocks_per_seq = meta->max_blocks_per_seq;
    a->rows_per_tile = meta->rows_per_tile;
    return PA_OK;
}

extern "C" int pa_prefill_varlen(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                 const int32_t *block_tables, float scale, void *out, const pa_prefill_meta *meta,
                                 const int32_t *tiles, pa_stream_t stream)
{
    PrefillArgs a;
    bool nothing = false;
    int rc = prepare_prefill("pa_prefill_varlen", dims, q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k,
                             block_tables, scale, out, meta, tiles, &a, &nothing);
    if (rc != PA_OK || nothing)
        return rc;
    return launch_prefill(a, stream);
}

extern "C" int pa_prefill_varlen_fused(const pa_dims *dims, const void *q, const void *k, const void *v,
                                       void *k_cache, void *v_cache, const int32_t *cu_seqlens_q,
                                       const int32_t *cu_seqlens_k, const int32_t *block_tables,
                                       const int32_t *slot_mapping, float scale, void *out,
                                       const pa_prefill_meta *meta, const int32_t *tiles, pa_stream_t stream)
{
    PrefillArgs a;
    bool nothing = false;
    int rc = prepare_prefill("pa_prefill_varlen_fused", dims, q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k,
                             block_tables, scale, out, meta, tiles, &a, &nothing);
    if (rc != PA_OK || nothing)
        return rc;
    if (!k || !v || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_varlen_fused: NULL pointer");
    if (misaligned(k) || misaligned(v))
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_varlen_fused: tensors must be 16-byte aligned");
    a.k_in = k;
    a.v_in = v;
    a.slot_mapping = slot_mapping;
    a.small_boxes = !meta->prefix_aligned;
    return launch_prefill(a, stream);
}

// INT8 prefill (plain and with the quantising store): the gather launch fills the
// plan's bf16 scratch cache from the INT8 cache (k_in set: after quantising the new
// rows into it), then the bf16 prefill kernel attends over the scratch cache through
// the scratch tables (128-token blocks).
static int prefill_int8(const char *fn, bool store, const pa_dims *dims, const void *q, const void *k, const void *v,
                        const void *k_cache, const void *v_cache, const void *k_scale, const void *v_scale,
                        const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, const int32_t *block_tables,
                        const int32_t *slot_mapping, const int32_t *scratch_tables, const int32_t *scratch_items,
                        float scale, void *out, const pa_prefill_meta *meta, const int32_t *tiles, void *workspace,
                        size_t workspace_bytes, pa_stream_t stream)
{
    PrefillArgs a;
    bool nothing = false;
    int rc = prepare_prefill(fn, dims, q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, scale, out,
                             meta, tiles, &a, &nothing);
    if (rc != PA_OK || nothing)
        return rc;
    const pa_dims &d = *dims;
    if (!k_scale || !v_scale || !scratch_tables || !scratch_items || !workspace)
        return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    if (misaligned(k_scale) || misaligned(v_scale) || misaligned(workspace) || misaligned(scratch_items))
        return fail(PA_ERR_INVALID_ARG, "%s: scales, scratch items and workspace must be 16-byte aligned", fn);
    if (meta->scratch_blocks < 1 || meta->scratch_pitch < 1 ||
        meta->workspace_bytes != (uint64_t)meta->scratch_blocks * kPrefillKeyTile * d.num_kv_heads * d.head_dim * 4)
        return fail(PA_ERR_INVALID_ARG, "%s: prefill meta was packed for other dims", fn);
    if (workspace_bytes < meta->workspace_bytes)
        return fail(PA_ERR_WORKSPACE, "%s: workspace has %zu bytes, needs %llu", fn, workspace_bytes,
                    (unsigned long long)meta->workspace_bytes);
    if (store) {
        if (!k || !v || !slot_mapping)
            return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", fn);
        if (misaligned(k) || misaligned(v))
            return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", fn);
    }
    const size_t half = (size_t)meta->scratch_blocks * kPrefillKeyTile * d.num_kv_heads * d.head_dim;
    GatherArgs g{};
    g.num_kv_heads = d.num_kv_heads;
    g.head_dim = d.head_dim;
    g.block_size = d.block_size;
    g.max_blocks = meta->max_blocks_per_seq;
    g.scratch_blocks = meta->scratch_blocks;
    g.num_slots = (int64_t)d.num_blocks * d.block_size;
    g.k_codes = static_cast<const int8_t *>(k_cache);
    g.v_codes = static_cast<const int8_t *>(v_cache);
    g.k_scale = static_cast<const uint16_t *>(k_scale);
    g.v_scale = static_cast<const uint16_t *>(v_scale);
    g.block_tables = block_tables;
    g.scratch_items = scratch_items;
    g.k_out = static_cast<uint16_t *>(workspace);
    g.v_out = g.k_out + half;
    g.out_v8 = (reinterpret_cast<uintptr_t>(workspace) & 31u) == 0 ? 1 : 0;
    if (store) {
        g.k_in = static_cast<const uint16_t *>(k);
        g.v_in = static_cast<const uint16_t *>(v);
        g.slot_mapping = slot_mapping;
        g.k_codes_w = static_cast<int8_t *>(const_cast<void *>(k_cache));
        g.v_codes_w = static_cast<int8_t *>(const_cast<void *>(v_cache));
        g.k_scale_w = static_cast<uint16_t *>(const_cast<void *>(k_scale));
        g.v_scale_w = static_cast<uint16_t *>(const_cast<void *>(v_scale));
    }
    if ((rc = launch_int8_gather(g, stream)) != PA_OK)
        return rc;
    a.dims.num_blocks = meta->scratch_blocks;
    a.dims.block_size = kPrefillKeyTile;
    a.k_cache = g.k_out;
    a.v_cache = g.v_out;
    a.block_tables = scratch_tables;
    a.max_blocks_per_seq = meta->scratch_pitch;
    a.scratch_cache = true;
    return launch_prefill(a, stream);
}

extern "C" int pa_prefill_varlen_int8(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                                      const void *k_scale, const void *v_scale, const int32_t *cu_seqlens_q,
                                      const int32_t *cu_seqlens_k, const int32_t *block_tables,
                                      const int32_t *scratch_tables, const int32_t *scratch_items, float scale,
                                      void *out, const pa_prefill_meta *meta, const int32_t *tiles, void *workspace,
                                      size_t workspace_bytes, pa_stream_t stream)
{
    return prefill_int8("pa_prefill_varlen_int8", false, dims, q, nullptr, nullptr, k_cache, v_cache, k_scale, v_scale,
                        cu_seqlens_q, cu_seqlens_k, block_tables, nullptr, scratch_tables, scratch_items, scale, out,
                        meta, tiles, workspace, workspace_bytes, stream);
}

extern "C" int pa_prefill_varlen_int8_fused(const pa_dims *dims, const void *q, const void *k, const void *v,
                                            void *k_cache, void *v_cache, void *k_scale, void *v_scale,
                                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                            const int32_t *block_tables, const int32_t *slot_mapping,
                                            const int32_t *scratch_tables, const int32_t *scratch_items, float scale,
                                            void *out, const pa_prefill_meta *meta, const int32_t *tiles,
                                            void *workspace, size_t workspace_bytes, pa_stream_t stream)
{
    return prefill_int8("pa_prefill_varlen_int8_fused", true, dims, q, k, v, k_cache, v_cache, k_scale, v_scale,
                        cu_seqlens_q, cu_seqlens_k, block_tables, slot_mapping, scratch_tables, scratch_items, scale,
                        out, meta, tiles, workspace, workspace_bytes, stream);
}

// Host-side checks shared by pa_decode and pa_decode_int8; fills `a`.  Sets
// *nothing when the plan has no work (then no launch happens).
static int prepare_decode(const char *fn, const pa_dims *dims, const void *q, const void *k_cache,
                          const void *v_cache, const int32_t *context_lens, const int32_t *block_tables, float scale,
                          void *out, const pa_decode_meta *meta, const int32_t *items, const int32_t *seq_items,
                          void *workspace, size_t workspace_bytes, DecodeArgs *a, bool *nothing)
{
    *nothing = false;
    int rc = check_dims(dims);
    if (rc != PA_OK)
        return rc;
    if (!meta)
        return fail(PA_ERR_INVALID_ARG, "meta is NULL");
    if (meta->num_items < 0 || meta->num_seqs < 0 || meta->max_blocks_per_seq < 1 || meta->max_splits < 1)
        return fail(PA_ERR_INVALID_ARG, "malformed decode meta");
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(PA_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (meta->num_items == 0) {
        *nothing = true;
        return PA_OK;
    }
    if (!q || !k_cache || !v_cache || !context_lens || !block_tables || !out || !items || !seq_items)
        return fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    if (misaligned(q) || misaligned(k_cache) || misaligned(v_cache) || misaligned(out))
        return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", fn);
    if (workspace_bytes < meta->workspace_bytes)
        return fail(PA_ERR_WORKSPACE, "decode workspace has %zu bytes, needs %llu", workspace_bytes,
                    (unsigned long long)meta->workspace_bytes);
    if (meta->workspace_bytes > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return fail(PA_ERR_INVALID_ARG, "decode workspace must be non-NULL and 256-byte aligned");
    *a = DecodeArgs{};
    a->dims = *dims;
    a->q = q;
    a->k_cache = k_cache;
    a->v_cache = v_cache;
    a->context_lens = context_lens;
    a->block_tables = block_tables;
    a->items = items;
    a->seq_items = seq_items;
    a->out = out;
    if (meta->num_partials < 0)
        return fail(PA_ERR_INVALID_ARG, "malformed decode meta");
    if (meta->num_partials > 0) {
        size_t per = (size_t)dims->num_heads * dims->head_dim * 4;
        size_t need = align_up((size_t)meta->num_partials * per, 256) +
                      align_up((size_t)meta->num_partials * dims->num_heads * 4, 256);
        if (need > meta->workspace_bytes)
            return fail(PA_ERR_INVALID_ARG, "decode meta workspace size inconsistent with its partial count");
        a->part_o = static_cast<float *>(workspace);
        a->part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                align_up((size_t)meta->num_partials * per, 256));
    }
    a->scale = scale;
    a->num_seqs = meta->num_seqs;
    a->num_items = meta->num_items;
    a->max_blocks_per_seq = meta->max_blocks_per_seq;
    a->max_splits = meta->max_splits;
    return PA_OK;
}

extern "C" int pa_decode(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *context_lens, const int32_t *block_tables, float scale, void *out,
                         const pa_decode_meta *meta, const int32_t *items, const int32_t *seq_items, void *workspace,
                         size_t workspace_bytes, pa_stream_t stream)
{
    DecodeArgs a;
    bool nothing = false;
    int rc = prepare_decode("pa_decode", dims, q, k_cache, v_cache, context_lens, block_tables, scale, out, meta,
                            items, seq_items, workspace, workspace_bytes, &a, &nothing);
    if (rc != PA_OK || nothing)
        return rc;
    return launch_decode(a, stream);
}

extern "C" int pa_decode_fused(const pa_dims *dims, const void *q, const void *k, const void *v, void *k_cache,
                               void *v_cache, const int32_t *slot_mapping, const int32_t *context_lens,
                               const int32_t *block_tables, float scale, void *out, const pa_decode_meta *meta,
                               const int32_t *items, const int32_t *seq_items, void *workspace,
                               size_t workspace_bytes, pa_stream_t stream)
{
    DecodeArgs a;
    bool nothing = false;
    int rc = prepare_decode("pa_decode_fused", dims, q, k_cache, v_cache, context_lens, block_tables, scale, out,
                            meta, items, seq_items, workspace, workspace_bytes, &a, &nothing);
    if (rc != PA_OK || nothing)
        return rc;
    if (!k || !v || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "pa_decode_fused: NULL pointer");
    if (misaligned(k) || misaligned(v))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_fused: tensors must be 16-byte aligned");
    a.k_new = k;
    a.v_new = v;
    a.slot_mapping = slot_mapping;
    return launch_decode(a, stream);
}

extern "C" int pa_decode_int8_fused(const pa_dims *dims, const void *q, const void *k, const void *v,
                                    void *k_cache, void *v_cache, void *k_scale, void *v_scale,
                                    const int32_t *slot_mapping, const int32_t *context_lens,
                                    const int32_t *block_tables, float scale, void *out, const pa_decode_meta *meta,
                                    const int32_t *items, const int32_t *seq_items, void *workspace,
                                    size_t workspace_bytes, pa_stream_t stream)
{
    DecodeArgs a;
    bool nothing = false;
    int rc = prepare_decode("pa_decode_int8_fused", dims, q, k_cache, v_cache, context_lens, block_tables, scale,
                            out, meta, items, seq_items, workspace, workspace_bytes, &a, &nothing);
    if (rc != PA_OK || nothing)
        return rc;
    if (!k || !v || !slot_mapping || !k_scale || !v_scale)
        return fail(PA_ERR_INVALID_ARG, "pa_decode_int8_fused: NULL pointer");
    if (misaligned(k) || misaligned(v) || misaligned(k_scale) || misaligned(v_scale))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_int8_fused: tensors must be 16-byte aligned");
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.k_new = k;
    a.v_new = v;
    a.slot_mapping = slot_mapping;
    return launch_decode_int8(a, stream);
}

extern "C" int pa_store_kvcache_int8(const pa_dims *dims, const void *k, const void *v, void *k_cache,
                                     void *v_cache, void *k_scale, void *v_scale, const int32_t *slot_mapping,
                                     int32_t num_tokens, pa_stream_t stream)
{
    int rc = check_dims(dims);
    if (rc != PA_OK)
        return rc;
    if (num_tokens < 0)
        return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0)
        return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "pa_store_kvcache_int8: NULL pointer");
    if (misaligned(k) || misaligned(v) || misaligned(k_cache) || misaligned(v_cache) || misaligned(k_scale) ||
        misaligned(v_scale))
        return fail(PA_ERR_INVALID_ARG, "pa_store_kvcache_int8: tensors must be 16-byte aligned");
    return launch_store_kvcache_int8(*dims, k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, num_tokens,
                                     stream);
}

extern "C" int pa_decode_int8(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                              const void *k_scale, const void *v_scale, const int32_t *context_lens,
                              const int32_t *block_tables, float scale, void *out, const pa_decode_meta *meta,
                              const int32_t *items, const int32_t *seq_items, void *workspace,
                              size_t workspace_bytes, pa_stream_t stream)
{
    DecodeArgs a;
    bool nothing = false;
    int rc = prepare_decode("pa_decode_int8", dims, q, k_cache, v_cache, context_lens, block_tables, scale, out,
                            meta, items, seq_items, workspace, workspace_bytes, &a, &nothing);
    if (rc != PA_OK || nothing)
        return rc;
    if (!k_scale || !v_scale)
        return fail(PA_ERR_INVALID_ARG, "pa_decode_int8: NULL scale pointer");
    if (misaligned(k_scale) || misaligned(v_scale))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_int8: scales must be 16-byte aligned");
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return launch_decode_int8(a, stream);
}

extern "C" int pa_copy_blocks(const pa_dims *dims, void *k_cache, void *v_cache, const int32_t *triples,
                              int32_t num_triples, pa_stream_t stream)
{
    int rc = check_dims(dims);
    if (rc != PA_OK)
        return rc;
    if (num_triples < 0)
        return fail(PA_ERR_INVALID_ARG, "num_triples < 0");
    if (num_triples == 0)
        return PA_OK;
    if (!k_cache || !v_cache || !triples)
        return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: NULL pointer");
    if (misaligned(k_cache) || misaligned(v_cache) || (reinterpret_cast<uintptr_t>(triples) & 3u))
        return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: misaligned pointer");
    return launch_copy_blocks(*dims, k_cache, v_cache, triples, num_triples, stream);
}

extern "C" int pa_copy_blocks_int8(const pa_dims *dims, void *k_cache, void *v_cache, void *k_scale, void *v_scale,
                                   const int32_t *triples, int32_t num_triples, pa_stream_t stream)
{
    int rc = check_dims(dims);
    if (rc != PA_OK)
        return rc;
    if (num_triples < 0)
        return fail(PA_ERR_INVALID_ARG, "num_triples < 0");
    if (num_triples == 0)
        return PA_OK;
    if (!k_cache || !v_cache || !k_scale || !v_scale || !triples)
        return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks_int8: NULL pointer");
    if (misaligned(k_cache) || misaligned(v_cache) || misaligned(k_scale) || misaligned(v_scale) ||
        (reinterpret_cast<uintptr_t>(triples) & 3u))
        return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks_int8: misaligned pointer");
    return launch_copy_blocks(*dims, k_cache, v_cache, triples, num_triples, stream, k_scale, v_scale);
}

// pa_decode for callers that cannot allocate: the workspace is the library's
// own scratch array (see the header for its limit, set-up and sharing rules).
extern "C" int pa_decode_static(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *context_lens, const int32_t *block_tables, float scale, void *out,
                                const pa_decode_meta *meta, const int32_t *items, const int32_t *seq_items,
                                pa_stream_t stream)
{
    if (!meta)
        return fail(PA_ERR_INVALID_ARG, "meta is NULL");
    if (meta->workspace_bytes > PA_DECODE_STATIC_SCRATCH_BYTES)
        return fail(PA_ERR_WORKSPACE,
                    "pa_decode_static: plan needs %llu bytes of scratch, the library array holds %u; "
                    "use pa_decode with a workspace or pack with larger splits",
                    (unsigned long long)meta->workspace_bytes, PA_DECODE_STATIC_SCRATCH_BYTES);
    void *scratch = nullptr;
    int rc = decode_static_scratch(&scratch);
    if (rc != PA_OK)
        return rc;
    DecodeArgs a;
    bool nothing = false;
    rc = prepare_decode("pa_decode_static", dims, q, k_cache, v_cache, context_lens, block_tables, scale, out, meta,
                        items, seq_items, scratch, PA_DECODE_STATIC_SCRATCH_BYTES, &a, &nothing);
    if (rc != PA_OK || nothing)
        return rc;
    return launch_decode(a, stream);
}

extern "C" int pa_read_device_error(uint32_t *code, pa_stream_t stream)
{
    if (!code)
        return fail(PA_ERR_INVALID_ARG, "code is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    *code = 0;
    int rc = read_store_error(code);
    if (rc == PA_OK)
        rc = read_prefill_error(code);
    if (rc == PA_OK)
        rc = read_copy_error(code);
    if (rc == PA_OK)
        rc = read_decode_error(code);
    if (rc == PA_OK)
        rc = read_fused_error(code);
    if (rc == PA_OK)
        rc = read_fused8_error(code);
    if (rc == PA_OK)
        rc = read_selftest_error(code);
    return rc;
}

extern "C" int pa_stream_read(const void *src, size_t bytes, uint32_t *sink, pa_stream_t stream)
{
    if (bytes && !src)
        return fail(PA_ERR_INVALID_ARG, "pa_stream_read: src is NULL");
    if (!sink)
        return fail(PA_ERR_INVALID_ARG, "pa_stream_read: sink is NULL");
    if ((reinterpret_cast<uintptr_t>(src) & 15u) || (bytes & 15u) || (reinterpret_cast<uintptr_t>(sink) & 3u))
        return fail(PA_ERR_INVALID_ARG, "pa_stream_read: src and bytes must be 16-byte aligned, sink 4-byte aligned");
    return launch_stream_read(src, bytes, sink, stream);
}

extern "C" int pa_selftest_bounded_wait(uint32_t timeout_us, int arrive_first, pa_stream_t stream)
{
    if (timeout_us < 1 || timeout_us > 10000000u)
        return fail(PA_ERR_INVALID_ARG, "timeout_us (%u) must be in [1, 10000000]", timeout_us);
    return launch_selftest_wait(timeout_us, arrive_first ? 1 : 0, stream);
}
