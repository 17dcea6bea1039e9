// Host-side metadata packing for libpagedattn.
//
// Everything the kernels need to find their work is computed here on the CPU,
// from host arrays, into one caller buffer that is then uploaded with a single
// asynchronous copy.  Sources (page title, section):
//  - "手搓 vLLM 推理引擎" (LLM-101-CN nano-vllm walkthrough), Step 5:
//    prepare_prefill() builds cu_seqlens_q/k as prefix sums of the query and
//    key lengths (query length = len - num_cached_tokens) and the slots of the
//    new tokens, block_table[pos / block_size]*block_size + pos % block_size;
//    prepare_decode() uses context_lens = len(seq) and the slot of the last
//    token.  Block tables are padded rows of physical block ids (-1 padding,
//    prepare_block_tables).
//  - "面试问答准备: nano-vLLM 推理引擎优化", Q1: the per-token index arrays of
//    the varlen kernel are built on the CPU next to the scheduling loop so no
//    device scalar is ever read back.  Here the same idea yields a tile work
//    list (prefill) and a split plan (decode).
#include <algorithm>
#include <cstring>
#include <numeric>
#include <vector>

#include <cuda_runtime.h>

#include "internal.h"

namespace pa {
namespace {

struct Layout {
    size_t off = 0;
    size_t take(size_t bytes)
    {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    }
};

int check_seq_blocks(const pa_dims &d, int32_t num_seqs, const int32_t *lens, const int32_t *block_offsets,
                     const int32_t *block_ids, int32_t *max_blocks)
{
    if (!block_offsets)
        return fail(PA_ERR_INVALID_ARG, "block_offsets is NULL");
    if (block_offsets[0] != 0)
        return fail(PA_ERR_INVALID_ARG, "block_offsets[0] must be 0");
    int32_t mb = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        int64_t have = (int64_t)block_offsets[b + 1] - block_offsets[b];
        if (have < 0)
            return fail(PA_ERR_INVALID_ARG, "block_offsets not non-decreasing at sequence %d", b);
        int64_t need = ((int64_t)lens[b] + d.block_size - 1) / d.block_size;
        if (need > have)
            return fail(PA_ERR_INVALID_ARG, "sequence %d needs %lld blocks, has %lld", b, (long long)need,
                        (long long)have);
        if (need > 0 && !block_ids)
            return fail(PA_ERR_INVALID_ARG, "block_ids is NULL");
        for (int64_t i = 0; i < need; ++i) {
            int32_t p = block_ids[block_offsets[b] + i];
            if (p < 0 || p >= d.num_blocks)
                return fail(PA_ERR_INVALID_ARG, "sequence %d block %lld: id %d outside [0, %d)", b, (long long)i, p,
                            d.num_blocks);
        }
        mb = std::max<int32_t>(mb, (int32_t)need);
    }
    *max_blocks = std::max<int32_t>(mb, 1);
    return PA_OK;
}

void write_block_tables(const pa_dims &d, int32_t num_seqs, const int32_t *lens, const int32_t *block_offsets,
                        const int32_t *block_ids, int32_t mb, int32_t *bt)
{
    for (int32_t b = 0; b < num_seqs; ++b) {
        int32_t need = (int32_t)(((int64_t)lens[b] + d.block_size - 1) / d.block_size);
        int32_t *row = bt + (size_t)b * mb;
        for (int32_t i = 0; i < mb; ++i)
            row[i] = i < need ? block_ids[block_offsets[b] + i] : -1;
    }
}

} // namespace
} // namespace pa

using namespace pa;

extern "C" int pa_pack_prefill(const pa_dims *dims, int32_t num_seqs, const int32_t *seq_lens,
                               const int32_t *query_lens, const int32_t *block_offsets, const int32_t *block_ids,
                               void *host_buf, size_t host_buf_bytes, pa_prefill_meta *meta)
{
    int rc = check_dims(dims);
    if (rc != PA_OK)
        return rc;
    if (!meta)
        return fail(PA_ERR_INVALID_ARG, "meta is NULL");
    if (num_seqs < 0)
        return fail(PA_ERR_INVALID_ARG, "num_seqs < 0");
    if (num_seqs > 0 && (!seq_lens || !query_lens))
        return fail(PA_ERR_INVALID_ARG, "seq_lens/query_lens is NULL");
    const pa_dims &d = *dims;
    const int group = d.num_heads / d.num_kv_heads;
    int64_t total_q = 0, total_k = 0;
    int32_t max_q = 0, max_k = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        if (query_lens[b] < 0 || seq_lens[b] < query_lens[b])
            return fail(PA_ERR_INVALID_ARG, "sequence %d: need 0 <= query_len (%d) <= seq_len (%d)", b,
                        query_lens[b], seq_lens[b]);
        total_q += query_lens[b];
        total_k += seq_lens[b];
        max_q = std::max(max_q, query_lens[b]);
        max_k = std::max(max_k, seq_lens[b]);
    }
    if (total_q > INT32_MAX || total_k > INT32_MAX)
        return fail(PA_ERR_INVALID_ARG, "total length exceeds int32");
    int32_t mb = 1;
    if (num_seqs > 0 && (rc = check_seq_blocks(d, num_seqs, seq_lens, block_offsets, block_ids, &mb)) != PA_OK)
        return rc;

    // work list: (sequence, first query row, KV head, key tiles), longest first.
    // One item = two query tiles of `rows` positions each (the kernel ping-pongs them).
    const int32_t rows = std::max(1, kPrefillRows / group);
    const int32_t span = kPrefillTilesPerItem * rows;
    struct Tile {
        int32_t seq, q0, kvh, nkt;
    };
    std::vector<Tile> tiles;
    for (int32_t b = 0; b < num_seqs; ++b) {
        const int32_t lq = query_lens[b], lk = seq_lens[b];
        for (int32_t q0 = 0; q0 < lq; q0 += span) {
            int32_t last = std::min(q0 + span, lq) - 1;       // last query row of the item
            int32_t visible = lk - lq + last + 1;             // keys that row sees
            int32_t nkt = (visible + kPrefillKeyTile - 1) / kPrefillKeyTile;
            for (int32_t g = 0; g < d.num_kv_heads; ++g)
                tiles.push_back({b, q0, g, nkt});
        }
    }
    std::stable_sort(tiles.begin(), tiles.end(), [](const Tile &x, const Tile &y) { return x.nkt > y.nkt; });
    if (tiles.size() > (size_t)INT32_MAX / kPrefillItemInts)
        return fail(PA_ERR_INVALID_ARG, "too many tiles");

    Layout L;
    meta->num_seqs = num_seqs;
    meta->total_q = (int32_t)total_q;
    meta->max_seqlen_q = max_q;
    meta->max_seqlen_k = max_k;
    meta->max_blocks_per_seq = mb;
    meta->num_tiles = (int32_t)tiles.size();
    meta->rows_per_tile = rows;
    // the fused store + prefill reads the new keys from the inputs in boxes of min(block
    // size, 128) keys: possible when no box straddles a cached prefix and the new keys
    int32_t aligned = 1;
    const int32_t box = std::min<int32_t>(d.block_size, kPrefillKeyTile);
    for (int32_t b = 0; b < num_seqs; ++b) // sequences without new tokens have no work items
        if (query_lens[b] > 0 && (seq_lens[b] - query_lens[b]) % box != 0)
            aligned = 0;
    meta->prefix_aligned = aligned;
    // INT8 prefill scratch: each sequence with new tokens gets ceil(seq_len / 128)
    // consecutive 128-token blocks of a bf16 cache (K and V), in sequence order
    int64_t sblocks = 0;
    int32_t spitch = 1;
    for (int32_t b = 0; b < num_seqs; ++b)
        if (query_lens[b] > 0) {
            const int32_t n = (seq_lens[b] + kPrefillKeyTile - 1) / kPrefillKeyTile;
            sblocks += n;
            spitch = std::max(spitch, n);
        }
    if (sblocks * kPrefillKeyTile > INT32_MAX)
        return fail(PA_ERR_INVALID_ARG, "INT8 prefill scratch exceeds int32 rows");
    meta->scratch_blocks = (int32_t)sblocks;
    meta->scratch_pitch = spitch;
    meta->workspace_bytes = (uint64_t)sblocks * kPrefillKeyTile * d.num_kv_heads * d.head_dim * 2 * 2;
    meta->off_cu_seqlens_q = L.take(sizeof(int32_t) * (num_seqs + 1));
    meta->off_cu_seqlens_k = L.take(sizeof(int32_t) * (num_seqs + 1));
    meta->off_block_tables = L.take(sizeof(int32_t) * (size_t)num_seqs * mb);
    meta->off_slot_mapping = L.take(sizeof(int32_t) * (size_t)total_q);
    meta->off_tiles = L.take(sizeof(int32_t) * kPrefillItemInts * tiles.size());
    meta->off_scratch_tables = L.take(sizeof(int32_t) * (size_t)num_seqs * spitch);
    meta->off_scratch_items = L.take(sizeof(int32_t) * 8 * (size_t)sblocks);
    meta->total_bytes = L.off;
    if (!host_buf)
        return PA_OK;
    if (host_buf_bytes < meta->total_bytes)
        return fail(PA_ERR_WORKSPACE, "metadata buffer has %zu bytes, needs %llu", host_buf_bytes,
                    (unsigned long long)meta->total_bytes);

    char *base = static_cast<char *>(host_buf);
    int32_t *cu_q = reinterpret_cast<int32_t *>(base + meta->off_cu_seqlens_q);
    int32_t *cu_k = reinterpret_cast<int32_t *>(base + meta->off_cu_seqlens_k);
    int32_t *bt = reinterpret_cast<int32_t *>(base + meta->off_block_tables);
    int32_t *slots = reinterpret_cast<int32_t *>(base + meta->off_slot_mapping);
    int32_t *tl = reinterpret_cast<int32_t *>(base + meta->off_tiles);
    int32_t *stab = reinterpret_cast<int32_t *>(base + meta->off_scratch_tables);
    int32_t *sitem = reinterpret_cast<int32_t *>(base + meta->off_scratch_items);
    cu_q[0] = cu_k[0] = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        cu_q[b + 1] = cu_q[b] + query_lens[b];
        cu_k[b + 1] = cu_k[b] + seq_lens[b];
    }
    for (int32_t b = 0, sb = 0; b < num_seqs; ++b) {
        const int32_t n = query_lens[b] > 0 ? (seq_lens[b] + kPrefillKeyTile - 1) / kPrefillKeyTile : 0;
        for (int32_t i = 0; i < spitch; ++i)
            stab[(size_t)b * spitch + i] = i < n ? sb + i : -1;
        for (int32_t i = 0; i < n; ++i) {
            int32_t *e = sitem + 8 * (size_t)(sb + i);
            const int32_t cached = seq_lens[b] - query_lens[b];
            e[0] = b;
            e[1] = i * kPrefillKeyTile;
            e[2] = seq_lens[b];
            e[3] = cached;
            e[4] = cu_q[b] - cached;
            e[5] = e[6] = e[7] = 0;
        }
        sb += n;
    }
    if (num_seqs > 0)
        write_block_tables(d, num_seqs, seq_lens, block_offsets, block_ids, mb, bt);
    int64_t t = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        const int32_t *blk = block_ids + block_offsets[b];
        for (int32_t pos = seq_lens[b] - query_lens[b]; pos < seq_lens[b]; ++pos)
            slots[t++] = blk[pos / d.block_size] * d.block_size + pos % d.block_size;
    }
    for (size_t i = 0; i < tiles.size(); ++i) {
        int32_t *e = tl + kPrefillItemInts * i;
        const int32_t b = tiles[i].seq;
        e[0] = b;
        e[1] = tiles[i].q0;
        e[2] = tiles[i].kvh;
        e[3] = tiles[i].nkt;
        e[4] = cu_q[b];       // first packed query row of the sequence
        e[5] = query_lens[b];
        e[6] = seq_lens[b];
        e[7] = block_ids[block_offsets[b]]; // physical block holding key 0
    }
    return PA_OK;
}

extern "C" int pa_pack_decode(const pa_dims *dims, int32_t num_seqs, const int32_t *context_lens,
                              const int32_t *block_offsets, const int32_t *block_ids, int32_t split_tokens,
                              void *host_buf, size_t host_buf_bytes, pa_decode_meta *meta)
{
    int rc = check_dims(dims);
    if (rc != PA_OK)
        return rc;
    if (!meta)
        return fail(PA_ERR_INVALID_ARG, "meta is NULL");
    if (num_seqs < 0)
        return fail(PA_ERR_INVALID_ARG, "num_seqs < 0");
    if (num_seqs > 0 && !context_lens)
        return fail(PA_ERR_INVALID_ARG, "context_lens is NULL");
    if (split_tokens < 0 || split_tokens % kDecodeStep != 0)
        return fail(PA_ERR_INVALID_ARG, "split_tokens (%d) must be 0 or a positive multiple of %d", split_tokens,
                    kDecodeStep);
    const pa_dims &d = *dims;
    int64_t total = 0;
    int32_t max_ctx = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        if (context_lens[b] < 0)
            return fail(PA_ERR_INVALID_ARG, "context_lens[%d] < 0", b);
        total += context_lens[b];
        max_ctx = std::max(max_ctx, context_lens[b]);
    }
    int32_t mb = 1;
    if (num_seqs > 0 && (rc = check_seq_blocks(d, num_seqs, context_lens, block_offsets, block_ids, &mb)) != PA_OK)
        return rc;

    if (split_tokens == 0) {
        // Enough CTAs for several full waves of the GPU, at least 512 keys each.
        int dev = 0, sms = 148;
        if (cudaGetDevice(&dev) == cudaSuccess)
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaGetLastError();
        const int group = d.num_heads / d.num_kv_heads;
        int64_t slots = (int64_t)sms * std::max(1, decode_ctas_per_sm(d.head_dim, group));
        int64_t target = 8 * slots;
        int64_t units = (int64_t)num_seqs * d.num_kv_heads;
        if (units >= target || total == 0) {
            split_tokens = (int32_t)align_up((size_t)std::max(max_ctx, 1), kDecodeStep);
        } else {
            int64_t per = (total * d.num_kv_heads + target - 1) / target;
            split_tokens = (int32_t)align_up((size_t)std::max<int64_t>(per, 512), 256);
        }
    }

    // split plan: each sequence's context cut into n near-equal ranges (multiples of 64)
    struct Item {
        int32_t seq, k0, k1, slot;
    };
    std::vector<Item> items;
    std::vector<int32_t> seq_items(num_seqs + 1, 0);
    int32_t max_splits = 1;
    for (int32_t b = 0; b < num_seqs; ++b) {
        const int32_t ctx = context_lens[b];
        int32_t n = std::max<int32_t>(1, (ctx + split_tokens - 1) / split_tokens);
        int32_t len = (int32_t)align_up((size_t)((ctx + n - 1) / n), kDecodeStep);
        if (len > 0)
            n = std::max<int32_t>(1, (ctx + len - 1) / len);
        max_splits = std::max(max_splits, n);
        seq_items[b + 1] = seq_items[b] + (n > 1 ? n : 0);
        for (int32_t s = 0; s < n; ++s) {
            int32_t k0 = s * len, k1 = std::min(ctx, (s + 1) * len);
            items.push_back({b, k0, k1, n > 1 ? seq_items[b] + s : -1});
        }
    }
    std::stable_sort(items.begin(), items.end(),
                     [](const Item &x, const Item &y) { return x.k1 - x.k0 > y.k1 - y.k0; });
    const int64_t partials = num_seqs > 0 ? seq_items[num_seqs] : 0;

    Layout L;
    meta->num_seqs = num_seqs;
    meta->max_blocks_per_seq = mb;
    meta->num_items = (int32_t)items.size();
    meta->split_tokens = split_tokens;
    meta->max_splits = max_splits;
    meta->num_partials = (int32_t)partials;
    meta->off_context_lens = L.take(sizeof(int32_t) * num_seqs);
    meta->off_block_tables = L.take(sizeof(int32_t) * (size_t)num_seqs * mb);
    meta->off_slot_mapping = L.take(sizeof(int32_t) * num_seqs);
    meta->off_items = L.take(sizeof(int32_t) * 4 * items.size());
    meta->off_seq_items = L.take(sizeof(int32_t) * (num_seqs + 1));
    meta->total_bytes = L.off;
    meta->workspace_bytes = partials > 0 ? align_up((size_t)partials * d.num_heads * d.head_dim * 4, 256) +
                                               align_up((size_t)partials * d.num_heads * 4, 256)
                                         : 0;
    if (!host_buf)
        return PA_OK;
    if (host_buf_bytes < meta->total_bytes)
        return fail(PA_ERR_WORKSPACE, "metadata buffer has %zu bytes, needs %llu", host_buf_bytes,
                    (unsigned long long)meta->total_bytes);

    char *base = static_cast<char *>(host_buf);
    int32_t *cl = reinterpret_cast<int32_t *>(base + meta->off_context_lens);
    int32_t *bt = reinterpret_cast<int32_t *>(base + meta->off_block_tables);
    int32_t *slots = reinterpret_cast<int32_t *>(base + meta->off_slot_mapping);
    int32_t *it = reinterpret_cast<int32_t *>(base + meta->off_items);
    int32_t *si = reinterpret_cast<int32_t *>(base + meta->off_seq_items);
    if (num_seqs > 0) {
        std::memcpy(cl, context_lens, sizeof(int32_t) * num_seqs);
        write_block_tables(d, num_seqs, context_lens, block_offsets, block_ids, mb, bt);
    }
    for (int32_t b = 0; b < num_seqs; ++b) {
        int32_t pos = context_lens[b] - 1; // the token being decoded
        slots[b] = pos < 0 ? -1 : block_ids[block_offsets[b] + pos / d.block_size] * d.block_size + pos % d.block_size;
    }
    for (size_t i = 0; i < items.size(); ++i) {
        it[4 * i + 0] = items[i].seq;
        it[4 * i + 1] = items[i].k0;
        it[4 * i + 2] = items[i].k1;
        it[4 * i + 3] = items[i].slot;
    }
    std::memcpy(si, seq_items.data(), sizeof(int32_t) * (num_seqs + 1));
    return PA_OK;
}

extern "C" int pa_pack_decode_fixed(const pa_dims *dims, int32_t num_seqs, const int32_t *context_lens,
                                    const int32_t *block_offsets, const int32_t *block_ids, int32_t max_context,
                                    int32_t split_tokens, void *host_buf, size_t host_buf_bytes,
                                    pa_decode_meta *meta)
{
    int rc = check_dims(dims);
    if (rc != PA_OK)
        return rc;
    if (!meta)
        return fail(PA_ERR_INVALID_ARG, "meta is NULL");
    if (num_seqs < 1)
        return fail(PA_ERR_INVALID_ARG, "num_seqs must be >= 1 for a fixed-shape plan");
    if (!context_lens)
        return fail(PA_ERR_INVALID_ARG, "context_lens is NULL");
    if (max_context < 1)
        return fail(PA_ERR_INVALID_ARG, "max_context must be >= 1");
    if (split_tokens < 0 || split_tokens % kDecodeStep != 0)
        return fail(PA_ERR_INVALID_ARG, "split_tokens (%d) must be 0 or a positive multiple of %d", split_tokens,
                    kDecodeStep);
    const pa_dims &d = *dims;
    for (int32_t b = 0; b < num_seqs; ++b)
        if (context_lens[b] < 0 || context_lens[b] > max_context)
            return fail(PA_ERR_INVALID_ARG, "context_lens[%d] = %d outside [0, max_context = %d]", b, context_lens[b],
                        max_context);
    int32_t mb_used = 1;
    if ((rc = check_seq_blocks(d, num_seqs, context_lens, block_offsets, block_ids, &mb_used)) != PA_OK)
        return rc;
    // every shape below depends on (dims, num_seqs, max_context, split_tokens) only
    const int32_t split = split_tokens == 0 ? (int32_t)align_up((size_t)max_context, kDecodeStep) : split_tokens;
    const int32_t S = (max_context + split - 1) / split;
    const int32_t mb = (int32_t)(((int64_t)max_context + d.block_size - 1) / d.block_size);
    const int64_t num_items = (int64_t)num_seqs * S;
    if (num_items > INT32_MAX / 4)
        return fail(PA_ERR_INVALID_ARG, "too many work items");
    const int64_t partials = S > 1 ? num_items : 0;

    Layout L;
    meta->num_seqs = num_seqs;
    meta->max_blocks_per_seq = mb;
    meta->num_items = (int32_t)num_items;
    meta->split_tokens = split;
    meta->max_splits = S;
    meta->num_partials = (int32_t)partials;
    meta->off_context_lens = L.take(sizeof(int32_t) * num_seqs);
    meta->off_block_tables = L.take(sizeof(int32_t) * (size_t)num_seqs * mb);
    meta->off_slot_mapping = L.take(sizeof(int32_t) * num_seqs);
    meta->off_items = L.take(sizeof(int32_t) * 4 * (size_t)num_items);
    meta->off_seq_items = L.take(sizeof(int32_t) * (num_seqs + 1));
    meta->total_bytes = L.off;
    meta->workspace_bytes = partials > 0 ? align_up((size_t)partials * d.num_heads * d.head_dim * 4, 256) +
                                               align_up((size_t)partials * d.num_heads * 4, 256)
                                         : 0;
    if (!host_buf)
        return PA_OK;
    if (host_buf_bytes < meta->total_bytes)
        return fail(PA_ERR_WORKSPACE, "metadata buffer has %zu bytes, needs %llu", host_buf_bytes,
                    (unsigned long long)meta->total_bytes);

    char *base = static_cast<char *>(host_buf);
    int32_t *cl = reinterpret_cast<int32_t *>(base + meta->off_context_lens);
    int32_t *bt = reinterpret_cast<int32_t *>(base + meta->off_block_tables);
    int32_t *slots = reinterpret_cast<int32_t *>(base + meta->off_slot_mapping);
    int32_t *it = reinterpret_cast<int32_t *>(base + meta->off_items);
    int32_t *si = reinterpret_cast<int32_t *>(base + meta->off_seq_items);
    std::memcpy(cl, context_lens, sizeof(int32_t) * num_seqs);
    write_block_tables(d, num_seqs, context_lens, block_offsets, block_ids, mb, bt);
    for (int32_t b = 0; b < num_seqs; ++b) {
        int32_t pos = context_lens[b] - 1; // the token being decoded; -1 (padding entry) writes nothing
        slots[b] = pos < 0 ? -1 : block_ids[block_offsets[b] + pos / d.block_size] * d.block_size + pos % d.block_size;
        si[b] = S > 1 ? b * S : 0;
        for (int32_t s = 0; s < S; ++s) {
            const int32_t k0 = s * split;
            const bool empty = k0 >= context_lens[b];
            int32_t *e = it + 4 * ((size_t)b * S + s);
            e[0] = b;
            e[1] = empty ? 0 : k0; // empty ranges are (0, 0): only one item ends at the last key
            e[2] = empty ? 0 : std::min(context_lens[b], k0 + split);
            e[3] = S > 1 ? b * S + s : -1;
        }
    }
    si[num_seqs] = S > 1 ? num_seqs * S : 0;
    return PA_OK;
}
