// Internal declarations shared by the host-side translation units of libpagedattn.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "pagedattn.h"

namespace pa {

// Key tile of the prefill kernel and query rows of one tile (tcgen05 M).
constexpr int kPrefillKeyTile = 128;
constexpr int kPrefillRows = 128;
constexpr int kPrefillTilesPerItem = 2; // query tiles per prefill work item
// work-list entry: sequence, first query row, KV head, key tiles, first packed
// query row of the sequence, query length, key length, physical block of key 0
constexpr int kPrefillItemInts = 8;
// Keys per warp step of the decode kernel and per CTA step (4 warps).
constexpr int kDecodeChunk = 16;
constexpr int kDecodeStep = 64;
constexpr int kMaxGroup = 16;

// Thread-local error text.
void set_error(const char *fmt, ...);
int fail(int code, const char *fmt, ...);

// Shape checks shared by every entry point; returns PA_OK or an error code.
int check_dims(const pa_dims *dims);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Raise a kernel's dynamic shared-memory limit once per device (the attribute is
// per device; a process may drive several GPUs).  One flag word per kernel.
template <auto Kernel>
int ensure_smem(int bytes, const char *what)
{
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t)1 << dev : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit))
        return PA_OK;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "%s shared-memory attribute: %s", what, cudaGetErrorString(e));
    done.fetch_or(bit, std::memory_order_release);
    return PA_OK;
}

// Number of SMs of the current device (looked up once per device).
inline int sm_count(int *n)
{
    static std::atomic<int> cached[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    const bool slot = dev >= 0 && dev < 64;
    if (slot && (*n = cached[dev].load(std::memory_order_relaxed)) > 0)
        return PA_OK;
    e = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || *n < 1)
        return fail(PA_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
    if (slot)
        cached[dev].store(*n, std::memory_order_relaxed);
    return PA_OK;
}

// 3-D TMA descriptor (dims innermost first, strides of dims 1 and 2 in bytes,
// box in elements); PA_ERR_CUDA if the driver rejects it.
int encode_tmap_3d(CUtensorMap *m, CUtensorMapDataType type, const void *base, uint64_t d0, uint64_t d1,
                   uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                   CUtensorMapSwizzle swizzle, const char *what);

// Launchers (defined in the .cu files).  Each returns PA_OK or PA_ERR_CUDA.
int launch_store_kvcache(const pa_dims &d, const void *k, const void *v, void *k_cache, void *v_cache,
                         const int32_t *slot_mapping, int32_t num_tokens, void *stream);

// INT8 prefill front end: dequantise the keys/values a prefill batch reads into a
// bf16 scratch cache of 128-token blocks (and, with k_in set, first quantise the new
// tokens' rows into the INT8 cache).
struct GatherArgs {
    int32_t num_kv_heads, head_dim, block_size, max_blocks;
    int32_t scratch_blocks;
    int32_t out_v8; // the scratch is 32-byte aligned: 32-byte stores
    int64_t num_slots;
    const int8_t *k_codes, *v_codes;      // INT8 cache
    const uint16_t *k_scale, *v_scale;    // fp16 bits
    const int32_t *block_tables;
    const int32_t *scratch_items; // [scratch_blocks][8], see pa_prefill_meta
    uint16_t *k_out, *v_out;              // bf16 scratch [scratch_blocks * 128][Hkv][D]
    // quantising store of the new tokens (NULL otherwise)
    const uint16_t *k_in, *v_in;
    const int32_t *slot_mapping;
    int8_t *k_codes_w, *v_codes_w;
    uint16_t *k_scale_w, *v_scale_w;
};
int launch_int8_gather(const GatherArgs &a, void *stream);

int launch_store_kvcache_int8(const pa_dims &d, const void *k, const void *v, void *k_cache, void *v_cache,
                              void *k_scale, void *v_scale, const int32_t *slot_mapping, int32_t num_tokens,
                              void *stream);

struct PrefillArgs {
    pa_dims dims;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *cu_seqlens_q;
    const int32_t *cu_seqlens_k;
    const int32_t *block_tables;
    const int32_t *tiles;
    void *out;
    float scale;
    int32_t num_tiles;
    int32_t total_q;
    int32_t max_blocks_per_seq;
    int32_t rows_per_tile;
    // fused store (NULL otherwise): new tokens' K/V [total_q][Hkv][D] bf16 and their slots
    const void *k_in;
    const void *v_in;
    const int32_t *slot_mapping;
    // fused store with a cached prefix that does not end on a box boundary: fetch keys in
    // boxes of 16 rows, so that the box straddling the prefix end has few rows to patch
    bool small_boxes;
    // the cache is the INT8 prefill's scratch (block tables: the plan's scratch tables,
    // so the work entries' block of key 0 does not apply)
    bool scratch_cache;
};
int launch_prefill(const PrefillArgs &a, void *stream);

struct DecodeArgs {
    pa_dims dims;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const void *k_scale; // INT8 cache only: fp16 [num_blocks][num_kv_heads][block_size]
    const void *v_scale;
    const int32_t *context_lens;
    const int32_t *block_tables;
    const int32_t *items;
    const int32_t *seq_items;
    void *out;
    float *part_o;   // [num_partials][Hq][D]
    float *part_lse; // [num_partials][Hq]
    float scale;
    int32_t num_seqs;
    int32_t num_items;
    int32_t max_blocks_per_seq;
    int32_t max_splits;
    // fused store + decode only (else NULL): new K/V rows [num_seqs][Hkv][D] and their slots
    const void *k_new;
    const void *v_new;
    const int32_t *slot_mapping;
};
int launch_decode(const DecodeArgs &a, void *stream);
int launch_decode_int8(const DecodeArgs &a, void *stream);
// LSE merge of the split partials into out (no-op for plans without partials).
int launch_decode_combine(const DecodeArgs &a, void *stream);

// Device address of the library-owned decode scratch on the current device
// (looked up once per device).  Used only by pa_decode_static.
int decode_static_scratch(void **ptr);

// Concurrent decode CTAs one SM holds (occupancy of the decode kernel).
int decode_ctas_per_sm(int head_dim, int group);

// k_scale / v_scale NULL: bf16 cache; else INT8 codes plus fp16 scales [blocks][Hkv][bs].
int launch_copy_blocks(const pa_dims &d, void *k_cache, void *v_cache, const int32_t *triples, int32_t n,
                       void *stream, void *k_scale = nullptr, void *v_scale = nullptr);

// Read and clear the device error words (store: bit 0, prefill waits: bit 1,
// block copy: bit 2, INT8 decode waits: bit 3).
int read_store_error(uint32_t *code);
int read_prefill_error(uint32_t *code);
int read_copy_error(uint32_t *code);
int read_decode_error(uint32_t *code);
int read_fused_error(uint32_t *code);
int read_fused8_error(uint32_t *code);
int launch_selftest_wait(uint32_t timeout_us, int arrive_first, void *stream);
int read_selftest_error(uint32_t *code);
int launch_stream_read(const void *src, size_t bytes, uint32_t *sink, void *stream);

} // namespace pa
