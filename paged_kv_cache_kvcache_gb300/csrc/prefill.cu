// Causal variable-length prefill over the paged KV cache on tcgen05 tensor cores.
//
// Sources (page title, section):
//  - "手搓 vLLM 推理引擎" (LLM-101-CN nano-vllm walkthrough), Step 4:
//    packed varlen prefill with cu_seqlens_q/k; with prefix-cache hits K/V are
//    read from the paged cache through block_table and cu_seqlens_k exceeds
//    cu_seqlens_q.
//  - "推理系统" (CS 与 LLM 学习知识库), KV-cache toy: the new tokens sit at the
//    end of the sequence; new token i of T sees the first S - T + i + 1 keys.
//  - "vLLM / SGLang 面试源码深挖", section 2 (causal prefill is still
//    Theta(N^2)): tiles entirely above the causal diagonal are skipped,
//    boundary tiles are masked, online softmax merges tiles so the N x N scores
//    never reach HBM, and large tiles keep the tensor cores busy.
//  - "面试问答准备: nano-vLLM 推理引擎优化", Q1: the BLOCK_M = 1, no-tensor-core
//    kernel loses to tiled attention once prompts get long; the fix named
//    there is query tiling with an in-tile causal mask.
//
// GB300 design (persistent: one CTA per SM, 12 warps, each CTA walking its
// share of the work items; every ring and barrier phase runs on across items):
//  * A work item is (sequence, 2 query tiles, KV head).  Query tile rows
//    r = pos * G + h pack the G query heads that share a KV head next to each
//    other, so one K/V stream feeds all of them (GQA reuse); a 3-D TMA box
//    {64 d, G heads, P positions} loads each tile straight into the
//    128B-swizzled K-major layout tcgen05 reads.  The two tiles cover
//    consecutive positions and share every K/V tile the CTA loads.
//  * Keys in tiles of 128, gathered through the block table with one TMA box
//    per physical block (or one per tile when a block holds >= 128 tokens)
//    into a K/V ring; boxes past the end of the pool read as zeros and the V
//    rows past the sequence end are zeroed before use.
//  * warp 8: K TMA producer; warp 10: V producer; warp 11: Q producer (it
//    refills a query tile as soon as the item's last score MMA of that tile
//    has read it); warp 9: TMEM owner and the MMA issuer.  In the bf16 kernel
//    the whole warp runs the issue loop, converged, and an elected lane issues
//    each tcgen05.mma and commit: a 128 x 128 x 16 product runs 64 cycles, and a
//    lone lane in a divergent branch spends nearly as long issuing it, which
//    left no slack for the waits and commits between products.  Each query tile t owns 256
//    TMEM columns: S_t (128 fp32 columns, reused for P_t) and O_t.  The issue
//    order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) keeps the tensor core busy on
//    one tile while the other tile's softmax runs (ping-pong).  Because the
//    MMAs of one thread execute in order, S_t(j+1) being complete means
//    PV_t(j) is too: O_t is stable and P_t consumed when the softmax sees
//    S_t(j+1).  Across items the stream simply continues: the next item's first
//    score MMAs follow the last PVs, so they run while the softmax warps write
//    the previous item's output.
//  * warps 0-3 and 4-7: one softmax warpgroup per query tile, one query row
//    per thread: one tcgen05.ld round trip of the score row, which on tiles
//    that do not cross the causal diagonal also returns the row max
//    (tcgen05.ld.red, sm_103a); diagonal tiles are masked and reduced in
//    registers; fp32 online softmax in base 2
//    (scale * log2 e folded into one packed FMA), lazy O rescale (only when
//    the running max grows by more than 2^8), P written back over S with
//    tcgen05.st and consumed by the PV MMA straight from tensor memory;
//    epilogue (once the item's last PV is complete) O / l -> bf16 -> each
//    thread's own output row, straight from registers.
//  * Fused store (pa_prefill_varlen_fused, bf16): the K/V producers take the
//    new keys' boxes from the k/v inputs instead of the cache (so nothing
//    the launch writes is read by it), and warp 11, between its query loads,
//    copies the K/V rows of its item's query positions into their slots.  A
//    box that starts in the cached prefix and ends among the new keys (chunked
//    prefill resumes at any token count) is loaded from the cache and its new
//    keys' rows are then copied over it from the inputs by the producer before
//    the MMAs may read it.
//  * mbarriers order every hand-off; every wait is bounded and reports a
//    timeout through a device error word instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace pa {

__device__ uint32_t g_prefill_error; // bit 0: a bounded wait timed out; bit 1: the fused store met a bad slot

namespace {

// warps 0-7: softmax (two warpgroups), 8: K TMA producer, 9: MMA issuer (and
// TMEM owner), 10: V TMA producer, 11: Q TMA producer.  Registers are granted
// per 4 warps: 168 per thread at launch (65536 / 384 threads, rounded down to
// the allocation unit of 8); setmaxnreg then moves part of warps 8-11's share
// to the softmax warpgroups (216 per softmax thread, 72 in warps 8-11).
// One thread issues the MMAs of both query tiles: its in-order stream keeps the
// two tiles half a key tile apart, so one tile's softmax always runs under the
// other's MMAs.
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr int kKProducerWarp = 8, kMmaWarp = 9, kVProducerWarp = 10, kLoaderWarp = 11;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f; // log2 units
// Release events, numbered per CTA across its work items: an item with nkt key
// tiles owns nkt + 1 consecutive events, the first for its opening score MMAs
// (K tile 0 read), event first + j + 1 for MMA iteration j (V tile j and K tile
// j + 1 read).  A producer refilling a ring of S slots waits for the event that
// released the tile S places back; the MMA thread cannot pass the event that
// needs the tile being loaded, and between the two lie at most 2S - 1 events
// (one extra per item boundary), so 8 barriers keep every parity wait
// unambiguous for rings of up to 4 slots.
constexpr int kIterRing = 8;

template <int D>
struct PfLayout {
    static constexpr int kPanels = D / 64;          // 64-element (128-byte) panels along head_dim
    static constexpr int kPanelBytes = 128 * 128;   // 128 rows x 128 bytes
    static constexpr int kTileBytes = kPanels * kPanelBytes;
    // K is released as soon as the two score MMAs have read it, V only after
    // both PV MMAs: K gets the deeper ring so its loads start earliest.
    static constexpr int kKStages = D == 128 ? 3 : 4;
    static constexpr int kVStages = D == 128 ? 2 : 4;
    static constexpr int kQ = 0;                    // two query tiles
    static constexpr int kK = kQ + 2 * kTileBytes;
    static constexpr int kV = kK + kKStages * kTileBytes;
    static constexpr int kBar = kV + kVStages * kTileBytes;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBytes = kBar + kBarBytes + 1024; // + alignment slack
    static_assert(kKStages <= 4 && kVStages <= 4, "barrier slots");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct PfParams {
    int32_t num_items;     // entries of `tiles` (the CTAs walk them persistently)
    int32_t out_v8;        // out is 32-byte aligned: the epilogue stores 32 bytes per instruction
    const int32_t *cu_seqlens_q;
    const int32_t *cu_seqlens_k;
    const int32_t *block_tables;
    const int4 *tiles;
    __nv_bfloat16 *out;
    float scale_log2;
    int32_t num_heads;
    int32_t group;
    int32_t rows_per_tile; // query positions per query tile
    int32_t block_size;
    int32_t box_rows;      // rows per TMA box of a key tile: min(block size, 128), or 16 (see launch)
    int32_t max_blocks;
    int32_t num_slots;     // num_blocks * block_size: first out-of-range row (reads as zeros)
    int32_t num_kv_heads;
    // fused store: the new tokens' K/V rows are read from k_in/v_in (tensor maps
    // tm_kin/tm_vin) instead of the cache, and written into the cache at slot_mapping
    // (field order: the register allocation of the kernel is sensitive to it; this one
    // spills least)
    uint4 *k_cache;
    uint4 *v_cache;
    int32_t fused;
    const int32_t *slot_mapping;
    const uint4 *k_in;
    const uint4 *v_in;
};

// barrier slots (uint64 each) inside the barrier area
struct Bars {
    uint32_t base;
    __device__ uint32_t q_full(int t) const { return base + 8 * t; }
    // the item's last score MMA of query tile t is complete: its Q buffer may be refilled
    __device__ uint32_t q_free(int t) const { return base + 8 * (2 + t); }
    __device__ uint32_t k_full(int s) const { return base + 8 * (4 + s); }
    __device__ uint32_t v_full(int s) const { return base + 8 * (8 + s); }
    __device__ uint32_t released(int e) const { return base + 8 * (12 + (e & (kIterRing - 1))); }
    __device__ uint32_t s_full(int t) const { return base + 8 * (20 + t); }
    __device__ uint32_t p_full(int t) const { return base + 8 * (22 + t); }
    // the item's last PV MMA of query tile t is complete: O_t is final
    __device__ uint32_t o_full(int t) const { return base + 8 * (24 + t); }
    // V slot s holds an item's last key tile with its rows past the sequence end zeroed
    __device__ uint32_t v_tail(int s) const { return base + 8 * (26 + s); }
    __device__ uint32_t tmem_slot() const { return base + 8 * 30; }
    // fused store: K slot s holds the key tile whose straddling box (cached prefix, then
    // new keys) has had its new keys' rows copied in from the inputs
    __device__ uint32_t k_fix(int s) const { return base + 8 * (44 + s); }
};
static_assert(kIterRing == 8, "barrier slots 12..19");
constexpr int kTmemSlotOffset = 8 * 30;
constexpr int kAbortOffset = 8 * 31;

// One work item: (sequence, two query tiles of P positions, KV head) and the
// key tiles each query tile sees.
struct Item {
    int ord;                // position in this CTA's sequence of items
    int b, q0, g, cq0, lq, lk;
    int npos0, npos1;       // valid positions of query tiles 0 and 1 (tile 1 may be empty)
    int nkt0, nkt1, nkt;    // key tiles of each query tile; nkt = max
    bool tail;              // the last key tile runs past the sequence end
    int blk0;               // physical block holding key 0 (read by the short-batch kernel only)
};

// The items of this CTA: rounds of gridDim.x consecutive entries of the list
// (sorted longest first), odd rounds walked backwards so that the CTAs' totals
// stay even.  The next item's entry is fetched while the current one runs
// (from its start, or where the caller asks, to keep it out of a register-heavy loop).
struct ItemIter {
    const int4 *tiles;
    int n, P, ord, idx;
    int4 a0, a1;
    __device__ static int index(int ord)
    {
        const int c = (int)gridDim.x;
        return ord * c + ((ord & 1) ? c - 1 - (int)blockIdx.x : (int)blockIdx.x);
    }
    __device__ ItemIter(const int4 *t, int n_, int P_) : tiles(t), n(n_), P(P_), ord(0), idx(index(0))
    {
        if (idx < n) {
            a0 = __ldg(tiles + 2 * idx);
            a1 = __ldg(tiles + 2 * idx + 1);
        }
    }
    __device__ bool more() const { return idx < n; }
    __device__ Item decode(int o) const
    {
        Item w;
        w.ord = o;
        w.b = a0.x, w.q0 = a0.y, w.g = a0.z;
        w.cq0 = a1.x, w.lq = a1.y, w.lk = a1.z, w.blk0 = a1.w;
        const int off = w.lk - w.lq; // absolute position of query row 0
        w.npos0 = min(P, w.lq - w.q0);
        w.npos1 = max(0, min(P, w.lq - w.q0 - P));
        w.nkt0 = (off + w.q0 + w.npos0 + 127) >> 7;
        w.nkt1 = w.npos1 > 0 ? (off + w.q0 + P + w.npos1 + 127) >> 7 : 0;
        w.nkt = max(w.nkt0, w.nkt1);
        w.tail = w.nkt * 128 > w.lk;
        return w;
    }
    // the current item; advances to the next and (unless told not to) starts fetching its entry
    __device__ Item next(bool fetch_now = true)
    {
        const Item w = decode(ord);
        idx = index(++ord);
        if (fetch_now)
            fetch();
        return w;
    }
    // issued where it stands, so that its latency hides behind the current item
    __device__ void fetch()
    {
        if (idx < n) {
            a0 = ptx::ld_nc_v4_now(tiles + 2 * idx);
            a1 = ptx::ld_nc_v4_now(tiles + 2 * idx + 1);
        }
    }
    // the item next() returns next (valid while more())
    __device__ Item peek() const { return decode(ord); }
};

// Fused store: the key tile of item w holding a box that starts in the cached prefix
// and ends among the new keys (the prefix length is not a multiple of the box), or -1.
// That box is loaded from the cache like the rest of the prefix; the producer then
// copies the new keys' rows over it from the k/v inputs, since the launch is writing
// those cache rows itself.
__device__ __forceinline__ int straddle_tile(const Item &w, int fused, int box_rows)
{
    const int off = w.lk - w.lq; // cached prefix
    return fused && w.lq > 0 && (off & (box_rows - 1)) != 0 ? off >> 7 : -1;
}

// Rows [off, min(box end, lk)) of the straddling box of key tile j: the new keys, copied
// from the inputs (16-byte vectors, one warp) into their 128B-swizzled places in the tile.
template <int D>
__device__ __forceinline__ void patch_new_keys(uint8_t *tile, const uint4 *in, const Item &w, int j, int box_rows,
                                               int num_kv_heads, int lane)
{
    constexpr int VPR = D / 8; // 16-byte vectors per row
    constexpr int kU = 4;      // vectors in flight per lane
    const int off = w.lk - w.lq;
    const int end = min(off - (off & (box_rows - 1)) + box_rows, w.lk);
    const int total = (end - off) * VPR;
    for (int i0 = lane; i0 < total; i0 += 32 * kU) {
        uint4 x[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = i0 + 32 * u;
            if (i < total)
                x[u] = __ldg(in + ((size_t)(w.cq0 + i / VPR) * num_kv_heads + w.g) * VPR + i % VPR);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = i0 + 32 * u;
            if (i < total) {
                const int rr = off + i / VPR - j * 128;  // row in the tile
                const int c16 = i % VPR;
                const int panel = c16 >> 3, c = c16 & 7; // 64-element panel, 16-byte chunk in its row
                *reinterpret_cast<uint4 *>(tile + panel * (128 * 128) + rr * 128 + ((c ^ (rr & 7)) << 4)) = x[u];
            }
        }
    }
}

// Release event of the key tile `back` places before global tile X (X >= back),
// given the current item's ordinal and the item-start bits of the last tiles
// (bit i: tile X - i opens its item).  K tile j of item i is released by event
// (its global index) + i, V tile j one event later.
__device__ __forceinline__ int release_event(int X, int back, int ord, uint32_t starts, int v)
{
    return X - back + ord - __popc(starts & ((1u << back) - 1u)) + v;
}

struct Waiter {
    volatile uint32_t *abort;
    __device__ bool operator()(uint32_t bar, uint32_t parity) const
    {
        if (ptx::mbar_try_wait(bar, parity)) // fast path: phase already complete
            return true;
        if (*abort)
            return false;
        if (ptx::mbar_wait(bar, parity))
            return true;
        *abort = 1u;
        atomicOr(&g_prefill_error, 1u);
        return false;
    }
};

// Fused store: the new K/V rows of item w's query positions, KV head w.g, copied
// from the inputs to their cache slots (one warp; each (token, KV head) row belongs
// to exactly one item): the positions first, first + step, ...  Warp 11 copies each
// item's rows in passes while it waits to load the next item's query tiles; the rows
// of a CTA's last item are split three ways with the K and V producers, which have
// nothing left to load by then.  The kernel itself reads the new keys from the
// inputs, so nothing here is waited for.

template <int D>
__device__ __forceinline__ int store_vectors(const Item &w, int first, int step)
{
    return (w.npos0 + w.npos1 - first + step - 1) / step * (D / 8);
}

// One pass: the warp's 32 * kU vectors from vector i0 - lane on, of `total` (16 bytes of K
// and of V each, kU of each in flight per lane; vector i is 16-byte piece i % (D / 8) of KV
// head g of packed token row0 + (i / (D / 8)) * step).
template <int D, int kU>
__device__ __forceinline__ void store_rows_pass(const PfParams &p, int row0, int g, int total, int i0, int step)
{
    constexpr int VPR = D / 8; // 16-byte vectors per row of one head
    const size_t hkv = (size_t)p.num_kv_heads;
    uint4 kx[kU], vx[kU];
    int slot[kU]; // -1: nothing to store
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int i = i0 + 32 * u;
        slot[u] = -1;
        if (i < total) {
            const int row = row0 + (i / VPR) * step;
            const int s = __ldg(p.slot_mapping + row);
            const size_t from = ((size_t)row * hkv + g) * VPR + i % VPR;
            kx[u] = __ldg(p.k_in + from);
            vx[u] = __ldg(p.v_in + from);
            if (s >= 0 && s < p.num_slots)
                slot[u] = s;
            else if (s != -1)
                atomicOr(&g_prefill_error, 2u);
        }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
        if (slot[u] >= 0) {
            const size_t to = ((size_t)slot[u] * hkv + g) * VPR + (i0 + 32 * u) % VPR;
            p.k_cache[to] = kx[u];
            p.v_cache[to] = vx[u];
        }
}

// All new K/V rows of item w copied by the 256 threads of the softmax warpgroups (thread
// tid: vectors tid, tid + 256, ...; 8 of K and 8 of V in flight per thread, slots checked as
// in store_rows_pass).
template <int D>
__device__ __forceinline__ void store_item_rows_wide(const PfParams &p, const Item &w, int tid)
{
    constexpr int VPR = D / 8, kU = 8, kThreadsW = 256;
    const size_t hkv = (size_t)p.num_kv_heads;
    const int total = store_vectors<D>(w, 0, 1);
    for (int i0 = tid; i0 < total; i0 += kThreadsW * kU) {
        uint4 kx[kU], vx[kU];
        int slot[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = i0 + kThreadsW * u;
            slot[u] = -1;
            if (i < total) {
                const int row = w.cq0 + w.q0 + i / VPR;
                const int s = __ldg(p.slot_mapping + row);
                const size_t from = ((size_t)row * hkv + w.g) * VPR + i % VPR;
                kx[u] = __ldg(p.k_in + from);
                vx[u] = __ldg(p.v_in + from);
                if (s >= 0 && s < p.num_slots)
                    slot[u] = s;
                else if (s != -1)
                    atomicOr(&g_prefill_error, 2u);
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (slot[u] >= 0) {
                const size_t to = ((size_t)slot[u] * hkv + w.g) * VPR + (i0 + kThreadsW * u) % VPR;
                p.k_cache[to] = kx[u];
                p.v_cache[to] = vx[u];
            }
    }
}

// a `first` past every item's positions: the call copies nothing
constexpr int kNoRows = 1 << 20;

// Short kernel, fused store: an item of at least 128 positions has its rows copied by the
// softmax warps at its start (measured: 8 x 128 prompts 10.7 -> 9.8 us per launch); a
// smaller one by the three loader warps as in the other kernel (8 x 32: 6.7 against 7.0).
template <int D>
__device__ __forceinline__ bool wide_copy(const Item &w)
{
    return store_vectors<D>(w, 0, 1) >= 128 * (D / 8);
}

template <int D>
__device__ __forceinline__ void store_item_rows(const PfParams &p, const Item &w, int lane, int first = 0,
                                                int step = 1)
{
    constexpr int kU = 2;
    const int total = store_vectors<D>(w, first, step);
    for (int i0 = lane; i0 < total; i0 += 32 * kU)
        store_rows_pass<D, kU>(p, w.cq0 + w.q0 + first, w.g, total, i0, step);
}

// Rows G*P..127 of each query tile receive no TMA data: zero them once so their
// (discarded) scores stay finite and cost the same as real rows.
template <int D>
__device__ __forceinline__ void zero_query_padding(uint8_t *sgen, int first, int lane)
{
    using L = PfLayout<D>;
    if (first >= 128)
        return;
    const int chunks = (128 - first) * 8;
    for (int t = 0; t < 2; ++t)
        for (int pp = 0; pp < L::kPanels; ++pp)
            for (int c = lane; c < chunks; c += 32)
                *reinterpret_cast<uint4 *>(sgen + L::kQ + t * L::kTileBytes + pp * L::kPanelBytes +
                                           (first + (c >> 3)) * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
    __syncwarp();
}

// Query tile t of item w: one 3-D box {64 d, G heads, P positions} per panel.
// Always issued, also for an empty tile 1 (its rows are never used).
template <int D>
__device__ __forceinline__ void load_query_tile(const CUtensorMap *tm_q, const Bars &bars, uint32_t sbase,
                                                const Item &w, int t, int G, int P)
{
    using L = PfLayout<D>;
    ptx::mbar_arrive_expect_tx(bars.q_full(t), (uint32_t)(L::kPanels * 128 * G * P));
    for (int pp = 0; pp < L::kPanels; ++pp)
        ptx::tma_load_3d(sbase + L::kQ + t * L::kTileBytes + pp * L::kPanelBytes, tm_q, bars.q_full(t), pp * 64,
                         w.g * G, w.cq0 + w.q0 + t * P);
}

// The next item's query tiles into L2, so that their loads (which must wait for
// the current item's last score MMAs) arrive sooner.
template <int D>
__device__ __forceinline__ void prefetch_query_tiles(const CUtensorMap *tm_q, const Item &w, int G, int P)
{
    using L = PfLayout<D>;
    for (int t = 0; t < 2; ++t)
        for (int pp = 0; pp < L::kPanels; ++pp)
            ptx::tma_prefetch_3d(tm_q, pp * 64, w.g * G, w.cq0 + w.q0 + t * P);
}

// kShort: the instantiation for batches of at most one work item per CTA (short
// prompts, where each item's start-up latency is the launch's time): its loaders
// fetch their tensor maps and the first work entry while the barriers are set up,
// and the first key box comes from the block named in the work entry (so not used
// over the INT8 prefill's scratch cache, whose blocks the entries do not name).  The large
// batches keep the other instantiation, whose register allocation those additions
// would disturb (measured 1.5-2 % slower there).
template <int D, bool kShort>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kin,
                   const __grid_constant__ CUtensorMap tm_vin, const PfParams p)
{
    using L = PfLayout<D>;
    // per-thread register budgets after the hand-over
    constexpr int kSoftmaxRegs = 216, kOtherRegs = 72;
    static_assert(128 * (2 * kSoftmaxRegs + kOtherRegs) == kThreads * kLaunchRegs, "register hand-over");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *sgen = smem_raw + (sbase - raw); // generic pointer to the aligned base

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Bars bars{sbase + L::kBar};
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sgen + L::kBar + kAbortOffset);
    const Waiter wait{abort_flag};
    const int G = p.group;
    const int P = p.rows_per_tile;

    if constexpr (kShort) {
        if (warp >= 8 && lane == 0) {
            if (warp == kLoaderWarp) {
                ptx::prefetch_tmap(&tm_q);
                ptx::prefetch_l1(p.tiles + 2 * ItemIter::index(0));
            } else if (warp == kKProducerWarp) {
                ptx::prefetch_tmap(&tm_k);
                if (p.fused)
                    ptx::prefetch_tmap(&tm_kin);
            } else if (warp == kVProducerWarp) {
                ptx::prefetch_tmap(&tm_v);
                if (p.fused)
                    ptx::prefetch_tmap(&tm_vin);
            }
        }
    }

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bars.q_full(t), 1);
            ptx::mbar_init(bars.q_free(t), 1);
            ptx::mbar_init(bars.s_full(t), 1);
            ptx::mbar_init(bars.p_full(t), 4); // one arrival per softmax warp
            ptx::mbar_init(bars.o_full(t), 1);
        }
        for (int s = 0; s < L::kKStages; ++s) {
            ptx::mbar_init(bars.k_full(s), 1);
            ptx::mbar_init(bars.k_fix(s), 1);
        }
        for (int s = 0; s < L::kVStages; ++s) {
            ptx::mbar_init(bars.v_full(s), 1);
            ptx::mbar_init(bars.v_tail(s), 1);
        }
        for (int s = 0; s < kIterRing; ++s)
            ptx::mbar_init(bars.released(s), 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(bars.tmem_slot(), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + L::kBar + kTmemSlotOffset);
    auto wwait = [&](uint32_t bar, uint32_t parity) { return __all_sync(0xffffffffu, wait(bar, parity)); };

    if (warp >= 8) {
        // warps 8-11 (copies, MMA issue) need fewer registers and hand part of theirs
        // to the softmax warpgroups (128 x (2 kSoftmaxRegs + kOtherRegs) = the launch's
        // registers)
        ptx::reg_dealloc<kOtherRegs>();
        const int bs = p.block_size;
        const int box_rows = p.box_rows;
        const int nsub = 128 / box_rows;
        // row coordinate of sub-box `lane` of key tile j of item w (one TMA box per lane):
        // a cache row, or -(r + 1) for row r of the new keys' input (fused store); a box that
        // starts in the cached prefix comes from the cache (its new rows are patched in later)
        auto sub_row = [&](const Item &w, const int32_t *bt, int j) -> int {
            const int key = j * 128 + lane * box_rows;
            if (lane >= nsub || key >= w.lk)
                return p.num_slots; // fully out of range: TMA fills zeros
            const int off = w.lk - w.lq; // cached prefix
            if (p.fused && key >= off)
                return -(w.cq0 + key - off + 1);
            const int phys = kShort && key < bs ? w.blk0 : __ldg(bt + key / bs);
            return phys * bs + (key & (bs - 1));
        };
        if (warp == kLoaderWarp) {
            // ------------------------------------------------------------ bf16: Q producer
            ItemIter items(p.tiles, p.num_items, P);
            zero_query_padding<D>(sgen, G * P, lane);
            if (!kShort && lane == 0)
                ptx::prefetch_tmap(&tm_q);
            bool ok = true;
            uint32_t early = 0; // bit t: query tile t of the current item was loaded during the previous item's copy
            while (ok && items.more()) {
                const Item w = items.next();
                for (int t = 0; t < 2; ++t) {
                    if (early >> t & 1u)
                        continue;
                    // refill after the previous item's last score MMA of this tile
                    if (w.ord > 0 && !(ok = wwait(bars.q_free(t), (w.ord - 1) & 1)))
                        break;
                    if (lane == 0)
                        load_query_tile<D>(&tm_q, bars, sbase, w, t, G, P);
                    __syncwarp();
                }
                early = 0;
                if (ok && lane == 0 && items.more())
                    prefetch_query_tiles<D>(&tm_q, items.peek(), G, P);
                if (ok && p.fused) {
                    if (items.more()) {
                        // this item's rows, pass by pass; a query buffer that frees meanwhile is
                        // refilled with the next item's tile at once
                        constexpr int kU = 2;
                        const int total = store_vectors<D>(w, 0, 1);
                        for (int i0 = lane; __any_sync(0xffffffffu, i0 < total); i0 += 32 * kU) {
                            store_rows_pass<D, kU>(p, w.cq0 + w.q0, w.g, total, i0, 1);
                            for (int t = 0; t < 2; ++t)
                                if (!(early >> t & 1u) && (t == 0 || early) &&
                                    __shfl_sync(0xffffffffu, (int)ptx::mbar_test_wait(bars.q_free(t), w.ord & 1), 0)) {
                                    if (lane == 0)
                                        load_query_tile<D>(&tm_q, bars, sbase, items.peek(), t, G, P);
                                    __syncwarp();
                                    early |= 1u << t;
                                }
                        }
                    } else { // the CTA's last item: a third of its rows (the producers copy the rest;
                             // the short kernel's softmax warps copy all of them: no row here)
                        store_item_rows<D>(p, w, lane, kShort && wide_copy<D>(w) ? kNoRows : 0, 3);
                    }
                }
            }
        } else if (warp == kKProducerWarp || warp == kVProducerWarp) {
            // ------------------------------------------------------------ bf16: K and V producers
            ItemIter items(p.tiles, p.num_items, P);
            const bool is_k = warp == kKProducerWarp;
            const int nstages = is_k ? L::kKStages : L::kVStages;
            const uint32_t ring = sbase + (is_k ? L::kK : L::kV);
            const CUtensorMap *tm = is_k ? &tm_k : &tm_v;
            const CUtensorMap *tm_in = is_k ? &tm_kin : &tm_vin;
            if (!kShort && lane == 0) {
                ptx::prefetch_tmap(tm);
                if (p.fused)
                    ptx::prefetch_tmap(tm_in);
            }
            uint32_t starts = 0; // bit i: global key tile X - i opens its item
            int X = 0;           // global key tile (this CTA, all items)
            bool ok = true;
            while (ok && items.more()) {
                const Item w = items.next();
                const int jfix = straddle_tile(w, p.fused, box_rows);
                const int32_t *bt = p.block_tables + (size_t)w.b * p.max_blocks;
                int next = sub_row(w, bt, 0);
                for (int j = 0; j < w.nkt; ++j, ++X) {
                    const int cur = next;
                    if (j + 1 < w.nkt)
                        next = sub_row(w, bt, j + 1);
                    starts = (starts << 1) | (j == 0 ? 1u : 0u);
                    const int st = X % nstages;
                    // slot reuse: free once the tile nstages back is released
                    if (X >= nstages) {
                        const int e = release_event(X, nstages, w.ord, starts, is_k ? 0 : 1);
                        if (!(ok = wwait(bars.released(e), (e / kIterRing) & 1)))
                            break;
                    }
                    const uint32_t full = is_k ? bars.k_full(st) : bars.v_full(st);
                    const uint32_t dst = ring + st * L::kTileBytes;
                    if (lane == 0)
                        ptx::mbar_arrive_expect_tx(full, (uint32_t)L::kTileBytes);
                    // lane i issues the boxes of sub-box i (its own row coordinate and source)
                    if (lane < nsub) {
                        const CUtensorMap *src = cur < 0 ? tm_in : tm;
                        const int row = cur < 0 ? -cur - 1 : cur;
                        for (int pp = 0; pp < L::kPanels; ++pp)
                            ptx::tma_load_3d(dst + pp * L::kPanelBytes + lane * box_rows * 128, src, full, pp * 64,
                                             w.g, row);
                    }
                    __syncwarp();
                    const bool fix = j == jfix, zero = !is_k && w.tail && j == w.nkt - 1;
                    if (fix || zero) {
                        if (!(ok = wwait(full, (X / nstages) & 1)))
                            break;
                        uint8_t *tile = sgen + (is_k ? L::kK : L::kV) + st * L::kTileBytes;
                        if (fix) // the straddling box's new keys, from the inputs
                            patch_new_keys<D>(tile, is_k ? p.k_in : p.v_in, w, j, box_rows, p.num_kv_heads, lane);
                        if (zero) {
                            // V rows of keys past the sequence end may hold anything (even NaN
                            // bit patterns); zero them so that P = 0 cannot turn them into NaN in O.
                            const int first = w.lk - j * 128;
                            const int chunks = (128 - first) * 8;
                            for (int pp = 0; pp < L::kPanels; ++pp)
                                for (int c = lane; c < chunks; c += 32)
                                    *reinterpret_cast<uint4 *>(tile + pp * L::kPanelBytes + (first + (c >> 3)) * 128 +
                                                               (c & 7) * 16) = make_uint4(0, 0, 0, 0);
                        }
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0)
                            ptx::mbar_arrive(is_k ? bars.k_fix(st) : bars.v_tail(st));
                    }
                }
            }
            // fused store: this producer's third of the rows of the CTA's last item (its work
            // entry is still the iterator's last one)
            if (ok && p.fused && items.ord > 0) {
                const Item last = items.decode(items.ord - 1);
                store_item_rows<D>(p, last, lane, kShort && wide_copy<D>(last) ? kNoRows : (is_k ? 1 : 2), 3);
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------ MMA issuer (the whole warp,
            // one elected lane issuing each MMA and commit)

            ItemIter items(p.tiles, p.num_items, P);
            constexpr uint32_t idesc_s = ptx::idesc_bf16(128, 128, 0);
            constexpr uint32_t idesc_o = ptx::idesc_bf16(128, D, 1);
            // Shared-memory descriptors: a constant upper word and a lower word of base
            // address + the k step's offset.  The base passes through an empty asm so that
            // it is rebuilt at each use instead of hoisting all 16 k-step descriptors into
            // registers (this warpgroup runs on few).
            const uint32_t hi_k = (uint32_t)(ptx::smem_desc(0, 16, 1024, ptx::kSwizzle128B) >> 32);
            const uint32_t hi_v = (uint32_t)(ptx::smem_desc(0, L::kPanelBytes, 1024, ptx::kSwizzle128B) >> 32);
            auto desc = [](uint32_t lo, uint32_t hi) { return ((uint64_t)hi << 32) | lo; };
            auto issue_s = [&](int t, int ks) {
                uint32_t qa = (uint32_t)ptx::smem_desc(sbase + L::kQ + t * L::kTileBytes, 16, 1024, ptx::kSwizzle128B);
                uint32_t kb = (uint32_t)ptx::smem_desc(sbase + L::kK + ks * L::kTileBytes, 16, 1024, ptx::kSwizzle128B);
                asm volatile("" : "+r"(qa), "+r"(kb));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = ((kk >> 2) * L::kPanelBytes + (kk & 3) * 32) >> 4;
                    ptx::mma_bf16_ss_warp(tmem + t * 256, desc(qa + o, hi_k), desc(kb + o, hi_k), idesc_s, kk > 0);
                }
            };
            auto issue_pv = [&](int t, int vs, bool first) {
                uint32_t vb = (uint32_t)ptx::smem_desc(sbase + L::kV + vs * L::kTileBytes, L::kPanelBytes, 1024,
                                                       ptx::kSwizzle128B);
                asm volatile("" : "+r"(vb));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_bf16_ts_warp(tmem + t * 256 + 128, tmem + t * 256 + kk * 8, desc(vb + kk * (2048 >> 4), hi_v),
                                     idesc_o, (!first || kk > 0) ? 1u : 0u);
            };
            // ring positions kept as counters (no division in the issue loop)
            int ks = 0, kph = 0, vs = 0, vph = 0;
            uint32_t np = 0;       // bit t: parity of the P tiles of query tile t consumed so far
            uint32_t tailpar = 0;  // bit s: parity of the tail (or patched) tiles V slot s has held
            uint32_t fixpar = 0;   // bit s: parity of the patched tiles K slot s has held
            int E = 0;             // first release event of the current item
            bool ok = true;
            while (ok && items.more()) {
                const Item w = items.next();
                const uint32_t qpar = w.ord & 1;
                const int jfix = straddle_tile(w, p.fused, box_rows);
                ok = wwait(bars.q_full(0), qpar) && wwait(bars.k_full(ks), kph);
                if (ok && jfix == 0) { // key tile 0's straddling box patched
                    ok = wwait(bars.k_fix(ks), (fixpar >> ks) & 1u);
                    fixpar ^= 1u << ks;
                }
                if (!ok)
                    break;
                ptx::tc_fence_after();
                issue_s(0, ks);
                ptx::mma_commit_warp(bars.s_full(0));
                // query tile 1 is waited for only now (also when empty: its buffer is
                // released below, and every load of it must be consumed first)
                if (!(ok = wwait(bars.q_full(1), qpar)))
                    break;
                if (w.nkt1 > 0) {
                    ptx::tc_fence_after();
                    issue_s(1, ks);
                    ptx::mma_commit_warp(bars.s_full(1));
                }
                ptx::mma_commit_warp(bars.released(E)); // K tile 0 read by both score MMAs
                if (w.nkt0 == 1)
                    ptx::mma_commit_warp(bars.q_free(0));
                if (w.nkt1 <= 1)
                    ptx::mma_commit_warp(bars.q_free(1));
                if (++ks == L::kKStages) {
                    ks = 0;
                    kph ^= 1;
                }
                for (int j = 0; ok && j < w.nkt; ++j) {
                    bool v_ready = false, k_next = false;
                    // one query tile: PV(t, j), then S(t, j + 1) into the same TMEM columns
                    auto step = [&](const int t, const int ntk) {
                        if (!(ok = wwait(bars.p_full(t), (np >> t) & 1u)))
                            return;
                        np ^= 1u << t;
                        if (!v_ready) {
                            if (!(ok = wwait(bars.v_full(vs), vph)))
                                return;
                            if ((w.tail && j == w.nkt - 1) || j == jfix) {
                                if (!(ok = wwait(bars.v_tail(vs), (tailpar >> vs) & 1u)))
                                    return;
                                tailpar ^= 1u << vs;
                            }
                            v_ready = true;
                        }
                        ptx::tc_fence_after();
                        issue_pv(t, vs, j == 0);
                        if (j + 1 == ntk)
                            ptx::mma_commit_warp(bars.o_full(t)); // O_t final
                        if (j + 1 < ntk) {
                            if (!k_next) {
                                if (!(ok = wwait(bars.k_full(ks), kph)))
                                    return;
                                if (j + 1 == jfix) { // that key tile's straddling box patched
                                    if (!(ok = wwait(bars.k_fix(ks), (fixpar >> ks) & 1u)))
                                        return;
                                    fixpar ^= 1u << ks;
                                }
                                ptx::tc_fence_after();
                                k_next = true;
                            }
                            issue_s(t, ks);
                            ptx::mma_commit_warp(bars.s_full(t));
                            if (j + 2 == ntk)
                                ptx::mma_commit_warp(bars.q_free(t)); // that was the last read of Q_t
                        }
                    };
                    if (j < w.nkt0)
                        step(0, w.nkt0);
                    if (ok && j < w.nkt1)
                        step(1, w.nkt1);
                    if (!ok)
                        break;
                    ptx::mma_commit_warp(bars.released(E + j + 1)); // V tile j and K tile j + 1 read
                    if (++vs == L::kVStages) {
                        vs = 0;
                        vph ^= 1;
                    }
                    if (k_next && ++ks == L::kKStages) {
                        ks = 0;
                        kph ^= 1;
                    }
                }
                E += w.nkt + 1;
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- softmax + epilogue
        ItemIter items(p.tiles, p.num_items, P);
        ptx::reg_alloc<kSoftmaxRegs>();
        const int t = warp >> 2;                   // query tile of this warpgroup (warps 0-3, 4-7)
        const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
        const int r = quarter * 32 + lane;         // query row of the tile
        const int rpos = r / G, rhead = r % G;     // its position in the tile and head in the group
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const uint32_t s_col = tmem + lane_addr + t * 256;
        const uint32_t o_col = s_col + 128;
        const float sl2 = p.scale_log2;
        uint32_t ns = 0, no = 0; // S tiles and items of this query tile so far (parities)
        bool ok = true;
        if constexpr (kShort) {
            // fused store, one item per CTA: the eight softmax warps copy its new K/V rows
            // while they wait for its first scores (one pass of 8 K and 8 V vectors per
            // thread covers 64 KB of rows), if it has at least 128 positions
            if (p.fused && items.more() && wide_copy<D>(items.peek()))
                store_item_rows_wide<D>(p, items.peek(), (int)threadIdx.x);
        }

        while (ok && items.more()) {
            const Item w = items.next(false);
            const int ntile = t == 0 ? w.nkt0 : w.nkt1;
            const int npos = t == 0 ? w.npos0 : w.npos1;
            const bool row_valid = r < G * npos;
            // keys visible to this row; rows that hold no query are never masked (their
            // output is discarded) so that a warp's rows all take the same path
            const int limit = row_valid ? w.lk - w.lq + w.q0 + t * P + rpos + 1 : 0x3fffffff;
            float m_ref = -INFINITY, l_sum = 0.f;
            for (int j = 0; j < ntile; ++j) {
                if (!(ok = wwait(bars.s_full(t), ns & 1)))
                    break;
                ns ^= 1;
                ptx::tc_fence_after();
                const int lim = limit - j * 128; // columns this row sees in this tile
                // the whole score row in registers: one TMEM round trip per tile.  Tiles no row
                // of the warp sees only in part take the row max from the loads themselves
                // (tcgen05.ld.red); tiles crossing the causal diagonal mask first, then reduce.
                uint32_t sr[128];
                float mx;
                if (__any_sync(0xffffffffu, lim < 128)) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        ptx::tmem_ld32(s_col + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * q]));
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        sr[c] = c < lim ? sr[c] : __float_as_uint(-INFINITY);
                    float m8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        m8[i] = ptx::max3(__uint_as_float(sr[16 * i]), __uint_as_float(sr[16 * i + 1]),
                                          __uint_as_float(sr[16 * i + 2]));
#pragma unroll
                    for (int c = 3; c < 16; c += 2)
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            m8[i] = c + 1 < 16 ? ptx::max3(m8[i], __uint_as_float(sr[16 * i + c]),
                                                           __uint_as_float(sr[16 * i + c + 1]))
                                               : fmaxf(m8[i], __uint_as_float(sr[16 * i + c]));
                    mx = fmaxf(fmaxf(ptx::max3(m8[0], m8[1], m8[2]), ptx::max3(m8[3], m8[4], m8[5])),
                               fmaxf(m8[6], m8[7]));
                } else {
                    float m4[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        m4[q] = ptx::tmem_ld32_max(s_col + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * q]));
                    ptx::tmem_wait_ld();
                    mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                }
                const float mt = mx * sl2;
                float alpha = 1.f;
                bool rescale = false;
                if (row_valid && (mt > m_ref + kRescaleThreshold || (m_ref == -INFINITY && mt != -INFINITY))) {
                    const float m_new = fmaxf(m_ref, mt);
                    alpha = ptx::ex2(m_ref - m_new); // 0 on the first tile
                    rescale = j > 0;
                    l_sum *= alpha;
                    m_ref = m_new;
                }
                // P = 2^(s * scale * log2 e - m) as bf16 pairs written over S; row sum
                const uint64_t sl2x2 = ptx::f2(sl2, sl2);
                const float negm = m_ref == -INFINITY ? 0.f : -m_ref;
                const uint64_t negm2 = ptx::f2(negm, negm);
                uint64_t sum2[4] = {ptx::f2(0.f, 0.f), ptx::f2(0.f, 0.f), ptx::f2(0.f, 0.f), ptx::f2(0.f, 0.f)};
#pragma unroll
                for (int h = 0; h < 2; ++h) { // two halves: P columns 32h..32h+31 hold keys 64h..64h+63
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 64 * h; c < 64 * h + 64; c += 2) {
                        float x0, x1;
                        ptx::f2_split(
                            ptx::f2_fma(ptx::f2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2, negm2), x0, x1);
                        const float e0 = ptx::ex2(x0), e1 = ptx::ex2(x1); // masked columns: 2^-inf = 0
                        sum2[(c >> 1) & 3] = ptx::f2_add(sum2[(c >> 1) & 3], ptx::f2(e0, e1));
                        pk[(c >> 1) & 31] = ptx::pack_bf16(e0, e1);
                    }
                    ptx::tmem_st32(s_col + 32 * h, pk);
                }
                float s0, s1, s2, s3, s4, s5, s6, s7;
                ptx::f2_split(sum2[0], s0, s1);
                ptx::f2_split(sum2[1], s2, s3);
                ptx::f2_split(sum2[2], s4, s5);
                ptx::f2_split(sum2[3], s6, s7);
                l_sum += ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
                // O is stable here: PV(j-1) completed before S(j) did (in-order MMAs), and
                // PV(j) waits for this thread's p_full arrival below
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        ptx::tmem_ld32(o_col + cc * 32, o);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        ptx::tmem_st32(o_col + cc * 32, o);
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp(); // 128 arrivals on one word serialise: one per warp instead
                if (lane == 0)
                    ptx::mbar_arrive(bars.p_full(t));
            }
            items.fetch();
            if (!ok || ntile == 0)
                continue;
            // epilogue: O / l -> bf16 -> this row's output, straight from registers.  The
            // MMAs meanwhile run the next item's score tiles; the next item's first PV
            // (which overwrites O_t) waits for this warpgroup's next P, issued after these reads.
            if (!(ok = wwait(bars.o_full(t), no & 1)))
                break;
            no ^= 1;
            ptx::tc_fence_after();
            const float inv = (row_valid && l_sum > 0.f) ? 1.f / l_sum : 0.f;
            __nv_bfloat16 *orow =
                p.out + ((size_t)(w.cq0 + w.q0 + t * P + rpos) * p.num_heads + (size_t)w.g * G + rhead) * D;
            // TMEM loads in batches of kBatch 32-column chunks, one wait per batch
            // (bf16: the whole row at once; the register budget allows it)
            constexpr int kBatch = D / 32;
#pragma unroll
            for (int c0 = 0; c0 < D / 32; c0 += kBatch) {
                uint32_t o[kBatch][32];
#pragma unroll
                for (int cc = 0; cc < kBatch; ++cc)
                    ptx::tmem_ld32(o_col + (c0 + cc) * 32, o[cc]);
                ptx::tmem_wait_ld();
                if (row_valid && !*abort_flag) {
#pragma unroll
                    for (int cc = 0; cc < kBatch; ++cc)
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const uint32_t *x = o[cc] + 16 * c;
                            uint32_t w[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                w[i] = ptx::pack_bf16(__uint_as_float(x[2 * i]) * inv, __uint_as_float(x[2 * i + 1]) * inv);
                            __nv_bfloat16 *dst = orow + (c0 + cc) * 32 + c * 16;
                            // 32-byte stores when out allows (rows are 128 or 256 bytes, so each
                            // row keeps the base's alignment): each thread writes whole sectors,
                            // half the store instructions in the memory pipeline the MMA
                            // thread's barrier polls share
                            if (p.out_v8) {
                                ptx::st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                            } else {
                                reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                                reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                            }
                        }
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool kShort>
int launch(const PrefillArgs &a, cudaStream_t stream, int sms)
{
    using L = PfLayout<D>;
    if (int rc = ensure_smem<prefill_kernel<D, kShort>>(L::kSmemBytes, "prefill"))
        return rc;
    // The register hand-over inside the kernel assumes kLaunchRegs per thread at
    // launch; with fewer the softmax warpgroups' request could never be granted.
    static std::atomic<int> launch_regs{0};
    int nreg = launch_regs.load(std::memory_order_acquire);
    if (nreg == 0) {
        cudaFuncAttributes fa{};
        const cudaError_t e = cudaFuncGetAttributes(&fa, prefill_kernel<D, kShort>);
        if (e != cudaSuccess)
            return fail(PA_ERR_CUDA, "prefill kernel attributes: %s", cudaGetErrorString(e));
        launch_regs.store(nreg = fa.numRegs, std::memory_order_release);
    }
    if (nreg != kLaunchRegs)
        return fail(PA_ERR_UNSUPPORTED, "prefill kernel built with %d registers per thread, needs %d", nreg,
                    kLaunchRegs);
    const pa_dims &d = a.dims;
    const int G = d.num_heads / d.num_kv_heads;
    const uint64_t rows = (uint64_t)d.num_blocks * d.block_size;
    CUtensorMap tq, tk, tv;
    int rc;
    constexpr CUtensorMapDataType bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    constexpr CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if ((rc = encode_tmap_3d(&tq, bf16, a.q, D, d.num_heads, (uint64_t)a.total_q, (uint64_t)D * 2,
                             (uint64_t)d.num_heads * D * 2, 64, (uint32_t)G, (uint32_t)a.rows_per_tile, sw, "q")) !=
        PA_OK)
        return rc;
    // One box per physical block (or per 128-key tile); for a fused store whose cached
    // prefixes end inside a box, boxes of 16 rows, so a straddling box has at most 15 new
    // rows for the producer to patch in.
    const uint32_t box_rows = a.k_in && a.small_boxes ? 16u : d.block_size < 128 ? (uint32_t)d.block_size : 128u;
    if ((rc = encode_tmap_3d(&tk, bf16, a.k_cache, D, d.num_kv_heads, rows, (uint64_t)D * 2,
                             (uint64_t)d.num_kv_heads * D * 2, 64, 1, box_rows, sw, "k_cache")) != PA_OK)
        return rc;
    if ((rc = encode_tmap_3d(&tv, bf16, a.v_cache, D, d.num_kv_heads, rows, (uint64_t)D * 2,
                             (uint64_t)d.num_kv_heads * D * 2, 64, 1, box_rows, sw, "v_cache")) != PA_OK)
        return rc;
    CUtensorMap tkin = tk, tvin = tv; // fused store: the new keys' inputs, same box as the cache's
    if (a.k_in) {
        if ((rc = encode_tmap_3d(&tkin, bf16, a.k_in, D, d.num_kv_heads, (uint64_t)a.total_q, (uint64_t)D * 2,
                                 (uint64_t)d.num_kv_heads * D * 2, 64, 1, box_rows, sw, "k")) != PA_OK)
            return rc;
        if ((rc = encode_tmap_3d(&tvin, bf16, a.v_in, D, d.num_kv_heads, (uint64_t)a.total_q, (uint64_t)D * 2,
                                 (uint64_t)d.num_kv_heads * D * 2, 64, 1, box_rows, sw, "v")) != PA_OK)
            return rc;
    }
    PfParams p{};
    p.cu_seqlens_q = a.cu_seqlens_q;
    p.cu_seqlens_k = a.cu_seqlens_k;
    p.block_tables = a.block_tables;
    p.tiles = reinterpret_cast<const int4 *>(a.tiles);
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.scale_log2 = a.scale * kLog2e;
    p.num_heads = d.num_heads;
    p.group = G;
    p.rows_per_tile = a.rows_per_tile;
    p.block_size = d.block_size;
    p.box_rows = (int32_t)box_rows;
    p.max_blocks = a.max_blocks_per_seq;
    p.num_slots = (int32_t)rows;
    p.num_kv_heads = d.num_kv_heads;
    p.num_items = a.num_tiles;
    p.out_v8 = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0 ? 1 : 0;
    p.fused = a.k_in ? 1 : 0;
    p.slot_mapping = a.slot_mapping;
    p.k_in = static_cast<const uint4 *>(a.k_in);
    p.v_in = static_cast<const uint4 *>(a.v_in);
    p.k_cache = static_cast<uint4 *>(const_cast<void *>(a.k_cache));
    p.v_cache = static_cast<uint4 *>(const_cast<void *>(a.v_cache));
    // persistent: one CTA per SM (shared memory and TMEM admit one), each walking its items
    const int grid = a.num_tiles < sms ? a.num_tiles : sms;
    prefill_kernel<D, kShort><<<(unsigned)grid, kThreads, L::kSmemBytes, stream>>>(tq, tk, tv, tkin, tvin, p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    }
    return PA_OK;
}

} // namespace

int launch_prefill(const PrefillArgs &a, void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int sms = 0;
    if (int rc = sm_count(&sms))
        return rc;
    if (a.num_tiles <= sms && !a.scratch_cache) // at most one work item per CTA
        return a.dims.head_dim == 128 ? launch<128, true>(a, s, sms) : launch<64, true>(a, s, sms);
    return a.dims.head_dim == 128 ? launch<128, false>(a, s, sms) : launch<64, false>(a, s, sms);
}

int read_prefill_error(uint32_t *code)
{
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof v);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof zero);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "reading prefill error word: %s", cudaGetErrorString(e));
    *code |= (v & 1u) << 1; // a bounded wait timed out
    *code |= (v & 2u) >> 1; // the fused store met a slot outside [-1, num_slots): the store's bit
    return PA_OK;
}

} // namespace pa
