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
// GB300 design (one CTA per work-list tile, 6 warps, 1 CTA per SM):
//  * Query tile = 128 rows of one KV-head group: rows r = pos * G + h packs the
//    G query heads that share a KV head next to each other, so one K/V stream
//    feeds all of them (GQA reuse).  A 3-D TMA box {64 d, G heads, P positions}
//    loads it straight into the 128B-swizzled K-major layout tcgen05 reads.
//  * Keys in tiles of 128.  Each K/V tile is gathered through the block table
//    with one TMA box per physical block (or one per tile when a block holds
//    >= 128 tokens) into a 2-stage ring; boxes past the end of the pool read
//    as zeros.
//  * warp 0: TMA producer.  warp 1: TMEM allocation + single-thread tcgen05.mma
//    issue: S = Q K^T (M=128, N=128, K=D) into one of two TMEM score buffers,
//    then O += P V (M=128, N=D, K=128) into a TMEM accumulator, with V read
//    MN-major straight from its TMA layout.  warps 2-5: one query row per
//    thread — tcgen05.ld of the score row, causal mask on boundary tiles
//    only, fp32 online softmax in base 2 (scale * log2 e folded into one FMA),
//    lazy rescaling of O (only when the running max grows by more than 2^8),
//    P rounded to bf16 into swizzled shared memory, then the epilogue (O / l,
//    bf16, coalesced row stores).
//  * S double buffering lets the tensor core compute S_{j+1} while the softmax
//    warps work on S_j; mbarriers order every hand-off; every wait is bounded
//    and reports a timeout through a device error word instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace pa {

__device__ uint32_t g_prefill_error; // bit 0: a bounded wait timed out

namespace {

constexpr int kThreads = 192;
constexpr int kSoftmaxWarp0 = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f; // log2 units

template <int D>
struct PfLayout {
    static constexpr int kPanels = D / 64;          // 64-element (128-byte) panels along head_dim
    static constexpr int kPanelBytes = 128 * 128;   // 128 rows x 128 bytes
    static constexpr int kTileBytes = kPanels * kPanelBytes;
    static constexpr int kStages = D == 128 ? 2 : 3;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTileBytes;
    static constexpr int kV = kK + kStages * kTileBytes;
    static constexpr int kP = kV + kStages * kTileBytes;
    static constexpr int kPBytes = 2 * kPanelBytes; // 128 rows x 128 keys bf16; reused as O staging
    static constexpr int kBar = kP + kPBytes;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes = kBar + kBarBytes + 1024; // + alignment slack
    static_assert(128 * D * 2 <= kPBytes, "O staging must fit in the P buffer");
};

struct PfParams {
    const int32_t *cu_seqlens_q;
    const int32_t *cu_seqlens_k;
    const int32_t *block_tables;
    const int4 *tiles;
    __nv_bfloat16 *out;
    float scale_log2;
    int32_t num_heads;
    int32_t group;
    int32_t rows_per_tile; // query positions per tile
    int32_t block_size;
    int32_t max_blocks;
    int32_t num_slots;     // num_blocks * block_size: first out-of-range row (reads as zeros)
};

// barrier slots (uint64 each) inside the barrier area
struct Bars {
    uint32_t base;
    __device__ uint32_t q_full() const { return base; }
    __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
    __device__ uint32_t v_full(int s) const { return base + 8 * (4 + s); }
    __device__ uint32_t kv_empty(int s) const { return base + 8 * (7 + s); }
    __device__ uint32_t s_full(int b) const { return base + 8 * (10 + b); }
    __device__ uint32_t s_free(int b) const { return base + 8 * (12 + b); }
    __device__ uint32_t p_full() const { return base + 8 * 14; }
    __device__ uint32_t pv_done() const { return base + 8 * 15; }
    __device__ uint32_t tmem_slot() const { return base + 8 * 16; }
    __device__ uint32_t abort_slot() const { return base + 8 * 17; }
};

struct Waiter {
    volatile uint32_t *abort;
    __device__ bool operator()(uint32_t bar, uint32_t parity) const
    {
        if (*abort)
            return false;
        if (ptx::mbar_wait(bar, parity))
            return true;
        *abort = 1u;
        atomicOr(&g_prefill_error, 1u);
        return false;
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PfParams p)
{
    using L = PfLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *sgen = smem_raw + (sbase - raw); // generic pointer to the aligned base

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Bars bars{sbase + L::kBar};
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sgen + L::kBar + 8 * 17);
    const Waiter wait{abort_flag};

    const int4 tile = p.tiles[blockIdx.x];
    const int b = tile.x, q0 = tile.y, g = tile.z;
    const int cq0 = p.cu_seqlens_q[b];
    const int lq = p.cu_seqlens_q[b + 1] - cq0;
    const int lk = p.cu_seqlens_k[b + 1] - p.cu_seqlens_k[b];
    const int G = p.group;
    const int P = p.rows_per_tile;
    const int npos = min(P, lq - q0);     // valid query positions in this tile
    const int off = lk - lq;              // absolute position of query row 0
    const int nkt = (off + q0 + npos + 127) >> 7;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bars.q_full(), 1);
        for (int s = 0; s < L::kStages; ++s) {
            ptx::mbar_init(bars.k_full(s), 1);
            ptx::mbar_init(bars.v_full(s), 1);
            ptx::mbar_init(bars.kv_empty(s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(bars.s_full(s), 1);
            ptx::mbar_init(bars.s_free(s), 128);
        }
        ptx::mbar_init(bars.p_full(), 128);
        ptx::mbar_init(bars.pv_done(), 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(bars.tmem_slot(), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + L::kBar + 8 * 16);

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        const int bs = p.block_size;
        const int box_rows = bs < 128 ? bs : 128;
        const int nsub = 128 / box_rows;
        const int32_t *bt = p.block_tables + (size_t)b * p.max_blocks;
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_q);
            ptx::prefetch_tmap(&tm_k);
            ptx::prefetch_tmap(&tm_v);
            ptx::mbar_arrive_expect_tx(bars.q_full(), (uint32_t)(L::kPanels * 128 * G * P));
            for (int pp = 0; pp < L::kPanels; ++pp)
                ptx::tma_load_3d(sbase + L::kQ + pp * L::kPanelBytes, &tm_q, bars.q_full(), pp * 64, g * G,
                                 cq0 + q0);
        }
        // row coordinate of sub-box `lane` of key tile j (all lanes compute their own)
        auto sub_row = [&](int j) -> int {
            const int key = j * 128 + lane * box_rows;
            if (lane >= nsub || key >= lk)
                return p.num_slots; // fully out of range: TMA fills zeros
            const int phys = __ldg(bt + key / bs);
            return phys * bs + (key & (bs - 1));
        };
        int next = sub_row(0);
        for (int j = 0; j < nkt; ++j) {
            const int cur = next;
            if (j + 1 < nkt)
                next = sub_row(j + 1);
            const int st = j % L::kStages;
            if (j >= L::kStages && !__all_sync(0xffffffffu, wait(bars.kv_empty(st), ((j / L::kStages) - 1) & 1)))
                break;
            const uint32_t kdst = sbase + L::kK + st * L::kTileBytes;
            const uint32_t vdst = sbase + L::kV + st * L::kTileBytes;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bars.k_full(st), (uint32_t)L::kTileBytes);
                ptx::mbar_arrive_expect_tx(bars.v_full(st), (uint32_t)L::kTileBytes);
            }
            for (int i = 0; i < nsub; ++i) {
                const int row = __shfl_sync(0xffffffffu, cur, i);
                if (lane == 0) {
                    for (int pp = 0; pp < L::kPanels; ++pp) {
                        const uint32_t o = pp * L::kPanelBytes + i * box_rows * 128;
                        ptx::tma_load_3d(kdst + o, &tm_k, bars.k_full(st), pp * 64, g, row);
                        ptx::tma_load_3d(vdst + o, &tm_v, bars.v_full(st), pp * 64, g, row);
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = ptx::idesc_bf16(128, 128, 0);
            constexpr uint32_t idesc_o = ptx::idesc_bf16(128, D, 1);
            bool ok = wait(bars.q_full(), 0);
            for (int j = 0; ok && j <= nkt; ++j) {
                if (j < nkt) {
                    const int st = j % L::kStages;
                    if (!wait(bars.k_full(st), (j / L::kStages) & 1))
                        break;
                    if (j >= 2 && !wait(bars.s_free(j & 1), ((j - 2) >> 1) & 1))
                        break;
                    ptx::tc_fence_after();
                    const uint32_t d_s = tmem + ((j & 1) ? kColS1 : kColS0);
                    const uint32_t qa = sbase + L::kQ, kb = sbase + L::kK + st * L::kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
                        ptx::mma_bf16_ss(d_s, ptx::smem_desc(qa + o, 16, 1024, ptx::kSwizzle128B),
                                         ptx::smem_desc(kb + o, 16, 1024, ptx::kSwizzle128B), idesc_s, kk > 0);
                    }
                    ptx::mma_commit(bars.s_full(j & 1));
                }
                if (j >= 1) {
                    const int jj = j - 1, st = jj % L::kStages;
                    if (!wait(bars.p_full(), jj & 1))
                        break;
                    if (!wait(bars.v_full(st), (jj / L::kStages) & 1))
                        break;
                    ptx::tc_fence_after();
                    const uint32_t pa_ = sbase + L::kP, vb = sbase + L::kV + st * L::kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t oa = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
                        ptx::mma_bf16_ss(tmem + kColO, ptx::smem_desc(pa_ + oa, 16, 1024, ptx::kSwizzle128B),
                                         ptx::smem_desc(vb + kk * 2048, L::kPanelBytes, 1024, ptx::kSwizzle128B),
                                         idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(bars.pv_done());
                    ptx::mma_commit(bars.kv_empty(st));
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- softmax + epilogue
        const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
        const int r = quarter * 32 + lane;         // query row of the tile
        const int tid = (warp - kSoftmaxWarp0) * 32 + lane;
        const bool row_valid = r < G * npos;
        const int limit = off + q0 + r / G + 1;    // keys visible to this row
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY, l_sum = 0.f;
        uint8_t *prow = sgen + L::kP;
        bool ok = true;
        // all lanes poll the same barrier; agree on the outcome so .sync.aligned ops never diverge
        auto wwait = [&](uint32_t bar, uint32_t parity) {
            return __all_sync(0xffffffffu, wait(bar, parity));
        };

        for (int j = 0; j < nkt; ++j) {
            if (!(ok = wwait(bars.s_full(j & 1), (j >> 1) & 1)))
                break;
            ptx::tc_fence_after();
            uint32_t s[128];
            const uint32_t sa = tmem + lane_addr + ((j & 1) ? kColS1 : kColS0);
            ptx::tmem_ld32(sa + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
            ptx::tmem_ld32(sa + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
            ptx::tmem_ld32(sa + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
            ptx::tmem_ld32(sa + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bars.s_free(j & 1));

            const int kbase = j * 128;
            const int lim = limit - kbase;
            uint32_t pk[64];
            float alpha = 1.f;
            bool rescale = false;
            if (row_valid) {
                float mx = -INFINITY;
                if (lim >= 128) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        mx = fmaxf(mx, __uint_as_float(s[c]));
                } else {
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        const float v = c < lim ? __uint_as_float(s[c]) : -INFINITY;
                        s[c] = __float_as_uint(v);
                        mx = fmaxf(mx, v);
                    }
                }
                const float mt = mx * sl2;
                if (mt > m_ref + kRescaleThreshold || m_ref == -INFINITY) {
                    const float m_new = fmaxf(m_ref, mt);
                    alpha = ptx::ex2(m_ref - m_new); // 0 on the first tile
                    rescale = j > 0;
                    l_sum *= alpha;
                    m_ref = m_new;
                }
                float rs = 0.f;
#pragma unroll
                for (int c = 0; c < 128; c += 2) {
                    const float e0 = ptx::ex2(fmaf(__uint_as_float(s[c]), sl2, -m_ref));
                    const float e1 = ptx::ex2(fmaf(__uint_as_float(s[c + 1]), sl2, -m_ref));
                    rs += e0 + e1;
                    pk[c >> 1] = ptx::pack_bf16(e0, e1);
                }
                l_sum += rs;
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    pk[c] = 0u;
            }

            if (j > 0 && !(ok = wwait(bars.pv_done(), (j - 1) & 1)))
                break;
            ptx::tc_fence_after();
            if (__any_sync(0xffffffffu, rescale)) {
                const uint32_t oa = tmem + lane_addr + kColO;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    ptx::tmem_ld32(oa + cc * 32, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    ptx::tmem_st32(oa + cc * 32, o);
                }
                ptx::tmem_wait_st();
            }
            if (j == nkt - 1 && kbase + 128 > lk) {
                // keys past the sequence end: zero their V rows so 0 * garbage cannot poison O
                const int st = j % L::kStages;
                if (!(ok = wwait(bars.v_full(st), (j / L::kStages) & 1)))
                    break;
                if (r >= lk - kbase) {
                    uint8_t *vrow = sgen + L::kV + st * L::kTileBytes + r * 128;
#pragma unroll
                    for (int pp = 0; pp < L::kPanels; ++pp)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4 *>(vrow + pp * L::kPanelBytes + c * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            // P row r: keys 0-63 in panel 0, 64-127 in panel 1, 16-byte chunks XOR-swizzled by row
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int panel = c >> 3, chunk = c & 7;
                uint8_t *dst = prow + panel * L::kPanelBytes + r * 128 + ((chunk ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bars.p_full());
        }

        const bool good = ok && wwait(bars.pv_done(), (nkt - 1) & 1);
        // epilogue: O / l -> bf16 -> staging (row pitch 2*D bytes, chunk-swizzled) -> global
        uint8_t *stg = sgen + L::kP;
        if (good) {
            ptx::tc_fence_after();
            const float inv = (row_valid && l_sum > 0.f) ? 1.f / l_sum : 0.f;
            const uint32_t oa = tmem + lane_addr + kColO;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                ptx::tmem_ld32(oa + cc * 32, o);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = cc * 4 + c;
                    uint4 v;
                    v.x = ptx::pack_bf16(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv);
                    v.y = ptx::pack_bf16(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv);
                    v.z = ptx::pack_bf16(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv);
                    v.w = ptx::pack_bf16(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv);
                    *reinterpret_cast<uint4 *>(stg + r * (2 * D) + ((chunk ^ (r & 7)) << 4)) = v;
                }
            }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory"); // every softmax thread arrives exactly once
        if (!*abort_flag) {
            constexpr int CPR = D / 8; // 16-byte chunks per row
            const int nrows = G * npos;
            for (int idx = tid; idx < nrows * CPR; idx += 128) {
                const int rr = idx / CPR, c = idx % CPR;
                const int pos = q0 + rr / G, hl = rr % G;
                const size_t token = (size_t)cq0 + pos;
                uint4 v = *reinterpret_cast<const uint4 *>(stg + rr * (2 * D) + ((c ^ (rr & 7)) << 4));
                *reinterpret_cast<uint4 *>(p.out + (token * p.num_heads + (size_t)g * G + hl) * D + c * 8) = v;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        cudaGetLastError();
    }
    return fn;
}

int encode_3d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1,
              uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
              const char *what)
{
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
    return PA_OK;
}

template <int D>
int launch(const PrefillArgs &a, cudaStream_t stream)
{
    using L = PfLayout<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
        if (e != cudaSuccess)
            return fail(PA_ERR_CUDA, "prefill smem attribute: %s", cudaGetErrorString(e));
        configured = true;
    }
    auto enc = get_encoder();
    if (!enc)
        return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    const pa_dims &d = a.dims;
    const int G = d.num_heads / d.num_kv_heads;
    const uint64_t rows = (uint64_t)d.num_blocks * d.block_size;
    CUtensorMap tq, tk, tv;
    int rc;
    if ((rc = encode_3d(enc, &tq, a.q, D, d.num_heads, (uint64_t)a.total_q, (uint64_t)D * 2,
                        (uint64_t)d.num_heads * D * 2, 64, (uint32_t)G, (uint32_t)a.rows_per_tile, "q")) != PA_OK)
        return rc;
    const uint32_t box_rows = d.block_size < 128 ? (uint32_t)d.block_size : 128u;
    if ((rc = encode_3d(enc, &tk, a.k_cache, D, d.num_kv_heads, rows, (uint64_t)D * 2,
                        (uint64_t)d.num_kv_heads * D * 2, 64, 1, box_rows, "k_cache")) != PA_OK)
        return rc;
    if ((rc = encode_3d(enc, &tv, a.v_cache, D, d.num_kv_heads, rows, (uint64_t)D * 2,
                        (uint64_t)d.num_kv_heads * D * 2, 64, 1, box_rows, "v_cache")) != PA_OK)
        return rc;
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
    p.max_blocks = a.max_blocks_per_seq;
    p.num_slots = (int32_t)rows;
    prefill_kernel<D><<<(unsigned)a.num_tiles, kThreads, L::kSmemBytes, stream>>>(tq, tk, tv, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

} // namespace

int launch_prefill(const PrefillArgs &a, void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return a.dims.head_dim == 128 ? launch<128>(a, s) : launch<64>(a, s);
}

int read_prefill_error(uint32_t *code)
{
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof v);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof zero);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "reading prefill error word: %s", cudaGetErrorString(e));
    *code |= v << 1;
    return PA_OK;
}

} // namespace pa
