// decode.cu - paged, absorbed MLA decode on sm_103a.
//
// What it computes ("DeepSeek-V3 MLA deep engineering", sec. 2.4 and 4.3;
// "FlashMLA: efficient MLA decode kernel for Hopper GPUs", usage example):
// for every query row (b, s, h), scores against the paged latent cache
// score_t = scale * q'[0:576] . kv_t[0:576], an online softmax over the
// visible keys, o = sum_t p_t kv_t[0:512] and lse = ln sum_t exp(score_t).
//
// Work decomposition. One 2-CTA cluster owns one schedule part for one query
// token s (all H heads = the 128 rows of every MMA). The fp32 latent output of
// 128 rows x 512 columns is exactly one SM's tensor memory, so the pair splits
// it: CTA r keeps O[:, 256r : 256r+256] in TMEM. Both need the full score tile,
// so the score contraction (576 deep) is split in K instead: CTA r computes
// the partial S_r over dims [288r, 288r+288) and the two partials are swapped
// through distributed shared memory and added (S_0 + S_1 in both CTAs, so the
// softmax is bit-identical on both sides).
//
// Each CTA therefore needs 5 of the 9 64-column chunks of every page
// (r = 0: chunks 0-4, r = 1: chunks 4-8; chunk 4 is shared) and of the query.
// Per page (64 tokens):
//   TMA      5 x [64 x 64] bf16 boxes of the page into a 2-stage ring
//            (128-byte swizzle), addressed through the block table;
//   tcgen05  S_r[128 x 64]   = Q'_r . K_r^T       (18 K-steps, fp32 in TMEM);
//   exchange S = S_0 + S_1 via DSMEM (32 KB each way);
//   softmax  one thread per row: mask, row max, lazy rescale (only when the
//            max grows by more than 2^8), p = exp2(x - m), P bf16 to smem;
//   tcgen05  O_r[128 x 256] += P . V_r            (V_r = chunks 0-3 of the stage,
//            read as an MN-major operand).
// Roles (8 warps): warp 0 TMA producer, warp 1 MMA issuer (and TMEM owner),
// warps 4-7 softmax + epilogue; warps 2-3 only join the final barriers.
// Every wait is bounded; on expiry the kernel records MLA_ERR_TIMEOUT, drains
// its copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <math.h>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 128;
constexpr int kChunks = 5;
constexpr int kStages = 2;

constexpr int kQChunkBytes = kRows * 128;   // 16 KB: 128 rows x 64 bf16
constexpr int kKVChunkBytes = kPage * 128;  // 8 KB: 64 tokens x 64 bf16
constexpr int kQBytes = kChunks * kQChunkBytes;
constexpr int kStageBytes = kChunks * kKVChunkBytes;
constexpr int kPBytes = kRows * 128;         // P: 128 rows x 64 bf16
constexpr int kXBytes = kRows * kPage * 4;   // partial scores: 128 x 64 fp32
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kQBytes;
constexpr int kOffP = kOffKV + kStages * kStageBytes;
constexpr int kOffX = kOffP + kPBytes;
constexpr int kOffBar = kOffX + kXBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;

constexpr uint32_t kTmemO = 0;     // 256 columns
constexpr uint32_t kTmemS = 256;   // 64 columns
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleThreshold = 8.0f;  // log2 units: tolerate growth up to 2^8 before rescaling O

struct Bars {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t q_full, q_empty;
    uint64_t s_full, s_free;
    uint64_t p_full, pv_done;
    uint64_t o_free;
    uint64_t x_full, peer_free;
    uint64_t drain;
    uint32_t tmem_slot;
    int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// One work item: the pages [lo, hi) of batch b inside this part.
struct Item {
    int b, lo, hi, piece, seqlen, nblk;
    bool split;
};

struct ItemIter {
    const DecodeArgs* a;
    int row[6];
    int b, k;
    __device__ void init(const DecodeArgs& args, int part) {
        a = &args;
        const int* r = args.tile_meta + 8 * part;
#pragma unroll
        for (int i = 0; i < 6; ++i) row[i] = r[i];
        b = row[0];
        k = 0;
    }
    __device__ bool next(Item& it) {
        if (row[5] == 0) return false;
        while (b <= row[2]) {
            const int sl = a->seqlens[b];
            const int n = sl > 0 ? (sl + kPage - 1) / kPage : 0;
            const int cur = b++;
            if (n == 0) continue;
            it.b = cur;
            it.lo = (cur == row[0]) ? row[1] : 0;
            it.hi = (cur == row[2]) ? row[3] : n;
            it.piece = row[4] + k++;
            it.seqlen = sl;
            it.nblk = n;
            it.split = (a->num_splits[cur + 1] - a->num_splits[cur]) > 1;
            return true;
        }
        return false;
    }
};

__device__ __forceinline__ int visible_keys(int seqlen, int s_q, int s, int causal) {
    int n = causal ? seqlen - s_q + s + 1 : seqlen;
    return n < 0 ? 0 : (n > seqlen ? seqlen : n);
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv, DecodeArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sKV = smem + kOffKV;
    uint8_t* sP = smem + kOffP;
    float4* sX = reinterpret_cast<float4*>(smem + kOffX);
    Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
    volatile int* abort = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int cluster_id = blockIdx.x >> 1;
    const int part = cluster_id / args.s_q;
    const int s = cluster_id % args.s_q;
    int* err = args.err;
    const long long wait_ns = args.wait_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bars->kv_full[i], 1);
            mbar_init(&bars->kv_empty[i], 1);
        }
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_free, kRows);
        mbar_init(&bars->p_full, kRows);
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->o_free, kRows);
        mbar_init(&bars->x_full, kRows);     // arrivals come from the peer CTA
        mbar_init(&bars->peer_free, kRows);  // arrivals come from the peer CTA
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_kv);
    }
    if (args.H < kRows) {
        // query rows >= H are never loaded: keep them zero for every item
        for (int i = threadIdx.x; i < kChunks * (kRows - args.H) * 8; i += kThreads) {
            const int c = i / ((kRows - args.H) * 8);
            const int rem = i % ((kRows - args.H) * 8);
            const int r = args.H + rem / 8;
            reinterpret_cast<uint4*>(sQ + c * kQChunkBytes + r * 128)[rem % 8] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------- producer --
        if (lane == 0) {
            ItemIter iter;
            iter.init(args, part);
            Item it;
            int g = 0, n_items = 0;
            bool ok = true;
            const uint32_t q_bytes = (uint32_t)(kChunks * args.H * 128);
            while (ok && iter.next(it)) {
                if (n_items > 0) ok = mbar_wait(&bars->q_empty, (n_items - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                mbar_arrive_expect_tx(&bars->q_full, q_bytes);
                for (int c = 0; c < kChunks; ++c)
                    tma_load_3d(sQ + c * kQChunkBytes, &tm_q, &bars->q_full, 64 * (4 * (int)rank + c), 0,
                                it.b * args.s_q + s);
                ++n_items;
                for (int j = it.lo; j < it.hi; ++j, ++g) {
                    const int st = g % kStages;
                    if (g >= kStages) ok = mbar_wait(&bars->kv_empty[st], ((g / kStages) - 1) & 1, abort, err, wait_ns);
                    if (!ok) break;
                    int blk = j < args.mbps ? args.block_table[(size_t)it.b * args.mbps + j] : -1;
                    if (blk < 0 || blk >= args.num_blocks) {
                        record_error(err, kErrBadBlock);
                        blk = 0;
                    }
                    mbar_arrive_expect_tx(&bars->kv_full[st], (uint32_t)kStageBytes);
                    uint8_t* dst = sKV + st * kStageBytes;
                    for (int c = 0; c < kChunks; ++c)
                        tma_load_2d(dst + c * kKVChunkBytes, &tm_kv, &bars->kv_full[st], 64 * (4 * (int)rank + c),
                                    blk * kPage);
                }
            }
            // drain: wait for the last load issued into each buffer
            for (int gg = g - kStages > 0 ? g - kStages : 0; gg < g; ++gg)
                mbar_wait(&bars->kv_full[gg % kStages], (gg / kStages) & 1, nullptr, err, kDrainNs);
            if (n_items > 0) mbar_wait(&bars->q_full, (n_items - 1) & 1, nullptr, err, kDrainNs);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer --
        constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kPage, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, 256, false, true);
        ItemIter iter;
        iter.init(args, part);
        Item it;
        int g = 0, n_items = 0;
        bool ok = true;
        bool issued_any = false;
        // the page whose P.V product is still to be issued
        bool pend = false;
        int pend_st = 0, pend_g = 0, pend_item = 0;
        bool pend_first = false;

        auto issue_pv = [&]() -> bool {
            if (!warp_wait(&bars->p_full, pend_g & 1, abort, err, wait_ns)) return false;
            if (pend_first && pend_item >= 1 &&
                !warp_wait(&bars->o_free, (pend_item - 1) & 1, abort, err, wait_ns))
                return false;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t p_base = smem_u32(sP);
                const uint32_t v_base = smem_u32(sKV + pend_st * kStageBytes);
#pragma unroll
                for (int kk = 0; kk < kPage / 16; ++kk) {
                    const uint64_t ad = desc_sw128(p_base + kk * 32, 0, 1024);
                    const uint64_t bd = desc_sw128(v_base + kk * 2048, kKVChunkBytes, 1024);
                    mma_bf16_ss(tmem + kTmemO, ad, bd, idesc_pv, (!pend_first || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bars->pv_done);
                mma_commit(&bars->kv_empty[pend_st]);
            }
            __syncwarp();
            pend = false;
            return true;
        };

        while (ok && iter.next(it)) {
            ok = warp_wait(&bars->q_full, n_items & 1, abort, err, wait_ns);
            if (!ok) break;
            for (int j = it.lo; j < it.hi && ok; ++j, ++g) {
                const int st = g % kStages;
                ok = warp_wait(&bars->kv_full[st], (g / kStages) & 1, abort, err, wait_ns);
                if (!ok) break;
                uint8_t* stage = sKV + st * kStageBytes;
                const int tail_rows = (j == it.nblk - 1) ? it.seqlen - j * kPage : kPage;
                if (tail_rows < kPage) {
                    // rows past seqlen hold arbitrary bytes: zero them so that
                    // 0-probability columns cannot inject NaN/Inf into P.V
                    const int per_chunk = (kPage - tail_rows) * 8;  // 16-byte words
                    for (int i = lane; i < kChunks * per_chunk; i += 32) {
                        const int c = i / per_chunk, w = i % per_chunk;
                        reinterpret_cast<uint4*>(stage + c * kKVChunkBytes + tail_rows * 128)[w] = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (g >= 1) ok = warp_wait(&bars->s_free, (g - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t q_base = smem_u32(sQ);
                    const uint32_t k_base = smem_u32(stage);
                    // partial score over 18 K-steps of 16 dims: [288 r, 288 r + 288)
                    const int step0 = rank == 0 ? 0 : 2;  // first K-step inside local chunk 0
#pragma unroll
                    for (int t = 0; t < 18; ++t) {
                        const int ls = step0 + t;  // local K-step index
                        const int c = ls >> 2, kk = ls & 3;
                        const uint64_t ad = desc_sw128(q_base + c * kQChunkBytes + kk * 32, 0, 1024);
                        const uint64_t bd = desc_sw128(k_base + c * kKVChunkBytes + kk * 32, 0, 1024);
                        mma_bf16_ss(tmem + kTmemS, ad, bd, idesc_s, t > 0 ? 1u : 0u);
                    }
                    mma_commit(&bars->s_full);
                    if (j == it.hi - 1) mma_commit(&bars->q_empty);
                }
                __syncwarp();
                issued_any = true;
                if (pend) ok = issue_pv();
                if (!ok) break;
                pend = true;
                pend_st = st;
                pend_g = g;
                pend_item = n_items;
                pend_first = (j == it.lo);
            }
            ++n_items;
        }
        if (ok && pend) ok = issue_pv();
        // drain: every MMA this thread issued has completed before TMEM is freed
        if (issued_any) {
            if (lane == 0) mma_commit(&bars->drain);
            __syncwarp();
            warp_wait(&bars->drain, 0, nullptr, err, kDrainNs);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------- softmax + epilogue --
        const int row = threadIdx.x - 128;
        const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
        const uint32_t x_remote = mapa_shared(smem_u32(sX), peer);
        const uint32_t xfull_remote = mapa_shared(smem_u32(&bars->x_full), peer);
        const uint32_t pfree_remote = mapa_shared(smem_u32(&bars->peer_free), peer);
        ItemIter iter;
        iter.init(args, part);
        Item it;
        int g = 0, n_items = 0;
        bool ok = true;
        while (ok && iter.next(it)) {
            const int n_valid = visible_keys(it.seqlen, args.s_q, s, args.causal);
            float m = -INFINITY, l = 0.f;
            for (int j = it.lo; j < it.hi && ok; ++j, ++g) {
                ok = warp_wait(&bars->s_full, g & 1, abort, err, wait_ns);
                if (!ok) break;
                tc_fence_after();
                float x[kPage];
                {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + kTmemS, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(v[c]);
                    tmem_ld32(tmem + lane_base + kTmemS + 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) x[32 + c] = __uint_as_float(v[c]);
                }
                tc_fence_before();
                mbar_arrive(&bars->s_free);
                // swap partial scores with the peer
                if (g >= 1) ok = warp_wait<true>(&bars->peer_free, (g - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
#pragma unroll
                for (int q = 0; q < kPage / 4; ++q)
                    st_cluster_v4(x_remote + (uint32_t)((q * kRows + row) * 16), x[4 * q], x[4 * q + 1], x[4 * q + 2],
                                  x[4 * q + 3]);
                mbar_arrive_remote(xfull_remote);
                ok = warp_wait<true>(&bars->x_full, g & 1, abort, err, wait_ns);
                if (!ok) break;
                const int vcount = min(max(n_valid - j * kPage, 0), kPage);
                float mx = -INFINITY;
#pragma unroll
                for (int q = 0; q < kPage / 4; ++q) {
                    const float4 w = sX[q * kRows + row];
                    const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 4 * q + e;
                        // S_0 + S_1 in this order on both CTAs
                        const float sc = rank == 0 ? x[c] + wv[e] : wv[e] + x[c];
                        x[c] = c < vcount ? sc * args.scale_log2 : -INFINITY;
                        mx = fmaxf(mx, x[c]);
                    }
                }
                mbar_arrive_remote(pfree_remote);
                bool pv_waited = false;
                // lazy rescale: a row moves its reference max only when the new
                // max exceeds it by more than 2^8. The TMEM read-modify-write of O
                // is warp-collective, so the whole warp takes it when any of its
                // rows needs it; rows that do not scale by 1.
                const bool need = mx > m + kRescaleThreshold;
                const float alpha = need ? exp2f(m - mx) : 1.f;  // 0 when m = -inf
                if (j > it.lo && __any_sync(0xffffffffu, need)) {
                    ok = warp_wait(&bars->pv_done, (g - 1) & 1, abort, err, wait_ns);
                    if (!ok) break;
                    pv_waited = true;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 256; c += 32) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_base + kTmemO + c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(tmem + lane_base + kTmemO + c, v);
                    }
                    tmem_wait_st();
                }
                if (need) {
                    l *= alpha;
                    m = mx;
                }
                const float m_use = m == -INFINITY ? 0.f : m;
                uint32_t pk[kPage / 2];
#pragma unroll
                for (int c = 0; c < kPage / 2; ++c) {
                    // the row sum takes the fp32 probabilities; only the P.V operand is bf16
                    const float p0 = exp2f(x[2 * c] - m_use), p1 = exp2f(x[2 * c + 1] - m_use);
                    l += p0 + p1;
                    pk[c] = pack_bf16x2(p0, p1);
                }
                if (g >= 1 && !pv_waited) ok = warp_wait(&bars->pv_done, (g - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                uint8_t* prow = sP + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) * 16)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bars->p_full);
            }
            if (!ok) break;
            // epilogue of the item
            ok = warp_wait(&bars->pv_done, (g - 1) & 1, abort, err, wait_ns);
            if (!ok) break;
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const bool row_ok = row < args.H;
            const size_t orow = ((size_t)it.b * args.s_q + s) * args.H + row;
            const size_t prow_idx = ((size_t)it.piece * args.s_q + s) * args.H + row;
#pragma unroll 1
            for (int c = 0; c < 256; c += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kTmemO + c, v);
                tmem_wait_ld();
                if (!row_ok) continue;
                if (it.split) {
                    float4* dst = reinterpret_cast<float4*>(args.o_part + prow_idx * kDLatent + 256 * rank + c);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(__uint_as_float(v[4 * e]) * inv_l, __uint_as_float(v[4 * e + 1]) * inv_l,
                                             __uint_as_float(v[4 * e + 2]) * inv_l, __uint_as_float(v[4 * e + 3]) * inv_l);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.o_lat) + orow * kDLatent +
                                                          256 * rank + c);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * e + 0]) * inv_l, __uint_as_float(v[8 * e + 1]) * inv_l),
                                            pack_bf16x2(__uint_as_float(v[8 * e + 2]) * inv_l, __uint_as_float(v[8 * e + 3]) * inv_l),
                                            pack_bf16x2(__uint_as_float(v[8 * e + 4]) * inv_l, __uint_as_float(v[8 * e + 5]) * inv_l),
                                            pack_bf16x2(__uint_as_float(v[8 * e + 6]) * inv_l, __uint_as_float(v[8 * e + 7]) * inv_l));
                }
            }
            tc_fence_before();
            mbar_arrive(&bars->o_free);
            if (rank == 0 && row_ok) {
                const float lse_v = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
                if (it.split)
                    args.lse_part[prow_idx] = lse_v;
                else
                    args.lse[orow] = lse_v;
            }
            ++n_items;
        }
    }

    tc_fence_before();
    __syncthreads();
    // the peer may still arrive on our barriers / write our buffers until it
    // has finished its last page: leave together
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

cudaError_t prepare_kernel() {
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

cudaLaunchConfig_t make_config(int clusters, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

}  // namespace

cudaError_t launch_decode(const CUtensorMap* tm_q, const CUtensorMap* tm_kv, const DecodeArgs& args,
                          cudaStream_t stream) {
    cudaError_t e = prepare_kernel();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_config(args.num_parts * args.s_q, stream, attr);
    return cudaLaunchKernelEx(&cfg, decode_kernel, *tm_q, *tm_kv, args);
}

// Clusters of the decode kernel that can be resident at once on the current device.
int decode_max_active_clusters(int /*device*/) {
    if (prepare_kernel() != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_config(1024, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_kernel, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace mla
