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
// (r = 0: chunks 0-4, r = 1: chunks 4-8; chunk 4 is shared).
// Tensor memory of a CTA (512 columns): O_r [0, 256), its 288 query dims as
// the A operand [256, 400), S_r [416, 480), P in bf16 [480, 512).
// Per page (64 tokens):
//   TMA      5 x [64 x 64] bf16 boxes of the page into a 4-stage ring
//            (128-byte swizzle), addressed through the block table;
//   tcgen05  S_r[128 x 64] = Q'_r . K_r^T (18 K-steps, A from TMEM);
//   exchange the fp32 partial, scaled to log2 units, is staged in shared
//            memory and sent to the peer with one 32 KB bulk DSMEM copy that
//            completes on the peer's mbarrier; both CTAs then add the same two
//            values in the same order (x_0 + x_1), so the softmax is
//            bit-identical on both sides (fp16 partials were tried: their
//            rounding moves lse by up to 1.3e-3 on N(0,1) absorbed queries);
//   softmax  one thread per row: mask, row max, lazy rescale (only when the
//            max grows by more than 2^8), p = exp2(x - m), P bf16 to TMEM;
//   tcgen05  O_r[128 x 256] += P . V_r (A = P from TMEM; V_r = chunks 0-3 of
//            the stage, read as an MN-major operand).
// Roles (10 warps): warps 0-3 exchange (S from TMEM -> staged -> bulk copy;
// page g+1 goes out while the softmax of page g runs), warps 4-7 query load, softmax and
// epilogue, warp 8 TMA producer, warp 9 MMA issuer and TMEM owner. The MMA
// issuer polls its inputs and issues whichever of the next score product and
// the oldest pending P.V product is ready, so score products run ahead.
// Every wait is bounded; on expiry the kernel records MLA_ERR_TIMEOUT, drains
// its copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <math.h>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 320;
constexpr int kRows = 128;
constexpr int kChunks = 5;
constexpr int kStages = 4;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;

constexpr int kKVChunkBytes = kPage * 128;  // 8 KB: 64 tokens x 64 bf16
constexpr int kStageBytes = kChunks * kKVChunkBytes;
constexpr int kXBytes = kRows * kPage * 4;   // one page of partial scores: 128 x 64 fp32
constexpr int kOffKV = 0;
constexpr int kOffSend = kOffKV + kStages * kStageBytes;  // this CTA's partial
constexpr int kOffRecv = kOffSend + kXBytes;               // the peer's partial
constexpr int kOffBar = kOffRecv + kXBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;

constexpr uint32_t kTmemO = 0;     // 256 columns
constexpr uint32_t kTmemQ = 256;   // 144 columns: 288 bf16 query dims per row
constexpr uint32_t kTmemS = 416;   // 64 columns
constexpr uint32_t kTmemP = 480;   // 32 columns: 64 bf16 probabilities per row
constexpr uint32_t kTmemCols = 512;
constexpr int kQWords = 144;       // 32-bit words of one row's query slice

constexpr float kRescaleThreshold = 8.0f;  // log2 units: tolerate growth up to 2^8 before rescaling O

struct Bars {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t q_full, q_empty;
    uint64_t s_full, s_free;
    uint64_t p_full, pv_done;
    uint64_t o_free;
    uint64_t x_full;     // own expect_tx arrival + the peer's copy bytes
    uint64_t sx_ready;   // one arrival per exchange warp: own partial staged
    uint64_t c_done;     // one arrival per softmax warp: both partials read
    uint64_t send_free;  // local softmax done + peer softmax done with the buffer pair
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

// Walks the pages of a part in order, with their item context.
struct PageIter {
    ItemIter items;
    Item it;
    int j, g, n_items;  // page within the batch, page counter, items started
    bool valid;
    __device__ void init(const DecodeArgs& args, int part) {
        items.init(args, part);
        g = 0;
        n_items = 0;
        valid = items.next(it);
        j = valid ? it.lo : 0;
        if (valid) n_items = 1;
    }
    __device__ bool first_of_item() const { return j == it.lo; }
    __device__ bool last_of_item() const { return j == it.hi - 1; }
    __device__ void advance() {
        ++g;
        if (++j >= it.hi) {
            valid = items.next(it);
            if (valid) {
                j = it.lo;
                ++n_items;
            }
        }
    }
};

__device__ __forceinline__ int visible_keys(int seqlen, int s_q, int s, int causal) {
    int n = causal ? seqlen - s_q + s + 1 : seqlen;
    return n < 0 ? 0 : (n > seqlen ? seqlen : n);
}

__device__ __forceinline__ const uint4* query_row(const DecodeArgs& args, int b, int s, int row, uint32_t rank) {
    return reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(args.q_abs) +
                                          (((size_t)b * args.s_q + s) * args.H + row) * kDQK + 288 * rank);
}

// Query slice of one row into TMEM (the A operand of the score MMA): this CTA's
// 288 dims as 144 words of bf16 pairs; rows >= H get zeros. All 36 loads are
// in flight together (one memory latency, not nine).
__device__ __forceinline__ void load_query(const DecodeArgs& args, const Item& it, int s, int row, uint32_t rank,
                                           uint32_t taddr) {
    const bool live = row < args.H;
    const uint4* src = query_row(args, it.b, s, live ? row : 0, rank);
    uint32_t v[kQWords];
#pragma unroll
    for (int i = 0; i < kQWords / 4; ++i) {
        const uint4 w = live ? src[i] : make_uint4(0, 0, 0, 0);
        v[4 * i] = w.x;
        v[4 * i + 1] = w.y;
        v[4 * i + 2] = w.z;
        v[4 * i + 3] = w.w;
    }
#pragma unroll
    for (int c = 0; c < kQWords; c += 16) tmem_st16(taddr + (uint32_t)c, v + c);
    tmem_wait_st();
}

// Warm L2 with the query slice of a row that will be loaded one item later.
__device__ __forceinline__ void prefetch_query(const DecodeArgs& args, int b, int s, int row, uint32_t rank) {
    if (row >= args.H) return;
    const char* p = reinterpret_cast<const char*>(query_row(args, b, s, row, rank));
#pragma unroll
    for (int i = 0; i < 576; i += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + i));
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_kv, DecodeArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sKV = smem + kOffKV;
    float4* sSend = reinterpret_cast<float4*>(smem + kOffSend);  // [16][128] float4
    float4* sRecv = reinterpret_cast<float4*>(smem + kOffRecv);  // [16][128] float4
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
        mbar_init(&bars->q_full, kRows);
        mbar_init(&bars->q_empty, 1);
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_free, kRows);
        mbar_init(&bars->p_full, kRows);
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->o_free, kRows);
        mbar_init(&bars->x_full, 1);
        mbar_init(&bars->sx_ready, 4);
        mbar_init(&bars->c_done, 4);
        mbar_init(&bars->send_free, 2);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tm_kv);
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote arrive or copy
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;

    if (warp == kWarpProducer) {
        // ------------------------------------------------------- producer --
        if (lane == 0) {
            PageIter pg;
            pg.init(args, part);
            bool ok = true;
            for (; pg.valid; pg.advance()) {
                const int g = pg.g, st = g % kStages;
                if (g >= kStages) ok = mbar_wait(&bars->kv_empty[st], ((g / kStages) - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                const int j = pg.j;
                int blk = j < args.mbps ? args.block_table[(size_t)pg.it.b * args.mbps + j] : -1;
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
            const int g = pg.g;
            // drain: wait for the last load issued into each buffer
            for (int gg = g - kStages > 0 ? g - kStages : 0; gg < g; ++gg)
                mbar_wait(&bars->kv_full[gg % kStages], (gg / kStages) & 1, nullptr, err, kDrainNs);
        }
    } else if (warp == kWarpMma) {
        // ----------------------------------------------------- MMA issuer --
        constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kPage, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, 256, false, true);
        PageIter ps, pp;  // next score product, next P.V product
        ps.init(args, part);
        pp.init(args, part);
        bool ok = true, issued_any = false, q_ready = false;
        uint64_t t_last = globaltimer_ns();
        while (ok && pp.valid) {
            bool progressed = false;
            // --- score product of page ps.g
            if (ps.valid) {
                const int g = ps.g, st = g % kStages;
                bool ready = true;
                if (lane == 0) {
                    if (!q_ready && ps.first_of_item()) q_ready = mbar_test(smem_u32(&bars->q_full), (ps.n_items - 1) & 1);
                    ready = (q_ready || !ps.first_of_item()) && mbar_test(smem_u32(&bars->kv_full[st]), (g / kStages) & 1) &&
                            (g == 0 || mbar_test(smem_u32(&bars->s_free), (g - 1) & 1));
                }
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (ready) {
                    uint8_t* stage = sKV + st * kStageBytes;
                    const int tail_rows = (ps.j == ps.it.nblk - 1) ? ps.it.seqlen - ps.j * kPage : kPage;
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
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t k_base = smem_u32(stage);
                        // partial score over 18 K-steps of 16 dims: [288 r, 288 r + 288);
                        // the query slice in TMEM holds exactly those dims
                        const int step0 = rank == 0 ? 0 : 2;  // first K-step inside local chunk 0
#pragma unroll
                        for (int t = 0; t < 18; ++t) {
                            const int ls = step0 + t;
                            const int c = ls >> 2, kk = ls & 3;
                            const uint64_t bd = desc_sw128(k_base + c * kKVChunkBytes + kk * 32, 0, 1024);
                            mma_bf16_ts(tmem + kTmemS, tmem + kTmemQ + 8u * t, bd, idesc_s, t > 0 ? 1u : 0u);
                        }
                        mma_commit(&bars->s_full);
                        if (ps.last_of_item()) mma_commit(&bars->q_empty);
                    }
                    __syncwarp();
                    issued_any = true;
                    if (ps.last_of_item()) q_ready = false;
                    ps.advance();
                    progressed = true;
                }
            }
            // --- P.V product of page pp.g (its score product was issued earlier)
            if (pp.g < ps.g || !ps.valid) {
                const int g = pp.g, st = g % kStages;
                const bool first = pp.first_of_item();
                bool ready = true;
                if (lane == 0)
                    ready = mbar_test(smem_u32(&bars->p_full), g & 1) &&
                            (!first || pp.n_items == 1 || mbar_test(smem_u32(&bars->o_free), (pp.n_items - 2) & 1));
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (ready) {
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t v_base = smem_u32(sKV + st * kStageBytes);
#pragma unroll
                        for (int kk = 0; kk < kPage / 16; ++kk) {
                            const uint64_t bd = desc_sw128(v_base + kk * 2048, kKVChunkBytes, 1024);
                            mma_bf16_ts(tmem + kTmemO, tmem + kTmemP + 8u * kk, bd, idesc_pv, (!first || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&bars->pv_done);
                        mma_commit(&bars->kv_empty[st]);
                    }
                    __syncwarp();
                    pp.advance();
                    progressed = true;
                }
            }
            if (progressed) {
                t_last = globaltimer_ns();
            } else {
                if (*abort) ok = false;
                else if ((long long)(globaltimer_ns() - t_last) > wait_ns) {
                    record_error(err, kErrTimeout);
                    *abort = 1;
                    ok = false;
                }
                ok = __all_sync(0xffffffffu, ok);
            }
        }
        // drain: every MMA this thread issued has completed before TMEM is freed
        if (issued_any) {
            if (lane == 0) mma_commit(&bars->drain);
            __syncwarp();
            warp_wait(&bars->drain, 0, nullptr, err, kDrainNs);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------- exchange --
        const int row = threadIdx.x;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        PageIter pg;
        pg.init(args, part);
        bool ok = true;
        for (; ok && pg.valid; pg.advance()) {
            const int g = pg.g;
            ok = warp_wait(&bars->s_full, g & 1, abort, err, wait_ns);
            if (!ok) break;
            tc_fence_after();
            float x[kPage];
            {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kTmemS, v);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(v[c]) * args.scale_log2;
                tmem_ld32(tmem + lane_base + kTmemS + 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) x[32 + c] = __uint_as_float(v[c]) * args.scale_log2;
            }
            tc_fence_before();
            mbar_arrive(&bars->s_free);
            // the buffer pair was last used by page g - 1: both softmax sides must have read it
            if (g >= 1) ok = warp_wait(&bars->send_free, (g - 1) & 1, abort, err, wait_ns);
            if (!ok) break;
#pragma unroll
            for (int q = 0; q < kPage / 4; ++q) sSend[q * kRows + row] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->sx_ready);
            if (row == 0 && mbar_wait(&bars->sx_ready, g & 1, abort, err, wait_ns)) {
                mbar_arrive_expect_tx(&bars->x_full, (uint32_t)kXBytes);
                bulk_copy_to_peer(mapa_shared(smem_u32(sRecv), peer), sSend, (uint32_t)kXBytes,
                                  mapa_shared(smem_u32(&bars->x_full), peer));
            }
        }
    } else if (warp < 8) {
        // ------------------------------------ query load, softmax, epilogue --
        const int row = threadIdx.x - 128;
        const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
        ItemIter iter;
        iter.init(args, part);
        Item it, nxt;
        int g = 0, n_items = 0;
        bool ok = true;
        bool have = iter.next(it);
        if (have) {
            load_query(args, it, s, row, rank, tmem + lane_base + kTmemQ);
            tc_fence_before();
            mbar_arrive(&bars->q_full);
        }
        ItemIter ahead = iter;  // one item ahead of `it`, for L2 prefetch of its query rows
        while (ok && have) {
            {
                Item pf;
                ItemIter probe = ahead;
                if (probe.next(pf)) prefetch_query(args, pf.b, s, row, rank);
            }
            const int n_valid = visible_keys(it.seqlen, args.s_q, s, args.causal);
            float m = -INFINITY, l = 0.f;
            for (int j = it.lo; j < it.hi && ok; ++j, ++g) {
                ok = warp_wait(&bars->sx_ready, g & 1, abort, err, wait_ns);
                if (ok) ok = warp_wait(&bars->x_full, g & 1, abort, err, wait_ns);
                if (!ok) break;
                const int vcount = min(max(n_valid - j * kPage, 0), kPage);
                float x[kPage];
                float mx = -INFINITY;
#pragma unroll
                for (int q = 0; q < kPage / 4; ++q) {
                    const float4 a = sSend[q * kRows + row];
                    const float4 b = sRecv[q * kRows + row];
                    const float av[4] = {a.x, a.y, a.z, a.w};
                    const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 4 * q + e;
                        // x_0 + x_1 in this order on both CTAs
                        const float sc = rank == 0 ? av[e] + bv[e] : bv[e] + av[e];
                        x[c] = c < vcount ? sc : -INFINITY;
                        mx = fmaxf(mx, x[c]);
                    }
                }
                // both partials of this page are read: hand the buffer pair back.
                // The remote arrival only reports that our reads are complete (they
                // are ordered before it through c_done); the peer's next write into
                // our receive buffer is its bulk copy, so no cluster-scope release.
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->c_done);
                if (row == 0 && mbar_wait(&bars->c_done, g & 1, abort, err, wait_ns)) {
                    mbar_arrive(&bars->send_free);
                    fence_proxy_async_smem();
                    mbar_arrive_remote_relaxed(mapa_shared(smem_u32(&bars->send_free), peer));
                }
                bool pv_waited = false;
                // lazy rescale: a row moves its reference max only when the new
                // max exceeds it by more than 2^8. The TMEM read-modify-write of O
                // is warp-collective, so the whole warp takes it when any of its
                // rows needs it; rows that do not scale by 1.
                const bool need = mx > m + kRescaleThreshold;
                const float alpha = need ? fast_exp2(m - mx) : 1.f;  // 0 when m = -inf
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
                    const float p0 = fast_exp2(x[2 * c] - m_use), p1 = fast_exp2(x[2 * c + 1] - m_use);
                    l += p0 + p1;
                    pk[c] = pack_bf16x2(p0, p1);
                }
                if (g >= 1 && !pv_waited) ok = warp_wait(&bars->pv_done, (g - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                tmem_st32(tmem + lane_base + kTmemP, pk);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars->p_full);
            }
            if (!ok) break;
            // the next item's query slice goes in as soon as this item's last score
            // MMA is done: this item's last P.V product may be issued after the
            // next item's first score product
            const bool have_next = iter.next(nxt);
            ahead = iter;
            if (have_next) {
                ok = warp_wait(&bars->q_empty, n_items & 1, abort, err, wait_ns);
                if (!ok) break;
                tc_fence_after();
                load_query(args, nxt, s, row, rank, tmem + lane_base + kTmemQ);
                tc_fence_before();
                mbar_arrive(&bars->q_full);
            }
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
                // lse in natural log: x is in log2 units of the scaled score
                const float lse_v = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
                if (it.split)
                    args.lse_part[prow_idx] = lse_v;
                else
                    args.lse[orow] = lse_v;
            }
            ++n_items;
            it = nxt;
            have = have_next;
        }
    }

    tc_fence_before();
    __syncthreads();
    // the peer may still arrive on our barriers / copy into our buffers until it
    // has finished its last page: leave together
    cluster_sync_all();
    if (warp == kWarpMma) {
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

cudaError_t launch_decode(const CUtensorMap* tm_kv, const DecodeArgs& args,
                          cudaStream_t stream) {
    cudaError_t e = prepare_kernel();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_config(args.num_parts * args.s_q, stream, attr);
    return cudaLaunchKernelEx(&cfg, decode_kernel, *tm_kv, args);
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
