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
//   exchange each thread scales its row of S_r to log2 units (fp32) and
//            st.async's it into the peer's receive buffer (double-buffered);
//            the bytes complete on the peer's mbarrier, so no fence or flag
//            write is needed. Both CTAs add the same two values in the same
//            order (x_0 + x_1): the softmax is bit-identical on both sides;
//   softmax  one thread per row: mask, row max, lazy rescale (only when the
//            max grows by more than 2^8), p = exp2(x - m), P bf16 to TMEM;
//   tcgen05  O_r[128 x 256] += P . V_r (A = P from TMEM; V_r = chunks 0-3 of
//            the stage, read as an MN-major operand).
// The softmax threads run one page ahead on the exchange: while page g is
// being normalised, the partial scores of page g+1 are already in flight.
// Roles (10 warps): warps 0-7 query load, exchange, softmax and epilogue -
// two warps per TMEM lane quadrant, each owning 32 of a page's 64 columns (and
// half of the query words and of O); the pair combines its row maxima and row
// sums through two TMEM columns around a pair barrier - warp 8 TMA producer,
// warp 9 MMA issuer and TMEM owner. The MMA issuer polls its inputs and issues
// whichever of the next score product and the oldest pending P.V product is
// ready.
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
constexpr int kSoftmaxThreads = 256;  // warps 0-7
constexpr int kChunks = 5;
constexpr int kStages = 4;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;

constexpr int kKVChunkBytes = kPage * 128;  // 8 KB: 64 tokens x 64 bf16
constexpr int kStageBytes = kChunks * kKVChunkBytes;
constexpr int kXBytes = kRows * kPage * 4;   // one page of partial scores: 128 x 64 fp32
constexpr int kOffKV = 0;
constexpr int kOffRecv = kOffKV + kStages * kStageBytes;  // 2 buffers: the peer's partials
constexpr int kOffBar = kOffRecv + 2 * kXBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;

constexpr uint32_t kTmemO = 0;     // 256 columns
constexpr uint32_t kTmemQ = 256;   // 144 columns: 288 bf16 query dims per row
constexpr uint32_t kTmemX = 400;   // 4 columns: the warp pair's row max (400, 401) and row sum (402, 403)
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
    uint64_t x_full[2];     // own expect_tx arrival + the peer's st.async bytes
    uint64_t c_done[2];     // one arrival per softmax warp (8): receive buffer read
    uint64_t peer_free[2];  // the peer has read its receive buffer: we may write it again
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

// Half `half` of one row's query slice into TMEM (the A operand of the score
// MMA): of this CTA's 288 dims (144 words of bf16 pairs), words
// [72 half, 72 half + 72); rows >= H get zeros. All 18 loads are in flight
// together.
__device__ __forceinline__ void load_query(const DecodeArgs& args, const Item& it, int s, int row, uint32_t rank,
                                           int half, uint32_t taddr) {
    constexpr int kHalfWords = kQWords / 2;
    const bool live = row < args.H;
    const uint4* src = query_row(args, it.b, s, live ? row : 0, rank) + half * (kHalfWords / 4);
    uint32_t v[kHalfWords];
#pragma unroll
    for (int i = 0; i < kHalfWords / 4; ++i) {
        const uint4 w = live ? src[i] : make_uint4(0, 0, 0, 0);
        v[4 * i] = w.x;
        v[4 * i + 1] = w.y;
        v[4 * i + 2] = w.z;
        v[4 * i + 3] = w.w;
    }
    const uint32_t dst = taddr + (uint32_t)(half * kHalfWords);
    tmem_st16(dst, v);
    tmem_st16(dst + 16, v + 16);
    tmem_st16(dst + 32, v + 32);
    tmem_st16(dst + 48, v + 48);
    tmem_st8(dst + 64, v + 64);
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
    float4* sRecv = reinterpret_cast<float4*>(smem + kOffRecv);  // [2][16][128] float4
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
        mbar_init(&bars->q_full, kSoftmaxThreads);
        mbar_init(&bars->q_empty, 1);
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_free, kSoftmaxThreads);
        mbar_init(&bars->p_full, kSoftmaxThreads);
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->o_free, kSoftmaxThreads);
        for (int k = 0; k < 2; ++k) {
            mbar_init(&bars->x_full[k], 1);
            mbar_init(&bars->c_done[k], kSoftmaxThreads / 32);
            mbar_init(&bars->peer_free[k], 1);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tm_kv);
        // receive slots of pages 0 and 1 are armed up front; later ones are armed
        // when the slot has been read
        mbar_arrive_expect_tx(&bars->x_full[0], (uint32_t)kXBytes);
        mbar_arrive_expect_tx(&bars->x_full[1], (uint32_t)kXBytes);
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote store or arrive
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    // everything above overlaps the previous kernel on the stream; nothing it
    // may have written is read before this point
    griddep_wait();
    griddep_launch_dependents();

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
                // non-blocking probes: a suspended try_wait on one barrier would hold
                // back a product whose inputs became ready on another
                if (lane == 0) {
                    if (!q_ready && ps.first_of_item()) q_ready = mbar_probe(smem_u32(&bars->q_full), (ps.n_items - 1) & 1);
                    ready = (q_ready || !ps.first_of_item()) && mbar_probe(smem_u32(&bars->kv_full[st]), (g / kStages) & 1) &&
                            (g == 0 || mbar_probe(smem_u32(&bars->s_free), (g - 1) & 1));
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
                    ready = mbar_probe(smem_u32(&bars->p_full), g & 1) &&
                            (!first || pp.n_items == 1 || mbar_probe(smem_u32(&bars->o_free), (pp.n_items - 2) & 1));
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
    } else {
        // ------------------------- query load, exchange, softmax, epilogue --
        const int quad = warp & 3, half = warp >> 2;
        const int row = quad * 32 + lane;
        const int pair_bar = 1 + quad;  // named barrier of the two warps sharing these rows
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        // peer addresses of slot 0; slot 1 is a fixed offset away
        const uint32_t recv_remote0 = mapa_shared(smem_u32(sRecv + row), peer);
        const uint32_t xfull_remote0 = mapa_shared(smem_u32(&bars->x_full[0]), peer);
        const uint32_t pfree_remote0 = mapa_shared(smem_u32(&bars->peer_free[0]), peer);
        constexpr uint32_t kSlotBytes = 16 * kRows * 16;
        PageIter ps, pc;  // page whose partial is sent next, page processed next
        ps.init(args, part);
        pc.init(args, part);
        bool ok = true;
        float xs[32];  // own partial (log2 units) of this warp's 32 columns of the page sent last

        // reads this warp's half of S of page ps.g, frees S for the next score
        // product and sends the half to the peer
        auto send_page = [&]() -> bool {
            const int g = ps.g, k = g & 1;
            if (!warp_wait(&bars->s_full, g & 1, abort, err, wait_ns)) return false;
            tc_fence_after();
            {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kTmemS + 32u * half, v);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) xs[c] = __uint_as_float(v[c]) * args.scale_log2;
            }
            tc_fence_before();
            mbar_arrive(&bars->s_free);
            // the peer's slot k held page g - 2: it must have read it
            if (g >= 2 && !warp_wait(&bars->peer_free[k], ((g - 2) >> 1) & 1, abort, err, wait_ns)) return false;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                st_async_v4(recv_remote0 + k * kSlotBytes + (uint32_t)((8 * half + q) * kRows * 16), xs[4 * q],
                            xs[4 * q + 1], xs[4 * q + 2], xs[4 * q + 3], xfull_remote0 + k * (uint32_t)sizeof(uint64_t));
            ps.advance();
            return true;
        };

        ItemIter ahead;  // the item after the one being loaded, for an L2 prefetch of its query rows
        if (pc.valid) {
            load_query(args, pc.it, s, row, rank, half, tmem + lane_base + kTmemQ);
            tc_fence_before();
            mbar_arrive(&bars->q_full);
            ahead = pc.items;
            ok = send_page();
        }
        float m = -INFINITY, l = 0.f;  // l: this warp's half of the row sum
        int n_valid = 0;
        while (pc.valid) {
            // every exit goes through a pair barrier, so both warps of a pair leave together
            const int g = pc.g, k = g & 1;
            const Item it = pc.it;
            const int j = pc.j;
            const bool first = pc.first_of_item(), last = pc.last_of_item();
            if (first) {
                m = -INFINITY;
                l = 0.f;
                n_valid = visible_keys(it.seqlen, args.s_q, s, args.causal);
                Item pf;
                ItemIter probe = ahead;
                if (half == 0 && probe.next(pf)) prefetch_query(args, pf.b, s, row, rank);
            }
            float x[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) x[c] = xs[c];
            // (A) the next page's partial goes out before this page is normalised
            if (ok && ps.valid) {
                if (ps.first_of_item()) {
                    // a new item starts there: its query slice replaces this one as
                    // soon as this item's last score product is done
                    ok = warp_wait(&bars->q_empty, (ps.n_items - 2) & 1, abort, err, wait_ns);
                    if (ok) {
                        tc_fence_after();
                        load_query(args, ps.it, s, row, rank, half, tmem + lane_base + kTmemQ);
                        tc_fence_before();
                        mbar_arrive(&bars->q_full);
                        ahead = ps.items;
                    }
                }
                if (ok) ok = send_page();
            }
            // (B) page g: own partial + the peer's, for this warp's 32 columns
            if (ok) ok = warp_wait(&bars->x_full[k], (g >> 1) & 1, abort, err, wait_ns);
            float mh = -INFINITY;
            if (ok) {
                const float4* rv = sRecv + k * (16 * kRows) + 8 * half * kRows;
                const int vcount = min(max(n_valid - j * kPage - 32 * half, 0), 32);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 w = rv[q * kRows + row];
                    const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 4 * q + e;
                        // x_0 + x_1 in this order on both CTAs
                        x[c] = rank == 0 ? x[c] + wv[e] : wv[e] + x[c];
                    }
                }
                if (vcount < 32) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) x[c] = c < vcount ? x[c] : -INFINITY;
                }
#pragma unroll
                for (int c = 0; c < 32; ++c) mh = fmaxf(mh, x[c]);
                // slot k is read: re-arm it for page g + 2 and tell the peer it may write it
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->c_done[k]);
                if (warp == 0 && lane == 0 && mbar_wait(&bars->c_done[k], (g >> 1) & 1, abort, err, wait_ns)) {
                    mbar_arrive_expect_tx(&bars->x_full[k], (uint32_t)kXBytes);
                    fence_proxy_async_smem();
                    mbar_arrive_remote_relaxed(pfree_remote0 + k * (uint32_t)sizeof(uint64_t));
                }
                tmem_st1(tmem + lane_base + kTmemX + half, __float_as_uint(mh));
                tmem_wait_st();
            }
            tc_fence_before();
            ok = barrier_and(pair_bar, 64, ok);
            if (!ok) break;
            tc_fence_after();
            const float mx = fmaxf(mh, __uint_as_float(tmem_ld1(tmem + lane_base + kTmemX + (half ^ 1))));
            tmem_wait_ld();
            bool pv_waited = false;
            // lazy rescale: a row moves its reference max only when the new max
            // exceeds it by more than 2^8. Both warps of the pair see the same
            // mx and m, so they take the same decisions; the TMEM read-modify-
            // write of O is warp-collective, so a warp takes it when any of its
            // rows needs it (rows that do not scale by 1), each warp over its
            // half of O's columns.
            const bool need = mx > m + kRescaleThreshold;
            const float alpha = need ? fast_exp2(m - mx) : 1.f;  // 0 when m = -inf
            if (!first && __any_sync(0xffffffffu, need)) {
                ok = warp_wait(&bars->pv_done, (g - 1) & 1, abort, err, wait_ns);
                pv_waited = true;
                if (ok) {
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 128; c += 32) {
                        uint32_t v[32];
                        const uint32_t col = tmem + lane_base + kTmemO + 128u * half + c;
                        tmem_ld32(col, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(col, v);
                    }
                    tmem_wait_st();
                }
            }
            if (need) {
                l *= alpha;
                m = mx;
            }
            const float m_use = m == -INFINITY ? 0.f : m;
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                // the row sum takes the fp32 probabilities; only the P.V operand is bf16
                const float p0 = fast_exp2(x[2 * c] - m_use), p1 = fast_exp2(x[2 * c + 1] - m_use);
                l += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
            }
            if (ok && g >= 1 && !pv_waited) ok = warp_wait(&bars->pv_done, (g - 1) & 1, abort, err, wait_ns);
            if (ok) {
                tmem_st16(tmem + lane_base + kTmemP + 16u * half, pk);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars->p_full);
            }

            if (last) {
                // (C) epilogue of the item: the pair adds its two half sums (half 0 + half 1)
                if (ok) ok = warp_wait(&bars->pv_done, g & 1, abort, err, wait_ns);
                if (ok) {
                    tmem_st1(tmem + lane_base + kTmemX + 2 + half, __float_as_uint(l));
                    tmem_wait_st();
                }
                tc_fence_before();
                ok = barrier_and(pair_bar, 64, ok);
                if (!ok) break;
                tc_fence_after();
                const float l_other = __uint_as_float(tmem_ld1(tmem + lane_base + kTmemX + 2 + (half ^ 1)));
                tmem_wait_ld();
                const float l_row = half == 0 ? l + l_other : l_other + l;
                const float inv_l = l_row > 0.f ? 1.f / l_row : 0.f;
                const bool row_ok = row < args.H;
                const size_t orow = ((size_t)it.b * args.s_q + s) * args.H + row;
                const size_t prow_idx = ((size_t)it.piece * args.s_q + s) * args.H + row;
                const int ocol = 256 * rank + 128 * half;  // this warp's 128 latent columns
                // 32-byte stores: every store fills whole sectors
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + kTmemO + 128u * half + c, v);
                    tmem_wait_ld();
                    if (!row_ok) continue;
                    if (it.split) {
                        float* dst = args.o_part + prow_idx * kDLatent + ocol + c;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint32_t w[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(__uint_as_float(v[8 * e + i]) * inv_l);
                            st_global_v8(dst + 8 * e, w);
                        }
                    } else {
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(args.o_lat) + orow * kDLatent + ocol + c;
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            uint32_t w[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                w[i] = pack_bf16x2(__uint_as_float(v[16 * e + 2 * i]) * inv_l,
                                                   __uint_as_float(v[16 * e + 2 * i + 1]) * inv_l);
                            st_global_v8(dst + 16 * e, w);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars->o_free);
                if (rank == 0 && half == 0 && row_ok) {
                    // lse in natural log: x is in log2 units of the scaled score
                    const float lse_v = l_row > 0.f ? (m + log2f(l_row)) * 0.69314718055994530942f : -INFINITY;
                    if (it.split)
                        args.lse_part[prow_idx] = lse_v;
                    else
                        args.lse[orow] = lse_v;
                }
            }
            pc.advance();
        }
    }

    tc_fence_before();
    __syncthreads();
    // the peer may still store into our buffers or arrive on our barriers until
    // it has finished its last page: leave together
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

cudaLaunchConfig_t make_config(int clusters, cudaStream_t stream, cudaLaunchAttribute* attr, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cfg;
}

}  // namespace

cudaError_t launch_decode(const CUtensorMap* tm_kv, const DecodeArgs& args,
                          cudaStream_t stream) {
    cudaError_t e = prepare_kernel();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = make_config(args.num_parts * args.s_q, stream, attr, true);
    return cudaLaunchKernelEx(&cfg, decode_kernel, *tm_kv, args);
}

// Clusters of the decode kernel that can be resident at once on the current device.
int decode_max_active_clusters(int /*device*/) {
    if (prepare_kernel() != cudaSuccess) return 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = make_config(1024, nullptr, attr, false);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_kernel, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace mla
