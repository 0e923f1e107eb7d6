// decode.cu - paged, absorbed MLA decode on sm_103a.
//
// What it computes ("DeepSeek-V3 MLA deep engineering", sec. 2.4 and 4.3;
// "FlashMLA: efficient MLA decode kernel for Hopper GPUs", usage example):
// for every query row (b, s, h), scores against the paged latent cache
// score_t = scale * q'[0:576] . kv_t[0:576], an online softmax over the
// visible keys, o = sum_t p_t kv_t[0:512] and lse = ln sum_t exp(score_t).
//
// Work decomposition. One 2-CTA cluster owns one schedule part for one query
// token s; all H heads are the 128 rows of every MMA. The two CTAs split the
// work by role:
//  * the score CTA (rank 0) holds the whole absorbed query of the part's
//    current batch - dims [0, 512) in TMEM as the A operand, the 64 rope dims
//    in shared memory - and computes S = Q' K^T for two pages at a time
//    (N = 128 keys) into one of two TMEM buffers. Its softmax threads (one
//    per row and page) mask, take the row max, rescale lazily, exponentiate
//    and ship P (bf16, 128-byte-swizzled like an MMA operand) together with
//    the per-row rescale factor straight into the value CTA's shared memory
//    (st.async, counted on the value CTA's mbarrier);
//  * the value CTA (rank 1) keeps the fp32 output O [128 x 512] in its TMEM
//    (all 512 columns), loads its own copy of the value rows of each page
//    (mostly L2 hits: the score CTA has just read the same page), accumulates
//    O += P . V, rescales O rows when the score CTA moved their reference
//    max, and writes the normalised rows through shared memory with TMA
//    stores.
// Only P crosses between the CTAs (16 KB per page plus 1 KB of factors per
// pair); no score or exponential is computed twice.
//
// Loads are few and large: the TMA engine streams whole 24-32 KB boxes at
// close to HBM speed but only about half of that as 8 KB boxes. Key tiles use
// a 4-D view of the cache, [8-key group][64-dim chunk][8 keys][64 dims], so
// one 24 KB box brings three chunks of a page; the two pages of a pair go
// back to back into one 48 KB ring slot, which is then a valid 128-key MMA
// operand (8-key groups 3 KB apart). A batch's query comes through the same
// ring (three 48 KB boxes of 128 rows) and tcgen05.cp moves it into TMEM.
// Value CTA per page: two 32 KB boxes of [64 keys x 256 value columns], read
// as an MN-major operand.
// Roles (10 warps per CTA): warps 0-7 softmax (score CTA) or O rescale and
// epilogue (value CTA), two warps per TMEM lane quadrant - on the score CTA
// warp half h owns page h of a pair, on the value CTA O columns
// [256 h, 256 h + 256); warp 8 TMA producer; warp 9 MMA issuer and TMEM owner.
// Every wait is bounded; on expiry the kernel records MLA_ERR_TIMEOUT, tells
// the peer CTA, drains its copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <math.h>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 320;
constexpr int kRows = 128;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;

// ---- shared memory (offsets from a 1024-byte-aligned base) ----
constexpr int kChunkBytes = kPage * 128;         // [64 rows x 64 bf16], 128-byte swizzle
constexpr int kGroupChunks = 3;                  // 64-dim chunks per key box
constexpr int kBoxBytes = kGroupChunks * kChunkBytes;  // one page, three chunks: [8 groups][3 chunks][8 x 128 B]
constexpr int kSlotBytes = 2 * kBoxBytes;        // two pages (or 128 query rows), three chunks
constexpr int kGroupStride = kGroupChunks * 1024;      // bytes between 8-row groups inside a slot
constexpr int kQRopeBytes = kRows * 128;         // [128 rows x 64 rope dims]
constexpr int kOffBars = 0;
constexpr int kOffX = 1024;                      // score: row-stat exchange; value: rescale factors and 1/l
constexpr int kOffRole = 3072;
// score CTA
constexpr int kRing = 4;
constexpr int kOffQRope = kOffRole;              // 2 buffers (batch parity) of the 64 rope query dims
constexpr int kOffRing = kOffQRope + 2 * kQRopeBytes;
constexpr int kSmemScore = kOffRing + kRing * kSlotBytes;
// value CTA
constexpr int kPSlotBytes = 2 * kRows * 128;     // P of a page pair: two K-chunks [128 rows x 64 keys] bf16
constexpr int kVRing = 4;
constexpr int kVSlotBytes = 4 * kChunkBytes;     // [64 keys x 256 value columns]
constexpr int kOffP = kOffRole;
constexpr int kOffV = kOffP + 2 * kPSlotBytes;
constexpr int kSmemValue = kOffV + kVRing * kVSlotBytes;
constexpr int kSmemBytes = kSmemScore > kSmemValue ? kSmemScore : kSmemValue;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
// one P message: P (32 KB) + rescale factor and 1/l per row (fp32)
constexpr uint32_t kPMsgBytes = kPSlotBytes + 2 * kRows * 4;

// ---- tensor memory ----
constexpr uint32_t kTmemQ = 0;      // score CTA: query dims [0, 512) as bf16 pairs (256 columns)
constexpr uint32_t kTmemS0 = 256;   // score CTA: S buffers, 128 columns each
constexpr uint32_t kTmemS1 = 384;
constexpr uint32_t kTmemCols = 512; // value CTA: O, all columns

constexpr int kPrefetchPairs = 3;  // L2 prefetch distance of the score CTA's producer, in page pairs

constexpr float kRescaleThreshold = 8.0f;  // log2 units: tolerate growth up to 2^8 before rescaling O

struct Bars {
    // score CTA
    uint64_t ring_full[kRing], ring_empty[kRing];
    uint64_t qr_full[2], qr_empty[2];
    uint64_t q_drained;
    uint64_t s_full[2], s_free[2];
    uint64_t p_free[2];  // score CTA; arrivals come from the value CTA
    // value CTA
    uint64_t p_full[2];  // own arrive + expect_tx, bytes from the score CTA
    uint64_t v_full[kVRing], v_empty[kVRing];
    uint64_t pv_done, o_full, o_ack[2], o_free[2], stage_done;  // o_ack per P slot: the O warps can run one
                                                                 // pair ahead, never two on the same slot
    uint64_t drain;
    uint32_t tmem_slot;
    int abort;
};
static_assert(sizeof(Bars) <= kOffX, "barrier block");

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

// Walks the page pairs of a part in order: pages [j, j + np) of item `it`,
// np in {1, 2}; pairs never straddle two items.
struct PairIter {
    ItemIter items;
    Item it;
    int j, np, n, n_items;  // first page, pages in the pair, pair counter, items started
    bool valid;
    __device__ void init(const DecodeArgs& args, int part) {
        items.init(args, part);
        n = 0;
        n_items = 0;
        valid = items.next(it);
        if (valid) {
            n_items = 1;
            j = it.lo;
            np = min(2, it.hi - j);
        }
    }
    __device__ bool first_of_item() const { return j == it.lo; }
    __device__ bool last_of_item() const { return j + np >= it.hi; }
    __device__ void advance() {
        ++n;
        j += np;
        if (j >= it.hi) {
            valid = items.next(it);
            if (!valid) return;
            j = it.lo;
            ++n_items;
        }
        np = min(2, it.hi - j);
    }
};

__device__ __forceinline__ int visible_keys(int seqlen, int s_q, int s, int causal) {
    int n = causal ? seqlen - s_q + s + 1 : seqlen;
    return n < 0 ? 0 : (n > seqlen ? seqlen : n);
}

__device__ __forceinline__ int checked_block(const DecodeArgs& args, int b, int j, int* err) {
    int blk = j < args.mbps ? args.block_table[(size_t)b * args.mbps + j] : -1;
    if (blk < 0 || blk >= args.num_blocks) {
        record_error(err, kErrBadBlock);
        blk = 0;
    }
    return blk;
}

// Waits for the last TMA load issued into each of the `slots` buffers of a
// ring that has seen `issued` loads, so that no copy is in flight at exit.
__device__ __forceinline__ void drain_ring(uint64_t* full, int slots, int issued, int* err) {
    for (int r = issued - slots > 0 ? issued - slots : 0; r < issued; ++r)
        mbar_wait(&full[r % slots], (r / slots) & 1, nullptr, err, kDrainNs);
}

// ============================================================== score CTA ==
__device__ void score_producer(const DecodeMaps& maps, const DecodeArgs& args, Bars* bars, uint8_t* smem, int part,
                               int s, volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    uint8_t* ring = smem + kOffRing;
    const int hq = min(args.H, kRows);
    const uint32_t qbytes = (uint32_t)hq * 128;                    // rope box
    const uint32_t qgbytes = (uint32_t)hq * 128 * kGroupChunks;   // query chunk-group box
    PairIter pi;
    pi.init(args, part);
    // The ring holds 1.3 pairs, far less than HBM latency times this CTA's share
    // of the bandwidth; whole pages (contiguous 72 KB) are therefore requested
    // into L2 kPrefetchPairs ahead, and the ring refills from L2.
    PairIter pf;
    pf.init(args, part);
    auto prefetch_pair = [&]() {
        if (!pf.valid) return;
        for (int p = 0; p < pf.np; ++p) {
            const int j = pf.j + p;
            const int blk = j < args.mbps ? args.block_table[(size_t)pf.it.b * args.mbps + j] : -1;
            if (blk >= 0 && blk < args.num_blocks)
                prefetch_l2_bulk(static_cast<const uint8_t*>(args.kv) + (size_t)blk * kPage * kDQK * 2, kPage * kDQK * 2);
        }
        pf.advance();
    };
    for (int i = 0; i < kPrefetchPairs; ++i) prefetch_pair();
    bool ok = true;
    int r = 0, nq = 0;  // ring loads issued, rope query loads issued
    for (; ok && pi.valid; pi.advance()) {
        prefetch_pair();
        const int bs = pi.it.b * args.s_q + s;
        if (pi.first_of_item()) {
            // the batch's query: dims [0, 576) through the ring, three chunks per
            // slot (the MMA warp moves dims [0, 512) into TMEM), and the rope dims
            // into the rope buffer of its parity
            for (int g = 0; g < 3; ++g, ++r) {
                if (r >= kRing) ok = mbar_wait(&bars->ring_empty[r % kRing], ((r / kRing) - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                uint64_t* bar = &bars->ring_full[r % kRing];
                mbar_arrive_expect_tx(bar, qgbytes);
                tma_load_4d(ring + (r % kRing) * kSlotBytes, &maps.qg, bar, 0, 0, kGroupChunks * g, bs * args.H / 8);
            }
            if (!ok) break;
            const int qi = pi.n_items - 1;
            if (qi >= 2) ok = mbar_wait(&bars->qr_empty[qi & 1], ((qi >> 1) - 1) & 1, abort, err, wait_ns);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars->qr_full[qi & 1], qbytes);
            tma_load_3d(smem + kOffQRope + (qi & 1) * kQRopeBytes, &maps.q, &bars->qr_full[qi & 1], 512, 0, bs);
            ++nq;
        }
        const int blk0 = checked_block(args, pi.it.b, pi.j, err);
        const int blk1 = pi.np == 2 ? checked_block(args, pi.it.b, pi.j + 1, err) : 0;
        for (int g = 0; g < 3; ++g, ++r) {
            if (r >= kRing) ok = mbar_wait(&bars->ring_empty[r % kRing], ((r / kRing) - 1) & 1, abort, err, wait_ns);
            if (!ok) break;
            uint8_t* dst = ring + (r % kRing) * kSlotBytes;
            uint64_t* bar = &bars->ring_full[r % kRing];
            mbar_arrive_expect_tx(bar, (uint32_t)pi.np * kBoxBytes);
            tma_load_4d(dst, &maps.kg, bar, 0, 0, kGroupChunks * g, blk0 * (kPage / 8));
            if (pi.np == 2) tma_load_4d(dst + kBoxBytes, &maps.kg, bar, 0, 0, kGroupChunks * g, blk1 * (kPage / 8));
        }
    }
    drain_ring(bars->ring_full, kRing, r, err);
    drain_ring(bars->qr_full, 2, nq, err);
}

// Returns false when it gave up (timeout or abort).
__device__ bool score_mma(const DecodeArgs& args, Bars* bars, uint8_t* smem, uint32_t tmem, int part,
                          volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    const int lane = threadIdx.x & 31;
    uint8_t* ring = smem + kOffRing;
    constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, 2 * kPage, false, false);
    PairIter pi;
    pi.init(args, part);
    bool ok = true, issued = false;
    int r = 0;
    for (; ok && pi.valid; pi.advance()) {
        const int n = pi.n, buf = n & 1, qi = pi.n_items - 1;
        if (pi.first_of_item()) {
            // the previous batch's last score product has finished reading the query
            if (qi > 0) ok = warp_wait(&bars->q_drained, (qi - 1) & 1, abort, err, wait_ns);
            for (int g = 0; ok && g < 3; ++g, ++r) {
                ok = warp_wait(&bars->ring_full[r % kRing], (r / kRing) & 1, abort, err, wait_ns);
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t base = smem_u32(ring + (r % kRing) * kSlotBytes);
                    // chunks 3g .. 3g + 2 of the query; chunk 8 (rope) stays in shared memory
                    for (int cc = 0; cc < kGroupChunks; ++cc) {
                        const int c = kGroupChunks * g + cc;
                        if (c >= 8) break;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tmem_cp_128x256b(tmem + kTmemQ + 32u * c + 8u * kk,
                                             desc_sw128(base + cc * 1024 + 32 * kk, 0, kGroupStride));
                    }
                    mma_commit(&bars->ring_empty[r % kRing]);
                }
                __syncwarp();
                issued = true;
            }
            if (ok) ok = warp_wait(&bars->qr_full[qi & 1], (qi >> 1) & 1, abort, err, wait_ns);
            if (!ok) break;
        }
        // S buffer `buf` was read by the softmax of pair n - 2
        if (n >= 2) ok = warp_wait(&bars->s_free[buf], ((n >> 1) - 1) & 1, abort, err, wait_ns);
        if (!ok) break;
        const uint32_t d = tmem + (buf ? kTmemS1 : kTmemS0);
        const uint32_t rope = smem_u32(smem + kOffQRope + (qi & 1) * kQRopeBytes);
        for (int g = 0; g < 3; ++g, ++r) {
            ok = warp_wait(&bars->ring_full[r % kRing], (r / kRing) & 1, abort, err, wait_ns);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t base = smem_u32(ring + (r % kRing) * kSlotBytes);
#pragma unroll
                for (int cc = 0; cc < kGroupChunks; ++cc) {
                    const int c = kGroupChunks * g + cc;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // keys 0-63 from the first page, 64-127 from the second (8-key groups 3 KB apart)
                        const uint64_t bd = desc_sw128(base + cc * 1024 + 32 * kk, 0, kGroupStride);
                        const uint32_t acc = (c | kk) != 0 ? 1u : 0u;
                        if (c < 8)
                            mma_bf16_ts(d, tmem + kTmemQ + 32u * c + 8u * kk, bd, idesc_s, acc);
                        else
                            mma_bf16_ss(d, desc_sw128(rope + 32 * kk, 0, 1024), bd, idesc_s, acc);
                    }
                }
                mma_commit(&bars->ring_empty[r % kRing]);
            }
            __syncwarp();
            issued = true;
        }
        if (!ok) break;
        if (lane == 0) {
            mma_commit(&bars->s_full[buf]);
            if (pi.last_of_item()) {
                mma_commit(&bars->q_drained);
                mma_commit(&bars->qr_empty[qi & 1]);
            }
        }
        __syncwarp();
    }
    // every MMA and copy this warp issued has completed before TMEM is freed
    if (issued) {
        if (lane == 0) mma_commit(&bars->drain);
        __syncwarp();
        warp_wait(&bars->drain, 0, nullptr, err, kDrainNs);
    }
    return ok;
}

__device__ bool score_softmax(const DecodeArgs& args, Bars* bars, uint8_t* smem, uint32_t tmem, int part, int s,
                              uint32_t peer, volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    const int pair_bar = 1 + quad;  // named barrier of the two warps sharing these rows
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    // the value CTA's P slots, factor arrays and P barriers (same offsets there)
    const uint32_t p_remote = mapa_shared(smem_u32(smem + kOffP), peer);
    const uint32_t x_remote = mapa_shared(smem_u32(smem + kOffX), peer);
    const uint32_t pfull_remote = mapa_shared(smem_u32(&bars->p_full[0]), peer);
    float* xch = reinterpret_cast<float*>(smem + kOffX);  // [2 episodes][2 halves][128 rows]
    PairIter pi;
    pi.init(args, part);
    float m = -INFINITY, l = 0.f;
    int n_valid = 0, xe = 0;
    bool ok = true;
    for (; pi.valid; pi.advance()) {
        // every exit goes through a pair barrier, so both warps of a pair leave together
        const int n = pi.n, buf = n & 1, k = n & 1;
        const bool first = pi.first_of_item(), last = pi.last_of_item();
        if (first) {
            m = -INFINITY;
            l = 0.f;
            n_valid = visible_keys(pi.it.seqlen, args.s_q, s, args.causal);
        }
        float x[64];
        if (ok) ok = warp_wait(&bars->s_full[buf], (n >> 1) & 1, abort, err, wait_ns);
        if (ok) {
            tc_fence_after();
            const uint32_t col = tmem + lane_base + (buf ? kTmemS1 : kTmemS0) + 64u * half;
            uint32_t v[32];
            tmem_ld32(col, v);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(v[c]) * args.scale_log2;
            tmem_ld32(col + 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) x[32 + c] = __uint_as_float(v[c]) * args.scale_log2;
            tc_fence_before();
            mbar_arrive(&bars->s_free[buf]);
        }
        // keys of this half: page j + half; columns past the visible keys (or of a
        // missing second page) are masked by selection, so garbage never leaks
        const int vcount = half < pi.np ? min(max(n_valid - (pi.j + half) * kPage, 0), kPage) : 0;
        float mh = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            x[c] = c < vcount ? x[c] : -INFINITY;
            mh = fmaxf(mh, x[c]);
        }
        float* xb = xch + (xe & 1) * (2 * kRows);
        ++xe;
        xb[half * kRows + row] = mh;
        ok = barrier_and(pair_bar, 64, ok);
        if (!ok) break;
        const float mx = fmaxf(mh, xb[(half ^ 1) * kRows + row]);
        // lazy rescale: the reference max moves only when the row max exceeds it
        // by more than 2^8; both warps of a pair take the same decision
        const bool need = mx > m + kRescaleThreshold;
        const float alpha = need ? fast_exp2(m - mx) : 1.f;  // 0 when m = -inf
        if (need) {
            l *= alpha;
            m = mx;
        }
        const float m_use = m == -INFINITY ? 0.f : m;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            // the row sum takes the fp32 probabilities; only the P.V operand is bf16
            const float p0 = fast_exp2(x[2 * c] - m_use), p1 = fast_exp2(x[2 * c + 1] - m_use);
            l += p0 + p1;
            pk[c] = pack_bf16x2(p0, p1);
        }
        // slot k held pair n - 2 until the value CTA released it
        if (ok && n >= 2) ok = warp_wait(&bars->p_free[k], ((n >> 1) - 1) & 1, abort, err, wait_ns);
        const uint32_t mbar = pfull_remote + (uint32_t)k * 8u;
        if (ok) {
            // row `row` of K-chunk `half`: 16-byte word q at position q ^ (row % 8)
            const uint32_t dst = p_remote + (uint32_t)(k * kPSlotBytes + half * kRows * 128 + row * 128);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                st_async_u4(dst + (uint32_t)((q ^ (row & 7)) << 4), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                            pk[4 * q + 3], mbar);
            if (half == 0)
                st_async_b32(x_remote + (uint32_t)(k * 1024 + row * 4), __float_as_uint(row < args.H ? alpha : 1.f),
                             mbar);
        }
        if (last) {
            // the pair adds its two half sums (half 0 + half 1) for 1/l and lse
            xb = xch + (xe & 1) * (2 * kRows);
            ++xe;
            xb[half * kRows + row] = l;
            ok = barrier_and(pair_bar, 64, ok);
            if (!ok) break;
            const float lo = xb[(half ^ 1) * kRows + row];
            const float l_row = half == 0 ? l + lo : lo + l;
            if (half == 0) {
                const float inv_l = l_row > 0.f ? 1.f / l_row : 0.f;
                st_async_b32(x_remote + (uint32_t)(k * 1024 + 512 + row * 4), __float_as_uint(inv_l), mbar);
                if (row < args.H) {
                    // lse in natural log: x is in log2 units of the scaled score
                    const float lse_v = l_row > 0.f ? (m + log2f(l_row)) * 0.69314718055994530942f : -INFINITY;
                    if (pi.it.split)
                        args.lse_part[((size_t)pi.it.piece * args.s_q + s) * args.H + row] = lse_v;
                    else
                        args.lse[((size_t)pi.it.b * args.s_q + s) * args.H + row] = lse_v;
                }
            }
        } else if (ok && half == 0) {
            st_async_b32(x_remote + (uint32_t)(k * 1024 + 512 + row * 4), 0u, mbar);
        }
    }
    return ok;
}

// ============================================================== value CTA ==
__device__ void value_producer(const DecodeMaps& maps, const DecodeArgs& args, Bars* bars, uint8_t* smem, int part,
                               volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    uint8_t* vring = smem + kOffV;
    PairIter pi;
    pi.init(args, part);
    bool ok = true;
    int v = 0;
    for (; ok && pi.valid; pi.advance()) {
        for (int p = 0; ok && p < pi.np; ++p) {
            const int blk = checked_block(args, pi.it.b, pi.j + p, err);
            for (int h = 0; h < 2; ++h, ++v) {
                if (v >= kVRing) ok = mbar_wait(&bars->v_empty[v % kVRing], ((v / kVRing) - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                uint8_t* dst = vring + (v % kVRing) * kVSlotBytes;
                uint64_t* bar = &bars->v_full[v % kVRing];
                mbar_arrive_expect_tx(bar, (uint32_t)kVSlotBytes);
                tma_load_3d(dst, &maps.v, bar, 0, blk * kPage, 4 * h);
            }
        }
    }
    drain_ring(bars->v_full, kVRing, v, err);
}

__device__ bool value_mma(const DecodeArgs& args, Bars* bars, uint8_t* smem, uint32_t tmem, int part,
                          volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    const int lane = threadIdx.x & 31;
    uint8_t* vring = smem + kOffV;
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, 256, false, true);
    PairIter pi;
    pi.init(args, part);
    bool ok = true, issued = false;
    int v = 0;
    for (; ok && pi.valid; pi.advance()) {
        const int n = pi.n, k = n & 1, qi = pi.n_items - 1;
        const bool first = pi.first_of_item(), last = pi.last_of_item();
        ok = warp_wait<true>(&bars->p_full[k], (n >> 1) & 1, abort, err, wait_ns);
        if (!ok) break;
        if (lane == 0) {
            // P was written by the peer's generic stores: make it visible to the
            // tensor pipe, then arm the slot for pair n + 2 (its bytes can only
            // come after this pair has released the slot)
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars->p_full[k], kPMsgBytes);
        }
        __syncwarp();
        // the O warps have read this message's factors (and rescaled O if asked)
        ok = warp_wait(&bars->o_ack[k], (n >> 1) & 1, abort, err, wait_ns);
        if (!ok) break;
        for (int p = 0; ok && p < pi.np; ++p) {
            const int page = pi.j + p;
            const int tail = page == pi.it.nblk - 1 ? pi.it.seqlen - page * kPage : kPage;
            for (int h = 0; h < 2; ++h, ++v) {
                // a batch's first product overwrites O: its previous epilogue must have read it
                if (first && p == 0 && qi > 0) ok = warp_wait(&bars->o_free[h], (qi - 1) & 1, abort, err, wait_ns);
                if (ok) ok = warp_wait(&bars->v_full[v % kVRing], (v / kVRing) & 1, abort, err, wait_ns);
                if (!ok) break;
                uint8_t* vs = vring + (v % kVRing) * kVSlotBytes;
                if (tail < kPage) {
                    // rows past seqlen hold arbitrary bytes: zero them so that
                    // 0-probability keys cannot inject NaN/Inf into P.V
                    const int per_chunk = (kPage - tail) * 8;  // 16-byte words
                    for (int i = lane; i < 4 * per_chunk; i += 32) {
                        const int c = i / per_chunk, w = i % per_chunk;
                        reinterpret_cast<uint4*>(vs + c * kChunkBytes + tail * 128)[w] = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a_base = smem_u32(smem + kOffP + k * kPSlotBytes + p * kRows * 128);
                    const uint32_t v_base = smem_u32(vs);
#pragma unroll
                    for (int kk = 0; kk < kPage / 16; ++kk)
                        mma_bf16_ss(tmem + 256u * h, desc_sw128(a_base + 32 * kk, 0, 1024),
                                    desc_sw128(v_base + 2048 * kk, kChunkBytes, 1024), idesc_pv,
                                    (first && p == 0 && kk == 0) ? 0u : 1u);
                    mma_commit(&bars->v_empty[v % kVRing]);
                }
                __syncwarp();
                issued = true;
            }
        }
        if (!ok) break;
        if (lane == 0) {
            mma_commit(&bars->pv_done);
            if (last)
                mma_commit(&bars->o_full);  // the epilogue hands the slot back after staging in it
            else
                mma_commit_multicast(&bars->p_free[k], (uint16_t)1u);  // arrives on the score CTA (rank 0)
        }
        __syncwarp();
    }
    if (issued) {
        if (lane == 0) mma_commit(&bars->drain);
        __syncwarp();
        warp_wait(&bars->drain, 0, nullptr, err, kDrainNs);
    }
    return ok;
}

__device__ bool value_owarps(const DecodeMaps& maps, const DecodeArgs& args, Bars* bars, uint8_t* smem,
                             uint32_t tmem, int part, int s, uint32_t peer, volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float* xv = reinterpret_cast<const float*>(smem + kOffX);  // [slot][factor 128 | 1/l 128]
    const uint32_t ocol = tmem + lane_base + 256u * (uint32_t)half;
    PairIter pi;
    pi.init(args, part);
    bool ok = true;
    bool stored = false;
    for (; ok && pi.valid; pi.advance()) {
        const int n = pi.n, k = n & 1, qi = pi.n_items - 1;
        const bool first = pi.first_of_item(), last = pi.last_of_item();
        ok = warp_wait<true>(&bars->p_full[k], (n >> 1) & 1, abort, err, wait_ns);
        if (!ok) break;
        const float inv_l = xv[k * 256 + 128 + row];
        if (!first) {
            const float alpha = xv[k * 256 + row];
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
                // O rows of this warp move to the new reference max (after the
                // previous P.V product has landed)
                ok = warp_wait(&bars->pv_done, (n - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 256; c += 32) {
                    uint32_t v[32];
                    tmem_ld32(ocol + c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st32(ocol + c, v);
                }
                tmem_wait_st();
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_ack[k]);
        if (!last) continue;

        // ---- epilogue of the item: O * (1/l) -> staging (the pair's P slot) -> TMA store
        ok = warp_wait(&bars->o_full, qi & 1, abort, err, wait_ns);
        if (!ok) break;
        tc_fence_after();
        const Item& it = pi.it;
        const bool store = quad * 32 < args.H;
        uint8_t* stage = smem + kOffP + k * kPSlotBytes + warp * 4096;  // [32 rows x 128 B], 128-byte swizzle
        uint8_t* srow = stage + lane * 128;
        if (!it.split) {
            const int z = it.b * args.s_q + s;
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                const int col = 64 * i;
                uint32_t v0[32], v1[32];
                tmem_ld32(ocol + col, v0);
                tmem_ld32(ocol + col + 32, v1);
                tmem_wait_ld();
                if (!store) continue;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 w0, w1;
                    w0.x = pack_bf16x2(__uint_as_float(v0[8 * q + 0]) * inv_l, __uint_as_float(v0[8 * q + 1]) * inv_l);
                    w0.y = pack_bf16x2(__uint_as_float(v0[8 * q + 2]) * inv_l, __uint_as_float(v0[8 * q + 3]) * inv_l);
                    w0.z = pack_bf16x2(__uint_as_float(v0[8 * q + 4]) * inv_l, __uint_as_float(v0[8 * q + 5]) * inv_l);
                    w0.w = pack_bf16x2(__uint_as_float(v0[8 * q + 6]) * inv_l, __uint_as_float(v0[8 * q + 7]) * inv_l);
                    w1.x = pack_bf16x2(__uint_as_float(v1[8 * q + 0]) * inv_l, __uint_as_float(v1[8 * q + 1]) * inv_l);
                    w1.y = pack_bf16x2(__uint_as_float(v1[8 * q + 2]) * inv_l, __uint_as_float(v1[8 * q + 3]) * inv_l);
                    w1.z = pack_bf16x2(__uint_as_float(v1[8 * q + 4]) * inv_l, __uint_as_float(v1[8 * q + 5]) * inv_l);
                    w1.w = pack_bf16x2(__uint_as_float(v1[8 * q + 6]) * inv_l, __uint_as_float(v1[8 * q + 7]) * inv_l);
                    *reinterpret_cast<uint4*>(srow + ((q ^ (lane & 7)) << 4)) = w0;
                    *reinterpret_cast<uint4*>(srow + (((q + 4) ^ (lane & 7)) << 4)) = w1;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&maps.o, stage, 256 * half + col, quad * 32, z);
                    bulk_commit_group();
                    bulk_wait_group_read0();
                }
                __syncwarp();
                stored = true;
            }
        } else {
            const int z = it.piece * args.s_q + s;
#pragma unroll 1
            for (int i = 0; i < 8; ++i) {
                const int col = 32 * i;
                uint32_t v0[32];
                tmem_ld32(ocol + col, v0);
                tmem_wait_ld();
                if (!store) continue;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float4 w;
                    w.x = __uint_as_float(v0[4 * q + 0]) * inv_l;
                    w.y = __uint_as_float(v0[4 * q + 1]) * inv_l;
                    w.z = __uint_as_float(v0[4 * q + 2]) * inv_l;
                    w.w = __uint_as_float(v0[4 * q + 3]) * inv_l;
                    *reinterpret_cast<float4*>(srow + ((q ^ (lane & 7)) << 4)) = w;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&maps.op, stage, 256 * half + col, quad * 32, z);
                    bulk_commit_group();
                    bulk_wait_group_read0();
                }
                __syncwarp();
                stored = true;
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&bars->o_free[half]);
            mbar_arrive(&bars->stage_done);
        }
        if (warp == 0) {
            // all eight warps are done with the staging area: give the P slot back
            ok = warp_wait(&bars->stage_done, qi & 1, abort, err, wait_ns);
            if (ok && lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&bars->p_free[k]), peer));
            __syncwarp();
        }
    }
    if (stored && lane == 0) bulk_wait_group0();
    return ok;
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeMaps maps, DecodeArgs args) {
    extern __shared__ __align__(16) uint8_t smem[];
    Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);
    volatile int* abort = &bars->abort;

    const int warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int cluster_id = blockIdx.x >> 1;
    const int part = cluster_id / args.s_q;
    const int s = cluster_id % args.s_q;

    // the layout needs 1024-byte-aligned swizzle atoms and leaves no room to
    // realign; both CTAs see the same base and leave together
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) record_error(args.err, kErrUnsupported);
        cluster_sync_all();
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bars->ring_full[i], 1);
            mbar_init(&bars->ring_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->qr_full[i], 1);
            mbar_init(&bars->qr_empty[i], 1);
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_free[i], 256);
            mbar_init(&bars->p_free[i], 1);
            mbar_init(&bars->p_full[i], 1);
            mbar_init(&bars->o_free[i], 4);
            mbar_init(&bars->o_ack[i], 8);
        }
        mbar_init(&bars->q_drained, 1);
        for (int i = 0; i < kVRing; ++i) {
            mbar_init(&bars->v_full[i], 1);
            mbar_init(&bars->v_empty[i], 1);
        }
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->o_full, 1);
        mbar_init(&bars->stage_done, 8);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init_cluster();
        if (rank == 0) {
            tma_prefetch_desc(&maps.kg);
            tma_prefetch_desc(&maps.qg);
            tma_prefetch_desc(&maps.q);
        } else {
            tma_prefetch_desc(&maps.v);
            tma_prefetch_desc(&maps.o);
            tma_prefetch_desc(&maps.op);
            // the first two P messages may arrive as soon as the cluster is up
            mbar_arrive_expect_tx(&bars->p_full[0], kPMsgBytes);
            mbar_arrive_expect_tx(&bars->p_full[1], kPMsgBytes);
        }
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

    bool ok = true;
    if (rank == 0) {
        if (warp == kWarpProducer) {
            if ((threadIdx.x & 31) == 0) score_producer(maps, args, bars, smem, part, s, abort);
        } else if (warp == kWarpMma) {
            ok = score_mma(args, bars, smem, tmem, part, abort);
        } else {
            ok = score_softmax(args, bars, smem, tmem, part, s, peer, abort);
        }
    } else {
        if (warp == kWarpProducer) {
            if ((threadIdx.x & 31) == 0) value_producer(maps, args, bars, smem, part, abort);
        } else if (warp == kWarpMma) {
            ok = value_mma(args, bars, smem, tmem, part, abort);
        } else {
            ok = value_owarps(maps, args, bars, smem, tmem, part, s, peer, abort);
        }
    }
    // a role that gave up tells the peer, whose waits then end promptly
    if (!ok || *abort) st_cluster_b32(mapa_shared(smem_u32(&bars->abort), peer), 1u);

    tc_fence_before();
    __syncthreads();
    // the peer may still store into our buffers or arrive on our barriers until
    // it has finished its last pair: leave together
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

cudaError_t launch_decode(const DecodeMaps& maps, const DecodeArgs& args, cudaStream_t stream) {
    cudaError_t e = prepare_kernel();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = make_config(args.num_parts * args.s_q, stream, attr, true);
    return cudaLaunchKernelEx(&cfg, decode_kernel, maps, args);
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
