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
//    current batch in TMEM (576 dims as the A operand), computes S = Q' K^T
//    page by page (N = 64 keys) into one of three TMEM buffers, and its softmax
//    threads mask, take the row max, rescale lazily, exponentiate and ship P
//    (bf16, as a K-major operand tile without swizzle, so that every warp
//    instruction writes 512 contiguous bytes) together with the per-row
//    rescale factor straight into one of the value CTA's three P slots
//    (st.async, counted on the value CTA's mbarrier);
//  * the value CTA (rank 1) keeps the fp32 output O [128 x 512] in its TMEM
//    (all 512 columns), loads its own copy of the page's value columns (mostly
//    L2 hits: the score CTA has just read the same page), accumulates
//    O += P . V, rescales O rows when the score CTA moved their reference max,
//    and writes the normalised rows with 64 KB TMA stores, staged in the value
//    slot of the item's last page (free once its P.V product is done).
// Only P crosses between the CTAs (16 KB plus 1 KB of factors per page); no
// score or exponential is computed twice.
//
// Loads are few and large: the TMA engine of an SM works through boxes with a
// high fixed cost per box, so a whole page (9 chunks of [64 keys x 64 dims],
// one 3-D box over a [dims, keys, chunk] view of the cache) is a single load;
// 8 KB boxes would stream at a fifth of the rate. The query of a new batch
// arrives the same way (two boxes of 64 rows) and the softmax threads move it
// into TMEM.
// Roles (19 warps per CTA). Score CTA: warps 0-15 softmax in two groups of
// eight that take alternate pages (page n goes to group n % 2), two warps of a
// group per TMEM lane quadrant, warp half h owning keys [32 h, 32 h + 32) of a
// page; warp 16 TMA producer; warp 17 issues the score products and owns
// TMEM (warp 18 can take the odd pages: kScoreMmaWarps). Value CTA: warps 0-7 O rescale and
// epilogue, two per lane quadrant, warp half h owning O columns
// [256 h, 256 h + 256); warp 16 TMA producer; warp 17 P.V issuer and TMEM
// owner; over the INT8 cache warps 8-15 expand the value codes to bf16 in
// place; in the instantiation that runs when no merge kernel follows, warp 18
// writes the rows of empty sequences; the other warps have no role.
// Over the INT8 cache (records of 512 codes + 64 bf16 rope columns and a
// per-token scale) both CTAs load the records and expand them to bf16 in
// shared memory before their products.
// Every wait is bounded; on expiry the kernel records MLA_ERR_TIMEOUT, tells
// the peer CTA, drains its copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

#include "mla_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace mla {
namespace {

// Warps: 0-15 softmax (score CTA; two groups of eight, one per page parity)
// or 0-7 O rescale and epilogue (value CTA), 16 TMA producer, 17 MMA issuer
// and TMEM owner (score CTA: even pages), 18 second score MMA issuer (odd
// pages; idle on the value CTA).
constexpr int kThreads = 608;
constexpr int kRows = 128;
// Softmax groups on the score CTA: 2 (warps 0-15, alternate pages) or 1
// (warps 0-7 take every page; 8-15 have no role).
constexpr int kSoftmaxGroups = 2;
constexpr int kSoftmaxWarps = 8 * kSoftmaxGroups;
constexpr int kOWarps = 8;
constexpr int kWarpProducer = 16;
constexpr int kWarpMma = 17;
constexpr int kWarpMma2 = 18;
// Score-MMA issuing warps: 1 (warp 17 issues every page) or 2 (warps 17 and
// 18 take the even and odd pages). Issued warp-uniformly, one warp keeps the
// tensor pipe at its N = 64 rate (about 33 cycles a product), and one issuer
// finishes each page's products soonest, which frees its ring slot soonest.
constexpr int kScoreMmaWarps = 1;
constexpr int kChunks = kDQK / 64;  // 9 chunks of 64 dims

// ---- shared memory (offsets from a 1024-byte-aligned base) ----
constexpr int kChunkBytes = kPage * 128;           // [64 rows x 64 bf16], 128-byte swizzle
constexpr int kPageBytes = kChunks * kChunkBytes;  // a page (or 64 query rows): [9 chunks][64 rows][64 dims]
constexpr int kOffBars = 0;
constexpr int kOffX = 1024;                        // score: row-stat exchange; value: rescale factors and 1/l
// score CTA exchange area (floats, from kOffX):
constexpr int kXPair = 0;                          // [group][episode 2][half 2][128]: the pair's half-row values
constexpr int kXRef = kXPair + 2 * 2 * 2 * kRows;  // [page parity][128]: reference max after a page
constexpr int kXLSum = kXRef + 2 * kRows;          // [group][half][128]: a group's share of the row sum
constexpr int kXLMax = kXLSum + 2 * 2 * kRows;     // [group][128]: the reference max that share is relative to
constexpr int kXFloats = kXLMax + 2 * kRows;
static_assert(kOffX + 4 * kXFloats <= 9216, "exchange area");
// INT8 cache: the per-token scales of the page in each ring (or value) slot, 64 floats a slot
constexpr int kOffScale = 9216;
constexpr int kScaleBytes = kPage * 4;
constexpr int kOffRole = 10240;
// score CTA
constexpr int kRing = 3;
constexpr int kOffRing = kOffRole;
constexpr int kSmemScore = kOffRing + kRing * kPageBytes;
// value CTA
// P of a page, [128 rows x 64 keys] bf16, K-major without swizzle: eight key
// blocks of 8 keys, each [128 rows][16 B] (core matrices of 8 rows x 16 B are
// 128 contiguous bytes, 128 B apart along the rows and kPBlockBytes apart
// along K). One 16-byte word of P for each of a softmax warp's 32 rows is then
// 512 contiguous bytes.
constexpr int kPSlotBytes = kRows * 128;
constexpr int kPBlockBytes = kRows * 16;
constexpr int kVBytes = 8 * kChunkBytes;           // a page's value columns: [8 chunks][64 keys][64 dims]
constexpr int kVRing = 2;
constexpr int kOffXV = kOffX;                      // value: [P slot][rescale factor 128 | 1/l 128] fp32
constexpr int kOffP = kOffRole;                    // value: kPSlots P slots
// P slots: page n's message goes to slot n % kPSlots. Three let the softmax
// run a page further ahead of the P.V products (1 % faster on the multi-token
// workload; while P still crossed the cluster as 16-byte stores 128 bytes
// apart, a third slot made it 12 % slower).
constexpr int kPSlots = 3;
static_assert(kPSlots <= 3, "two pv_done barriers cover P slots up to three");
constexpr int kOffV = kOffP + kPSlots * kPSlotBytes;  // value: the value ring
constexpr int kSmemValue = kOffV + kVRing * kVBytes;
constexpr int kSmemUsed = kSmemScore > kSmemValue ? kSmemScore : kSmemValue;
constexpr int kSmemBytes = kSmemUsed + 1024;       // room to align the base to 1024 bytes
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kOffP % 1024 == 0 && kOffV % 1024 == 0 && kOffRing % 1024 == 0, "swizzle atoms");
static_assert(kOffXV + kPSlots * 1024 <= kOffScale, "value factor slots");
static_assert(kOffScale + kRing * kScaleBytes <= kOffRole && kOffScale + kVRing * kScaleBytes <= kOffRole, "scales");
// INT8 cache, in a page slot: the codes arrive as four planes [64 keys x 128 B]
// (128-byte swizzle) at kQ8Planes and are expanded in place into the bf16
// chunks 0-7; the score slot's rope key lands directly in chunk 8.
constexpr int kQ8Planes = 4 * kChunkBytes;             // byte offset of the code planes in a slot
constexpr uint32_t kQ8PageBytes = 4 * kChunkBytes + kChunkBytes + kScaleBytes;  // score slot: codes + rope + scales
constexpr uint32_t kQ8VBytes = 4 * kChunkBytes + kScaleBytes;                   // value slot: codes + scales
// one P message: P (16 KB) + rescale factor and 1/l per row (fp32)
constexpr uint32_t kPMsgBytes = kPSlotBytes + 2 * kRows * 4;

// ---- tensor memory ----
constexpr uint32_t kTmemQ = 0;       // score CTA: the 576 query dims as bf16 pairs (288 columns)
constexpr uint32_t kTmemS = 288;     // score CTA: kSBufs S buffers of 64 columns
// S buffers: page n's scores go to buffer n % kSBufs. With three, the score
// products can run two pages ahead of the softmax that frees a buffer.
constexpr int kSBufs = 3;
static_assert(kTmemS + 64 * kSBufs <= 512, "TMEM columns");
constexpr uint32_t kTmemCols = 512;  // value CTA: O, all columns

// After an abort the value CTA waits this long for P messages that may still
// be in flight towards its shared memory (a message lands within a few
// microseconds; one that was only partly sent never completes its phase).
constexpr long long kPDrainNs = 20000;

constexpr float kRescaleThreshold = 8.0f;  // log2 units: tolerate growth up to 2^8 before rescaling O

struct Bars {
    // score CTA
    uint64_t ring_full[kRing], ring_empty[kRing];
    uint64_t q_full, q_drained;
    uint64_t s_full[kSBufs], s_free[kSBufs];
    uint64_t p_free[kPSlots];  // score CTA; arrivals come from the value CTA
    uint64_t ref_full[2][4];  // [page parity][lane quadrant]: reference max of a page published
    uint64_t lsum_full[4];    // [lane quadrant]: the group without an item's last page published its row sums
    uint64_t drain2;          // second score MMA warp
    uint64_t deq_full[2];     // INT8 cache: [page parity] the page is expanded to bf16 in its ring slot
    // value CTA
    uint64_t p_full[kPSlots];  // own arrive + expect_tx, bytes from the score CTA
    uint64_t v_full[kVRing], v_empty[kVRing];
    // [page % 2]: the page's P.V products are done. The O warps wait for page
    // n - 1's before moving O to a new reference max at page n; P(n) arriving
    // means the products of page n - kPSlots are done, so with two barriers the
    // one waited on (last phase: page n - 3) is never two phases behind.
    uint64_t pv_done[2];
    uint64_t o_full;
    uint64_t o_ack[kPSlots];  // per P slot: the O warps have read the slot's factors
    uint64_t o_free[2];  // [O column half]: the epilogue's eight warps have read those columns
    uint64_t stage_full, stage_free;  // epilogue rounds: eight warps staged / staging read by the store
    uint64_t drain;
    uint64_t vdeq_full[kVRing];     // INT8 cache: the value slot is expanded to bf16
    uint32_t tmem_slot;
    int abort;
    int p_consumed;  // value CTA: P messages its MMA warp has taken (their successors are armed)
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

// Walks the pages of a part in order, with their item context.
struct PageIter {
    ItemIter items;
    Item it;
    int j, n, n_items;  // page within the batch, page counter, items started
    bool valid;
    __device__ void init(const DecodeArgs& args, int part) {
        items.init(args, part);
        n = 0;
        n_items = 0;
        valid = items.next(it);
        if (valid) {
            n_items = 1;
            j = it.lo;
        }
    }
    __device__ bool first_of_item() const { return j == it.lo; }
    __device__ bool last_of_item() const { return j == it.hi - 1; }
    __device__ void advance() {
        ++n;
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

// Tells both CTAs of the cluster to give up: every bounded wait of either
// CTA then returns within a few polls instead of running to its limit.
__device__ __forceinline__ void raise_abort(volatile int* abort) {
    *abort = 1;
    st_cluster_b32(mapa_shared(smem_u32(const_cast<int*>(abort)), cluster_ctarank() ^ 1u), 1u);
}

// Block id of page j of batch b. An id outside the pool (or a page past the
// table row) records MLA_ERR_BAD_BLOCK, aborts the cluster and returns block
// 0, so the load that follows stays inside the cache.
__device__ __forceinline__ int checked_block(const DecodeArgs& args, int b, int j, int* err, volatile int* abort) {
    int blk = j < args.mbps ? args.block_table[(size_t)b * args.mbps + j] : -1;
    if (blk < 0 || blk >= args.num_blocks) {
        record_error(err, kErrBadBlock);
        raise_abort(abort);
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

// ============================================================= INT8 cache ==
// Writes the 16 values of code unit u (plane p, key k) as bf16 into the page's
// chunk 2p + u / 4 (128-byte swizzle), or zeros for a key past the valid ones.
__device__ __forceinline__ void q8_store_unit(uint8_t* slot, int p, int k, int u, uint4 codes, float sc, bool live) {
    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
    if (live) q8_dequant16(codes, sc, lo, hi);
    uint8_t* row = slot + (2 * p + (u >> 2)) * kChunkBytes + k * 128;
    const int w0 = 2 * (u & 3);
    *reinterpret_cast<uint4*>(row + ((w0 ^ (k & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(row + (((w0 + 1) ^ (k & 7)) << 4)) = hi;
}

// Expands one page slot in place from INT8 codes to the bf16 page the MMAs read
// (the codes stand for code * scale, exactly representable in bf16). Code
// plane p (dims [128 p, 128 p + 128), [64 keys][128 B], 128-byte swizzle) sits at
// slot + kQ8Planes + 8 KB p and becomes bf16 chunks 2p and 2p + 1 at slot +
// 16 KB p; keys at or past `valid` become zeros. Eight warps share a page, warp
// w8 taking keys [8 w8, 8 w8 + 8) of every plane (8 units of 16 codes per lane).
// Row k of output chunk 4 + p is row k of code plane p, so a warp only
// overwrites code rows of its own keys: it loads all of its codes first, and
// needs no other warp.
__device__ __forceinline__ void q8_expand_warp(uint8_t* slot, const float* sc, int valid, int w8, int lane) {
    const int kr = lane >> 3, u = lane & 7;
    uint4 c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int p = i >> 1, k = 8 * w8 + 4 * (i & 1) + kr;
        c[i] = *reinterpret_cast<const uint4*>(slot + kQ8Planes + p * kChunkBytes + k * 128 + ((u ^ (k & 7)) << 4));
    }
    const float s0 = sc[8 * w8 + kr], s1 = sc[8 * w8 + 4 + kr];
    __syncwarp();  // every lane's codes are in registers before any lane overwrites code rows
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int p = i >> 1, k = 8 * w8 + 4 * (i & 1) + kr;
        q8_store_unit(slot, p, k, u, c[i], (i & 1) ? s1 : s0, k < valid);
    }
}

// ============================================================== score CTA ==
// Ring positions: every batch first takes two positions for its query (rows
// 0-63 and 64-127), then one per page; producer, MMA warp and softmax warps
// count them the same way.
template <bool kQ8>
__device__ void score_producer(const DecodeMaps& maps, const DecodeArgs& args, Bars* bars, uint8_t* smem, int part,
                               int s, volatile int* abort) {
    // the whole warp runs this loop (warp-uniform waits); lane 0 issues the loads
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    const int lane = threadIdx.x & 31;
    uint8_t* ring = smem + kOffRing;
    const uint32_t qbytes = (uint32_t)(kChunks * args.qrows * 128);
    // The part's first batch is the first entry of its schedule row (a part
    // never starts on an empty batch), so its query is requested right after
    // that one read, while the walk below still reads the batch's length.
    const int* trow = args.tile_meta + 8 * part;
    const int b_first = trow[0];
    const bool q_early = trow[5] > 0;
    if (q_early && lane == 0) {
        const int row0 = (b_first * args.s_q + s) * args.H;
        for (int h = 0; h < 2; ++h) {
            mbar_arrive_expect_tx(&bars->ring_full[h], qbytes);
            tma_load_3d(ring + h * kPageBytes, &maps.q, &bars->ring_full[h], 0, row0 + 64 * h, 0);
        }
    }
    __syncwarp();
    PageIter pi;
    pi.init(args, part);
    // a schedule from other sequence lengths could start elsewhere
    if (q_early && lane == 0 && (!pi.valid || pi.it.b != b_first)) {
        record_error(err, kErrBadBlock);
        raise_abort(abort);
    }
    bool ok = true;
    int r = 0;
    for (; ok && pi.valid; pi.advance()) {
        if (pi.first_of_item() && q_early && pi.n_items == 1) {
            r = 2;  // the first query went out above
        } else if (pi.first_of_item()) {
            const int row0 = (pi.it.b * args.s_q + s) * args.H;
            for (int h = 0; h < 2; ++h, ++r) {
                if (r >= kRing) ok = warp_wait(&bars->ring_empty[r % kRing], ((r / kRing) - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                if (lane == 0) {
                    uint64_t* bar = &bars->ring_full[r % kRing];
                    mbar_arrive_expect_tx(bar, qbytes);
                    tma_load_3d(ring + (r % kRing) * kPageBytes, &maps.q, bar, 0, row0 + 64 * h, 0);
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        if (r >= kRing) ok = warp_wait(&bars->ring_empty[r % kRing], ((r / kRing) - 1) & 1, abort, err, wait_ns);
        if (!ok) break;
        if (lane == 0) {
            const int blk = checked_block(args, pi.it.b, pi.j, err, abort);
            uint64_t* bar = &bars->ring_full[r % kRing];
            uint8_t* slot = ring + (r % kRing) * kPageBytes;
            if (kQ8) {
                // codes (four planes), the bf16 rope key straight into chunk 8, the scales
                mbar_arrive_expect_tx(bar, kQ8PageBytes);
                tma_load_3d(slot + kQ8Planes, &maps.kv8, bar, 0, blk * kPage, 0);
                tma_load_2d(slot + 8 * kChunkBytes, &maps.rope, bar, 0, blk * kPage);
                bulk_load(smem + kOffScale + (r % kRing) * kScaleBytes, args.kv_scale + (size_t)blk * kPage,
                          kScaleBytes, bar);
            } else {
                mbar_arrive_expect_tx(bar, (uint32_t)kPageBytes);
                tma_load_3d(slot, &maps.kv, bar, 0, blk * kPage, 0);
            }
        }
        __syncwarp();
        ++r;
    }
    if (q_early && r < 2) r = 2;  // the early query loads land before the CTA may leave
    if (lane == 0) drain_ring(bars->ring_full, kRing, r, err);
    __syncwarp();
}

// Score products of the pages with parity `parity` (0 or 1, when two warps
// share the pages), or of every page (parity < 0). Returns false when it gave
// up (timeout or abort).
template <bool kQ8>
__device__ bool score_mma(const DecodeArgs& args, Bars* bars, uint8_t* smem, uint32_t tmem, int part, int parity,
                          volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    const int lane = threadIdx.x & 31;
    uint8_t* ring = smem + kOffRing;
    constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kPage, false, false);
    uint64_t* drain = parity <= 0 ? &bars->drain : &bars->drain2;
    PageIter pi;
    pi.init(args, part);
    bool ok = true, issued = false;
    int r = 0;
    for (; ok && pi.valid; pi.advance()) {
        const int n = pi.n, buf = n & 1, qi = pi.n_items - 1;
        if (pi.first_of_item()) {
            // the softmax threads have moved the batch's query into TMEM and are
            // done reading its two ring slots
            ok = warp_wait(&bars->q_full, qi & 1, abort, err, wait_ns);
            if (!ok) break;
            if (parity <= 0 && lane == 0) {
                mbar_arrive(&bars->ring_empty[r % kRing]);
                mbar_arrive(&bars->ring_empty[(r + 1) % kRing]);
            }
            __syncwarp();
            r += 2;
        }
        if (parity < 0 || buf == parity) {
            // S buffer `buf` was read by the softmax of page n - 2
            const int sb = n % kSBufs;
            if (n >= kSBufs) ok = warp_wait(&bars->s_free[sb], ((n / kSBufs) - 1) & 1, abort, err, wait_ns);
            // the page has landed (INT8 cache: and its softmax group has expanded it)
            if (ok)
                ok = kQ8 ? warp_wait(&bars->deq_full[n & 1], (n >> 1) & 1, abort, err, wait_ns)
                         : warp_wait(&bars->ring_full[r % kRing], (r / kRing) & 1, abort, err, wait_ns);
            if (!ok) break;
            tc_fence_after();
            // the whole warp runs the issue loop (warp-uniform operands); one
            // elected lane issues. One descriptor per page; a K-step moves its
            // start address field (bytes / 16) by a constant.
            const uint64_t bdesc = desc_sw128(smem_u32(ring + (r % kRing) * kPageBytes), 0, 1024);
            const uint32_t d = tmem + kTmemS + 64u * (uint32_t)sb;
            // kept rolled: fully unrolled, the 36 products' code competes for
            // instruction fetch with the 18 other warps' (measured 21 % slower).
            // A chunk's four products go under one elect.sync (3.4 % faster on
            // the multi-token workload than one elect.sync per product).
#pragma unroll 1
            for (int c = 0; c < kChunks; ++c)
                mma_bf16_ts4(d, tmem + kTmemQ + 32u * c, bdesc + (uint64_t)((c * kChunkBytes) >> 4), idesc_s,
                             c != 0 ? 1u : 0u);
            mma_commit(&bars->ring_empty[r % kRing]);
            mma_commit(&bars->s_full[sb]);
            issued = true;
        }
        // both warps report when their products of the item no longer read the query
        if (pi.last_of_item()) mma_commit(&bars->q_drained);
        ++r;
    }
    // every MMA this warp issued has completed before TMEM is freed
    if (issued) {
        mma_commit(drain);
        warp_wait(drain, 0, nullptr, err, kDrainNs);
    }
    return ok;
}

// Softmax of the score CTA. Two groups of eight warps take alternate pages of
// the part (group g the pages with n % 2 == g); in a group, the two warps of a
// TMEM lane quadrant share its 32 rows, each taking 32 of the page's 64 keys.
// The online softmax needs one reference max per row for the whole item (O
// accumulates P . V with P taken relative to it), so the reference max moves
// along the page chain: the group of page n reads the value after page n - 1
// (published by the other group), decides whether the row max of page n moves
// it (lazily: only by more than 2^8) and publishes the value after page n.
// Each group keeps its own share of the row sum; at an item's end the group
// without the last page publishes its share, and the group with it adds both
// for 1/l and lse.
template <bool kQ8>
__device__ bool score_softmax(const DecodeArgs& args, Bars* bars, uint8_t* smem, uint32_t tmem, int part, int s,
                              uint32_t peer, volatile int* abort) {
    static_assert(!kQ8 || kSoftmaxGroups == 2, "the INT8 expansion is done by the group that owns the page");
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp >> 3;  // page parity of this group
    const int quad = warp & 3, half = (warp >> 2) & 1;
    const int row = quad * 32 + lane;
    const int pair_bar = 1 + 4 * g + quad;  // named barrier of the two warps of this group sharing these rows
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    uint8_t* ring = smem + kOffRing;
    // the value CTA's P slots, factor arrays and P barriers (same offsets there)
    const uint32_t p_remote = mapa_shared(smem_u32(smem + kOffP), peer);
    const uint32_t x_remote = mapa_shared(smem_u32(smem + kOffXV), peer);
    const uint32_t pfull_remote = mapa_shared(smem_u32(&bars->p_full[0]), peer);
    float* xf = reinterpret_cast<float*>(smem + kOffX);
    float* xpair = xf + kXPair + g * (2 * 2 * kRows);  // this group's [episode][half][128]
    float* xref = xf + kXRef;                          // [page parity][128]
    float* xlsum = xf + kXLSum;                        // [group][half][128]
    float* xlmax = xf + kXLMax;                        // [group][128]
    // this thread's query row inside the two 64-row query boxes, and the query
    // chunks this warp moves into TMEM (the four warps of a quadrant share them)
    const int qbox = quad >> 1, qrow = 32 * (quad & 1) + lane;
    const int qpart = kSoftmaxGroups == 2 ? 2 * g + half : half;  // the quadrant's warps split the 9 chunks
    const float* scales = reinterpret_cast<const float*>(smem + kOffScale);
    PageIter pi;
    pi.init(args, part);
    // scores stay unscaled (x = q' . k; reference maxima in the same units); the
    // scale goes into the exponent's FMA: p = 2^(x s - m s), s = scale * log2(e)
    const float sc = args.scale_log2;
    const float thr = kRescaleThreshold / sc;  // the lazy-rescale margin in unscaled units
    float m_own = -INFINITY, l = 0.f;  // this thread's share of the row sum, relative to m_own
    int n_valid = 0, xe = 0, r = 0;
    bool ok = true;
    for (; pi.valid; pi.advance()) {
        // every exit goes through a pair barrier, so both warps of a pair leave together
        const int n = pi.n, buf = n & 1, qi = pi.n_items - 1;
        const bool first = pi.first_of_item(), last = pi.last_of_item();
        if (first) {
            m_own = -INFINITY;
            l = 0.f;
            n_valid = visible_keys(pi.it.seqlen, args.s_q, s, args.causal);
            // the batch's query into TMEM (row -> lane), once the previous
            // batch's last score products have stopped reading the old one
            if (ok && qi > 0) ok = warp_wait(&bars->q_drained, (qi - 1) & 1, abort, err, wait_ns);
            const int rq = r + qbox;
            if (ok) ok = warp_wait(&bars->ring_full[rq % kRing], (rq / kRing) & 1, abort, err, wait_ns);
            if (ok) {
                tc_fence_after();
                const bool have = qrow < args.qrows;  // fewer than 64 query rows in the whole call
                const uint8_t* src = ring + (rq % kRing) * kPageBytes + qrow * 128;
#pragma unroll 1
                for (int c = qpart; c < kChunks; c += 2 * kSoftmaxGroups) {
                    uint32_t v[32];
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const uint4 x = have ? *reinterpret_cast<const uint4*>(src + c * args.qrows * 128 +
                                                                               ((w ^ (qrow & 7)) << 4))
                                             : make_uint4(0, 0, 0, 0);
                        v[4 * w] = x.x;
                        v[4 * w + 1] = x.y;
                        v[4 * w + 2] = x.z;
                        v[4 * w + 3] = x.w;
                    }
                    tmem_st32(tmem + lane_base + kTmemQ + 32u * c, v);
                }
                tmem_wait_st();
                fence_proxy_async_smem();  // the slots are refilled by TMA after this release
                tc_fence_before();
                mbar_arrive(&bars->q_full);
            }
            // both groups pass an item start together, so neither runs an item ahead
            if (ok) ok = warp_wait(&bars->q_full, qi & 1, abort, err, wait_ns);
            r += 2;
        }
        ++r;
        if (kSoftmaxGroups == 2 && buf != g) {
            // the other group's page; at the item's last page, hand over this
            // group's share of the row sum (complete: its last page was n - 1)
            if (last) {
                xlsum[(g * 2 + half) * kRows + row] = l;
                if (half == 0) xlmax[g * kRows + row] = m_own;
                mbar_arrive(&bars->lsum_full[quad]);
            }
            continue;
        }
        if (kQ8) {
            // this group's page: expand its codes in the ring slot before its
            // score products can be issued (slot of ring position r - 1)
            const int rp = r - 1, slot = rp % kRing;
            if (ok) ok = warp_wait(&bars->ring_full[slot], (rp / kRing) & 1, abort, err, wait_ns);
            if (ok) {
                const int valid = min(kPage, pi.it.seqlen - pi.j * kPage);
                q8_expand_warp(ring + slot * kPageBytes, scales + slot * kPage, valid, warp & 7, lane);
                fence_proxy_async_smem();  // the tensor pipe reads the expanded page next
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->deq_full[g]);
            }
        }
        float x[32];
        const int sb = n % kSBufs;
        if (ok) ok = warp_wait(&bars->s_full[sb], (n / kSBufs) & 1, abort, err, wait_ns);
        if (ok) {
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + kTmemS + 64u * (uint32_t)sb + 32u * (uint32_t)half, v);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(v[c]);
            tc_fence_before();
            mbar_arrive(&bars->s_free[sb]);
        }
        // keys of this half; columns past the visible keys are masked by
        // selection, so whatever the tail rows of the page hold never leaks
        const int vcount = min(max(n_valid - pi.j * kPage - 32 * half, 0), 32);
        if (vcount < 32) {  // (only a sequence's last page has such keys)
#pragma unroll
            for (int c = 0; c < 32; ++c) x[c] = c < vcount ? x[c] : -INFINITY;
        }
        float mh = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; ++c) mh = fmaxf(mh, x[c]);
        // the reference max before this page: none at an item's first page,
        // else the value the other group published after page n - 1. Both warps
        // of the pair read it before the pair barrier, and the half-0 warp
        // publishes this page's value only after that barrier. The next
        // publication on the same barrier (page n + 1, whose group waits for
        // this page's, or passes an item start with both groups) therefore
        // cannot come before both warps have taken page n - 1's: a warp that
        // fell behind its partner would otherwise find the barrier two phases
        // on and wait for a phase that never completes.
        float m_prev = -INFINITY;
        if (!first) {
            if (ok) ok = warp_wait(&bars->ref_full[buf ^ 1][quad], ((n - 1) >> 1) & 1, abort, err, wait_ns);
            m_prev = xref[(buf ^ 1) * kRows + row];
        }
        float* xb = xpair + (xe & 1) * (2 * kRows);
        ++xe;
        xb[half * kRows + row] = mh;
        ok = barrier_and(pair_bar, 64, ok);
        if (!ok) break;
        const float mx = fmaxf(mh, xb[(half ^ 1) * kRows + row]);
        // lazy rescale: the reference max moves only when the row max exceeds it
        // by more than 2^8; both warps of a pair take the same decision
        const bool need = mx > m_prev + thr;
        const float m_new = need ? mx : m_prev;
        const float alpha = need ? fast_exp2((m_prev - mx) * sc) : 1.f;  // 0 when m_prev = -inf
        if (half == 0) {
            xref[buf * kRows + row] = m_new;
            mbar_arrive(&bars->ref_full[buf][quad]);
        }
        if (m_new != m_own) {
            if (l > 0.f) l *= fast_exp2((m_own - m_new) * sc);
            m_own = m_new;
        }
        const float ms = m_new == -INFINITY ? 0.f : m_new * sc;
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            // the row sum takes the fp32 probabilities; only the P.V operand is bf16
            const float p0 = fast_exp2(fmaf(x[2 * c], sc, -ms)), p1 = fast_exp2(fmaf(x[2 * c + 1], sc, -ms));
            l += p0 + p1;
            pk[c] = pack_bf16x2(p0, p1);
        }
        // slot buf held page n - 2 until the value CTA released it
        const int pb = n % kPSlots;  // P slot of this page
        if (ok && n >= kPSlots) ok = warp_wait(&bars->p_free[pb], ((n / kPSlots) - 1) & 1, abort, err, wait_ns);
        const uint32_t mbar = pfull_remote + (uint32_t)pb * 8u;
        if (ok) {
            // Word w of this row (keys 32 half + 8 w .. + 8) goes to key block
            // 4 half + w at row * 16: each st.async of the warp writes 512
            // contiguous bytes. (Cross-cluster stores of 32 rows' 16 bytes at a
            // 128-byte stride, as a 128-byte-swizzled tile would need, cost
            // about 10 % of the spec workload's call.)
            const uint32_t dst = p_remote + (uint32_t)(pb * kPSlotBytes + 4 * half * kPBlockBytes + row * 16);
#pragma unroll
            for (int w = 0; w < 4; ++w)
                st_async_u4(dst + (uint32_t)(w * kPBlockBytes), pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3],
                            mbar);
            if (half == 0)
                st_async_b32(x_remote + (uint32_t)(pb * 1024 + row * 4), __float_as_uint(row < args.H ? alpha : 1.f),
                             mbar);
        }
        if (last) {
            // the pair adds its two half sums (half 0 + half 1), then the other
            // group's share, moved to this reference max
            xb = xpair + (xe & 1) * (2 * kRows);
            ++xe;
            xb[half * kRows + row] = l;
            ok = barrier_and(pair_bar, 64, ok);
            if (!ok) break;
            const float lo = xb[(half ^ 1) * kRows + row];
            const float l_pair = half == 0 ? l + lo : lo + l;
            float l_row = l_pair;
            if (kSoftmaxGroups == 2) {
                if (ok) ok = warp_wait(&bars->lsum_full[quad], qi & 1, abort, err, wait_ns);
                const float l_oth = xlsum[((g ^ 1) * 2) * kRows + row] + xlsum[((g ^ 1) * 2 + 1) * kRows + row];
                const float m_oth = xlmax[(g ^ 1) * kRows + row];
                l_row += l_oth > 0.f ? l_oth * fast_exp2((m_oth - m_new) * sc) : 0.f;
            }
            if (ok && half == 0) {
                const float inv_l = l_row > 0.f ? 1.f / l_row : 0.f;
                st_async_b32(x_remote + (uint32_t)(pb * 1024 + 512 + row * 4), __float_as_uint(inv_l), mbar);
                if (row < args.H) {
                    // lse in natural log of the scaled scores: m s + log2 l is in log2 units
                    const float lse_v =
                        l_row > 0.f ? (m_new * sc + log2f(l_row)) * 0.69314718055994530942f : -INFINITY;
                    if (pi.it.split)
                        args.lse_part[((size_t)pi.it.piece * args.s_q + s) * args.H + row] = lse_v;
                    else
                        args.lse[((size_t)pi.it.b * args.s_q + s) * args.H + row] = lse_v;
                }
            }
        } else if (ok && half == 0) {
            st_async_b32(x_remote + (uint32_t)(pb * 1024 + 512 + row * 4), 0u, mbar);
        }
    }
    return ok;
}

// ============================================================== value CTA ==
template <bool kQ8>
__device__ void value_producer(const DecodeMaps& maps, const DecodeArgs& args, Bars* bars, uint8_t* smem, int part,
                               volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    uint8_t* vring = smem + kOffV;
    PageIter pi;
    pi.init(args, part);
    bool ok = !args.withhold;  // test hook: issue nothing, so that the P.V warp's first wait runs out
    int v = 0;
    for (; ok && pi.valid; pi.advance()) {
        if (v >= kVRing) ok = mbar_wait(&bars->v_empty[v % kVRing], ((v / kVRing) - 1) & 1, abort, err, wait_ns);
        if (!ok) break;
        const int blk = checked_block(args, pi.it.b, pi.j, err, abort);
        uint64_t* bar = &bars->v_full[v % kVRing];
        if (kQ8) {
            mbar_arrive_expect_tx(bar, kQ8VBytes);
            tma_load_3d(vring + (v % kVRing) * kVBytes + kQ8Planes, &maps.kv8, bar, 0, blk * kPage, 0);
            bulk_load(smem + kOffScale + (v % kVRing) * kScaleBytes, args.kv_scale + (size_t)blk * kPage, kScaleBytes,
                      bar);
        } else {
            mbar_arrive_expect_tx(bar, (uint32_t)kVBytes);
            tma_load_3d(vring + (v % kVRing) * kVBytes, &maps.v, bar, 0, blk * kPage, 0);
        }
        ++v;
    }
    drain_ring(bars->v_full, kVRing, v, err);
}

template <bool kQ8>
__device__ bool value_mma(const DecodeArgs& args, Bars* bars, uint8_t* smem, uint32_t tmem, int part,
                          volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    const int lane = threadIdx.x & 31;
    uint8_t* vring = smem + kOffV;
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, 256, false, true);
    PageIter pi;
    pi.init(args, part);
    bool ok = true, issued = false;
    int consumed = 0;
    for (; ok && pi.valid; pi.advance()) {
        const int n = pi.n, k = n % kPSlots, qi = pi.n_items - 1;
        const bool first = pi.first_of_item(), last = pi.last_of_item();
        ok = warp_wait<true>(&bars->p_full[k], (n / kPSlots) & 1, abort, err, wait_ns);
        if (!ok) break;
        consumed = n + 1;
        if (lane == 0) {
            // P was written by the peer's generic stores: make it visible to the
            // tensor pipe, then arm the slot for page n + kPSlots (its bytes can
            // only come after this page has released the slot)
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars->p_full[k], kPMsgBytes);
        }
        __syncwarp();
        // the O warps have read this message's factors (and rescaled O if asked)
        ok = warp_wait(&bars->o_ack[k], (n / kPSlots) & 1, abort, err, wait_ns);
        if (ok)
            ok = kQ8 ? warp_wait(&bars->vdeq_full[n % kVRing], (n / kVRing) & 1, abort, err, wait_ns)
                     : warp_wait(&bars->v_full[n % kVRing], (n / kVRing) & 1, abort, err, wait_ns);
        if (!ok) break;
        uint8_t* vs = vring + (n % kVRing) * kVBytes;
        const int tail = pi.j == pi.it.nblk - 1 ? pi.it.seqlen - pi.j * kPage : kPage;
        if (!kQ8 && tail < kPage) {  // (the INT8 expansion writes those rows as zeros)
            // rows past seqlen hold arbitrary bytes: zero them so that
            // 0-probability keys cannot inject NaN/Inf into P.V
            const int per_chunk = (kPage - tail) * 8;  // 16-byte words
            for (int i = lane; i < 8 * per_chunk; i += 32) {
                const int c = i / per_chunk, w = i % per_chunk;
                reinterpret_cast<uint4*>(vs + c * kChunkBytes + tail * 128)[w] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        tc_fence_after();
        {
            // whole warp, one elected lane issues; K-step kk reads key blocks
            // 2 kk and 2 kk + 1 of P
            const uint64_t adesc = desc_noswz(smem_u32(smem + kOffP + k * kPSlotBytes), kPBlockBytes, 128);
            const uint64_t vdesc = desc_sw128(smem_u32(vs), kChunkBytes, 1024);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // a batch's first products overwrite O: the previous epilogue
                // must have read this half of it (the other half may still be
                // in its hands)
                if (first && qi > 0) {
                    ok = warp_wait(&bars->o_free[h], (qi - 1) & 1, abort, err, wait_ns);
                    if (!ok) break;
                    tc_fence_after();
                }
                // the page's four 16-key K-steps under one elect.sync (P: two
                // key blocks further per step; V: 16 key rows further)
                static_assert(kPage == 64, "four K-steps per page");
                mma_bf16_ss4(tmem + 256u * h, adesc, (uint64_t)((2 * kPBlockBytes) >> 4),
                             vdesc + (uint64_t)((4 * h * kChunkBytes) >> 4), (uint64_t)(2048 >> 4), idesc_pv,
                             first ? 0u : 1u);
            }
            if (!ok) break;
            // the last page's slot becomes the epilogue's staging area, which
            // hands it back to the producer
            if (!last) mma_commit(&bars->v_empty[n % kVRing]);
            mma_commit(&bars->pv_done[n & 1]);
            if (last) mma_commit(&bars->o_full);
            mma_commit_multicast(&bars->p_free[k], (uint16_t)1u);  // arrives on the score CTA (rank 0)
        }
        issued = true;
    }
    if (issued) {
        mma_commit(&bars->drain);
        warp_wait(&bars->drain, 0, nullptr, err, kDrainNs);
    }
    if (lane == 0) bars->p_consumed = consumed;
    return ok;
}

// INT8 cache: warps 8-15 of the value CTA expand each value slot's codes to
// bf16 (rows past the sequence as zeros) before its P.V products.
__device__ bool value_expand(const DecodeArgs& args, Bars* bars, uint8_t* smem, int part, volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* vring = smem + kOffV;
    const float* scales = reinterpret_cast<const float*>(smem + kOffScale);
    PageIter pi;
    pi.init(args, part);
    bool ok = true;
    for (; ok && pi.valid; pi.advance()) {
        const int n = pi.n, slot = n % kVRing;
        ok = warp_wait(&bars->v_full[slot], (n / kVRing) & 1, abort, err, wait_ns);
        if (!ok) break;
        const int valid = min(kPage, pi.it.seqlen - pi.j * kPage);
        q8_expand_warp(vring + slot * kVBytes, scales + slot * kPage, valid, warp - 8, lane);
        fence_proxy_async_smem();  // the tensor pipe reads the expanded values next
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->vdeq_full[slot]);
    }
    return ok;
}

// Empty sequences (no keys) have no pages and no piece, so no item writes their
// rows. Where no merge kernel follows (which writes them otherwise), an
// otherwise idle warp of the value CTA gives them o = 0 and lse = -inf for the
// cluster's query token. An empty batch belongs to the part holding page 0 of
// the next non-empty batch (that part zeros the empty batches just before each
// of its items that starts at page 0), trailing empty batches to the part
// holding the last page of the last non-empty one, and, with every sequence
// empty, all batches to part 0 (then without work): each is written once.
__device__ void zero_empty_batches(const DecodeArgs& args, int part, int s) {
    const int t = threadIdx.x & 31;  // one warp
    auto empty = [&](int b) { return args.seqlens[b] <= 0; };
    auto zero = [&](int b) {
        const size_t row0 = ((size_t)b * args.s_q + s) * args.H;
        uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.o_lat) + row0 * kDLatent);
        const int words = args.H * kDLatent / 8;  // 16-byte words of the batch's H rows
        for (int i = t; i < words; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
        for (int h = t; h < args.H; h += 32) args.lse[row0 + h] = -INFINITY;
    };
    ItemIter items;
    items.init(args, part);
    Item it;
    bool any = false;
    int last_b = -1, last_hi = 0, last_n = 0;
    while (items.next(it)) {
        any = true;
        if (it.lo == 0)
            for (int b = it.b - 1; b >= 0 && empty(b); --b) zero(b);
        last_b = it.b;
        last_hi = it.hi;
        last_n = it.nblk;
    }
    if (!any) {
        if (part == 0)
            for (int b = 0; b < args.B; ++b) zero(b);  // no part has work: every sequence is empty
        return;
    }
    if (last_hi == last_n) {
        int b = last_b + 1;
        while (b < args.B && empty(b)) ++b;
        if (b == args.B)
            for (int e = last_b + 1; e < args.B; ++e) zero(e);
    }
}

__device__ bool value_owarps(const DecodeMaps& maps, const DecodeArgs& args, Bars* bars, uint8_t* smem,
                             uint32_t tmem, int part, int s, volatile int* abort) {
    int* err = args.err;
    const long long wait_ns = args.wait_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float* xv = reinterpret_cast<const float*>(smem + kOffXV);  // [slot][factor 128 | 1/l 128]
    const uint32_t ocol = tmem + lane_base + 256u * (uint32_t)half;
    PageIter pi;
    pi.init(args, part);
    bool ok = true;
    bool stored = false;
    bool acked = false;  // this page's message was acknowledged ahead (see below)
    int erounds = 0;     // epilogue rounds so far (phase of stage_full / stage_free)
    for (; ok && pi.valid; pi.advance()) {
        const int n = pi.n, k = n % kPSlots, qi = pi.n_items - 1;
        const bool first = pi.first_of_item(), last = pi.last_of_item();
        if (acked) {
            acked = false;
            continue;
        }
        ok = warp_wait<true>(&bars->p_full[k], (n / kPSlots) & 1, abort, err, wait_ns);
        if (!ok) break;
        const float inv_l = xv[k * 256 + 128 + row];
        if (!first) {
            const float alpha = xv[k * 256 + row];
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
                // O rows of this warp move to the new reference max (after the
                // previous P.V product has landed)
                ok = warp_wait(&bars->pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, abort, err, wait_ns);
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
        {
            // The next item's first page needs nothing from its message (no
            // rescale of O, no 1/l unless it is also that item's last page):
            // acknowledge it now, so that its P.V products can start on each
            // half of O as soon as this epilogue has read that half. (Its slot's
            // previous message, page n - 2, was acknowledged before this one.)
            PageIter nx = pi;
            nx.advance();
            if (nx.valid && !nx.last_of_item()) {
                if (lane == 0) mbar_arrive(&bars->o_ack[nx.n % kPSlots]);
                acked = true;
            }
        }

        // ---- epilogue of the item: O * (1/l) -> staging -> TMA store. The
        // staging area is the value slot of this last page: 64 KB, i.e. 256 bf16
        // columns of all rows per round (a split sequence's piece goes to the
        // partial buffer in bf16 too, beside its fp32 lse), stored as one box
        // [4 chunks][rows][128 B] (128-byte swizzle) by thread 0 once the eight
        // warps have written their parts (stage_full), after which the area is
        // free for the next round (stage_free).
        ok = warp_wait(&bars->o_full, qi & 1, abort, err, wait_ns);
        if (!ok) break;
        tc_fence_after();
        const Item& it = pi.it;
        const bool row_ok = row < args.H;
        const int hrows = min(args.H, kRows);
        // after the part's last item no page is loaded any more and both value
        // slots can stage: one round of eight chunks instead of two of four
        const bool wide = it.b == pi.items.row[2];
        uint8_t* stage = wide ? smem + kOffV : smem + kOffV + (n % kVRing) * kVBytes;
        const int cpr = wide ? 8 : 4;  // 128-byte chunks (64 bf16 columns) per round
        const int rounds = 8 / cpr;
        const int z = it.split ? it.piece * args.s_q + s : it.b * args.s_q + s;
        for (int rnd = 0; rnd < rounds; ++rnd) {
            // this warp: chunks [cpr/2 half, cpr/2 half + cpr/2) of the round
#pragma unroll 1
            for (int cc = 0; cc < cpr / 2; ++cc) {
                const int chunk = (cpr / 2) * half + cc;
                uint8_t* dst = stage + chunk * hrows * 128 + row * 128;
                {
                    // 64 bf16 columns = one 128-byte row, read from TMEM 32 columns
                    // (four 16-byte words) at a time
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t col = (uint32_t)(64 * (cpr * rnd + chunk) + 32 * hh);  // absolute O column
                        uint32_t v0[32];
                        tmem_ld32(tmem + lane_base + col, v0);
                        tmem_wait_ld();
                        if (row_ok) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint4 w0;
                                w0.x = pack_bf16x2(__uint_as_float(v0[8 * q + 0]) * inv_l, __uint_as_float(v0[8 * q + 1]) * inv_l);
                                w0.y = pack_bf16x2(__uint_as_float(v0[8 * q + 2]) * inv_l, __uint_as_float(v0[8 * q + 3]) * inv_l);
                                w0.z = pack_bf16x2(__uint_as_float(v0[8 * q + 4]) * inv_l, __uint_as_float(v0[8 * q + 5]) * inv_l);
                                w0.w = pack_bf16x2(__uint_as_float(v0[8 * q + 6]) * inv_l, __uint_as_float(v0[8 * q + 7]) * inv_l);
                                *reinterpret_cast<uint4*>(dst + (((q + 4 * hh) ^ (row & 7)) << 4)) = w0;
                            }
                        }
                    }
                }
            }
            {
                // columns of O read so far: the next item's products may
                // overwrite each half once all eight warps have read it
                const int per_round = cpr * 64;
                const int done = (rnd + 1) * per_round, before = rnd * per_round;
                if (before < 256 && done >= 256) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->o_free[0]);
                }
                if (done >= 512) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->o_free[1]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->stage_full);
            if (warp == 0) {
                ok = warp_wait(&bars->stage_full, erounds & 1, abort, err, wait_ns);
                if (ok && lane == 0) {
                    // boxes of four chunks
                    for (int b4 = 0; b4 < cpr / 4; ++b4) {
                        uint8_t* src = stage + b4 * 4 * hrows * 128;
                        if (it.split)
                            tma_store_4d(&maps.op, src, 0, 0, cpr * rnd + 4 * b4, z);
                        else
                            tma_store_4d(&maps.o, src, 0, 0, cpr * rnd + 4 * b4, z);
                    }
                    bulk_commit_group();
                    bulk_wait_group_read0();  // the next round rewrites the staging area
                    stored = true;
                    mbar_arrive(&bars->stage_free);
                }
                __syncwarp();
            }
            if (ok) ok = warp_wait(&bars->stage_free, erounds & 1, abort, err, wait_ns);
            ++erounds;
            if (!ok) break;
        }
        if (!ok) break;
        // staging read by the last store: the slot goes back to the producer
        if (threadIdx.x == 0) mbar_arrive(&bars->v_empty[n % kVRing]);
    }
    if (stored) bulk_wait_group0();
    return ok;
}

// kEmpty: this launch also writes the rows of empty sequences (no merge kernel
// follows it). It is a separate instantiation because the extra role, though
// it never runs beside the pages, measurably slows the kernel that lacks it.
template <bool kQ8, bool kEmpty>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeMaps maps, DecodeArgs args) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms; both CTAs run the same
    // kernel, so the offsets used for remote addresses agree
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);
    volatile int* abort = &bars->abort;

    const int warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int cluster_id = blockIdx.x >> 1;
    const int part = cluster_id / args.s_q;
    const int s = cluster_id % args.s_q;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bars->ring_full[i], 1);
            mbar_init(&bars->ring_empty[i], 1);
        }
        mbar_init(&bars->q_full, 32 * kSoftmaxWarps);
        mbar_init(&bars->q_drained, kScoreMmaWarps);
        for (int i = 0; i < kSBufs; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_free[i], 256);
        }
        for (int i = 0; i < kPSlots; ++i) {
            mbar_init(&bars->p_free[i], 1);
            mbar_init(&bars->p_full[i], 1);
            mbar_init(&bars->o_ack[i], 8);
        }
        for (int i = 0; i < 2; ++i) {
            for (int q = 0; q < 4; ++q) mbar_init(&bars->ref_full[i][q], 32);
            mbar_init(&bars->o_free[i], kOWarps);
        }
        for (int i = 0; i < kVRing; ++i) {
            mbar_init(&bars->v_full[i], 1);
            mbar_init(&bars->v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&bars->pv_done[i], 1);
        mbar_init(&bars->o_full, 1);
        for (int q = 0; q < 4; ++q) mbar_init(&bars->lsum_full[q], 64);
        mbar_init(&bars->stage_full, kOWarps);
        mbar_init(&bars->stage_free, 1);
        mbar_init(&bars->drain, 1);
        mbar_init(&bars->drain2, 1);
        for (int i = 0; i < 2; ++i) mbar_init(&bars->deq_full[i], 8);
        for (int i = 0; i < kVRing; ++i) mbar_init(&bars->vdeq_full[i], 8);
        bars->abort = 0;
        bars->p_consumed = 0;
        fence_mbarrier_init_cluster();
        if (rank == 0) {
            if (kQ8) {
                tma_prefetch_desc(&maps.kv8);
                tma_prefetch_desc(&maps.rope);
            } else {
                tma_prefetch_desc(&maps.kv);
            }
            tma_prefetch_desc(&maps.q);
        } else {
            tma_prefetch_desc(kQ8 ? &maps.kv8 : &maps.v);
            tma_prefetch_desc(&maps.o);
            tma_prefetch_desc(&maps.op);
            // the first kPSlots P messages may arrive as soon as the cluster is up
            for (int i = 0; i < kPSlots; ++i) mbar_arrive_expect_tx(&bars->p_full[i], kPMsgBytes);
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
            score_producer<kQ8>(maps, args, bars, smem, part, s, abort);
        } else if (warp == kWarpMma) {
            ok = score_mma<kQ8>(args, bars, smem, tmem, part, kScoreMmaWarps == 1 ? -1 : 0, abort);
        } else if (warp == kWarpMma2) {
            if (kScoreMmaWarps == 2) ok = score_mma<kQ8>(args, bars, smem, tmem, part, 1, abort);
        } else if (warp < kSoftmaxWarps) {
            ok = score_softmax<kQ8>(args, bars, smem, tmem, part, s, peer, abort);
        }
    } else {
        if (warp == kWarpProducer) {
            if ((threadIdx.x & 31) == 0) value_producer<kQ8>(maps, args, bars, smem, part, abort);
        } else if (warp == kWarpMma) {
            ok = value_mma<kQ8>(args, bars, smem, tmem, part, abort);
        } else if (warp < kOWarps) {
            ok = value_owarps(maps, args, bars, smem, tmem, part, s, abort);
        } else if (kQ8 && warp < 16) {
            ok = value_expand(args, bars, smem, part, abort);
        } else if (kEmpty && warp == kWarpMma2) {
            zero_empty_batches(args, part, s);
        }
    }
    // a role that gave up tells the peer, whose waits then end promptly
    if (!ok || *abort) st_cluster_b32(mapa_shared(smem_u32(&bars->abort), peer), 1u);

    tc_fence_before();
    __syncthreads();
    // the peer may still store into our buffers or arrive on our barriers until
    // it has finished its last page: leave together
    cluster_sync_all();
    if (rank == 1 && warp == kWarpMma && (threadIdx.x & 31) == 0 && *abort) {
        // The score CTA has stopped sending, but the st.async stores of the
        // armed P messages (pages c .. c + kPSlots - 1) may still be landing in this
        // CTA's shared memory: wait for their phases, briefly, before leaving.
        const int c = bars->p_consumed;
        for (int n = c; n < c + kPSlots; ++n)
            mbar_wait(&bars->p_full[n % kPSlots], (n / kPSlots) & 1, nullptr, nullptr, kPDrainNs);
    }
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Sets the kernel's shared-memory attribute once per device (thread-safe).
template <bool kQ8, bool kEmpty>
cudaError_t prepare_kernel() {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(decode_kernel<kQ8, kEmpty>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess) done[dev] = true;
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
    const bool q8 = args.kv_scale != nullptr, own = args.own_empty != 0;
    cudaError_t e = q8 ? (own ? prepare_kernel<true, true>() : prepare_kernel<true, false>())
                       : (own ? prepare_kernel<false, true>() : prepare_kernel<false, false>());
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = make_config(args.num_parts * args.s_q, stream, attr, true);
    if (q8) return own ? cudaLaunchKernelEx(&cfg, decode_kernel<true, true>, maps, args)
                       : cudaLaunchKernelEx(&cfg, decode_kernel<true, false>, maps, args);
    return own ? cudaLaunchKernelEx(&cfg, decode_kernel<false, true>, maps, args)
               : cudaLaunchKernelEx(&cfg, decode_kernel<false, false>, maps, args);
}

// Clusters of the decode kernel that can be resident at once on the current device.
int decode_max_active_clusters(int /*device*/) {
    // both cache formats use the same threads and shared memory
    if (prepare_kernel<false, false>() != cudaSuccess) return 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = make_config(1024, nullptr, attr, false);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_kernel<false, false>, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace mla
