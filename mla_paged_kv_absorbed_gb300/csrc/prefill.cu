// prefill.cu - prefill over the paged latent cache in the naive (decompress)
// form: the per-head keys and values are up-projected from the cached latent,
// then ordinary causal attention runs per head.
//
// What it computes ("DeepSeek-V3 MLA deep engineering", sec. 2.2: k = W_UK c,
// v = W_UV c; sec. 3.1: the rope key is shared by the heads; sec. 4.3: the
// paged module decompresses K and V per head before attention; the SC11
// article's opening: prefill processes a whole prompt, decode one token):
// for sequence b with seqlen L and s_q query tokens (its last s_q positions),
// head h and query s:
//   K_t = [W_UK[h] c_t | k_rope_t] (192), V_t = W_UV[h]^T c_t (128), t < L
//   out[b,s,h,:] = softmax_t(scale * q[b,s,h,:] . K_t) V_t over t <= L - s_q + s
//   lse[b,s,h]   = ln sum_t exp(scale * q . K_t)
// The naive form costs 2 * (192 + 128) flops per (query, key, head) against
// 2 * (576 + 512) for the absorbed form, so it is the cheaper form once a
// sequence has many query tokens; the up-projections cost 2 * 512 * 256 flops
// per (token, head), once.
//
// Kernels here: the gather of the sequence's latent rows and rope keys into
// contiguous buffers (the two up-projections then run as batched head GEMMs,
// gemm.cu), and the attention: one CTA per (b, h, two 128-query tiles),
// 64-key tiles of K and V streaming through a TMA ring and shared by both query
// tiles, S = Q K^T and O += P V on tcgen05 with S (double-buffered), P and O in
// TMEM, two softmax threads per query row (online softmax, lazy rescaling of O).
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {

__device__ int g_prefill_error = 0;

namespace {

// ------------------------------------------------------------------ gather --
// One CTA per (b, page j): rows t = 64 j .. 64 j + 63 of sequence b. For t <
// seqlen: C[b Lmax + t] = c_t[0:512], Kbuf[h][b Lmax + t][128:192] = k_rope_t for
// every head; for t >= seqlen both are zero, so padding keys contribute
// nothing finite-unsafe (their K and V rows are exact zeros after the GEMMs).
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads)
    prefill_gather_kernel(const __nv_bfloat16* __restrict__ kv, int num_blocks, const int32_t* __restrict__ table,
                          int mbps, const int32_t* __restrict__ seqlens, int H, size_t R, __nv_bfloat16* __restrict__ C,
                          __nv_bfloat16* __restrict__ Kbuf) {
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.y, j = blockIdx.x;
    const int L = seqlens[b];
    if (j == 0 && threadIdx.x == 0 && L > mbps * kPage) record_error(&g_prefill_error, kErrBadBlock);
    int blk = -1;
    if (j * kPage < L) {
        blk = table[(size_t)b * mbps + j];
        if (blk < 0 || blk >= num_blocks) {
            if (threadIdx.x == 0) record_error(&g_prefill_error, kErrBadBlock);
            blk = -1;
        }
    }
    const size_t row0 = (size_t)b * mbps * kPage + (size_t)j * kPage;
    // latent: 64 rows x 64 words of 16 bytes
    for (int i = threadIdx.x; i < kPage * 64; i += kGatherThreads) {
        const int r = i >> 6, w = i & 63;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (blk >= 0 && j * kPage + r < L)
            v = reinterpret_cast<const uint4*>(kv + ((size_t)blk * kPage + r) * kDQK)[w];
        reinterpret_cast<uint4*>(C + (row0 + r) * kDLatent)[w] = v;
    }
    // rope key: 64 rows x 8 words, copied into every head's K rows
    for (int i = threadIdx.x; i < kPage * 8 * H; i += kGatherThreads) {
        const int w = i & 7, r = (i >> 3) & (kPage - 1), h = i >> 9;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (blk >= 0 && j * kPage + r < L)
            v = reinterpret_cast<const uint4*>(kv + ((size_t)blk * kPage + r) * kDQK + kDLatent)[w];
        reinterpret_cast<uint4*>(Kbuf + ((size_t)h * R + row0 + r) * kDQ + kDNope)[w] = v;
    }
}

// --------------------------------------------------------------- attention --
// One CTA per (b, h, block of 256 query rows) = two 128-row query tiles (t = 0,
// 1) that share every 64-key tile of K and V, so each K/V byte loaded feeds
// twice the products. Warps 8t .. 8t + 7 run tile t's softmax and epilogue,
// two per TMEM lane quadrant: warp w owns rows 32 (w % 4) .. + 31 of its tile
// and keys [32 ((w / 4) % 2), + 32) of every key tile, and the two warps of a
// quadrant exchange their half-row maxima (and, at the end, their half sums)
// through shared memory. Warp 16 is the TMA producer, warp 17 issues the
// products and owns TMEM (all 512 columns: per tile two 64-column S buffers
// and a 128-column O). S_t = Q_t K^T goes to one of tile t's S buffers; the
// softmax writes P (bf16 pairs) back over the first 32 columns of the same
// buffer, and O_t += P V takes P as the A operand straight from TMEM. The
// tensor pipe runs a CTA's products in issue order, so S_t of key tile j + 2
// (issued after P V of tile j) never overwrites P before it has been read, and
// P is written only after both halves of a row have read their scores.
constexpr int kATiles = 2;
constexpr int kAThreads = 576;
constexpr int kAWarpProducer = 16;
constexpr int kAWarpMma = 17;
constexpr int kARows = 128;     // query rows per tile
constexpr int kAKeys = 64;      // keys per tile
constexpr int kAStages = 3;
constexpr int kQBytes = 3 * kARows * 128;   // [3 chunks][128 rows][64]
constexpr int kKBytes = 3 * kAKeys * 128;   // [3 chunks][64 keys][64]
constexpr int kVBytesA = 2 * kAKeys * 128;  // [2 chunks][64 keys][64]
constexpr int kAXBytes = 2 * 2 * kARows * 4;  // per tile: [2 episodes][2 halves][128 rows] floats
constexpr int kAOffX = 1024;
constexpr int kAOffQ = 6144;
constexpr int kAOffK = kAOffQ + kATiles * kQBytes;
constexpr int kAOffV = kAOffK + kAStages * kKBytes;
constexpr int kASmem = kAOffV + kAStages * kVBytesA + 1024;  // + alignment slack
static_assert(kASmem <= 232448, "prefill attention shared memory");
static_assert(kAOffX + kATiles * kAXBytes <= kAOffQ, "exchange area");
static_assert(kAOffQ % 1024 == 0 && kAOffK % 1024 == 0 && kAOffV % 1024 == 0, "swizzle atoms");
constexpr uint32_t kATmemCols = 512;
// tile t: S buffers at 128 t and 128 t + 64 (P over the first 32 of each), O at 256 + 128 t
__device__ __forceinline__ uint32_t tmem_s(int t, int sb) { return (uint32_t)(128 * t + 64 * sb); }
__device__ __forceinline__ uint32_t tmem_o(int t) { return (uint32_t)(256 + 128 * t); }
constexpr float kARescale = 8.0f;

struct ABars {
    uint64_t q_full;
    uint64_t kv_full[kAStages], kv_empty[kAStages];
    uint64_t s_full[kATiles][2], p_full[kATiles][2];
    uint64_t pv_done[kATiles], drain;
    uint32_t tmem_slot;
    int abort;
};
static_assert(sizeof(ABars) <= kAOffX, "prefill barriers");

struct PrefillArgs {
    const int32_t* seqlens;
    int s_q, H, Lmax;
    float scale_log2;
    int causal;
    __nv_bfloat16* out;  // [B, s_q, H, 128]
    float* lse;          // [B, s_q, H]
    int* err;
    long long wait_ns;
};
struct PrefillMaps {
    CUtensorMap q, k, v;
};

__device__ __forceinline__ int visible(int L, int s_q, int s, int causal) {
    int n = causal ? L - s_q + s + 1 : L;
    return n < 0 ? 0 : (n > L ? L : n);
}

// Key tiles query tile t (rows q0 + 128 t ..) needs: up to the last visible key
// of its last valid row (0 when it has no valid row).
__device__ __forceinline__ int tile_count(int L, const PrefillArgs& args, int q0, int t) {
    const int first = q0 + kARows * t;
    const int last_row = min(first + kARows, args.s_q) - 1;
    const int n_max = last_row >= first ? visible(L, args.s_q, last_row, args.causal) : 0;
    return (n_max + kAKeys - 1) / kAKeys;
}

__global__ void __launch_bounds__(kAThreads, 1)
    prefill_attn_kernel(const __grid_constant__ PrefillMaps maps, PrefillArgs args) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    ABars* bars = reinterpret_cast<ABars*>(smem);
    volatile int* abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grid (query blocks, H, B), launched x fastest: the blocks of one (sequence,
    // head) run side by side and share its K and V in L2 (launching the longest
    // blocks of every head first measured slower: their K/V outgrew the L2)
    const int h = blockIdx.y, b = blockIdx.z;
    const int q0 = blockIdx.x * (kATiles * kARows);
    int* err = args.err;
    const long long wait_ns = args.wait_ns;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int i = 0; i < kAStages; ++i) {
            mbar_init(&bars->kv_full[i], 1);
            mbar_init(&bars->kv_empty[i], 1);
        }
        for (int t = 0; t < kATiles; ++t) {
            for (int i = 0; i < 2; ++i) {
                mbar_init(&bars->s_full[t][i], 1);
                mbar_init(&bars->p_full[t][i], 256);
            }
            mbar_init(&bars->pv_done[t], 1);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
    }
    if (warp == kAWarpMma) {
        tmem_alloc(&bars->tmem_slot, kATmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    griddep_wait();
    griddep_launch_dependents();

    const int L = min(max(args.seqlens[b], 0), args.Lmax);  // longer sequences were reported by the gather
    int tiles_t[kATiles];
#pragma unroll
    for (int t = 0; t < kATiles; ++t) tiles_t[t] = tile_count(L, args, q0, t);
    const int tiles = max(tiles_t[0], tiles_t[1]);  // key tiles the block loads (causal: tile 1's count)
    const int key_row0 = b * args.Lmax;  // first key row of this sequence in the K/V buffers

    bool ok = true;
    if (warp == kAWarpProducer) {
        // producer: both query tiles once, then K and V tiles through the ring
        if (lane == 0 && tiles > 0) {
            mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(kATiles * kQBytes));
            for (int t = 0; t < kATiles; ++t)
                tma_load_4d(smem + kAOffQ + t * kQBytes, &maps.q, &bars->q_full, 0, h, b * args.s_q + q0 + kARows * t,
                            0);
            int issued = 0;
            for (int j = 0; j < tiles; ++j) {
                const int st = j % kAStages;
                if (j >= kAStages && !mbar_wait(&bars->kv_empty[st], ((j / kAStages) - 1) & 1, abort, err, wait_ns)) break;
                mbar_arrive_expect_tx(&bars->kv_full[st], (uint32_t)(kKBytes + kVBytesA));
                tma_load_4d(smem + kAOffK + st * kKBytes, &maps.k, &bars->kv_full[st], 0, key_row0 + j * kAKeys, 0, h);
                tma_load_4d(smem + kAOffV + st * kVBytesA, &maps.v, &bars->kv_full[st], 0, key_row0 + j * kAKeys, 0, h);
                issued = j + 1;
            }
            // every load this thread issued has landed before the CTA may leave
            mbar_wait(&bars->q_full, 0, nullptr, err, kDrainNs);
            for (int j = issued - kAStages > 0 ? issued - kAStages : 0; j < issued; ++j)
                mbar_wait(&bars->kv_full[j % kAStages], (j / kAStages) & 1, nullptr, err, kDrainNs);
        }
        __syncwarp();
    } else if (warp == kAWarpMma) {
        // MMA issuer (whole warp; one elected lane issues)
        const uint32_t idesc_s = idesc_bf16_f32(kARows, kAKeys, false, false);
        const uint32_t idesc_o = idesc_bf16_f32(kARows, 128, false, true);
        bool issued = false;
        if (tiles > 0) ok = warp_wait(&bars->q_full, 0, abort, err, wait_ns);
        // K(j) has landed once kv_full was seen for it; S products of both tiles
        auto issue_s = [&](int t, int j) {
            const int st = j % kAStages, sb = j & 1;
            const uint64_t qdesc = desc_sw128(smem_u32(smem + kAOffQ + t * kQBytes), 0, 1024);
            const uint64_t kdesc = desc_sw128(smem_u32(smem + kAOffK + st * kKBytes), 0, 1024);
#pragma unroll
            for (int c = 0; c < 3; ++c)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tmem + tmem_s(t, sb), qdesc + (uint64_t)((c * kARows * 128 + 32 * kk) >> 4),
                                kdesc + (uint64_t)((c * kAKeys * 128 + 32 * kk) >> 4), idesc_s, (c | kk) != 0);
            mma_commit(&bars->s_full[t][sb]);
        };
        auto load_ready = [&](int j) -> bool {
            if (!warp_wait(&bars->kv_full[j % kAStages], (j / kAStages) & 1, abort, err, wait_ns)) return false;
            tc_fence_after();
            return true;
        };
        for (int j = 0; ok && j < 2 && j < tiles; ++j) {
            ok = load_ready(j);
            if (!ok) break;
            issued = true;
            for (int t = 0; t < kATiles; ++t)
                if (j < tiles_t[t]) issue_s(t, j);
        }
        for (int j = 0; ok && j < tiles; ++j) {
            const int st = j % kAStages, sb = j & 1;
            const uint64_t vdesc = desc_sw128(smem_u32(smem + kAOffV + st * kVBytesA), kAKeys * 128, 1024);
            for (int t = 0; ok && t < kATiles; ++t) {
                if (j >= tiles_t[t]) continue;
                ok = warp_wait(&bars->p_full[t][sb], (j >> 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kAKeys / 16; ++kk)
                    mma_bf16_ts(tmem + tmem_o(t), tmem + tmem_s(t, sb) + 8u * (uint32_t)kk,
                                vdesc + (uint64_t)((2048 * kk) >> 4), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bars->pv_done[t]);
            }
            if (!ok) break;
            mma_commit(&bars->kv_empty[st]);  // K(j) and V(j) read by every product of tile j
            if (j + 2 < tiles) {
                ok = load_ready(j + 2);
                if (!ok) break;
                for (int t = 0; t < kATiles; ++t)
                    if (j + 2 < tiles_t[t]) issue_s(t, j + 2);
            }
        }
        if (issued) {
            mma_commit(&bars->drain);
            warp_wait(&bars->drain, 0, nullptr, err, kDrainNs);
        }
    } else if (warp < 8 * kATiles) {
        // softmax and epilogue of query tile t: thread = (query row, half of each key tile)
        const int t = warp >> 3;
        const int quad = warp & 3, half = (warp >> 2) & 1;
        const int row = quad * 32 + lane, s = q0 + kARows * t + row;
        const bool valid_row = s < args.s_q;
        const int n_vis = valid_row ? visible(L, args.s_q, s, args.causal) : 0;
        const int tiles_my = tiles_t[t];
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const uint32_t ocol = tmem + lane_base + tmem_o(t) + 64u * (uint32_t)half;  // this half's 64 O columns
        const int pair_bar = 1 + 4 * t + quad;  // named barrier of this quadrant's two warps
        float* xch = reinterpret_cast<float*>(smem + kAOffX + t * kAXBytes);
        int xe = 0;
        // scores stay unscaled (x = q . k, m their running max); the scale goes
        // into the exponent's FMA: p = 2^(x s - m s), s = softmax scale * log2(e)
        const float sc = args.scale_log2;
        const float thr = kARescale / sc;  // the lazy-rescale margin in unscaled units
        float m = -INFINITY, l = 0.f;  // l: this half's share of the row sum, relative to m
        for (int j = 0; j < tiles_my; ++j) {
            const int sb = j & 1;
            const uint32_t sbuf = tmem + lane_base + tmem_s(t, sb);
            float x[32];
            if (ok) ok = warp_wait(&bars->s_full[t][sb], (j >> 1) & 1, abort, err, wait_ns);
            if (ok) {
                tc_fence_after();
                uint32_t v[32];
                tmem_ld32(sbuf + 32u * (uint32_t)half, v);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(v[c]);
            }
            // keys past the visible ones are masked by selection (only the tiles
            // on the diagonal and past the sequence have any)
            const int vcount = min(max(n_vis - j * kAKeys - 32 * half, 0), 32);
            if (vcount < 32) {
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] = c < vcount ? x[c] : -INFINITY;
            }
            float mh = -INFINITY;
#pragma unroll
            for (int c = 0; c < 32; ++c) mh = fmaxf(mh, x[c]);
            // both halves of the row have read their scores after this barrier
            float* xb = xch + (xe & 1) * (2 * kARows);
            ++xe;
            xb[half * kARows + row] = mh;
            ok = barrier_and(pair_bar, 64, ok);
            if (!ok) break;
            const float mx = fmaxf(mh, xb[(half ^ 1) * kARows + row]);
            // lazy rescale: move the reference max only when the row max grows by
            // more than 2^8 (both halves take the same decision)
            const bool need = mx > m + thr;
            const float alpha = need ? fast_exp2((m - mx) * sc) : 1.f;  // 0 when m = -inf
            if (need) {
                l *= alpha;
                m = mx;
            }
            // this half's O columns move to the new reference (warp-uniform
            // decision) once P V of key tile j - 1 has landed; S(j) completing
            // implies P V of tile j - 2 has, so the barrier is at most one phase
            // behind this wait. Both warps of the pair see the same maxima, so
            // they take this branch together.
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                ok = warp_wait(&bars->pv_done[t], (j - 1) & 1, abort, err, wait_ns);
                if (ok) {
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 64; c += 32) {
                        uint32_t v[32];
                        tmem_ld32(ocol + (uint32_t)c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(ocol + (uint32_t)c, v);
                    }
                    tmem_wait_st();
                }
                ok = barrier_and(pair_bar, 64, ok);  // the pair leaves together
                if (!ok) break;
            }
            const float ms = m == -INFINITY ? 0.f : m * sc;
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float p0 = fast_exp2(fmaf(x[2 * c], sc, -ms)), p1 = fast_exp2(fmaf(x[2 * c + 1], sc, -ms));
                l += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
            }
            // P of keys [32 half, 32 half + 32) as bf16 pairs in columns [16 half, 16 half + 16)
            tmem_st16(sbuf + 16u * (uint32_t)half, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_full[t][sb]);
        }
        // epilogue: O / l -> out (bf16), lse. P V of the last two key tiles may
        // both be outstanding: wait for their phases in order (a parity wait
        // must never run two phases ahead of the barrier)
        if (ok && tiles_my > 1) ok = warp_wait(&bars->pv_done[t], (tiles_my - 2) & 1, abort, err, wait_ns);
        if (ok && tiles_my > 0) ok = warp_wait(&bars->pv_done[t], (tiles_my - 1) & 1, abort, err, wait_ns);
        // the row sum: this half's share plus the other's (both relative to m)
        float* xb = xch + (xe & 1) * (2 * kARows);
        xb[half * kARows + row] = l;
        ok = barrier_and(pair_bar, 64, ok);
        if (ok) {
            const float l_row = half == 0 ? l + xb[kARows + row] : xb[row] + l;
            tc_fence_after();
            const float inv_l = l_row > 0.f ? 1.f / l_row : 0.f;
            __nv_bfloat16* dst = args.out + (((size_t)b * args.s_q + s) * args.H + h) * kDV + 64 * half;
#pragma unroll 1
            for (int c = 0; c < 64; c += 32) {
                uint32_t v[32];
                if (tiles_my > 0) {
                    tmem_ld32(ocol + (uint32_t)c, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
                if (valid_row) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint4 o;
                        o.x = pack_bf16x2(__uint_as_float(v[8 * w + 0]) * inv_l, __uint_as_float(v[8 * w + 1]) * inv_l);
                        o.y = pack_bf16x2(__uint_as_float(v[8 * w + 2]) * inv_l, __uint_as_float(v[8 * w + 3]) * inv_l);
                        o.z = pack_bf16x2(__uint_as_float(v[8 * w + 4]) * inv_l, __uint_as_float(v[8 * w + 5]) * inv_l);
                        o.w = pack_bf16x2(__uint_as_float(v[8 * w + 6]) * inv_l, __uint_as_float(v[8 * w + 7]) * inv_l);
                        reinterpret_cast<uint4*>(dst + c)[w] = o;
                    }
                }
            }
            if (valid_row && half == 0)
                args.lse[((size_t)b * args.s_q + s) * args.H + h] =
                    l_row > 0.f ? (m * sc + log2f(l_row)) * 0.69314718055994530942f : -INFINITY;
        }
    }
    if (!ok) *abort = 1;
    tc_fence_before();
    __syncthreads();
    if (warp == kAWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kATmemCols);
    }
}

cudaError_t prepare_attn() {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kASmem);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

}  // namespace

cudaError_t launch_prefill_gather(const void* kv, int num_blocks, const int32_t* table, int mbps,
                                  const int32_t* seqlens, int B, int H, void* C, void* Kbuf, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)mbps, (unsigned)B, 1);
    cfg.blockDim = dim3(kGatherThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const size_t R = (size_t)B * mbps * kPage;
    return cudaLaunchKernelEx(&cfg, prefill_gather_kernel, static_cast<const __nv_bfloat16*>(kv), num_blocks, table,
                              mbps, seqlens, H, R, static_cast<__nv_bfloat16*>(C), static_cast<__nv_bfloat16*>(Kbuf));
}

cudaError_t launch_prefill_attn(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                                const int32_t* seqlens, int B, int s_q, int H, int Lmax, float scale, int causal,
                                void* out, float* lse, long long wait_ns, cudaStream_t stream) {
    cudaError_t e = prepare_attn();
    if (e != cudaSuccess) return e;
    PrefillMaps maps;
    maps.q = *tq;
    maps.k = *tk;
    maps.v = *tv;
    PrefillArgs a;
    a.seqlens = seqlens;
    a.s_q = s_q;
    a.H = H;
    a.Lmax = Lmax;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.causal = causal;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.err = &g_prefill_error;
    a.wait_ns = wait_ns;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((s_q + kATiles * kARows - 1) / (kATiles * kARows)), (unsigned)H, (unsigned)B);
    cfg.blockDim = dim3(kAThreads, 1, 1);
    cfg.dynamicSmemBytes = kASmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_attn_kernel, maps, a);
}

// Reads this file's error word into *out and clears it, in stream order.
cudaError_t prefill_error_fetch(int* out, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_prefill_error, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    static const int zero = 0;
    return cudaMemcpyToSymbolAsync(g_prefill_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
}

}  // namespace mla
