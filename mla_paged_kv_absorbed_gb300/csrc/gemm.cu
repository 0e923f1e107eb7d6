// gemm.cu - per-head batched bf16 GEMM on tcgen05, used by both projections
// around the attention:
//   absorb   q_abs[r,h,0:512] = q[r,h,0:128] . W_UK[h]   (K = 128, N = 512)
//            q_abs[r,h,512:576] = q[r,h,128:192]          (rope part, copied)
//   out-proj out[r,h,:]       = o_lat[r,h,:] . W_UV[h]    (K = 512, N = 128)
// ("DeepSeek-V3 MLA deep engineering", sec. 2.2 and sec. 2.4.)
//
// head_gemm_kernel (the out-projection; also usable for any K that is a
// multiple of 128) - one CTA computes a [128 rows x n_cta] tile of one head: rows are the
// B * s_q query tokens (TMA zero-fills rows past the end), the accumulator
// lives in TMEM (n_cta fp32 columns), A (activations, K-major) and B (the
// head's weight, N-major) stream through a TMA ring of 128-deep K stages in
// 128-byte-swizzled shared memory. Each stage is two boxes only - A as
// [2 chunks][128 rows][64], B as [n_cta/64 chunks][128 k][64] through 4-D
// views - because the TMA engine of an SM spends a large fixed time per box
// (8-16 KB boxes stream at 20-35 GB/s per SM, 64 KB boxes at ~110).
// Warp 0 produces, one thread of warp 1 issues the MMAs, and all four warps
// run the epilogue: TMEM -> bf16 -> the (now idle) stage buffers in the same
// swizzled layout -> one TMA tensor store.
//
// absorb_kernel (the absorb, K = 128) - further down: a persistent kernel over
// 128-column units that overlaps one unit's store with the next units' loads.
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {

__device__ int g_gemm_error = 0;

namespace {

constexpr int kThreads = 128;
constexpr int kBM = 128;
constexpr int kBK = 128;  // K per stage: two 64-wide swizzle chunks

template <int NCTA, int STAGES>
struct GemmSmem {
    static constexpr int kABytes = kBM * kBK * 2;          // 32 KB: [2][128 rows][64]
    static constexpr int kBBytes = kBK * NCTA * 2;         // [NCTA/64][128 k][64]
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kBarOffset = STAGES * kStageBytes;
    static constexpr int kBytes = kBarOffset + 256 + 1024;  // + barriers + alignment slack
    static_assert(kStageBytes * STAGES >= kBM * NCTA * 2, "epilogue staging fits the stage buffers");
};

template <int NCTA, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    head_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_out, GemmArgs args, long long wait_ns) {
    using L = GemmSmem<NCTA, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
    uint64_t* empty = full + STAGES;
    uint64_t* done = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * NCTA;
    const int m0 = blockIdx.y * kBM;
    const int h = blockIdx.z;
    const int num_k = args.K / kBK;
    int* err = &g_gemm_error;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort = 0;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_out);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, NCTA);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // launched as a programmatic dependent: the set-up above overlaps the
    // previous kernel; no global memory is touched before it has completed
    griddep_wait();
    griddep_launch_dependents();

    if (warp == 0 && lane == 0) {
        // producer
        int issued = 0;
        for (int kc = 0; kc < num_k; ++kc) {
            const int s = kc % STAGES;
            if (kc >= STAGES && !mbar_wait(&empty[s], ((kc / STAGES) - 1) & 1, abort, err, wait_ns)) break;
            uint8_t* a_dst = smem + s * L::kStageBytes;
            uint8_t* b_dst = a_dst + L::kABytes;
            mbar_arrive_expect_tx(&full[s], L::kStageBytes);
            tma_load_4d(a_dst, &tm_a, &full[s], 0, m0, 2 * kc, args.a_shared ? 0 : h);
            if (args.b_kmajor)  // [NCTA rows][2 K chunks][64] as [chunk][row][64]
                tma_load_4d(b_dst, &tm_b, &full[s], 0, n0, 2 * kc, h);
            else
                tma_load_4d(b_dst, &tm_b, &full[s], 0, kc * kBK, n0 / 64, h);
            issued = kc + 1;
        }
        // never leave with a copy in flight: wait for the last load of every stage
        for (int kc = issued - STAGES > 0 ? issued - STAGES : 0; kc < issued; ++kc)
            mbar_wait(&full[kc % STAGES], (kc / STAGES) & 1, nullptr, err, kDrainNs);
    } else if (warp >= 2 && args.rope_src != nullptr) {
        // rope columns (absorb): q[r,h,128:192] -> q_abs[r,h,512:576], 128 bytes per
        // row. The CTAs of the head's n tiles share the tile's rows; eight
        // consecutive threads move one row, so each warp instruction covers four
        // whole 128-byte rows. Done by the two idle warps while the stage loads.
        const int nt = (int)gridDim.x;
        const int rows_per = (kBM + nt - 1) / nt;
        const int r0 = m0 + (int)blockIdx.x * rows_per;
        const int r1 = min(min(r0 + rows_per, m0 + kBM), args.R);
        const int tt = threadIdx.x - 64;  // 0..63
        for (int base = r0 * 8; base < r1 * 8; base += 64 * 8) {
            uint4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int idx = base + i * 64 + tt;  // row * 8 + 16-byte word
                if (idx < r1 * 8) {
                    const int row = idx >> 3, w = idx & 7;
                    v[i] = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(args.rope_src) +
                                                          ((size_t)row * args.H + h) * kDQ + kDNope)[w];
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int idx = base + i * 64 + tt;
                if (idx < r1 * 8) {
                    const int row = idx >> 3, w = idx & 7;
                    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.out) +
                                             ((size_t)row * args.H + h) * args.out_row_elems + kDLatent)[w] = v[i];
                }
            }
        }
    } else if (warp == 1) {
        // MMA issuer
        const uint32_t idesc = idesc_bf16_f32(kBM, NCTA, false, args.b_kmajor == 0);
        bool ok = true;
        for (int kc = 0; kc < num_k && ok; ++kc) {
            const int s = kc % STAGES;
            ok = warp_wait(&full[s], (kc / STAGES) & 1, abort, err, wait_ns);
            if (!ok) break;
            tc_fence_after();
            {
                // whole warp, one elected lane issues (warp-uniform operands)
                const uint32_t a_base = smem_u32(smem + s * L::kStageBytes);
                const uint32_t b_base = a_base + L::kABytes;
                const uint64_t ad0 = desc_sw128(a_base, 0, 1024);
                // N-major B: n-chunks are 128 k-rows apart, a K-step is 16 k-rows;
                // K-major B: like A, a K-step is 32 bytes inside the 128-byte rows
                const uint64_t bd0 = args.b_kmajor ? desc_sw128(b_base, 0, 1024) : desc_sw128(b_base, kBK * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t ad = ad0 + (uint64_t)(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
                    const uint64_t bd = args.b_kmajor
                                            ? bd0 + (uint64_t)(((kk >> 2) * (NCTA * 128) + (kk & 3) * 32) >> 4)
                                            : bd0 + (uint64_t)((kk * 2048) >> 4);
                    mma_bf16_ss(tmem, ad, bd, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
        }
        mma_commit(done);  // also covers the partial run on abort
    }

    // epilogue: thread t owns tile row t (output row m0 + t). Every load and MMA
    // is complete once `done` fires, so the stage buffers take the bf16 tile as
    // [NCTA/64 chunks][128 rows][128 B] (swizzled), which one TMA box stores
    // (rows past R are clipped).
    const bool ok = mbar_wait(done, 0, nullptr, err, kDrainNs) && !*abort;
    tc_fence_after();
    const int t = threadIdx.x;
#pragma unroll 1
    for (int c = 0; c < NCTA / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c * 32), v);
        tmem_wait_ld();
        uint8_t* box = smem + (c / 2) * (kBM * 128) + t * 128;  // chunk of 64 columns, row t
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gidx = (c & 1) * 4 + i;  // 16-byte granule inside the 128-byte row
            *reinterpret_cast<uint4*>(box + ((gidx ^ (t & 7)) * 16)) =
                make_uint4(pack_bf16x2(__uint_as_float(v[8 * i + 0]), __uint_as_float(v[8 * i + 1])),
                           pack_bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                           pack_bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                           pack_bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
        }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (t == 0 && ok) {
        tma_store_4d(&tm_out, smem, 0, m0, n0 / 64, h);
        bulk_commit_group();
        bulk_wait_group_read0();
    }
    if (t == 0 && ok) bulk_wait_group0();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, NCTA);
}

template <int NCTA, int STAGES>
cudaError_t launch_variant(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const CUtensorMap* tm_out,
                           const GemmArgs& args, long long wait_ns, cudaStream_t stream) {
    using L = GemmSmem<NCTA, STAGES>;
    auto kern = head_gemm_kernel<NCTA, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(args.N / NCTA, (args.R + kBM - 1) / kBM, args.H);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, *tm_a, *tm_b, *tm_out, args, wait_ns);
}

// ---------------------------------------------------------------------------
// wres_gemm_kernel: the K = 512, N = 128 head GEMMs (the out-projection and the
// prefill's two decompression GEMMs) with the head's weight resident. One CTA
// per (head, group of 128-row tiles) loads W[h] (512 x 128 bf16 = 128 KB, four
// 128-deep K-stages, the same boxes as head_gemm_kernel) once, then streams its
// tiles' A rows through a two-slot ring of 32 KB K-stages. The accumulator is
// double-buffered in TMEM (2 x 128 columns), so the products of tile t + 1 run
// while four epilogue warps move tile t through a 32 KB staging buffer to a TMA
// store. Against one CTA per (head, tile), the weight is read once per CTA
// instead of once per tile, and a few tiles per head (B * s_q = 264 rows: 3
// tiles) run in one wave instead of 2.5.
// Warps: 0 TMA producer, 1 MMA issuer and TMEM owner, 2-5 epilogue (warp w
// reads TMEM lane quadrant w % 4, one thread per tile row).
constexpr int kWrThreads = 192;
constexpr int kWrStages = 4;           // K = 512 as four stages of 128
constexpr int kWrStageBytes = 32768;   // [2 chunks][128 rows][64] bf16
constexpr int kWrRing = 2;
constexpr int kWrOffA = kWrStages * kWrStageBytes;          // after the weight
constexpr int kWrOffStage = kWrOffA + kWrRing * kWrStageBytes;
constexpr int kWrOffBar = kWrOffStage + kWrStageBytes;
constexpr int kWrBytes = kWrOffBar + 256 + 1024;            // + barriers + alignment slack
static_assert(kWrBytes <= 232448, "shared memory per CTA");

struct WrBars {
    uint64_t w_full, a_full[kWrRing], a_empty[kWrRing], acc_full[2], acc_free[2], drain;
    uint32_t tmem_slot;
    int abort;
};
static_assert(sizeof(WrBars) <= 256, "barrier block");

__global__ void __launch_bounds__(kWrThreads, 1)
    wres_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_out, GemmArgs args, int tiles_per_cta, long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    WrBars* bars = reinterpret_cast<WrBars*>(smem + kWrOffBar);
    volatile int* abort = &bars->abort;
    int* err = &g_gemm_error;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x;
    const int mtiles = (args.R + kBM - 1) / kBM;
    const int t0 = (int)blockIdx.y * tiles_per_cta;
    const int ntiles = max(0, min(mtiles, t0 + tiles_per_cta) - t0);

    if (threadIdx.x == 0) {
        mbar_init(&bars->w_full, 1);
        for (int i = 0; i < kWrRing; ++i) {
            mbar_init(&bars->a_full[i], 1);
            mbar_init(&bars->a_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->acc_full[i], 1);
            mbar_init(&bars->acc_free[i], 4);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_out);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    griddep_wait();
    griddep_launch_dependents();

    if (warp == 0) {
        if (lane == 0 && ntiles > 0) {
            mbar_arrive_expect_tx(&bars->w_full, kWrStages * kWrStageBytes);
            for (int kc = 0; kc < kWrStages; ++kc) {
                uint8_t* dst = smem + kc * kWrStageBytes;
                if (args.b_kmajor)  // [2 K chunks][128 n rows][64]
                    tma_load_4d(dst, &tm_b, &bars->w_full, 0, 0, 2 * kc, h);
                else                // [2 n chunks][128 k rows][64]
                    tma_load_4d(dst, &tm_b, &bars->w_full, 0, kc * kBK, 0, h);
            }
            int q = 0;
            bool ok = true;
            for (int t = 0; t < ntiles && ok; ++t) {
                const int m0 = (t0 + t) * kBM;
                for (int kc = 0; kc < kWrStages; ++kc, ++q) {
                    const int slot = q % kWrRing;
                    if (q >= kWrRing) ok = mbar_wait(&bars->a_empty[slot], ((q / kWrRing) - 1) & 1, abort, err, wait_ns);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&bars->a_full[slot], kWrStageBytes);
                    tma_load_4d(smem + kWrOffA + slot * kWrStageBytes, &tm_a, &bars->a_full[slot], 0, m0, 2 * kc,
                                args.a_shared ? 0 : h);
                }
            }
            // never leave with a copy in flight
            mbar_wait(&bars->w_full, 0, nullptr, err, kDrainNs);
            for (int r = q - kWrRing > 0 ? q - kWrRing : 0; r < q; ++r)
                mbar_wait(&bars->a_full[r % kWrRing], (r / kWrRing) & 1, nullptr, err, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        const uint32_t idesc = idesc_bf16_f32(kBM, 128, false, args.b_kmajor == 0);
        bool ok = ntiles > 0 && warp_wait(&bars->w_full, 0, abort, err, wait_ns);
        bool issued = false;
        int q = 0;
        for (int t = 0; t < ntiles && ok; ++t) {
            const int buf = t & 1;
            // the epilogue has read this buffer's tile t - 2
            if (t >= 2) ok = warp_wait(&bars->acc_free[buf], ((t >> 1) - 1) & 1, abort, err, wait_ns);
            for (int kc = 0; kc < kWrStages && ok; ++kc, ++q) {
                const int slot = q % kWrRing;
                ok = warp_wait(&bars->a_full[slot], (q / kWrRing) & 1, abort, err, wait_ns);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a_base = smem_u32(smem + kWrOffA + slot * kWrStageBytes);
                const uint32_t b_base = smem_u32(smem + kc * kWrStageBytes);
                const uint64_t ad0 = desc_sw128(a_base, 0, 1024);
                const uint64_t bd0 = args.b_kmajor ? desc_sw128(b_base, 0, 1024) : desc_sw128(b_base, kBK * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t ad = ad0 + (uint64_t)(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
                    const uint64_t bd = args.b_kmajor ? bd0 + (uint64_t)(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4)
                                                      : bd0 + (uint64_t)((kk * 2048) >> 4);
                    mma_bf16_ss(tmem + 128u * (uint32_t)buf, ad, bd, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bars->a_empty[slot]);
                issued = true;
            }
            if (ok) mma_commit(&bars->acc_full[buf]);
        }
        // every product has completed before TMEM is freed
        if (issued) {
            mma_commit(&bars->drain);
            warp_wait(&bars->drain, 0, nullptr, err, kDrainNs);
        }
    } else {
        // epilogue: TMEM -> bf16 -> staging ([2 chunks][128 rows][128 B], swizzled) -> TMA store
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint8_t* stage = smem + kWrOffStage;
        const bool leader = threadIdx.x == 64;
        bool stored = false, ok = true;
        for (int t = 0; t < ntiles && ok; ++t) {
            const int buf = t & 1;
            ok = warp_wait(&bars->acc_full[buf], (t >> 1) & 1, abort, err, wait_ns);
            // the staging buffer is free once the previous tile's store has read it
            if (leader && stored) bulk_wait_group_read0();
            ok = barrier_and(1, 128, ok);
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + 128u * (uint32_t)buf + (uint32_t)(c * 32), v);
                tmem_wait_ld();
                uint8_t* box = stage + (c >> 1) * (kBM * 128) + row * 128;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int gidx = (c & 1) * 4 + i;
                    *reinterpret_cast<uint4*>(box + ((gidx ^ (row & 7)) * 16)) =
                        make_uint4(pack_bf16x2(__uint_as_float(v[8 * i + 0]), __uint_as_float(v[8 * i + 1])),
                                   pack_bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                                   pack_bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                                   pack_bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
                }
            }
            // TMEM buffer read: the products of tile t + 2 may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->acc_free[buf]);
            fence_proxy_async_smem();
            ok = barrier_and(1, 128, ok);
            if (ok && leader) {
                tma_store_4d(&tm_out, stage, 0, (t0 + t) * kBM, 0, h);
                bulk_commit_group();
                stored = true;
            }
        }
        if (leader && stored) bulk_wait_group0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

cudaError_t launch_wres(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const CUtensorMap* tm_out,
                        const GemmArgs& args, long long wait_ns, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(wres_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWrBytes);
    if (e != cudaSuccess) return e;
    const int sm_count = device_sm_count();
    if (sm_count <= 0) return cudaErrorInvalidDevice;
    const int mtiles = (args.R + kBM - 1) / kBM;
    // one CTA per SM: as many row-tile groups per head as the SMs beyond one
    // per head allow (1 at 128 heads), each group one contiguous run of tiles
    const int groups = max(1, min(mtiles, sm_count / args.H));
    const int per = (mtiles + groups - 1) / groups;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)args.H, (unsigned)((mtiles + per - 1) / per), 1);
    cfg.blockDim = dim3(kWrThreads, 1, 1);
    cfg.dynamicSmemBytes = kWrBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, wres_gemm_kernel, *tm_a, *tm_b, *tm_out, args, per, wait_ns);
}

// ---------------------------------------------------------------------------
// absorb_kernel: the absorb projection (K = 128) as a persistent kernel. Work
// units are (head, 128-row tile, 128-column quarter of the 512 outputs); each
// CTA (one per SM) walks a contiguous range of them, so it keeps the head's
// query tile across its units, and the units' stages overlap: the weight tile
// of a later unit loads while an earlier unit's output is being stored. (One
// CTA per 256-column tile loaded, multiplied and stored in lockstep with all
// the others, so HBM saw a read phase and then a write phase.)
// Warps: 0 TMA producer, 1 MMA issuer and TMEM owner, 2-5 epilogue (one
// thread per tile row: TMEM -> bf16 -> swizzled staging -> TMA store), 6 the
// rope columns of the units with quarter 0.
constexpr int kAbsThreads = 224;
constexpr int kAbsN = 128;      // output columns per unit
constexpr int kAbsQuarters = 4; // 512 / kAbsN
constexpr int kAbsBSlots = 3;

struct AbsSmem {
    static constexpr int kA = kBM * 128 * 2;       // [2 chunks][128 rows][64]: the query tile (K = 128)
    static constexpr int kB = 128 * kAbsN * 2;     // [2 n-chunks][128 k][64]
    static constexpr int kStage = kBM * kAbsN * 2; // [2 chunks][128 rows][64] bf16 output
    static constexpr int kOffA = 0;                // two query slots
    static constexpr int kOffB = kOffA + 2 * kA;   // weight ring
    static constexpr int kOffS = kOffB + kAbsBSlots * kB;  // two staging buffers
    static constexpr int kOffBar = kOffS + 2 * kStage;
    static constexpr int kBytes = kOffBar + 256 + 1024;    // + barriers + alignment slack
};
static_assert(AbsSmem::kBytes <= 232448, "absorb kernel shared memory");

// At most one bulk store group of this thread still reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

struct AbsUnit {
    int h, mt, nq, g;  // head, row tile, column quarter, group = (h, mt)
};
__device__ __forceinline__ AbsUnit abs_unit(int u, int mtiles) {
    AbsUnit x;
    x.g = u / kAbsQuarters;
    x.nq = u % kAbsQuarters;
    x.h = x.g / mtiles;
    x.mt = x.g % mtiles;
    return x;
}

__global__ void __launch_bounds__(kAbsThreads, 1)
    absorb_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                  const __grid_constant__ CUtensorMap tm_out, GemmArgs args, long long wait_ns) {
    using L = AbsSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
    uint64_t* a_empty = a_full + 2;
    uint64_t* b_full = a_empty + 2;
    uint64_t* b_empty = b_full + kAbsBSlots;
    uint64_t* acc_full = b_empty + kAbsBSlots;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* done = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mtiles = (args.R + kBM - 1) / kBM;
    const int units = args.H * mtiles * kAbsQuarters;
    const int u0 = (int)(((long long)blockIdx.x * units) / gridDim.x);
    const int u1 = (int)(((long long)(blockIdx.x + 1) * units) / gridDim.x);
    int* err = &g_gemm_error;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 1);
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);  // one arrival per epilogue warp
        }
        for (int i = 0; i < kAbsBSlots; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        mbar_init(done, 1);
        *abort = 0;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_out);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 2 * kAbsN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // launched as a programmatic dependent: the set-up above overlaps the
    // previous kernel; no global memory is touched before it has completed
    griddep_wait();
    griddep_launch_dependents();

    if (warp == 0) {
        // producer: the whole warp walks the units (uniform waits), lane 0 loads
        bool ok = true;
        int gi = -1, prev_g = -1, issued = 0;
        for (int u = u0; ok && u < u1; ++u) {
            const int i = u - u0;
            const AbsUnit x = abs_unit(u, mtiles);
            if (x.g != prev_g) {
                prev_g = x.g;
                ++gi;
                const int sa = gi & 1;
                // the query slot held group gi - 2 until its last product
                if (gi >= 2) ok = warp_wait(&a_empty[sa], ((gi >> 1) - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&a_full[sa], L::kA);
                    tma_load_4d(smem + L::kOffA + sa * L::kA, &tm_a, &a_full[sa], 0, x.mt * kBM, 0, x.h);
                }
                __syncwarp();
            }
            const int sb = i % kAbsBSlots;
            if (i >= kAbsBSlots) ok = warp_wait(&b_empty[sb], ((i / kAbsBSlots) - 1) & 1, abort, err, wait_ns);
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&b_full[sb], L::kB);
                tma_load_4d(smem + L::kOffB + sb * L::kB, &tm_b, &b_full[sb], 0, 0, x.nq * (kAbsN / 64), x.h);
            }
            __syncwarp();
            issued = i + 1;
        }
        // never leave with a copy in flight: the last load of every slot has landed
        if (lane == 0) {
            for (int i = issued - kAbsBSlots > 0 ? issued - kAbsBSlots : 0; i < issued; ++i)
                mbar_wait(&b_full[i % kAbsBSlots], (i / kAbsBSlots) & 1, nullptr, err, kDrainNs);
            for (int g = gi - 1 > 0 ? gi - 1 : 0; g <= gi; ++g)
                mbar_wait(&a_full[g & 1], (g >> 1) & 1, nullptr, err, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // MMA issuer: unit i into accumulator i % 2
        constexpr uint32_t idesc = idesc_bf16_f32(kBM, kAbsN, false, true);
        bool ok = true, issued = false;
        int gi = -1, prev_g = -1;
        for (int u = u0; ok && u < u1; ++u) {
            const int i = u - u0;
            const AbsUnit x = abs_unit(u, mtiles);
            if (x.g != prev_g) {
                prev_g = x.g;
                ++gi;
            }
            const int sa = gi & 1, sb = i % kAbsBSlots, ac = i & 1;
            ok = warp_wait(&a_full[sa], (gi >> 1) & 1, abort, err, wait_ns);
            if (ok) ok = warp_wait(&b_full[sb], (i / kAbsBSlots) & 1, abort, err, wait_ns);
            // the epilogue has read unit i - 2 out of this accumulator
            if (ok && i >= 2) ok = warp_wait(&acc_empty[ac], ((i >> 1) - 1) & 1, abort, err, wait_ns);
            if (!ok) break;
            tc_fence_after();
            {
                // whole warp, one elected lane issues (warp-uniform operands)
                const uint64_t ad0 = desc_sw128(smem_u32(smem + L::kOffA + sa * L::kA), 0, 1024);
                const uint64_t bd0 = desc_sw128(smem_u32(smem + L::kOffB + sb * L::kB), 128 * 128, 1024);  // n-chunks 128 k-rows apart
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = ad0 + (uint64_t)(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
                    const uint64_t bd = bd0 + (uint64_t)((kk * 2048) >> 4);
                    mma_bf16_ss(tmem + (uint32_t)(ac * kAbsN), ad, bd, idesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(&b_empty[sb]);
                mma_commit(&acc_full[ac]);
                const bool last_of_group = (u + 1 == u1) || ((u + 1) / kAbsQuarters != x.g);
                if (last_of_group) mma_commit(&a_empty[sa]);
            }
            issued = true;
        }
        if (issued) {
            mma_commit(done);
            warp_wait(done, 0, nullptr, err, kDrainNs);
        }
        if (!ok) *abort = 1;
    } else if (warp >= 2 && warp < 6) {
        // epilogue: thread = tile row 32 (warp % 4) + lane (TMEM lane quadrant of the warp)
        const int row = 32 * (warp & 3) + lane;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const bool storer = warp == 2 && lane == 0;
        bool ok = true, stored = false;
        for (int u = u0; u < u1; ++u) {
            const int i = u - u0;
            const AbsUnit x = abs_unit(u, mtiles);
            const int ac = i & 1;
            uint8_t* stage = smem + L::kOffS + ac * L::kStage;
            // the store of unit i - 2 has read this staging buffer (at most one store outstanding)
            if (storer && i >= 2) bulk_wait_group_read1();
            ok = barrier_and(1, 128, ok);
            if (!ok) break;
            ok = warp_wait(&acc_full[ac], (i >> 1) & 1, abort, err, wait_ns);
            ok = barrier_and(2, 128, ok);
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < kAbsN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + (uint32_t)(ac * kAbsN + c * 32), v);
                tmem_wait_ld();
                uint8_t* box = stage + (c / 2) * (kBM * 128) + row * 128;  // chunk of 64 columns, this row
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int gidx = (c & 1) * 4 + q;  // 16-byte granule inside the 128-byte row
                    *reinterpret_cast<uint4*>(box + ((gidx ^ (row & 7)) * 16)) =
                        make_uint4(pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                                   pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                   pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                   pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                }
            }
            // the accumulator may take unit i + 2
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ac]);
            fence_proxy_async_smem();
            ok = barrier_and(3, 128, ok);
            if (!ok) break;
            if (storer) {
                tma_store_4d(&tm_out, stage, 0, x.mt * kBM, x.nq * (kAbsN / 64), x.h);
                bulk_commit_group();
                stored = true;
            }
        }
        if (storer && stored) bulk_wait_group0();
    } else if (warp == 6 && args.rope_src != nullptr) {
        // rope columns q[r,h,128:192] -> q_abs[r,h,512:576] of the units with
        // quarter 0: eight lanes per 128-byte row, eight words per lane in flight
        for (int u = u0; u < u1; ++u) {
            const AbsUnit x = abs_unit(u, mtiles);
            if (x.nq != 0) continue;
            const int r0 = x.mt * kBM, r1 = min(r0 + kBM, args.R);
            for (int base = r0 * 8; base < r1 * 8; base += 32 * 8) {
                uint4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int idx = base + j * 32 + lane;  // row * 8 + 16-byte word
                    if (idx < r1 * 8) {
                        const int r = idx >> 3, w = idx & 7;
                        v[j] = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(args.rope_src) +
                                                              ((size_t)r * args.H + x.h) * kDQ + kDNope)[w];
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int idx = base + j * 32 + lane;
                    if (idx < r1 * 8) {
                        const int r = idx >> 3, w = idx & 7;
                        reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.out) +
                                                 ((size_t)r * args.H + x.h) * args.out_row_elems + kDLatent)[w] = v[j];
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 2 * kAbsN);
}

cudaError_t launch_absorb(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const CUtensorMap* tm_out,
                          const GemmArgs& args, long long wait_ns, cudaStream_t stream) {
    const int sm_count = device_sm_count();
    if (sm_count <= 0) return cudaErrorInvalidDevice;
    cudaError_t e = cudaFuncSetAttribute(absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AbsSmem::kBytes);
    if (e != cudaSuccess) return e;
    const int units = args.H * ((args.R + kBM - 1) / kBM) * kAbsQuarters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units < sm_count ? units : sm_count, 1, 1);
    cfg.blockDim = dim3(kAbsThreads, 1, 1);
    cfg.dynamicSmemBytes = AbsSmem::kBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, absorb_kernel, *tm_a, *tm_b, *tm_out, args, wait_ns);
}

}  // namespace

// Reads the projection kernels' error word into *out and clears it, in stream order
// (the caller synchronises).
cudaError_t gemm_error_fetch(int* out, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_gemm_error, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    static const int zero = 0;
    return cudaMemcpyToSymbolAsync(g_gemm_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
}

cudaError_t launch_head_gemm(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const CUtensorMap* tm_out,
                             const GemmArgs& args, long long wait_ns, cudaStream_t stream) {
    // absorb: K = 128, the persistent kernel over 128-column units; out-proj:
    // K = 512 through three stages, one CTA per head and row tile
    if (args.K == 128 && args.N == kAbsN * kAbsQuarters && args.n_cta == kAbsN)
        return launch_absorb(tm_a, tm_b, tm_out, args, wait_ns, stream);
    // K = 512, N = 128 with several row tiles per head: the weight-resident
    // kernel (one tile per head is faster as one CTA per (head, tile) with a
    // three-stage ring of A and weight stages: 10.7 against 12.4 us on the
    // DeepSeek-V3 decode batch)
    if (args.K == kWrStages * kBK && args.N == 128 && args.n_cta == 128 && args.rope_src == nullptr &&
        args.R > kBM)
        return launch_wres(tm_a, tm_b, tm_out, args, wait_ns, stream);
    if (args.n_cta == 128) return launch_variant<128, 3>(tm_a, tm_b, tm_out, args, wait_ns, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mla
