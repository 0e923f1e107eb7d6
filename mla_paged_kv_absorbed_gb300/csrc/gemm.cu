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
    if (args.n_cta == 128) return launch_variant<128, 3>(tm_a, tm_b, tm_out, args, wait_ns, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mla
