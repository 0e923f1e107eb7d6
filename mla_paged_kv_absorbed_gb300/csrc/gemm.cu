// gemm.cu - per-head batched bf16 GEMM on tcgen05, used by both projections
// around the attention:
//   absorb   q_abs[r,h,0:512] = q[r,h,0:128] . W_UK[h]   (K = 128, N = 512)
//            q_abs[r,h,512:576] = q[r,h,128:192]          (rope part, copied)
//   out-proj out[r,h,:]       = o_lat[r,h,:] . W_UV[h]    (K = 512, N = 128)
// ("DeepSeek-V3 MLA deep engineering", sec. 2.2 and sec. 2.4.)
//
// One CTA computes a [128 rows x n_cta] tile of one head: rows are the
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
            tma_load_4d(a_dst, &tm_a, &full[s], 0, m0, 2 * kc, h);
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
        constexpr uint32_t idesc = idesc_bf16_f32(kBM, NCTA, false, true);
        bool ok = true;
        for (int kc = 0; kc < num_k && ok; ++kc) {
            const int s = kc % STAGES;
            ok = warp_wait(&full[s], (kc / STAGES) & 1, abort, err, wait_ns);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t a_base = smem_u32(smem + s * L::kStageBytes);
                const uint32_t b_base = a_base + L::kABytes;
                const uint64_t ad0 = desc_sw128(a_base, 0, 1024);
                const uint64_t bd0 = desc_sw128(b_base, kBK * 128, 1024);  // n-chunks are 128 k-rows apart
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t ad = ad0 + (uint64_t)(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
                    const uint64_t bd = bd0 + (uint64_t)((kk * 2048) >> 4);
                    mma_bf16_ss(tmem, ad, bd, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
            __syncwarp();
        }
        if (lane == 0) mma_commit(done);  // also covers the partial run on abort
        __syncwarp();
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
    // absorb: K = 128, one stage (two CTAs fit an SM); out-proj: K = 512 through three stages
    if (args.n_cta == 256) return launch_variant<256, 1>(tm_a, tm_b, tm_out, args, wait_ns, stream);
    if (args.n_cta == 128) return launch_variant<128, 3>(tm_a, tm_b, tm_out, args, wait_ns, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mla
