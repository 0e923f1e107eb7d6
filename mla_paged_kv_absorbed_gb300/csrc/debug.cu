// debug.cu - test hooks exposing single building blocks of the decode path:
//  * a paged gather that loads each page as one whole-page TMA box through the
//    decode kernel's own tensor map (the 3-D [dims, keys, chunk] view of the
//    cache, 128-byte swizzle, built by the same host helper), then un-swizzles
//    the page to HBM;
//  * a one-tile tcgen05 product D[128 x N] = A[128 x K] . B with the same
//    shared-memory layouts and descriptors as the decode kernel (K-major B
//    like the key tile, MN-major B like the value tile); A is read from
//    shared memory, or from tensor memory filled by tcgen05.st (a_tmem = 1)
//    or by tcgen05.cp from the swizzled shared tile (a_tmem = 2).
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

// ------------------------------------------------------------------ gather --
constexpr int kGatherThreads = 256;
constexpr int kGatherChunks = kDQK / 64;  // 9 boxes of [64 tokens x 64 columns]
constexpr int kGatherSmem = kGatherChunks * 8192 + 64 + 1024;

__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(const __grid_constant__ CUtensorMap tm_kv, const int32_t* __restrict__ block_table, int mbps,
                  const int32_t* __restrict__ seqlens, int max_tokens, int num_blocks, __nv_bfloat16* __restrict__ out) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kGatherChunks * 8192);
    const int page = blockIdx.x, b = blockIdx.y;
    const int sl = seqlens[b];
    const int limit = sl < max_tokens ? sl : max_tokens;
    const int t0 = page * kPage;
    if (t0 >= limit || page >= mbps) return;
    const int blk = block_table[(size_t)b * mbps + page];
    if (blk < 0 || blk >= num_blocks) return;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbarrier_init_cluster();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // one box {64 dims, 64 keys, 9 chunks} = the whole page, as the decode kernel loads it
        mbar_arrive_expect_tx(bar, kGatherChunks * 8192);
        tma_load_3d(smem, &tm_kv, bar, 0, blk * kPage, 0);
    }
    // every thread waits (bounded); a timeout leaves out untouched
    const bool ok = mbar_wait(bar, 0, nullptr, nullptr, 2000000000LL);
    if (!ok) return;
    const int rows = limit - t0 < kPage ? limit - t0 : kPage;
    // one 16-byte word per thread step: word w of row t in chunk c sits at
    // position w ^ (t % 8) inside the 128-byte row (128-byte swizzle)
    for (int i = threadIdx.x; i < rows * kGatherChunks * 8; i += kGatherThreads) {
        const int t = i / (kGatherChunks * 8);
        const int rem = i % (kGatherChunks * 8);
        const int c = rem / 8, w = rem % 8;
        const uint4 v = *reinterpret_cast<const uint4*>(smem + c * 8192 + t * 128 + ((w ^ (t & 7)) * 16));
        *reinterpret_cast<uint4*>(out + ((size_t)b * max_tokens + t0 + t) * kDQK + c * 64 + w * 8) = v;
    }
}

// --------------------------------------------------------------------- mma --
constexpr int kMmaThreads = 128;
constexpr int kMmaSmem = 16384 + 32768 + 64 + 1024;

__global__ void __launch_bounds__(kMmaThreads, 1)
    mma_tile_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, int K, int N,
                    int b_kmajor, int a_tmem, const __nv_bfloat16* __restrict__ a_glob, float* __restrict__ d) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;              // [128 rows x 64] K-major, 16 KB
    uint8_t* sB = smem + 16384;      // K-major: [N rows x 64]; MN-major: N/64 atoms of [64 K-rows x 64]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 16384 + 32768);
    uint64_t* full = bars;
    uint64_t* done = bars + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(done, 1);
        fence_mbarrier_init_cluster();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);  // D in columns [0, N), A (when in TMEM) in [256, 288)
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t idesc = idesc_bf16_f32(128, N, false, b_kmajor == 0);
    bool ok = true;
    for (int kc = 0; kc < K / 64 && ok; ++kc) {
        if (threadIdx.x == 0) {
            const uint32_t bytes = 16384 + (uint32_t)N * 128;
            mbar_arrive_expect_tx(full, bytes);
            tma_load_2d(sA, &tm_a, full, 64 * kc, 0);
            if (b_kmajor) {
                tma_load_2d(sB, &tm_b, full, 64 * kc, 0);  // box [64 cols x N rows]
            } else {
                for (int j = 0; j < N / 64; ++j) tma_load_2d(sB + j * 8192, &tm_b, full, 64 * j, 64 * kc);
            }
        }
        if (a_tmem == 1) {
            // row t of this K chunk -> TMEM lane t, 32 columns of bf16 pairs
            const uint32_t* src = reinterpret_cast<const uint32_t*>(a_glob + (size_t)threadIdx.x * K + 64 * kc);
            uint32_t v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = src[i];
            tmem_st32(tmem + ((uint32_t)(warp * 32) << 16) + 256u, v);
            tmem_wait_st();
            tc_fence_before();
        }
        ok = __syncthreads_and(mbar_wait(full, kc & 1, nullptr, nullptr, 2000000000LL));
        tc_fence_after();
        if (ok && warp == 0) {
            // the whole warp runs the issue code; one elected lane issues
            const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
            if (a_tmem == 2) {
                // the A tile goes from shared to tensor memory on the tensor pipe
                // (tcgen05.cp), ahead of the MMAs that read it
                for (int kk = 0; kk < 4; ++kk)
                    tmem_cp_128x256b(tmem + 256u + 8u * kk, desc_sw128(a_base + kk * 32, 0, 1024));
            }
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = b_kmajor ? desc_sw128(b_base + kk * 32, 0, 1024)
                                             : desc_sw128(b_base + kk * 2048, 8192, 1024);
                if (a_tmem) {
                    mma_bf16_ts(tmem, tmem + 256u + 8u * kk, bd, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                } else {
                    const uint64_t ad = desc_sw128(a_base + kk * 32, 0, 1024);
                    mma_bf16_ss(tmem, ad, bd, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                }
            }
            mma_commit(done);
        }
        // the buffers are reused by the next chunk: wait for this chunk's MMAs
        if (ok) ok = mbar_wait(done, kc & 1, nullptr, nullptr, 2000000000LL);
        ok = __syncthreads_and(ok);
    }
    tc_fence_after();
    for (int c = 0; c < N; c += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
        tmem_wait_ld();
        if (ok)
            for (int e = 0; e < 32; ++e) d[(size_t)threadIdx.x * N + c + e] = __uint_as_float(v[e]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_debug_gather(const CUtensorMap* tm_kv, const int32_t* block_table, int mbps, const int32_t* seqlens,
                                int B, int max_tokens, int num_blocks, void* out, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGatherSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((max_tokens + kPage - 1) / kPage, B);
    gather_kernel<<<grid, kGatherThreads, kGatherSmem, stream>>>(*tm_kv, block_table, mbps, seqlens, max_tokens,
                                                                 num_blocks, static_cast<__nv_bfloat16*>(out));
    return cudaGetLastError();
}

cudaError_t launch_debug_mma(const CUtensorMap* tm_a, const CUtensorMap* tm_b, int K, int N, int b_kmajor, int a_tmem,
                             const void* a, float* d, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(mma_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem);
    if (e != cudaSuccess) return e;
    mma_tile_kernel<<<1, kMmaThreads, kMmaSmem, stream>>>(*tm_a, *tm_b, K, N, b_kmajor, a_tmem,
                                                         static_cast<const __nv_bfloat16*>(a), d);
    return cudaGetLastError();
}

}  // namespace mla
