// finalize.cu - the decode's split merge fused with the output projection.
//
// What it computes: out[b,s,h,:] = o[b,s,h,:] . W_UV[h] ("DeepSeek-V3 MLA deep
// engineering", sec. 2.2: the value up-projection applied on the latent side
// after attention), where o is the attention output of the row. For a row
// whose sequence the decode split into pieces i (each normalised by its own
// softmax sum, with log-sum-exp lse_i):
//   L = max_i lse_i,  lse = L + ln sum_i exp(lse_i - L),  o = sum_i exp(lse_i - lse) o_i,
// the standard merge of softmax pieces (the pages name num_splits and the
// returned lse - "FlashMLA: efficient MLA decode kernel for Hopper GPUs", usage
// example - but not the formula). Rows of unsplit sequences were written by the
// decode as bf16 and are read as they are; rows of empty sequences are zero with
// lse = -inf. The SC11 article ("MLA decode fused operator", Fig. 1 text) fuses
// the output projection into the attention operator to save the round trip of
// the attention output; here the merged rows of split sequences go straight
// into the projection's operand and are never written to memory.
//
// Work decomposition: one CTA per (head, group of 128-row tiles), like the
// weight-resident projection: W_UV[h] (512 x 128 bf16, 128 KB) is loaded once;
// eight merge warps build each tile's A operand stage by stage (four K-stages
// of 128 latent columns, a two-slot ring) in the 128-byte-swizzled K-major
// layout a TMA box would give, one MMA warp issues the products into a
// double-buffered TMEM accumulator, and four epilogue warps store the tile.
// Warps: 0 weight load, 1 MMA issuer and TMEM owner, 2-5 epilogue (warp w reads
// TMEM lane quadrant w % 4), 6-13 merge (warp m owns tile rows 16 m .. 16 m + 15).
// A merge lane holds four rows x four pieces of loads in flight (four bf16
// values each), so that the partial rows (L2 hits: the decode wrote them just
// before) stream at a useful rate through registers alone; the shared memory
// holds the weight.
#include <cuda_bf16.h>
#include <math.h>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kFBM = 128;             // rows per tile
constexpr int kFBK = 128;             // latent columns per K-stage
constexpr int kFStages = 4;           // K = 512
constexpr int kFStageBytes = 32768;   // [2 chunks of 64 columns][128 rows][128 B]
constexpr int kFRing = 2;
constexpr int kFMergeWarps = 8;
constexpr int kFFirstMerge = 6;
constexpr int kFThreads = (kFFirstMerge + kFMergeWarps) * 32;
constexpr int kFRowsPerWarp = kFBM / kFMergeWarps;  // 16
constexpr int kFOffA = kFStages * kFStageBytes;     // after the weight
constexpr int kFOffStage = kFOffA + kFRing * kFStageBytes;
constexpr int kFOffBar = kFOffStage + kFStageBytes;
constexpr int kFBytes = kFOffBar + 256 + 1024;      // + barriers + alignment slack
static_assert(kFBytes <= 232448, "shared memory per CTA");
static_assert(kFRowsPerWarp == 16 && kFBK == 4 * 32, "a merge lane owns 4 columns of a stage; 16 rows per warp");

struct FinBars {
    uint64_t w_full, a_full[kFRing], a_empty[kFRing], acc_full[2], acc_free[2], drain;
    uint32_t tmem_slot;
    int abort;
};
static_assert(sizeof(FinBars) <= 256, "barrier block");

__device__ __forceinline__ float4 f4_zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }

// Four bf16 partial values (8 bytes) widened to fp32.
__device__ __forceinline__ float4 ld_part4(const void* base, size_t elem) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + elem);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
}

__device__ __forceinline__ void fma4(float4& acc, float w, const float4& v) {
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
}

// Writes this lane's four columns (stage columns 4 lane .. 4 lane + 3) of tile
// row `row` into the stage: chunk lane / 16, 16-byte granule (lane % 16) / 2
// at position granule ^ (row % 8), half (lane % 2).
__device__ __forceinline__ void put4(uint8_t* stage, int row, int lane, uint2 v) {
    const int c = lane >> 4, g = (lane & 15) >> 1;
    *reinterpret_cast<uint2*>(stage + c * (kFBM * 128) + row * 128 + ((g ^ (row & 7)) << 4) + (lane & 1) * 8) = v;
}

__device__ __forceinline__ uint2 pack4(const float4& a) {
    return make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
}

__global__ void __launch_bounds__(kFThreads, 1)
    finalize_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_out, FinArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    FinBars* bars = reinterpret_cast<FinBars*>(smem + kFOffBar);
    volatile int* abort = &bars->abort;
    int* err = a.err;
    const long long wait_ns = a.wait_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x;
    const int mtiles = (a.R + kFBM - 1) / kFBM;
    const int t0 = (int)blockIdx.y * a.tiles_per_cta;
    const int ntiles = max(0, min(mtiles, t0 + a.tiles_per_cta) - t0);

    if (threadIdx.x == 0) {
        mbar_init(&bars->w_full, 1);
        for (int i = 0; i < kFRing; ++i) {
            mbar_init(&bars->a_full[i], kFMergeWarps);
            mbar_init(&bars->a_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->acc_full[i], 1);
            mbar_init(&bars->acc_free[i], 4);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tm_w);
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
    // the weight does not depend on the previous kernel: request it before waiting
    if (warp == 0 && lane == 0 && ntiles > 0) {
        mbar_arrive_expect_tx(&bars->w_full, kFStages * kFStageBytes);
        for (int kc = 0; kc < kFStages; ++kc)  // [2 column chunks][128 latent rows][64]
            tma_load_4d(smem + kc * kFStageBytes, &tm_w, &bars->w_full, 0, kc * kFBK, 0, h);
    }
    griddep_wait();
    griddep_launch_dependents();

    if (warp == 0) {
        // never leave with the weight copy in flight
        if (lane == 0 && ntiles > 0) mbar_wait(&bars->w_full, 0, nullptr, err, kDrainNs);
        __syncwarp();
    } else if (warp == 1) {
        const uint32_t idesc = idesc_bf16_f32(kFBM, 128, false, true);
        bool ok = ntiles > 0 && warp_wait(&bars->w_full, 0, abort, err, wait_ns);
        bool issued = false;
        int q = 0;
        for (int t = 0; t < ntiles && ok; ++t) {
            const int buf = t & 1;
            // the epilogue has read this buffer's tile t - 2
            if (t >= 2) ok = warp_wait(&bars->acc_free[buf], ((t >> 1) - 1) & 1, abort, err, wait_ns);
            for (int kc = 0; kc < kFStages && ok; ++kc, ++q) {
                const int slot = q % kFRing;
                ok = warp_wait(&bars->a_full[slot], (q / kFRing) & 1, abort, err, wait_ns);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ad0 = desc_sw128(smem_u32(smem + kFOffA + slot * kFStageBytes), 0, 1024);
                const uint64_t bd0 = desc_sw128(smem_u32(smem + kc * kFStageBytes), kFBK * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < kFBK / 16; ++kk) {
                    const uint64_t ad = ad0 + (uint64_t)(((kk >> 2) * (kFBM * 128) + (kk & 3) * 32) >> 4);
                    const uint64_t bd = bd0 + (uint64_t)((kk * 2048) >> 4);
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
        if (!ok) *abort = 1;
    } else if (warp < kFFirstMerge) {
        // epilogue: TMEM -> bf16 -> staging ([2 chunks][128 rows][128 B], swizzled) -> TMA store
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint8_t* stage = smem + kFOffStage;
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
                uint8_t* box = stage + (c >> 1) * (kFBM * 128) + row * 128;
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
                tma_store_4d(&tm_out, stage, 0, (t0 + t) * kFBM, 0, h);
                bulk_commit_group();
                stored = true;
            }
        }
        if (leader && stored) bulk_wait_group0();
    } else {
        // merge warps: this warp's 16 rows of every tile, stage by stage
        const int mw = warp - kFFirstMerge;
        const int H = a.H, s_q = a.s_q;
        bool ok = true;
        int q = 0;
        for (int t = 0; t < ntiles && ok; ++t) {
            const int m0 = (t0 + t) * kFBM + mw * kFRowsPerWarp;
            // lane j < 16: row m0 + j's first piece, piece count and merged lse
            // (rows past R: no pieces, written as zeros and never stored)
            int first = 0, n = 0, s = 0;
            float total = -INFINITY;
            if (lane < kFRowsPerWarp && m0 + lane < a.R) {
                const int r = m0 + lane;
                const int b = r / s_q;
                s = r - b * s_q;
                first = a.num_splits[b];
                n = a.num_splits[b + 1] - first;
                if (n != 1) {
                    float L = -INFINITY;
                    for (int i = 0; i < n; ++i) L = fmaxf(L, a.lse_part[((size_t)(first + i) * s_q + s) * H + h]);
                    if (L != -INFINITY) {
                        float sum = 0.f;
                        for (int i = 0; i < n; ++i) sum += expf(a.lse_part[((size_t)(first + i) * s_q + s) * H + h] - L);
                        total = L + logf(sum);
                    }
                    a.lse[(size_t)r * H + h] = total;
                }
            }
            for (int kc = 0; kc < kFStages && ok; ++kc, ++q) {
                const int slot = q % kFRing;
                // the products of stage q - 2 have read this slot
                if (q >= kFRing) ok = warp_wait(&bars->a_empty[slot], ((q / kFRing) - 1) & 1, abort, err, wait_ns);
                if (!ok) break;
                uint8_t* stage = smem + kFOffA + slot * kFStageBytes;
                const int col = kc * kFBK + 4 * lane;  // this lane's four latent columns
#pragma unroll 1
                for (int j0 = 0; j0 < kFRowsPerWarp; j0 += 4) {
                    int rf[4], rn[4], rs[4];
                    float rt[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        rf[jj] = __shfl_sync(0xffffffffu, first, j0 + jj);
                        rn[jj] = __shfl_sync(0xffffffffu, n, j0 + jj);
                        rs[jj] = __shfl_sync(0xffffffffu, s, j0 + jj);
                        rt[jj] = __shfl_sync(0xffffffffu, total, j0 + jj);
                    }
                    // issue every load of the four rows (first four pieces) before any use
                    float4 v[4][4];
                    float w[4][4];
                    uint2 u[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const size_t orow = (size_t)(m0 + j0 + jj) * H + h;
                        u[jj] = make_uint2(0u, 0u);
                        if (rn[jj] == 1)
                            u[jj] = *reinterpret_cast<const uint2*>(
                                static_cast<const __nv_bfloat16*>(a.o_lat) + orow * kDLatent + col);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            w[jj][i] = -INFINITY;
                            v[jj][i] = f4_zero();
                            if (rn[jj] >= 2 && i < rn[jj] && rt[jj] != -INFINITY) {
                                const size_t prow = ((size_t)(rf[jj] + i) * s_q + rs[jj]) * H + h;
                                w[jj][i] = a.lse_part[prow];
                                v[jj][i] = ld_part4(a.o_part, prow * kDLatent + col);
                            }
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        if (rn[jj] == 1) {
                            put4(stage, mw * kFRowsPerWarp + j0 + jj, lane, u[jj]);
                            continue;
                        }
                        float4 acc = f4_zero();
                        if (rn[jj] >= 2 && rt[jj] != -INFINITY) {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                if (i < rn[jj]) fma4(acc, expf(w[jj][i] - rt[jj]), v[jj][i]);
                            // pieces 4, 5, ... (long sequences), in ascending order
                            for (int i = 4; i < rn[jj]; ++i) {
                                const size_t prow = ((size_t)(rf[jj] + i) * s_q + rs[jj]) * H + h;
                                fma4(acc, expf(a.lse_part[prow] - rt[jj]), ld_part4(a.o_part, prow * kDLatent + col));
                            }
                        }
                        put4(stage, mw * kFRowsPerWarp + j0 + jj, lane, pack4(acc));
                    }
                }
                // the tensor pipe reads the stage next
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->a_full[slot]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace

cudaError_t launch_finalize(const CUtensorMap* tm_w, const CUtensorMap* tm_out, const FinArgs& args,
                            cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFBytes);
    if (e != cudaSuccess) return e;
    const int sm_count = device_sm_count();
    if (sm_count <= 0) return cudaErrorInvalidDevice;
    const int mtiles = (args.R + kFBM - 1) / kFBM;
    // one CTA per SM: as many row-tile groups per head as the SMs beyond one per
    // head allow, each group one contiguous run of tiles
    const int groups = max(1, min(mtiles, sm_count / args.H));
    FinArgs a = args;
    a.tiles_per_cta = (mtiles + groups - 1) / groups;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)args.H, (unsigned)((mtiles + a.tiles_per_cta - 1) / a.tiles_per_cta), 1);
    cfg.blockDim = dim3(kFThreads, 1, 1);
    cfg.dynamicSmemBytes = kFBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, finalize_kernel, *tm_w, *tm_out, a);
}

}  // namespace mla
