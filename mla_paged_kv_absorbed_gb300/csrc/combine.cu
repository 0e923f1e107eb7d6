// combine.cu - split-KV log-sum-exp combine.
//
// For a query row whose sequence was split into pieces i (disjoint key ranges,
// each already normalised by its own softmax sum):
//   L = max_i lse_i,  lse = L + ln sum_i exp(lse_i - L),  o = sum_i exp(lse_i - lse) o_i.
// The pages name num_splits and the returned lse ("FlashMLA: efficient MLA
// decode kernel for Hopper GPUs", usage example) but not the formula; this is
// the standard merge of softmax pieces.
//
// One warp per query row (b, s, h). Rows are dealt to the warps of the grid
// round-robin (row r goes to warp r mod the grid's warp count), so the rows of
// the few split batches - contiguous in row order - spread evenly over every
// warp instead of queueing on the handful of warps whose range holds them.
// Each lane owns 16 of the 512 latent
// columns as four groups of four (the pieces are bf16: coalesced 256-byte
// rows per instruction, widened to fp32 for the sums). The
// lanes read the pieces' lse values and reduce max and sum by shuffles; the
// pieces are then accumulated in ascending order, four at a time so that 16
// loads per lane are in flight. Batches with a single piece were written
// directly by the decode kernel and are skipped; batches with no piece
// (seqlen 0) get o = 0, lse = -inf.
#include <cuda_bf16.h>
#include <math.h>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 128;
constexpr int kWarpsPerCta = kThreads / 32;

// Four bf16 partial values (8 bytes) widened to fp32.
__device__ __forceinline__ float4 ld_part4(const __nv_bfloat16* __restrict__ p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
}

__device__ void combine_row(const int32_t* __restrict__ num_splits, int row, int s_q, int H,
                            const __nv_bfloat16* __restrict__ o_part, const float* __restrict__ lse_part,
                            __nv_bfloat16* __restrict__ o_lat, float* __restrict__ lse) {
    const int lane = threadIdx.x & 31;
    const int h = row % H;
    const int s = (row / H) % s_q;
    const int b = row / (H * s_q);
    const int first = num_splits[b];
    const int n = num_splits[b + 1] - first;
    if (n == 1) return;
    // the first four pieces' lse and partial rows are requested first, with the
    // reduction's loads right after, so the common case (two to four pieces) costs
    // one memory round trip: none of these addresses depends on a loaded value
    float l4[4];
    float4 v4[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        l4[j] = -INFINITY;
#pragma unroll
        for (int k = 0; k < 4; ++k) v4[j][k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < n) {
            const size_t prow = ((size_t)(first + j) * s_q + s) * H + h;
            l4[j] = lse_part[prow];
            const __nv_bfloat16* src = o_part + prow * kDLatent;
#pragma unroll
            for (int k = 0; k < 4; ++k) v4[j][k] = ld_part4(src + 4 * (lane + 32 * k));
        }
    }
    // lse of piece i of this row
    auto lse_of = [&](int i) { return lse_part[((size_t)(first + i) * s_q + s) * H + h]; };
    float L = -INFINITY;
    for (int i = lane; i < n; i += 32) L = fmaxf(L, lse_of(i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L = fmaxf(L, __shfl_xor_sync(0xffffffffu, L, o));
    float total = -INFINITY;
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (L != -INFINITY) {
        float sum = 0.f;
        for (int i = lane; i < n; i += 32) sum += expf(lse_of(i) - L);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        total = L + logf(sum);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float w = j < n ? expf(l4[j] - total) : 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc[k].x += w * v4[j][k].x;
                acc[k].y += w * v4[j][k].y;
                acc[k].z += w * v4[j][k].z;
                acc[k].w += w * v4[j][k].w;
            }
        }
        // pieces 4, 5, ... (long sequences), four at a time, in ascending order
        for (int i0 = 4; i0 < n; i0 += 4) {
            float4 v[4][4];
            float w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j;
                w[j] = 0.f;
                if (i < n) {
                    const size_t prow = ((size_t)(first + i) * s_q + s) * H + h;
                    w[j] = expf(lse_part[prow] - total);
                    const __nv_bfloat16* src = o_part + prow * kDLatent;
#pragma unroll
                    for (int k = 0; k < 4; ++k) v[j][k] = ld_part4(src + 4 * (lane + 32 * k));
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) v[j][k] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc[k].x += w[j] * v[j][k].x;
                    acc[k].y += w[j] * v[j][k].y;
                    acc[k].z += w[j] * v[j][k].z;
                    acc[k].w += w[j] * v[j][k].w;
                }
        }
    }
    uint2* dst = reinterpret_cast<uint2*>(o_lat + (size_t)row * kDLatent);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x, acc[k].y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z, acc[k].w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        dst[lane + 32 * k] = u;
    }
    if (lane == 0) lse[row] = total;
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const int32_t* __restrict__ num_splits, int rows, int s_q,
                                                           int H, const __nv_bfloat16* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           __nv_bfloat16* __restrict__ o_lat,
                                                           float* __restrict__ lse) {
    // launched as a programmatic dependent of the decode kernel: wait for it
    griddep_wait();
    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stride = (int)gridDim.x * kWarpsPerCta;       // warps in the grid
    const int gw = (int)blockIdx.x * kWarpsPerCta + warp;
    for (long long base = gw; base < rows; base += 32LL * stride) {
        // the piece counts of this warp's next 32 rows, read at once (lane j:
        // row base + j * stride); only rows of split or empty batches have work
        const long long row_j = base + (long long)lane * stride;  // ((b * s_q) + s) * H + h
        int n_j = 1;
        if (row_j < rows) {
            const int b = (int)(row_j / (H * s_q));
            n_j = num_splits[b + 1] - num_splits[b];
        }
        unsigned todo = __ballot_sync(0xffffffffu, n_j != 1);
        while (todo) {
            const int j = __ffs(todo) - 1;
            todo &= todo - 1;
            combine_row(num_splits, (int)(base + (long long)j * stride), s_q, H, o_part, lse_part, o_lat, lse);
        }
    }
}

}  // namespace

cudaError_t launch_combine(const int32_t* num_splits, int B, int s_q, int H, const void* o_part,
                           const float* lse_part, void* o_lat, float* lse, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    const int rows = B * s_q * H;
    const int ctas = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
    const int sm_count = device_sm_count();
    if (sm_count <= 0) return cudaErrorInvalidDevice;
    // up to four CTAs (16 warps) per SM: each split row is a chain of two
    // dependent memory round trips (its pieces' lse, then their partial
    // outputs), so the rows of the whole grid are kept in flight at once
    cfg.gridDim = dim3(ctas < 1 ? 1 : (ctas < 4 * sm_count ? ctas : 4 * sm_count), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, num_splits, rows, s_q, H,
                              static_cast<const __nv_bfloat16*>(o_part), lse_part,
                              static_cast<__nv_bfloat16*>(o_lat), lse);
}

}  // namespace mla
