// combine.cu - split-KV log-sum-exp combine.
//
// For a query row whose sequence was split into pieces i (disjoint key ranges,
// each already normalised by its own softmax sum):
//   L = max_i lse_i,  lse = L + ln sum_i exp(lse_i - L),  o = sum_i exp(lse_i - lse) o_i.
// The pages name num_splits and the returned lse ("FlashMLA: efficient MLA
// decode kernel for Hopper GPUs", usage example) but not the formula; this is
// the standard merge of softmax pieces.
//
// One CTA per (batch, query token); one warp per head row; each lane owns 16
// of the 512 latent columns as four float4 (coalesced 512-byte rows). Batches
// with a single piece were written directly by the decode kernel and are
// skipped; batches with no piece (seqlen 0) get o = 0, lse = -inf.
#include <cuda_bf16.h>
#include <math.h>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) combine_kernel(const int32_t* __restrict__ num_splits, int s_q, int H,
                                                           const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           __nv_bfloat16* __restrict__ o_lat,
                                                           float* __restrict__ lse) {
    // launched as a programmatic dependent of the decode kernel: wait for it
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.x / s_q;
    const int s = blockIdx.x % s_q;
    const int first = num_splits[b];
    const int n = num_splits[b + 1] - first;
    if (n == 1) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int h = warp; h < H; h += kThreads / 32) {
        const size_t row = ((size_t)b * s_q + s) * H + h;
        float4 acc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        float total = -INFINITY;
        if (n > 1) {
            float L = -INFINITY;
            for (int i = 0; i < n; ++i) L = fmaxf(L, lse_part[((size_t)(first + i) * s_q + s) * H + h]);
            if (L != -INFINITY) {
                float sum = 0.f;
                for (int i = 0; i < n; ++i) sum += expf(lse_part[((size_t)(first + i) * s_q + s) * H + h] - L);
                total = L + logf(sum);
                for (int i = 0; i < n; ++i) {
                    const size_t prow = ((size_t)(first + i) * s_q + s) * H + h;
                    const float w = expf(lse_part[prow] - total);
                    const float4* src = reinterpret_cast<const float4*>(o_part + prow * kDLatent);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 v = src[lane + 32 * k];
                        acc[k].x += w * v.x;
                        acc[k].y += w * v.y;
                        acc[k].z += w * v.z;
                        acc[k].w += w * v.w;
                    }
                }
            }
        }
        uint2* dst = reinterpret_cast<uint2*>(o_lat + row * kDLatent);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x, acc[k].y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z, acc[k].w);
            uint2 v;
            v.x = *reinterpret_cast<uint32_t*>(&lo);
            v.y = *reinterpret_cast<uint32_t*>(&hi);
            dst[lane + 32 * k] = v;
        }
        if (lane == 0) lse[row] = total;
    }
}

}  // namespace

cudaError_t launch_combine(const int32_t* num_splits, int B, int s_q, int H, const float* o_part,
                           const float* lse_part, void* o_lat, float* lse, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B * s_q, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, num_splits, s_q, H, o_part, lse_part,
                              static_cast<__nv_bfloat16*>(o_lat), lse);
}

}  // namespace mla
