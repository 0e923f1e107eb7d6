// quant.cu - quantisation of bf16 cache rows into the INT8 record format
// (quant.cuh): [c_KV 512 | k_rope 64] bf16 -> [512 INT8 codes | 64 bf16] + a
// power-of-two scale per row.
//
// One warp per row: lane l holds the latent's 16-byte words l and l + 32
// (16 values), the row maximum is a shuffle reduction, and each lane writes its
// 16 codes as two 8-byte words; lanes 0-7 copy the rope part's eight words.
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "quant.cuh"

namespace mla {
namespace {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ uint2 codes8(uint4 v, float inv_s) {
    const uint32_t* u = reinterpret_cast<const uint32_t*>(&v);
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        c[2 * i] = q8_code(__uint_as_float(u[i] << 16), inv_s);
        c[2 * i + 1] = q8_code(__uint_as_float(u[i] & 0xFFFF0000u), inv_s);
    }
    return make_uint2(c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24), c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24));
}

__device__ __forceinline__ float amax8(uint4 v) {
    const uint32_t* u = reinterpret_cast<const uint32_t*>(&v);
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(u[i] << 16)), fabsf(__uint_as_float(u[i] & 0xFFFF0000u))));
    return m;
}

__global__ void __launch_bounds__(kQuantThreads)
    quantize_kernel(const __nv_bfloat16* __restrict__ kv, long long rows, uint8_t* __restrict__ rec,
                    float* __restrict__ scale) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const uint4* src = reinterpret_cast<const uint4*>(kv + row * kDQK);
    const uint4 a = src[lane], b = src[lane + 32];
    float m = fmaxf(amax8(a), amax8(b));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = q8_scale(m);
    const float inv_s = 1.f / s;  // exact: s is a power of two
    uint2* dst = reinterpret_cast<uint2*>(rec + row * kQ8Record);
    dst[lane] = codes8(a, inv_s);
    dst[lane + 32] = codes8(b, inv_s);
    if (lane < 8) reinterpret_cast<uint4*>(rec + row * kQ8Record + kDLatent)[lane] = src[kDLatent / 8 + lane];
    if (lane == 0) scale[row] = s;
}

}  // namespace

cudaError_t launch_quantize(const void* kv, long long rows, void* rec, float* scale, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int per = kQuantThreads / 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + per - 1) / per), 1, 1);
    cfg.blockDim = dim3(kQuantThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_kernel, static_cast<const __nv_bfloat16*>(kv), rows,
                              static_cast<uint8_t*>(rec), scale);
}

}  // namespace mla
