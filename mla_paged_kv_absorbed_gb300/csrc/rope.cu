// rope.cu - the step before the decode path: rotary encoding of the decoupled
// rope parts and the append of the new tokens to the paged latent cache.
//
// What it computes ("DeepSeek-V3 MLA deep engineering", sec. 3.1: the rope
// query part and the position key are rotated by a position-dependent angle,
// separately from the latent; sec. 3.2: the position key of token t is RoPE
// applied per token; sec. 4.3: only the latent goes into the paged cache,
// kv_cache.store(c_kv)). The pages describe the rotation in words only; it is
// the standard rotary encoding: the 64 rope dims are 32 adjacent pairs
// (x[2i], x[2i+1]), and pair i turns by t * theta_i, theta_i = base^(-2i/64).
//
// For token s of sequence b, at position t = cache_seqlens[b] - s_q + s (the
// lengths already count the new tokens):
//   q[b,s,h,128:192]  <- RoPE(q[b,s,h,128:192], t)        for every head h (in place)
//   kv_cache slot     <- [kv_new[b,s,0:512] | RoPE(kv_new[b,s,512:576], t)]
// where the slot is row t % 64 of block block_table[b][t / 64].
//
// One CTA per (b, s): the 32 angles t * theta_i (theta_i from the host) are
// reduced and turned into (cos, sin) once, in double precision (positions reach tens of thousands of radians, where a
// float angle would lose about a milli-radian), then every head's rope part and
// the new cache row are rotated in fp32 and rounded to bf16. All accesses are
// 16-byte words; the latent is copied unchanged.
//
// With an INT8 cache (quant.cuh) the slot is the token's 640-byte record: the
// latent's INT8 codes under its power-of-two scale (written to the scale
// array), then the rotated rope key in bf16.
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace mla {

__device__ int g_rope_error = 0;

namespace {

constexpr int kRopeThreads = 128;
constexpr int kPairs = kDRope / 2;  // 32
constexpr int kQWords = 128 * 8 / kRopeThreads;  // rope words of q per thread at H = 128

// theta_i = base^(-2i/64) for the 32 pairs, computed once on the host (the
// same double-precision formula for every token, so no CTA repeats it)
struct RopeTheta {
    double v[kPairs];
};

__device__ __forceinline__ uint32_t rotate_pair(uint32_t packed, float c, float s) {
    const float x0 = __uint_as_float(packed << 16), x1 = __uint_as_float(packed & 0xFFFF0000u);
    return pack_bf16x2(x0 * c - x1 * s, x0 * s + x1 * c);
}

// Rotates the four pairs of one 16-byte word (pairs 4 w .. 4 w + 3).
__device__ __forceinline__ uint4 rotate_word(uint4 v, const float2* cs, int w) {
    const float2 a = cs[4 * w], b = cs[4 * w + 1], c = cs[4 * w + 2], d = cs[4 * w + 3];
    return make_uint4(rotate_pair(v.x, a.x, a.y), rotate_pair(v.y, b.x, b.y), rotate_pair(v.z, c.x, c.y),
                      rotate_pair(v.w, d.x, d.y));
}

template <bool kQ8>
__global__ void __launch_bounds__(kRopeThreads)
    rope_append_kernel(__nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kv_new,
                       const int32_t* __restrict__ seqlens, const int32_t* __restrict__ block_table, int mbps,
                       __nv_bfloat16* __restrict__ kv_cache, uint8_t* __restrict__ kv8, float* __restrict__ kv_scale,
                       int num_blocks, int s_q, int H, const __grid_constant__ RopeTheta th) {
    __shared__ float2 cs[kPairs];
    __shared__ float red[2];
    griddep_wait();
    griddep_launch_dependents();
    const int row = blockIdx.x;  // b * s_q + s
    const int b = row / s_q, s = row % s_q;
    const int t = seqlens[b] - s_q + s;
    if (t < 0) return;  // no such token: the sequence is shorter than s_q
    // every head's rope part (8 words of 16 bytes per head) is requested before
    // the angles are computed, so the loads overlap the double-precision work
    auto qword = [&](int i) {
        return reinterpret_cast<uint4*>(q + ((size_t)row * H + (i >> 3)) * kDQ + kDNope) + (i & 7);
    };
    uint4 qw[kQWords];
#pragma unroll
    for (int k = 0; k < kQWords; ++k) {
        const int i = threadIdx.x + k * kRopeThreads;
        if (i < H * 8) qw[k] = *qword(i);
    }
    if (threadIdx.x < kPairs) {
        double sn, c;
        sincos((double)t * th.v[threadIdx.x], &sn, &c);
        cs[threadIdx.x] = make_float2((float)c, (float)sn);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kQWords; ++k) {
        const int i = threadIdx.x + k * kRopeThreads;
        if (i < H * 8) *qword(i) = rotate_word(qw[k], cs, i & 7);
    }

    // the new token's cache row: 64 words of latent (copied) + 8 words of rope (rotated)
    const int j = t / kPage;
    const int blk = j < mbps ? block_table[(size_t)b * mbps + j] : -1;
    if (blk < 0 || blk >= num_blocks) {
        if (threadIdx.x == 0) record_error(&g_rope_error, kErrBadBlock);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(kv_new + (size_t)row * kDQK);
    const size_t slot = (size_t)blk * kPage + t % kPage;
    if (!kQ8) {
        uint4* dst = reinterpret_cast<uint4*>(kv_cache + slot * kDQK);
        if (threadIdx.x < kDLatent / 8) {
            dst[threadIdx.x] = src[threadIdx.x];
        } else if (threadIdx.x < kDLatent / 8 + 8) {
            const int w = threadIdx.x - kDLatent / 8;
            dst[kDLatent / 8 + w] = rotate_word(src[kDLatent / 8 + w], cs, w);
        }
        return;
    }
    // INT8 record: threads 0-63 hold one latent word (8 values) each; the row
    // maximum over the two warps, then the codes; threads 64-71 rotate the rope words
    uint8_t* rec = kv8 + slot * kQ8Record;
    uint4 v = make_uint4(0, 0, 0, 0);
    float m = 0.f;
    if (threadIdx.x < kDLatent / 8) {
        v = src[threadIdx.x];
        const uint32_t* u = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(u[i] << 16)), fabsf(__uint_as_float(u[i] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x < kDLatent / 8 && (threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < kDLatent / 8) {
        const float sc = q8_scale(fmaxf(red[0], red[1]));
        const float inv = 1.f / sc;  // exact: a power of two
        const uint32_t* u = reinterpret_cast<const uint32_t*>(&v);
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            c[2 * i] = q8_code(__uint_as_float(u[i] << 16), inv);
            c[2 * i + 1] = q8_code(__uint_as_float(u[i] & 0xFFFF0000u), inv);
        }
        reinterpret_cast<uint2*>(rec)[threadIdx.x] =
            make_uint2(c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24), c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24));
        if (threadIdx.x == 0) kv_scale[slot] = sc;
    } else if (threadIdx.x < kDLatent / 8 + 8) {
        const int w = threadIdx.x - kDLatent / 8;
        reinterpret_cast<uint4*>(rec + kDLatent)[w] = rotate_word(src[kDLatent / 8 + w], cs, w);
    }
}

}  // namespace

cudaError_t launch_rope_append(void* q, const void* kv_new, const int32_t* seqlens, const int32_t* block_table,
                               int mbps, void* kv_cache, void* kv8, float* kv_scale, int num_blocks, int B, int s_q,
                               int H, double base, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * s_q), 1, 1);
    cfg.blockDim = dim3(kRopeThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    RopeTheta th;
    for (int i = 0; i < kPairs; ++i) th.v[i] = pow(base, -2.0 * (double)i / (double)kDRope);
    if (kv8 != nullptr)
        return cudaLaunchKernelEx(&cfg, rope_append_kernel<true>, static_cast<__nv_bfloat16*>(q),
                                  static_cast<const __nv_bfloat16*>(kv_new), seqlens, block_table, mbps,
                                  static_cast<__nv_bfloat16*>(nullptr), static_cast<uint8_t*>(kv8), kv_scale,
                                  num_blocks, s_q, H, th);
    return cudaLaunchKernelEx(&cfg, rope_append_kernel<false>, static_cast<__nv_bfloat16*>(q),
                              static_cast<const __nv_bfloat16*>(kv_new), seqlens, block_table, mbps,
                              static_cast<__nv_bfloat16*>(kv_cache), static_cast<uint8_t*>(nullptr),
                              static_cast<float*>(nullptr), num_blocks, s_q, H, th);
}

// Reads this file's error word into *out and clears it, in stream order.
cudaError_t rope_error_fetch(int* out, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_rope_error, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    static const int zero = 0;
    return cudaMemcpyToSymbolAsync(g_rope_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
}

}  // namespace mla
