// quant.cuh - the INT8 latent cache format and its arithmetic.
//
// "DeepSeek-V3 MLA deep engineering" (sec. 7.2) quantises the compressed latent
// to 8 bits, c_t = Quantize(W_DKV h_t, bits = 8); "DeepSeek tech explainer (1)"
// (sec. 3.1) names INT8 as the representative KV quantisation. Nothing else is
// fixed there; this library reads it as:
//  * one record of 640 bytes per token: the 512 latent dims as INT8 codes
//    (bytes 0..511), then the decoupled rope key unchanged as 64 bf16 values
//    (bytes 512..639; it is not part of c_KV);
//  * one fp32 scale per token, in a separate array [num_blocks, 64];
//  * symmetric codes in [-127, 127]; the scale is the smallest power of two s
//    with 127 s >= max |c| (an all-zero latent has s = 1); code = c / s rounded
//    to nearest, ties to even.
// With a power-of-two scale, c / s is exact (the rounding decision is the same
// whatever precision takes it) and code * s is exactly representable in bf16,
// so a dequantised page is bit for bit the bf16 page of the values the codes
// stand for.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace mla {

constexpr int kQ8Record = 640;  // bytes per token

// The smallest power of two s with 127 s >= amax, for a finite amax >= 0.
// amax = m 2^k with m in [0.5, 1): 127 * 2^(k-7) >= amax iff m <= 127/128,
// otherwise 2^(k-6).
__device__ __forceinline__ float q8_scale(float amax) {
    if (!(amax > 0.f)) return 1.f;
    int k;
    const float m = frexpf(amax, &k);
    return ldexpf(1.f, m <= 127.f / 128.f ? k - 7 : k - 6);
}

// Code of x under scale s (x * (1 / s) is exact: s is a power of two).
__device__ __forceinline__ uint32_t q8_code(float x, float inv_s) {
    return (uint32_t)(__float2int_rn(x * inv_s)) & 0xFFu;
}

// 16 INT8 codes (one 16-byte word) -> 16 bf16 values code * s (two 16-byte
// words), exactly. A code byte b, read with its sign bit flipped (b ^ 0x80 =
// code + 128), becomes the low byte of the float 2^23 + code + 128; one fused
// multiply-add by s and -(2^23 + 128) s (both exact for a power of two s) leaves
// code * s, which bf16 holds exactly.
__device__ __forceinline__ void q8_dequant16(uint4 src, float s, uint4& lo, uint4& hi) {
    const float off = -8388736.f * s;
    const uint32_t w[4] = {src.x ^ 0x80808080u, src.y ^ 0x80808080u, src.z ^ 0x80808080u, src.w ^ 0x80808080u};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float f0 = fmaf(__uint_as_float(__byte_perm(w[j], 0x4B000000u, 0x7540)), s, off);
        const float f1 = fmaf(__uint_as_float(__byte_perm(w[j], 0x4B000000u, 0x7541)), s, off);
        const float f2 = fmaf(__uint_as_float(__byte_perm(w[j], 0x4B000000u, 0x7542)), s, off);
        const float f3 = fmaf(__uint_as_float(__byte_perm(w[j], 0x4B000000u, 0x7543)), s, off);
        o[2 * j] = pack_bf16x2(f0, f1);
        o[2 * j + 1] = pack_bf16x2(f2, f3);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace mla
