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
// Each lane owns 16 of the 512 latent columns as four groups of four (the
// pieces are bf16: coalesced 256-byte rows per instruction, widened to fp32
// for the sums). A warp requests three rows before reducing any: for each,
// the lse of piece i on lane i and the first two pieces' partial rows (two
// pieces is the common split). A row of at most two pieces is then reduced
// by every lane from its registers; longer rows reduce the lanes' lse values
// by shuffles and load their further pieces four at a time. Pieces are
// accumulated in ascending order. Batches with a single piece were written
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

// One row's merge in two steps, so that a warp can keep three rows' loads in
// flight. The request issues the lse values and partial rows of the row's first
// kHeld pieces (no address depends on a loaded value: the piece range comes
// from the schedule read beforehand); the finish reduces, loads any further
// pieces four at a time, and stores. Two pieces is the common split; holding
// only those leaves the registers for a third row in flight.
constexpr int kHeld = 2;
struct RowMerge {
    int row, first, n;
    float ll;  // lse of piece `lane` (-inf past the row's pieces): rows of more pieces reduce these
    float l4[kHeld];
    uint2 v[kHeld][4];  // [piece][k]: this lane's columns 4 (lane + 32 k) .. + 3, bf16
};

__device__ __forceinline__ float4 widen4(uint2 u) {
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
}

__device__ __forceinline__ void merge_request(RowMerge& m, int row, int first, int n, int s_q, int H,
                                              const __nv_bfloat16* __restrict__ o_part,
                                              const float* __restrict__ lse_part, int lane) {
    m.row = row;
    m.first = first;
    m.n = n;
    const int h = row % H, s = (row / H) % s_q;
    m.ll = lane < n ? lse_part[((size_t)(first + lane) * s_q + s) * H + h] : -INFINITY;
#pragma unroll
    for (int j = 0; j < kHeld; ++j) {
        m.l4[j] = -INFINITY;
#pragma unroll
        for (int k = 0; k < 4; ++k) m.v[j][k] = make_uint2(0u, 0u);
        if (j < n) {
            const size_t prow = ((size_t)(first + j) * s_q + s) * H + h;
            m.l4[j] = lse_part[prow];
            const __nv_bfloat16* src = o_part + prow * kDLatent;
#pragma unroll
            for (int k = 0; k < 4; ++k) m.v[j][k] = *reinterpret_cast<const uint2*>(src + 4 * (lane + 32 * k));
        }
    }
}

__device__ __forceinline__ void merge_finish(const RowMerge& m, int s_q, int H, const __nv_bfloat16* __restrict__ o_part,
                                             const float* __restrict__ lse_part, __nv_bfloat16* __restrict__ o_lat,
                                             float* __restrict__ lse, int lane) {
    const int h = m.row % H, s = (m.row / H) % s_q, n = m.n, first = m.first;
    // lse of piece i of this row
    auto lse_of = [&](int i) { return lse_part[((size_t)(first + i) * s_q + s) * H + h]; };
    float L = -INFINITY;
    if (n <= kHeld) {
#pragma unroll
        for (int j = 0; j < kHeld; ++j)
            if (j < n) L = fmaxf(L, m.l4[j]);
    } else {
        L = m.ll;
        for (int i = lane + 32; i < n; i += 32) L = fmaxf(L, lse_of(i));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L = fmaxf(L, __shfl_xor_sync(0xffffffffu, L, o));
    }
    float total = -INFINITY;
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (L != -INFINITY) {
        float sum = 0.f;
        if (n <= kHeld) {
#pragma unroll
            for (int j = 0; j < kHeld; ++j)
                if (j < n) sum += expf(m.l4[j] - L);
        } else {
            if (lane < n) sum = expf(m.ll - L);
            for (int i = lane + 32; i < n; i += 32) sum += expf(lse_of(i) - L);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        }
        total = L + logf(sum);
#pragma unroll
        for (int j = 0; j < kHeld; ++j) {
            const float w = j < n ? expf(m.l4[j] - total) : 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 v = widen4(m.v[j][k]);
                acc[k].x += w * v.x;
                acc[k].y += w * v.y;
                acc[k].z += w * v.z;
                acc[k].w += w * v.w;
            }
        }
        // pieces kHeld, kHeld + 1, ... (longer splits), four at a time, in ascending order
        for (int i0 = kHeld; i0 < n; i0 += 4) {
            uint2 v[4][4];
            float w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j;
                w[j] = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) v[j][k] = make_uint2(0u, 0u);
                if (i < n) {
                    const size_t prow = ((size_t)(first + i) * s_q + s) * H + h;
                    w[j] = expf(lse_part[prow] - total);
                    const __nv_bfloat16* src = o_part + prow * kDLatent;
#pragma unroll
                    for (int k = 0; k < 4; ++k) v[j][k] = *reinterpret_cast<const uint2*>(src + 4 * (lane + 32 * k));
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 x = widen4(v[j][k]);
                    acc[k].x += w[j] * x.x;
                    acc[k].y += w[j] * x.y;
                    acc[k].z += w[j] * x.z;
                    acc[k].w += w[j] * x.w;
                }
        }
    }
    uint2* dst = reinterpret_cast<uint2*>(o_lat + (size_t)m.row * kDLatent);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x, acc[k].y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z, acc[k].w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        dst[lane + 32 * k] = u;
    }
    if (lane == 0) lse[m.row] = total;
}

__global__ void __launch_bounds__(kThreads, 4) combine_kernel(const int32_t* __restrict__ num_splits, int rows, int s_q,
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
        // the piece ranges of this warp's next 32 rows, read at once (lane j:
        // row base + j * stride); only rows of split or empty batches have work
        const long long row_j = base + (long long)lane * stride;  // ((b * s_q) + s) * H + h
        int n_j = 1, first_j = 0;
        if (row_j < rows) {
            const int b = (int)(row_j / (H * s_q));
            first_j = num_splits[b];
            n_j = num_splits[b + 1] - first_j;
        }
        unsigned todo = __ballot_sync(0xffffffffu, n_j != 1);
        // three rows at a time: all three rows' first loads are in flight
        // before any is reduced
        while (todo) {
            RowMerge m1, m2, m3;
            int j = __ffs(todo) - 1;
            todo &= todo - 1;
            merge_request(m1, (int)(base + (long long)j * stride), __shfl_sync(0xffffffffu, first_j, j),
                          __shfl_sync(0xffffffffu, n_j, j), s_q, H, o_part, lse_part, lane);
            const bool two = todo != 0;
            if (two) {
                j = __ffs(todo) - 1;
                todo &= todo - 1;
                merge_request(m2, (int)(base + (long long)j * stride), __shfl_sync(0xffffffffu, first_j, j),
                              __shfl_sync(0xffffffffu, n_j, j), s_q, H, o_part, lse_part, lane);
            }
            const bool three = todo != 0;
            if (three) {
                j = __ffs(todo) - 1;
                todo &= todo - 1;
                merge_request(m3, (int)(base + (long long)j * stride), __shfl_sync(0xffffffffu, first_j, j),
                              __shfl_sync(0xffffffffu, n_j, j), s_q, H, o_part, lse_part, lane);
            }
            merge_finish(m1, s_q, H, o_part, lse_part, o_lat, lse, lane);
            if (two) merge_finish(m2, s_q, H, o_part, lse_part, o_lat, lse, lane);
            if (three) merge_finish(m3, s_q, H, o_part, lse_part, o_lat, lse, lane);
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
