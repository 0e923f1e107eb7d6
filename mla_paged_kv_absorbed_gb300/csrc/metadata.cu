// metadata.cu - device construction of the split/tile schedule.
//
// Computes the same schedule as the walk documented at mla_get_metadata in
// include/mla.h, but in parallel: every batch derives, in closed form, the
// parts its pages fall into (keys are monotone in (b, page), so a batch's
// pages form contiguous runs of parts), and the part rows are filled by the
// batches that open and close them. Chunked block scans give the running
// batch starts, the previous batch's last key and the piece numbering, so any
// B fits one 256-thread block and nothing is stored per batch.
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename T, typename Op>
__device__ T block_exclusive_scan(T v, T identity, Op op, T* warp_tot, T* total_out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc = op(inc, n);
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        T w = lane < kWarps ? warp_tot[lane] : identity;
        T winc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            T n = __shfl_up_sync(0xffffffffu, winc, o);
            if (lane >= o) winc = op(winc, n);
        }
        if (lane < kWarps) warp_tot[lane] = winc;  // inclusive over warps
    }
    __syncthreads();
    T warp_prefix = warp == 0 ? identity : warp_tot[warp - 1];
    T excl_in_warp = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) excl_in_warp = identity;
    T result = op(warp_prefix, excl_in_warp);
    if (total_out) *total_out = warp_tot[kWarps - 1];
    __syncthreads();
    return result;
}

struct Add64 {
    __device__ long long operator()(long long a, long long b) const { return a + b; }
};
struct Max64 {
    __device__ long long operator()(long long a, long long b) const { return a > b ? a : b; }
};
struct Add32 {
    __device__ int operator()(int a, int b) const { return a + b; }
};

__device__ __forceinline__ long long pages_of(int seqlen) {
    return seqlen > 0 ? ((long long)seqlen + kPage - 1) / kPage : 0;
}

__global__ void __launch_bounds__(kThreads) metadata_kernel(const int32_t* __restrict__ seqlens, int B,
                                                            int num_parts, int ovh, int min_split,
                                                            int32_t* __restrict__ tile_meta,
                                                            int32_t* __restrict__ num_splits) {
    __shared__ long long s_tot64[kWarps];
    __shared__ int s_tot32[kWarps];
    __shared__ long long s_total;

    for (int i = threadIdx.x; i < num_parts * 8; i += kThreads) tile_meta[i] = 0;

    // pass 1: total cost
    long long acc = 0;
    for (int b = threadIdx.x; b < B; b += kThreads) {
        long long n = pages_of(seqlens[b]);
        if (n > 0) acc += n + ovh;
    }
    {
        long long dummy_total;
        (void)block_exclusive_scan<long long>(acc, 0LL, Add64(), s_tot64, &dummy_total);
        if (threadIdx.x == 0) s_total = dummy_total;
    }
    __syncthreads();
    const long long total = s_total;
    long long quota = (total + num_parts - 1) / num_parts;
    if (quota < 1) quota = 1;

    // pass 2: per batch, chunk by chunk
    long long carry_start = 0, carry_lastkey = -1;
    int carry_pieces = 0;
    for (int base = 0; base < B; base += kThreads) {
        const int b = base + threadIdx.x;
        const long long n = b < B ? pages_of(seqlens[b]) : 0;
        const long long cost = n > 0 ? n + ovh : 0;
        long long chunk_cost;
        const long long start = carry_start + block_exclusive_scan<long long>(cost, 0LL, Add64(), s_tot64, &chunk_cost);
        const bool is_long = n >= min_split;
        // key of the batch's last unit (-1 when the batch is empty)
        const long long lastkey = n == 0 ? -1 : ((is_long && n >= 2) ? start + ovh + n - 1 : start);
        long long chunk_max;
        long long prev_lastkey = block_exclusive_scan<long long>(lastkey, -1LL, Max64(), s_tot64, &chunk_max);
        prev_lastkey = prev_lastkey > carry_lastkey ? prev_lastkey : carry_lastkey;

        // parts touched: p0 (page 0) and the run [p1, pl] of pages 1..n-1
        long long p0 = start / quota, p1 = p0, pl = p0;
        if (n > 0 && is_long && n >= 2) {
            p1 = (start + ovh + 1) / quota;
            pl = (start + ovh + n - 1) / quota;
        }
        int splits = 0;
        if (n > 0) splits = (int)(pl - p1 + 1) + (p0 != p1 ? 1 : 0);
        int chunk_pieces;
        const int first_piece = carry_pieces + block_exclusive_scan<int>(splits, 0, Add32(), s_tot32, &chunk_pieces);
        if (b < B) num_splits[b] = first_piece;

        if (n > 0) {
            const long long prev_part = prev_lastkey >= 0 ? prev_lastkey / quota : -1;
            const long long next_start = start + cost;
            const long long next_part = next_start < total ? next_start / quota : (long long)num_parts;
            int k = 0;
            for (long long p = p0; p <= pl; ++p) {
                if (p > p0 && p < p1) continue;  // gap between page 0 and page 1
                long long lo, hi;
                if (!is_long || n == 1) {
                    lo = 0;
                    hi = n;
                } else {
                    lo = (p == p0) ? 0 : (p * quota - start - ovh);
                    if (lo < 1 && p != p0) lo = 1;
                    if (p == pl) {
                        hi = n;
                    } else if (p == p0 && p0 != p1) {
                        hi = 1;
                    } else {
                        hi = (p + 1) * quota - start - ovh;
                        if (hi > n) hi = n;
                    }
                }
                int32_t* row = tile_meta + 8 * p;
                const bool opens = (p > p0) || (p0 > prev_part);
                const bool closes = (p < pl) || (next_part > pl);
                if (opens) {
                    row[0] = b;
                    row[1] = (int32_t)lo;
                    row[4] = first_piece + k;
                }
                if (closes) {
                    row[2] = b;
                    row[3] = (int32_t)hi;
                }
                atomicAdd(&row[5], 1);
                ++k;
            }
        }
        carry_start += chunk_cost;
        carry_lastkey = chunk_max > carry_lastkey ? chunk_max : carry_lastkey;
        carry_pieces += chunk_pieces;
    }
    if (threadIdx.x == 0) num_splits[B] = carry_pieces;
}

}  // namespace

cudaError_t launch_metadata(const int32_t* seqlens, int B, int num_parts, int ovh, int min_split,
                            int32_t* tile_meta, int32_t* num_splits, cudaStream_t stream) {
    metadata_kernel<<<1, kThreads, 0, stream>>>(seqlens, B, num_parts, ovh, min_split, tile_meta, num_splits);
    return cudaGetLastError();
}

}  // namespace mla
