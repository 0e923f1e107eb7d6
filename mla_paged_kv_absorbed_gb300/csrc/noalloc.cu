// noalloc.cu - mla_decode_paged_noalloc: the paged decode for callers that may
// not allocate device memory.
//
// Some callers cannot call cudaMalloc: a plugin that a host inference engine
// hands only its input and output buffers (the host owns the memory pool and
// forbids foreign allocations), or a serving loop that must never block, where
// an allocation may synchronise the device. mla_decode_paged needs a
// caller-provided workspace for its split partials and its device error word;
// this entry point takes that scratch from a fixed array compiled into the
// library instead, so the caller passes only inputs and outputs.
//
// The scratch is a file-scope __device__ array of MLA_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads this part of the library holds it until the process
// exits; with lazy module loading (the CUDA default) that happens on the first
// call on a device, which is when the array is reserved. In host code the
// array's name is only a host-side stand-in, so every call looks up the device
// address with cudaGetSymbolAddress on the current device (a lookup, no
// allocation; after cudaDeviceReset it returns the new context's address, so
// no stale pointer is kept). The first call on a device loads the module, so
// it should come before any stream capture. Every call shares the one array:
// calls that overlap on the GPU (different streams, no ordering) race on it.
#include "mla.h"
#include "mla_internal.h"

// Holds the decode's device error word (first 256 bytes) and its split partials,
// laid out exactly like a mla_decode_paged workspace.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

namespace mla {
namespace {

// Device address of g_noalloc_scratch on the current device (nullptr on failure).
void* scratch_address() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    return p;
}

}  // namespace
}  // namespace mla

extern "C" int mla_decode_paged_noalloc(const mla_bf16_t* q_abs, const mla_bf16_t* kv_cache, int num_blocks,
                                        const int32_t* block_table, int max_blocks_per_seq,
                                        const int32_t* cache_seqlens, int B, int s_q, int H,
                                        const int32_t* tile_meta, const int32_t* num_splits, int num_parts,
                                        float softmax_scale, int causal, mla_bf16_t* o_lat, float* lse,
                                        int32_t* device_status, mla_stream_t stream) {
    const size_t need = mla_workspace_size(B, s_q, H, num_parts);
    if (need == 0 || need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_INVALID_ARG;
    // every argument is checked before the scratch is touched: a rejected call enqueues nothing
    const int bad = mla::decode_check_args(q_abs, kv_cache, nullptr, nullptr, num_blocks, block_table,
                                           max_blocks_per_seq, cache_seqlens, B, s_q, H, tile_meta, num_splits,
                                           num_parts, softmax_scale, causal, o_lat, lse, nullptr, nullptr);
    if (bad != MLA_OK) return bad;
    void* scratch = mla::scratch_address();
    if (scratch == nullptr) return MLA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the error word must start at zero; the partials are always written before they are read
    if (cudaMemsetAsync(scratch, 0, mla::kWorkspaceHeader, st) != cudaSuccess) return MLA_ERR_CUDA;
    const int rc = mla_decode_paged(q_abs, kv_cache, num_blocks, block_table, max_blocks_per_seq, cache_seqlens, B,
                                    s_q, H, tile_meta, num_splits, num_parts, softmax_scale, causal, o_lat, lse,
                                    scratch, (size_t)MLA_NOALLOC_SCRATCH_BYTES, stream);
    if (rc != MLA_OK) return rc;
    if (device_status != nullptr &&
        cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return MLA_ERR_CUDA;
    return MLA_OK;
}
