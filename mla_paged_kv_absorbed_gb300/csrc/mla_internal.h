// mla_internal.h - launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units. Not installed; the public interface is include/mla.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

constexpr int kPage = 64;
constexpr int kDLatent = 512;
constexpr int kDRope = 64;
constexpr int kDQK = 576;
constexpr int kDNope = 128;
constexpr int kDQ = 192;
constexpr int kDV = 128;
constexpr int kSchedOverhead = 7;
constexpr int kSchedMinSplitPages = 32;
constexpr size_t kWorkspaceHeader = 256;

// Workspace layout: [error word | pad to 256] [lse_part fp32 P*s_q*H, padded to
// 256 B] [o_part P*s_q*H*512 fp32-sized; the pieces are stored as bf16 in its first half],
// with P = B + num_parts.
struct WorkspaceLayout {
    size_t lse_offset, o_offset, total;
};
WorkspaceLayout workspace_layout(int B, int s_q, int H, int num_parts);

// SM count of the current device (cached per device ordinal), 0 on failure.
int device_sm_count();

cudaError_t launch_metadata(const int32_t* seqlens, int B, int num_parts, int ovh, int min_split,
                            int32_t* tile_meta, int32_t* num_splits, cudaStream_t stream);

struct GemmArgs {
    int R;            // rows = B * s_q
    int H;            // heads
    int K;            // contraction length (128 absorb, 512 out-proj)
    int N;            // output columns per head (512 absorb, 128 out-proj)
    int n_cta;        // output columns per CTA
    void* out;        // bf16 [R, H, out_row_elems]
    int out_row_elems;
    const void* rope_src;  // absorb only: q [R, H, 192]; rope part copied to out columns 512..575
    int a_shared;          // 1: every head reads the same A rows (the A map has one head)
    int b_kmajor;          // 1: B is stored [N rows][K] (K contiguous) instead of [K rows][N]
};
cudaError_t launch_head_gemm(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const CUtensorMap* tm_out,
                             const GemmArgs& args, long long wait_ns, cudaStream_t stream);

struct DecodeArgs {
    const void* q_abs;  // bf16 [B, s_q, H, 576]
    const int32_t* block_table;
    int mbps;
    const int32_t* seqlens;
    const int32_t* tile_meta;
    const int32_t* num_splits;
    int num_parts;
    int B, s_q, H, num_blocks;
    int qrows;         // rows of one query box: min(64, B * s_q * H)
    float scale_log2;  // softmax_scale * log2(e)
    int causal;
    void* o_lat;       // bf16 [B, s_q, H, 512]
    float* lse;        // [B, s_q, H]
    void* o_part;      // bf16 [P, s_q, H, 512]: the split pieces' normalised outputs
    float* lse_part;   // [P, s_q, H]
    int* err;
    long long wait_ns;
    int withhold;      // test hook: the value CTA never loads its first page (its consumer's wait runs out)
    const float* kv_scale;  // INT8 cache: per-token scales [num_blocks * 64]; nullptr for the bf16 cache
    int own_empty;  // no merge kernel follows: the decode writes the rows of empty sequences (o = 0, lse = -inf)
};
cudaError_t gemm_error_fetch(int* out, cudaStream_t stream);
int decode_max_active_clusters(int device);

// TMA descriptors of the decode kernel (all 128-byte swizzle; dims listed
// innermost first):
//  kv: the cache as {64 dims, num_blocks * 64 keys, 9 chunks}, strides {1152, 128} B;
//      box {64, 64, 9} = one whole page, [chunk][key][64 dims] in shared memory
//  v:  the same view, box {64, 64, 8} = the page's 512 value columns
//  q:  q_abs as {64 dims, B * s_q * H rows, 9 chunks}, strides {1152, 128} B;
//      box {64, qrows, 9} with qrows = min(64, B * s_q * H)
//  o:  o_lat as {64 cols, H rows, 8 chunks, B * s_q}, strides {1024, 128, H * 1024} B;
//      box {64, min(H, 128), 4, 1} (store)
//  op: o_part (bf16) as {64 cols, H rows, 8 chunks, pieces * s_q}, strides {1024, 128, H * 1024} B;
//      box {64, min(H, 128), 4, 1} (store), like o
struct DecodeMaps {
    CUtensorMap kv, v, q, o, op;
    CUtensorMap kv8, rope;  // INT8 cache only
};
cudaError_t launch_decode(const DecodeMaps& maps, const DecodeArgs& args, cudaStream_t stream);
// The decode entry points' host-side argument checks, apart from the workspace
// (api.cu; no device call): MLA_OK or MLA_ERR_INVALID_ARG.
int decode_check_args(const void* q_abs, const void* kv_cache, const void* kv8, const float* kv_scale,
                      int num_blocks, const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens,
                      int B, int s_q, int H, const int32_t* tile_meta, const int32_t* num_splits, int num_parts,
                      float softmax_scale, int causal, const void* o_lat, const float* lse, const void* w_uv,
                      const void* out);

// The split merge fused with the output projection (finalize.cu).
struct FinArgs {
    const int32_t* num_splits;  // [B + 1] piece offsets from the schedule
    int R;                      // rows = B * s_q
    int s_q, H;
    const void* o_part;         // bf16 [pieces, s_q, H, 512] split partials (workspace)
    const float* lse_part;      // fp32 [pieces, s_q, H]
    const void* o_lat;          // bf16 [B, s_q, H, 512]: rows of unsplit sequences (written by the decode)
    float* lse;                 // fp32 [B, s_q, H]: written here for split and empty rows
    int* err;                   // device error word
    long long wait_ns;
    int tiles_per_cta;          // set by launch_finalize
};
cudaError_t launch_finalize(const CUtensorMap* tm_w, const CUtensorMap* tm_out, const FinArgs& args,
                            cudaStream_t stream);

cudaError_t launch_rope_append(void* q, const void* kv_new, const int32_t* seqlens, const int32_t* block_table,
                               int mbps, void* kv_cache, void* kv8, float* kv_scale, int num_blocks, int B, int s_q,
                               int H, double base, cudaStream_t stream);
cudaError_t launch_quantize(const void* kv, long long rows, void* rec, float* scale, cudaStream_t stream);
cudaError_t rope_error_fetch(int* out, cudaStream_t stream);

// Prefill (naive form): gather + attention launchers (prefill.cu).
cudaError_t launch_prefill_gather(const void* kv, int num_blocks, const int32_t* table, int mbps,
                                  const int32_t* seqlens, int B, int H, void* C, void* Kbuf, cudaStream_t stream);
cudaError_t launch_prefill_attn(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                                const int32_t* seqlens, int B, int s_q, int H, int Lmax, float scale, int causal,
                                void* out, float* lse, long long wait_ns, cudaStream_t stream);
cudaError_t prefill_error_fetch(int* out, cudaStream_t stream);

cudaError_t launch_combine(const int32_t* num_splits, int B, int s_q, int H, const void* o_part,
                           const float* lse_part, void* o_lat, float* lse, cudaStream_t stream);

cudaError_t launch_debug_gather(const CUtensorMap* tm_kv, const int32_t* block_table, int mbps,
                                const int32_t* seqlens, int B, int max_tokens, int num_blocks, void* out,
                                cudaStream_t stream);

cudaError_t launch_debug_mma(const CUtensorMap* tm_a, const CUtensorMap* tm_b, int K, int N, int b_kmajor,
                             int a_tmem, const void* a, float* d, cudaStream_t stream);

}  // namespace mla
