/*
 * mla.h - C ABI of libmla: paged, absorbed Multi-head Latent Attention decode
 * on one GB300 (sm_103a).
 *
 * The hot path of one decode step, one call per row of the path:
 *
 *   mla_get_metadata   split/tile schedule from cache_seqlens (once per step)
 *   mla_absorb_q       q' = [W_UK^T q_nope | q_rope]          (per layer)
 *   mla_decode_paged   attention of q' over the paged latent cache, with
 *                      split-KV and the log-sum-exp combine     (per layer)
 *   mla_out_proj       out = W_UV^T o_lat                      (per layer)
 *
 * mla_decode_out_proj does the last two as the decode and one finalize kernel
 * (the split merge fused with the output projection; the attention output of
 * split sequences is never stored).
 *
 * Sources for what each call computes (page title, then section):
 *  [V3] "DeepSeek-V3 Multi-head Latent Attention (MLA) deep engineering: low-rank
 *       KV cache compression" (ybb.press): sec. 2.2 (k = W_UK c, v = W_UV c),
 *       sec. 2.4 (absorption trick), sec. 3.1 (decoupled RoPE), sec. 4.3 (paged,
 *       latent-only cache).
 *  [FM] "FlashMLA: efficient MLA decode kernel for Hopper GPUs" (wuwenjie.xyz):
 *       feature list (bf16 paged kv cache, block size 64) and usage example
 *       (get_mla_metadata(cache_seqlens, s_q*h_q/h_kv, h_kv) once per step;
 *       flash_mla_with_kvcache(q, kvcache, block_table, cache_seqlens, dv,
 *       metadata, num_splits, causal) -> (o, lse) per layer).
 *  [DS1] "DeepSeek tech explainer (1): MLA" (sunshychen.top), sec. 1 (causal mask).
 *  [SC] cshb120.cn/d/6765100, the SC11 MLA decode fused operator article: the
 *       absorb mode is used for decode; up-projection, attention and output
 *       projection are the decode steps; page loads overlap compute (Fig. 2 text).
 *
 * Conventions shared by every call
 *  - bf16 tensors are passed as `mla_bf16_t*` (raw 16-bit storage of IEEE
 *    bfloat16). All tensors are dense, row-major, contiguous in the layouts
 *    stated below, and device pointers unless said otherwise.
 *  - Every device pointer that is read by the tensor-memory accelerator
 *    (q, q_abs, kv_cache, w_uk, w_uv, o_lat) must be 16-byte aligned.
 *  - Ownership: the caller owns every buffer; the library allocates no device
 *    memory and keeps no pointer after a call returns (it caches only per-device
 *    properties).
 *  - Streams: `stream` is a cudaStream_t passed as `void*` (NULL = the legacy
 *    default stream). Every call only enqueues work on it and returns; none
 *    synchronises except mla_read_device_error.
 *  - Errors: argument errors are detected on the host, return a status and
 *    launch nothing. A failed launch returns MLA_ERR_CUDA. Problems only the
 *    device can see (a block id outside the pool, a sequence longer than its
 *    table row, a bounded wait that expired) are recorded in the error word
 *    at the start of the workspace and read with mla_read_device_error.
 *  - Shapes: H (query heads) in {16, 32, 64, 128}; s_q (query tokens per
 *    sequence) in {1, 2}; one shared latent kv head (h_kv = 1).
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mla_bf16_t;   /* IEEE bfloat16 bit pattern */
typedef void* mla_stream_t;    /* cudaStream_t */

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or shape */
    MLA_ERR_UNSUPPORTED = 2,  /* device is not sm_103, or shape outside the supported set */
    MLA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or a launch failed */
    MLA_ERR_TIMEOUT = 4,      /* (device) a bounded pipeline wait expired */
    MLA_ERR_BAD_BLOCK = 5     /* (device) block id outside [0, num_blocks) or seqlen past its table row */
} mla_status_t;

/* Fixed model geometry (DeepSeek-V3 MLA, [V3] sec. 2.3 and 3.1; page size [FM]). */
#define MLA_PAGE_SIZE 64      /* tokens per kv page */
#define MLA_D_LATENT 512      /* c_KV width d_c, also the latent value width */
#define MLA_D_ROPE 64         /* decoupled rope width */
#define MLA_D_QK 576          /* absorbed query / cached key width = 512 + 64 */
#define MLA_D_NOPE 128        /* per-head non-rope query width d_h */
#define MLA_D_Q 192           /* per-head query width = 128 + 64 */
#define MLA_D_V 128           /* per-head output width after W_UV */
#define MLA_TILE_META_INTS 8  /* int32 per schedule row */

/* Schedule constants used by mla_get_metadata (see there). */
#define MLA_SCHED_PIECE_OVERHEAD 7   /* cost of one piece, in page-equivalents */
#define MLA_SCHED_MIN_SPLIT_PAGES 32 /* sequences shorter than this are never split */

/* Human-readable name of a status code (static string). */
const char* mla_status_string(int status);

/* Library ABI version (major * 100 + minor). 1.0: the schedule, absorb,
 * decode and output-projection calls. 1.1 (101) adds the INT8 cache
 * (mla_quantize_cache, mla_decode_paged_q8, mla_rope_append_q8), the RoPE
 * append, the prefill, the fused decode + output projection and the
 * no-allocation decode; the 1.0 calls are unchanged. */
int mla_version(void);

/* The two schedule constants compiled into this library. */
void mla_schedule_constants(int* piece_overhead, int* min_split_pages);

/*
 * Default number of schedule parts for `device`: one part per pair of SMs
 * for each query token, i.e. floor(SM count / (2 * s_q)). Returns a positive
 * count, or minus a status code (e.g. -MLA_ERR_CUDA).
 */
int mla_default_num_parts(int device, int s_q);

/*
 * Bytes of device workspace mla_decode_paged needs for this shape: a 256-byte
 * error-word header, then the split partials (lse fp32 [P, s_q, H], and the
 * normalised piece outputs o as bf16 [P, s_q, H, 512] in a region sized for
 * fp32, for up to P = B + num_parts pieces). Returns 0 for bad
 * arguments. The workspace must be zero-filled before its first use.
 */
size_t mla_workspace_size(int B, int s_q, int H, int num_parts);

/*
 * mla_get_metadata - tile/split schedule of one decode step.
 * Pages: [FM] usage example (get_mla_metadata(cache_seqlens, s_q*h_q/h_kv, h_kv),
 * called once per step and reused by every layer). The pages fix only the
 * call shape; the schedule rule is this library's own:
 *
 *   nblk_b = ceil(seqlen_b / 64); cost_b = nblk_b + MLA_SCHED_PIECE_OVERHEAD
 *   (0 if nblk_b == 0); start_b = sum of earlier costs; total = sum of costs;
 *   quota = max(1, ceil(total / num_parts)).
 *   Unit (b, page j) has key start_b when the batch is short
 *   (nblk_b < MLA_SCHED_MIN_SPLIT_PAGES) or j == 0, else
 *   start_b + MLA_SCHED_PIECE_OVERHEAD + j; it belongs to part floor(key / quota).
 *   A piece is a maximal run of one batch's pages inside one part; pieces are
 *   numbered in part order.
 *
 * cache_seqlens: device int32 [B], kv length of each sequence including its
 *   s_q new tokens (negative values count as 0).
 * h_kv must be 1. s_q and H are validated like mla_decode_paged's.
 * tile_meta (out): device int32 [num_parts, 8]; row p =
 *   {begin_b, begin_page, end_b, end_page (exclusive), first_piece, n_pieces, 0, 0},
 *   all zeros for an empty part.
 * num_splits (out): device int32 [B + 1]; num_splits[b] = index of batch b's
 *   first piece, num_splits[B] = number of pieces (<= B + num_parts).
 * One small kernel, no host synchronisation.
 */
int mla_get_metadata(const int32_t* cache_seqlens, int B, int s_q, int H, int h_kv, int num_parts,
                     int32_t* tile_meta, int32_t* num_splits, mla_stream_t stream);

/*
 * mla_absorb_q - query absorption. Pages: [V3] sec. 2.4 (q' = W_UK^T q, so the
 * score is taken against the cached latent directly), [V3] sec. 3.1 (the rope
 * part of the query stays separate), [SC] (absorb mode for decode).
 *
 * q_abs[b,s,h, c]     = sum_{d<128} q[b,s,h,d] * w_uk[h,d,c]   (c < 512)
 * q_abs[b,s,h,512+i]  = q[b,s,h,128+i]                          (i < 64)
 * q: bf16 [B, s_q, H, 192] = [q_nope 128 | q_rope 64];  w_uk: bf16 [H, 128, 512];
 * q_abs (out): bf16 [B, s_q, H, 576]. fp32 accumulation, bf16 round-to-nearest-even.
 * Runs as a persistent tcgen05 GEMM: one CTA per SM walks a contiguous range of
 * (head, 128-row tile, 128-column quarter) units; the 64 rope columns are copied.
 */
int mla_absorb_q(const mla_bf16_t* q, const mla_bf16_t* w_uk, mla_bf16_t* q_abs, int B, int s_q, int H,
                 mla_stream_t stream);

/*
 * mla_decode_paged - absorbed attention over the paged latent cache.
 * Pages: [V3] sec. 2.4 (score = scale * q' . [c_KV | k_rope]), sec. 4.3 (only
 * the latent is cached, in pages), [FM] (bf16 cache, 64-token blocks, returns
 * o and lse, num_splits for long sequences), [DS1] sec. 1 (causal mask),
 * [SC] Fig. 2 text (page loads overlap compute).
 *
 * For every (b, s, h):  n = causal ? seqlen_b - s_q + s + 1 : seqlen_b (clamped
 * to [0, seqlen_b]); score_t = softmax_scale * q_abs[b,s,h,:] . kv(b,t)[0:576]
 * for t < n; o_lat[b,s,h,:] = sum_t softmax(score)_t * kv(b,t)[0:512];
 * lse[b,s,h] = ln sum_t exp(score_t). A row with n == 0 gets o = 0, lse = -inf.
 * kv(b,t) is row t % 64 of block block_table[b][t / 64].
 *
 * q_abs:        bf16 [B, s_q, H, 576] (from mla_absorb_q, or any absorbed query).
 * kv_cache:     bf16 [num_blocks, 64, 576]; row = [c_KV 512 | k_rope 64].
 * block_table:  int32 [B, max_blocks_per_seq]; entries past a sequence's last
 *               page are never read.
 * cache_seqlens:int32 [B]; must need at most max_blocks_per_seq pages.
 * tile_meta, num_splits, num_parts: from mla_get_metadata on the same
 *               cache_seqlens, B, s_q, H and num_parts.
 * softmax_scale > 0 (DeepSeek-V3: 1/sqrt(192)). causal: 0 or 1.
 * o_lat (out):  bf16 [B, s_q, H, 512]; lse (out): fp32 [B, s_q, H].
 * workspace:    device, >= mla_workspace_size(B, s_q, H, num_parts) bytes,
 *               256-byte aligned, zero-filled before first use; holds the
 *               device error word and the split partials. Calls that share a
 *               workspace must be ordered on one stream.
 * Launches the decode kernel (2-CTA clusters, TMA + tcgen05) and the split
 * combine kernel; with max_blocks_per_seq below the split threshold
 * (min_split_pages of mla_schedule_constants, 32 pages) no sequence can be
 * split and the decode kernel alone is launched (it then also writes the rows
 * of empty sequences).
 */
int mla_decode_paged(const mla_bf16_t* q_abs, const mla_bf16_t* kv_cache, int num_blocks,
                     const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens,
                     int B, int s_q, int H, const int32_t* tile_meta, const int32_t* num_splits, int num_parts,
                     float softmax_scale, int causal, mla_bf16_t* o_lat, float* lse,
                     void* workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * mla_decode_out_proj - mla_decode_paged followed by mla_out_proj, with the
 * split merge and the output projection fused into one finalize kernel.
 * Pages: as mla_decode_paged and mla_out_proj; the fusion follows [SC] Fig. 1
 * text (the output projection inside the attention operator, to save the
 * round trip of the attention output).
 *
 * out[b,s,h,j] = sum_{c<512} o[b,s,h,c] * w_uv[h,c,j], o the attention output
 * of mla_decode_paged (rounded to bf16, as o_lat is there); lse as there.
 * Arguments as mla_decode_paged, plus w_uv: bf16 [H, 512, 128] and out (out):
 * bf16 [B, s_q, H, 128]. o_lat: bf16 [B, s_q, H, 512] scratch: only the rows of
 * sequences that were not split (num_splits) are written there; the merged
 * rows of split sequences go straight into the projection and are never
 * stored. The workspace must be as large as mla_decode_paged's.
 * Launches the decode kernel and the finalize kernel (W_UV[h] resident in
 * shared memory; eight warps merge each 128-row tile's pieces into the
 * product's operand; tcgen05 products into TMEM; TMA stores of out).
 */
int mla_decode_out_proj(const mla_bf16_t* q_abs, const mla_bf16_t* kv_cache, int num_blocks,
                        const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens, int B,
                        int s_q, int H, const int32_t* tile_meta, const int32_t* num_splits, int num_parts,
                        float softmax_scale, int causal, const mla_bf16_t* w_uv, mla_bf16_t* o_lat, mla_bf16_t* out,
                        float* lse, void* workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * mla_out_proj - output up-projection. Pages: [V3] sec. 2.2 (v = W_UV c, applied
 * after attention on the latent side), [SC] (output projection step).
 * out[b,s,h,j] = sum_{c<512} o_lat[b,s,h,c] * w_uv[h,c,j]
 * o_lat: bf16 [B, s_q, H, 512]; w_uv: bf16 [H, 512, 128]; out (out): bf16 [B, s_q, H, 128].
 * fp32 accumulation, bf16 round-to-nearest-even. Batched tcgen05 GEMM.
 */
int mla_out_proj(const mla_bf16_t* o_lat, const mla_bf16_t* w_uv, mla_bf16_t* out, int B, int s_q, int H,
                 mla_stream_t stream);

/*
 * mla_rope_append - the step before the decode: rotary position encoding of
 * the decoupled rope parts and the append of the new tokens to the paged
 * latent cache. Pages: [V3] sec. 3.1 (the rope query part and the position
 * key are rotated by a position-dependent angle, apart from the latent),
 * sec. 3.2 (the position key of token t is RoPE applied per token), sec. 4.3
 * (only the latent is stored, page by page: kv_cache.store(c_kv)). The pages
 * describe the rotation in words only; this is the standard rotary encoding:
 * the 64 rope dims are 32 adjacent pairs (x[2i], x[2i+1]) and pair i turns by
 * the angle t * theta_i, theta_i = rope_base^(-2i/64).
 *
 * Token s of sequence b sits at position t = cache_seqlens[b] - s_q + s
 * (cache_seqlens already counts the s_q new tokens, as mla_decode_paged
 * expects). For every such token with t >= 0:
 *   q[b,s,h,128:192] <- RoPE(q[b,s,h,128:192], t) for every head h (in place;
 *                       q [B, s_q, H, 192] bf16, the nope part is untouched);
 *   row t % 64 of block block_table[b][t / 64] of kv_cache [num_blocks, 64, 576]
 *                    <- [kv_new[b,s,0:512] | RoPE(kv_new[b,s,512:576], t)]
 *                       (kv_new [B, s_q, 576] bf16: the new token's c_KV and
 *                       its not yet rotated k_rope; the latent is copied as is).
 * Angles are reduced in double precision; the rotation is done in fp32 and
 * rounded to bf16 (round to nearest even). rope_base > 1 (DeepSeek-V3: 10000).
 * A block id outside [0, num_blocks), or a position past the table row, is
 * recorded as MLA_ERR_BAD_BLOCK in the library's own error word (read by
 * mla_read_device_error) and that row is not written. One small launch (one
 * CTA per new token), no host synchronisation.
 */
int mla_rope_append(mla_bf16_t* q, const mla_bf16_t* kv_new, const int32_t* cache_seqlens, const int32_t* block_table,
                    int max_blocks_per_seq, mla_bf16_t* kv_cache, int num_blocks, int B, int s_q, int H,
                    float rope_base, mla_stream_t stream);

/*
 * INT8 latent cache. Pages: [V3] sec. 7.2 (the compressed latent is stored in
 * 8 bits, c_t = Quantize(W_DKV h_t, bits = 8)); [DS1] sec. 3.1 (INT8 as the
 * representative KV quantisation). The pages fix only the width; this library
 * reads it as:
 *   kv8      uint8 [num_blocks, 64, 640]: per token a 640-byte record, bytes
 *            0..511 the INT8 codes of c_KV, bytes 512..639 k_rope as 64 bf16
 *            values (the decoupled rope key is not part of c_KV), unchanged;
 *   kv_scale fp32 [num_blocks, 64]: one scale per token, the smallest power of
 *            two s with 127 s >= max_c |c_KV[c]| (s = 1 for an all-zero latent);
 *   code = c_KV / s rounded to nearest, ties to even, in [-127, 127].
 * The token stands for [code * s | k_rope]; with a power-of-two s every code * s
 * is exact in bf16, so the decode over kv8 equals the bf16 decode over the
 * cache of those values (bit for bit, same schedule). Latent values are
 * finite; their maximum is at least 2^-119 or all of them are zero.
 */

/*
 * mla_quantize_cache - bf16 cache rows -> INT8 records and scales.
 * kv: bf16 [tokens, 576] (e.g. a whole [num_blocks, 64, 576] cache); kv8 (out):
 * uint8 [tokens, 640]; kv_scale (out): fp32 [tokens]. All 16-byte aligned.
 * One warp per token, one launch.
 */
int mla_quantize_cache(const mla_bf16_t* kv, long long tokens, uint8_t* kv8, float* kv_scale, mla_stream_t stream);

/*
 * mla_rope_append_q8 - mla_rope_append into an INT8 cache: the same rotation
 * of q's rope parts, and the new token's slot receives its record (codes of
 * kv_new[b,s,0:512] under its scale, then RoPE(kv_new[b,s,512:576], t) in bf16)
 * and its scale. Same arguments and errors as mla_rope_append, with kv8 uint8
 * [num_blocks, 64, 640] and kv_scale fp32 [num_blocks, 64] in place of kv_cache.
 */
int mla_rope_append_q8(mla_bf16_t* q, const mla_bf16_t* kv_new, const int32_t* cache_seqlens,
                       const int32_t* block_table, int max_blocks_per_seq, uint8_t* kv8, float* kv_scale,
                       int num_blocks, int B, int s_q, int H, float rope_base, mla_stream_t stream);

/*
 * mla_decode_paged_q8 - mla_decode_paged over an INT8 cache (kv8, kv_scale as
 * above; both 16-byte aligned). Same arguments, outputs, workspace and errors
 * as mla_decode_paged. Each CTA loads a page's 32 KB of codes (plus, on the
 * score side, its 8 KB of rope keys and 256 bytes of scales) instead of 72 KB
 * and expands it to bf16 in shared memory before the tensor-core products.
 */
int mla_decode_paged_q8(const mla_bf16_t* q_abs, const uint8_t* kv8, const float* kv_scale, int num_blocks,
                        const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens, int B,
                        int s_q, int H, const int32_t* tile_meta, const int32_t* num_splits, int num_parts,
                        float softmax_scale, int causal, mla_bf16_t* o_lat, float* lse, void* workspace,
                        size_t workspace_bytes, mla_stream_t stream);

/*
 * mla_prefill_paged - prefill over the same paged latent cache, in the naive
 * (decompress) form. Pages: [V3] sec. 2.2 (k = W_UK c, v = W_UV c), sec. 3.1
 * (the rope key is shared by the heads), sec. 4.3 (the paged module
 * decompresses K and V per head before ordinary attention); [SC] opening
 * (prefill processes the prompt, decode one token at a time).
 *
 * The s_q query tokens of sequence b are its last s_q positions (a whole
 * prompt when s_q == cache_seqlens[b], a prompt chunk after earlier tokens
 * otherwise; cache_seqlens already counts them). For every (b, s, h):
 *   K_t = [W_UK[h] c_t | k_rope_t] (192), V_t = W_UV[h]^T c_t (128) for t < seqlen_b,
 *   n = causal ? seqlen_b - s_q + s + 1 : seqlen_b (clamped to [0, seqlen_b]),
 *   out[b,s,h,:] = sum_{t<n} softmax_t(softmax_scale * q[b,s,h,:] . K_t) V_t,
 *   lse[b,s,h] = ln sum_{t<n} exp(softmax_scale * q . K_t); n == 0 gives 0, -inf.
 * q: bf16 [B, s_q, H, 192] = [q_nope 128 | q_rope 64] (rope already applied);
 * kv_cache, block_table, cache_seqlens as mla_decode_paged; w_uk [H, 128, 512],
 * w_uv [H, 512, 128] bf16; out (out): bf16 [B, s_q, H, 128] (the per-head
 * output, already through W_UV); lse (out): fp32 [B, s_q, H].
 * workspace: device, >= mla_prefill_workspace_size(B, H, max_blocks_per_seq)
 * bytes, 1024-byte aligned (no zero-fill needed): holds the gathered latent and
 * the decompressed K and V (bf16) of every sequence, padded to
 * max_blocks_per_seq pages. Any s_q >= 1; H in {16, 32, 64, 128}.
 * Launches a gather, two batched head GEMMs (tcgen05, the head's weight resident
 * per CTA) and the attention kernel (one CTA per (sequence, head, 256 query
 * rows) as two 128-row tiles sharing each K/V tile; tcgen05 with S, P and O in
 * tensor memory). A block id outside the pool, or a sequence longer than its
 * table row, is recorded as MLA_ERR_BAD_BLOCK in the library's error word and
 * those rows read as zeros.
 */
size_t mla_prefill_workspace_size(int B, int H, int max_blocks_per_seq);
int mla_prefill_paged(const mla_bf16_t* q, const mla_bf16_t* kv_cache, int num_blocks, const int32_t* block_table,
                      int max_blocks_per_seq, const int32_t* cache_seqlens, int B, int s_q, int H,
                      const mla_bf16_t* w_uk, const mla_bf16_t* w_uv, float softmax_scale, int causal,
                      mla_bf16_t* out, float* lse, void* workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * Reads and clears the device error word of `workspace` (may be NULL) and the
 * library's own error words (projections, rope append, prefill); synchronises `stream`.
 * Returns MLA_OK, MLA_ERR_TIMEOUT or MLA_ERR_BAD_BLOCK as recorded by the
 * kernels since the last read, or MLA_ERR_CUDA if the read failed.
 */
int mla_read_device_error(void* workspace, mla_stream_t stream);

/*
 * Bound on every pipeline wait inside the kernels, in nanoseconds of device
 * wall-clock time (default 4e9, i.e. 4 s). A wait that runs out records
 * MLA_ERR_TIMEOUT in the error word (the workspace's, or the library's own
 * word for the projections) and the kernel drains its copies and MMAs, frees
 * its tensor memory and returns. `ns` <= 0 restores the default. Applies to
 * launches made after the call, process-wide.
 */
void mla_set_wait_limit_ns(long long ns);

/*
 * mla_decode_paged_noalloc - mla_decode_paged for callers that may not
 * allocate device memory. (No counterpart on the pages: this is a packaging
 * variant of the same decode, not part of the method.)
 *
 * Who needs it: code that is handed only its input and output buffers and must
 * not call cudaMalloc itself - e.g. a plugin inside a host inference engine that
 * owns the device memory pool, or a serving loop where an allocation could
 * synchronise the device. It computes exactly what mla_decode_paged computes,
 * with the same arguments and errors, except that the workspace (split
 * partials and device error word) lives in a fixed scratch array compiled into
 * the library, MLA_NOALLOC_SCRATCH_BYTES (about 64 MiB) per GPU that uses it,
 * held until the process exits. Limit: (B + num_parts) * s_q * H must not
 * exceed MLA_NOALLOC_MAX_ROWS (32768; e.g. B = 128, num_parts = 76, s_q = 1,
 * H = 128 uses 26112); larger shapes return MLA_ERR_INVALID_ARG and launch
 * nothing. The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 * device_status (optional, may be NULL): caller-owned device int32 that
 * receives, in stream order after the kernels, the device status of this call
 * (MLA_OK, MLA_ERR_TIMEOUT or MLA_ERR_BAD_BLOCK); the scratch error word is
 * cleared at the start of every call.
 * Every call looks up the scratch array's device address on the current
 * device (cudaGetSymbolAddress: a lookup, no allocation). Under lazy module
 * loading (the CUDA default) the first call on a device loads the library's
 * device code, and that is when the array is reserved on that device; make
 * that first call before any stream capture. All calls share the one array
 * and it keeps the last call's contents (each call clears the error word it
 * needs at zero; every partial is written before it is read): calls that
 * overlap on the GPU (on unordered streams) race on it and must be serialised
 * by the caller.
 */
#define MLA_NOALLOC_MAX_ROWS 32768
#define MLA_NOALLOC_SCRATCH_BYTES (256 + MLA_NOALLOC_MAX_ROWS * (4 + 4 * MLA_D_LATENT))
int mla_decode_paged_noalloc(const mla_bf16_t* q_abs, const mla_bf16_t* kv_cache, int num_blocks,
                             const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens,
                             int B, int s_q, int H, const int32_t* tile_meta, const int32_t* num_splits,
                             int num_parts, float softmax_scale, int causal, mla_bf16_t* o_lat, float* lse,
                             int32_t* device_status, mla_stream_t stream);

/* ----------------------------------------------------------------------------
 * Test hooks. They expose single building blocks of the path so tests can
 * check them on their own; they are not part of a decode step.
 * ------------------------------------------------------------------------- */

/*
 * Paged gather through TMA with mla_decode_paged's own page load: one
 * whole-page box through the same tensor map (3-D [dims, keys, chunk] view,
 * 128-byte swizzle), then un-swizzled to HBM:
 * out[b, t, :] = kv(b, t)[0:576] for t < min(seqlen_b, max_tokens); other rows
 * of out are left untouched. out: bf16 [B, max_tokens, 576]. Bit-exact copy.
 */
int mla_debug_gather(const mla_bf16_t* kv_cache, int num_blocks, const int32_t* block_table,
                     int max_blocks_per_seq, const int32_t* cache_seqlens, int B, int max_tokens,
                     mla_bf16_t* out, mla_stream_t stream);

/*
 * Failure-path check without any fault: with `enable` != 0, mla_decode_paged
 * launches made afterwards (process-wide) never issue the value CTA's first
 * page load, so the P.V warp's bounded wait for it runs out: the kernel
 * records MLA_ERR_TIMEOUT, aborts both CTAs of each cluster with work, drains
 * what is in flight, frees its tensor memory and returns (the outputs of that
 * call are undefined). Nothing is read or written out of bounds. 0 restores
 * normal operation.
 */
void mla_debug_withhold_value_load(int enable);

/*
 * One-tile tcgen05 check: D[128, N] = A[128, K] * B[K, N] in fp32, the same
 * operand layouts the decode kernel uses. A: bf16 [128, K] row-major
 * (K-major); a_tmem = 0 reads it from 128-byte-swizzled shared memory, a_tmem = 1
 * from tensor memory written by thread stores, a_tmem = 2 from tensor memory
 * filled by tcgen05.cp from the swizzled shared tile (row m in lane m, bf16
 * pairs per 32-bit column, as the decode kernel holds the absorbed query).
 * b_kmajor = 1: B given as bf16
 * [N, K] row-major (K-major, like the key tile); b_kmajor = 0: B given as bf16
 * [K, N] row-major (N-major, like the value tile). K in {64, 128, ..., 576},
 * N in {64, 128, 256}. d: fp32 [128, N].
 */
int mla_debug_mma(const mla_bf16_t* a, const mla_bf16_t* b, int K, int N, int b_kmajor, int a_tmem, float* d,
                  mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
