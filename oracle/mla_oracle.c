/*
 * mla_oracle.c - plain, slow CPU oracle for paged, absorbed MLA decode.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg may load this library. The CUDA path never
 * calls it and shares no source with it.
 *
 * Arithmetic: every input arrives as float (the exact widening of the bf16
 * values the GPU sees); every sum and every exp/log is done in double;
 * outputs are double. Scalar loops, two-pass softmax, no tiling, no fusion
 * beyond what the definitions below state. OpenMP only spreads independent
 * (b, s, h) rows over cores.
 *
 * Sources (page title, then section or equation):
 *  [V3]  "DeepSeek-V3 Multi-head Latent Attention (MLA) deep engineering:
 *        low-rank KV cache compression" (ybb.press):
 *        sec. 2.2 (k = W_UK c, v = W_UV c), sec. 2.4 (absorption: q^T W_UK c =
 *        (W_UK^T q)^T c), sec. 3.1 (decoupled RoPE: a per-head rope query part
 *        and a shared rope key part), sec. 4.1 (the tile-wise normalised online
 *        softmax recurrence), sec. 4.3 (only the latent is cached, pages).
 *  [FM]  "FlashMLA: efficient MLA decode kernel for Hopper GPUs" (wuwenjie.xyz):
 *        features list (bf16 paged kv cache, block size 64) and usage example
 *        (get_mla_metadata -> tile schedule + num_splits; flash_mla_with_kvcache
 *        returns (o, lse)).
 *  [DS1] "DeepSeek tech explainer (1): MLA" (sunshychen.top), sec. 1: causal
 *        attention with a lower-triangular mask.
 *
 * Readings where the pages are silent or garbled (each is stated once more at
 * the function that uses it):
 *  - The rope part enters the score by concatenation: score = q_nope.k_nope +
 *    q_rope.k_rope (the sum printed in [V3] sec. 3.1 adds vectors of different
 *    lengths and cannot be meant literally). The scale is a caller argument.
 *  - kv cache row layout: [c_KV (512) | k_rope (64)], one shared kv head.
 *  - W_UK is [H, 128, 512] and used as q'[c] = sum_d q_nope[d] W_UK[h,d,c];
 *    W_UV is [H, 512, 128] and used as out[j] = sum_c o_lat[c] W_UV[h,c,j].
 *  - Causal alignment is bottom-right: query s of s_q sees keys t with
 *    t <= seqlen - s_q + s.
 *  - lse is the natural log of sum_t exp(scaled score). A row with no visible
 *    key has o = 0 and lse = -inf.
 *  - Split-KV combine: L = max_i lse_i, lse = L + ln sum_i exp(lse_i - L),
 *    o = sum_i exp(lse_i - lse) o_i (the pages name num_splits and lse only).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_PAGE 64   /* tokens per page [FM] */
#define ORC_DC 512    /* latent c_KV width [V3] sec. 2.3 */
#define ORC_DR 64     /* decoupled rope width */
#define ORC_DQK 576   /* absorbed query / key width = DC + DR */
#define ORC_DN 128    /* per-head nope width d_h */
#define ORC_DQ 192    /* per-head query width = DN + DR */
#define ORC_DV 128    /* per-head value width after W_UV */

/* Pointer to kv row of logical token t of a sequence, through its block table row. */
static const float* kv_row(const float* kv, const int32_t* table_row, int64_t t) {
    int64_t blk = table_row[t / ORC_PAGE];
    return kv + (blk * ORC_PAGE + (t % ORC_PAGE)) * ORC_DQK;
}

/* Number of keys query s (of s_q) of a sequence with `seqlen` tokens may see. */
static int64_t visible_keys(int64_t seqlen, int s_q, int s, int causal) {
    int64_t n = causal ? seqlen - s_q + s + 1 : seqlen;
    if (n < 0) n = 0;
    if (n > seqlen) n = seqlen;
    return n;
}

/*
 * Absorption of the query [V3 sec. 2.4]: q'[c] = sum_d W_UK[h,d,c] q_nope[d]
 * for c < 512, followed by the untouched rope part q_rope (64) [V3 sec. 3.1].
 * q [R, H, 192] float, w_uk [H, 128, 512] float -> q_abs [R, H, 576] double.
 */
void orc_absorb_q(const float* q, const float* w_uk, int64_t R, int H, double* q_abs) {
    #pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int h = 0; h < H; ++h) {
            const float* qr = q + (r * H + h) * ORC_DQ;
            const float* w = w_uk + (int64_t)h * ORC_DN * ORC_DC;
            double* out = q_abs + (r * H + h) * ORC_DQK;
            for (int c = 0; c < ORC_DC; ++c) {
                double acc = 0.0;
                for (int d = 0; d < ORC_DN; ++d) acc += (double)qr[d] * (double)w[(int64_t)d * ORC_DC + c];
                out[c] = acc;
            }
            for (int i = 0; i < ORC_DR; ++i) out[ORC_DC + i] = (double)qr[ORC_DN + i];
        }
    }
}

/*
 * One absorbed query row against logical keys [t_lo, t_hi) of one sequence:
 * score_t = scale * (q' . kv_t[0:576]); p = softmax(score) in two passes;
 * o = sum_t p_t kv_t[0:512]; lse = max + ln sum exp(score - max).
 * [V3 sec. 2.4]: the absorbed query is dotted with the cached latent directly.
 */
static void attend_absorbed_row(const double* qa, const float* kv, const int32_t* table_row,
                                int64_t t_lo, int64_t t_hi, double scale, double* o, double* lse) {
    for (int c = 0; c < ORC_DC; ++c) o[c] = 0.0;
    if (t_hi <= t_lo) { *lse = -INFINITY; return; }
    int64_t n = t_hi - t_lo;
    double* sc = (double*)malloc((size_t)n * sizeof(double));
    double mx = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        const float* k = kv_row(kv, table_row, t_lo + i);
        double dot = 0.0;
        for (int c = 0; c < ORC_DQK; ++c) dot += qa[c] * (double)k[c];
        sc[i] = scale * dot;
        if (sc[i] > mx) mx = sc[i];
    }
    double l = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double p = exp(sc[i] - mx);
        l += p;
        const float* v = kv_row(kv, table_row, t_lo + i);
        for (int c = 0; c < ORC_DC; ++c) o[c] += p * (double)v[c];
    }
    for (int c = 0; c < ORC_DC; ++c) o[c] /= l;
    *lse = mx + log(l);
    free(sc);
}

/*
 * Absorbed-form paged attention for a whole batch.
 * q_abs [B, s_q, H, 576] double; kv [num_blocks, 64, 576] float;
 * block_table [B, mbps] int32; seqlens [B] int32 ->
 * o_lat [B, s_q, H, 512] double, lse [B, s_q, H] double.
 */
void orc_attend_absorbed(const double* q_abs, const float* kv, const int32_t* block_table, int mbps,
                         const int32_t* seqlens, int B, int s_q, int H, double scale, int causal,
                         double* o_lat, double* lse) {
    #pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < s_q; ++s)
            for (int h = 0; h < H; ++h) {
                int64_t row = ((int64_t)b * s_q + s) * H + h;
                int64_t n = visible_keys(seqlens[b], s_q, s, causal);
                attend_absorbed_row(q_abs + row * ORC_DQK, kv, block_table + (int64_t)b * mbps, 0, n,
                                    scale, o_lat + row * ORC_DC, lse + row);
            }
}

/*
 * Naive (decompress) form [V3 sec. 2.2, sec. 3.1, sec. 4.3]: for every visible
 * token materialise the per-head key K_t = [W_UK[h] c_t (128) | k_rope_t (64)]
 * and value V_t = W_UV[h]^T c_t (128), then ordinary softmax attention with the
 * un-absorbed query q [B, s_q, H, 192]. out [B, s_q, H, 128], lse [B, s_q, H].
 */
void orc_attend_naive(const float* q, const float* kv, const int32_t* block_table, int mbps,
                      const int32_t* seqlens, int B, int s_q, int H, const float* w_uk,
                      const float* w_uv, double scale, int causal, double* out, double* lse) {
    #pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < s_q; ++s)
            for (int h = 0; h < H; ++h) {
                int64_t row = ((int64_t)b * s_q + s) * H + h;
                const float* qr = q + row * ORC_DQ;
                const int32_t* trow = block_table + (int64_t)b * mbps;
                const float* wk = w_uk + (int64_t)h * ORC_DN * ORC_DC;
                const float* wv = w_uv + (int64_t)h * ORC_DC * ORC_DV;
                int64_t n = visible_keys(seqlens[b], s_q, s, causal);
                double* o = out + row * ORC_DV;
                for (int j = 0; j < ORC_DV; ++j) o[j] = 0.0;
                if (n == 0) { lse[row] = -INFINITY; continue; }
                double* sc = (double*)malloc((size_t)n * sizeof(double));
                double mx = -INFINITY;
                for (int64_t t = 0; t < n; ++t) {
                    const float* c = kv_row(kv, trow, t);
                    double dot = 0.0;
                    for (int d = 0; d < ORC_DN; ++d) {
                        double kd = 0.0;
                        for (int cc = 0; cc < ORC_DC; ++cc) kd += (double)wk[(int64_t)d * ORC_DC + cc] * (double)c[cc];
                        dot += (double)qr[d] * kd;
                    }
                    for (int i = 0; i < ORC_DR; ++i) dot += (double)qr[ORC_DN + i] * (double)c[ORC_DC + i];
                    sc[t] = scale * dot;
                    if (sc[t] > mx) mx = sc[t];
                }
                double l = 0.0;
                for (int64_t t = 0; t < n; ++t) {
                    double p = exp(sc[t] - mx);
                    l += p;
                    const float* c = kv_row(kv, trow, t);
                    for (int j = 0; j < ORC_DV; ++j) {
                        double vj = 0.0;
                        for (int cc = 0; cc < ORC_DC; ++cc) vj += (double)wv[(int64_t)cc * ORC_DV + j] * (double)c[cc];
                        o[j] += p * vj;
                    }
                }
                for (int j = 0; j < ORC_DV; ++j) o[j] /= l;
                lse[row] = mx + log(l);
                free(sc);
            }
}

/*
 * Prefill in the naive (decompress) form over the paged cache [V3 sec. 2.2: the
 * per-head key and value are up-projections of the cached latent, k = W_UK c,
 * v = W_UV c; sec. 3.1: the rope key part is shared by the heads; sec. 4.3:
 * the paged module decompresses K and V per head before ordinary attention].
 * The s_q query tokens of each sequence are its last s_q positions (a whole
 * prompt when s_q = seqlen, a prompt chunk after earlier tokens otherwise).
 * For each (b, h) the keys and values of every cached token t < seqlen_b are
 * materialised once:
 *   K_t = [sum_c W_UK[h,d,c] c_t[c] (d < 128) | k_rope_t (64)],  V_t[j] = sum_c c_t[c] W_UV[h,c,j],
 * then every query row takes a two-pass softmax over its visible keys
 * (bottom-right causal alignment) and out = sum_t p_t V_t.
 * q [B, s_q, H, 192] float -> out [B, s_q, H, 128], lse [B, s_q, H] double.
 */
void orc_prefill_naive(const float* q, const float* kv, const int32_t* block_table, int mbps,
                       const int32_t* seqlens, int B, int s_q, int H, const float* w_uk,
                       const float* w_uv, double scale, int causal, double* out, double* lse) {
    #pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const int64_t L = seqlens[b] > 0 ? seqlens[b] : 0;
            const int32_t* trow = block_table + (int64_t)b * mbps;
            const float* wk = w_uk + (int64_t)h * ORC_DN * ORC_DC;
            const float* wv = w_uv + (int64_t)h * ORC_DC * ORC_DV;
            double* K = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * ORC_DQ);
            double* V = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * ORC_DV);
            for (int64_t t = 0; t < L; ++t) {
                const float* c = kv_row(kv, trow, t);
                for (int d = 0; d < ORC_DN; ++d) {
                    double kd = 0.0;
                    for (int cc = 0; cc < ORC_DC; ++cc) kd += (double)wk[(int64_t)d * ORC_DC + cc] * (double)c[cc];
                    K[t * ORC_DQ + d] = kd;
                }
                for (int i = 0; i < ORC_DR; ++i) K[t * ORC_DQ + ORC_DN + i] = c[ORC_DC + i];
                for (int j = 0; j < ORC_DV; ++j) {
                    double vj = 0.0;
                    for (int cc = 0; cc < ORC_DC; ++cc) vj += (double)c[cc] * (double)wv[(int64_t)cc * ORC_DV + j];
                    V[t * ORC_DV + j] = vj;
                }
            }
            double* sc = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
            for (int s = 0; s < s_q; ++s) {
                const int64_t row = ((int64_t)b * s_q + s) * H + h;
                const float* qr = q + row * ORC_DQ;
                double* o = out + row * ORC_DV;
                for (int j = 0; j < ORC_DV; ++j) o[j] = 0.0;
                const int64_t n = visible_keys(L, s_q, s, causal);
                if (n == 0) { lse[row] = -INFINITY; continue; }
                double mx = -INFINITY;
                for (int64_t t = 0; t < n; ++t) {
                    double dot = 0.0;
                    for (int d = 0; d < ORC_DQ; ++d) dot += (double)qr[d] * K[t * ORC_DQ + d];
                    sc[t] = scale * dot;
                    if (sc[t] > mx) mx = sc[t];
                }
                double l = 0.0;
                for (int64_t t = 0; t < n; ++t) {
                    const double p = exp(sc[t] - mx);
                    l += p;
                    for (int j = 0; j < ORC_DV; ++j) o[j] += p * V[t * ORC_DV + j];
                }
                for (int j = 0; j < ORC_DV; ++j) o[j] /= l;
                lse[row] = mx + log(l);
            }
            free(sc);
            free(K);
            free(V);
        }
}

/*
 * Output up-projection [V3 sec. 2.2, W_UV side of the absorption]:
 * out[r,h,j] = sum_c o_lat[r,h,c] W_UV[h,c,j].
 * o_lat [R, H, 512] double, w_uv [H, 512, 128] float -> out [R, H, 128] double.
 */
void orc_out_proj(const double* o_lat, const float* w_uv, int64_t R, int H, double* out) {
    #pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int h = 0; h < H; ++h) {
            const double* o = o_lat + (r * H + h) * ORC_DC;
            const float* w = w_uv + (int64_t)h * ORC_DC * ORC_DV;
            double* dst = out + (r * H + h) * ORC_DV;
            for (int j = 0; j < ORC_DV; ++j) {
                double acc = 0.0;
                for (int c = 0; c < ORC_DC; ++c) acc += o[c] * (double)w[(int64_t)c * ORC_DV + j];
                dst[j] = acc;
            }
        }
}

/*
 * The pages' own streaming recurrence [V3 sec. 4.1], one key at a time, with a
 * normalised accumulator: m_new = max(m, s); e = exp(m - m_new) l + exp(s - m_new);
 * acc = acc * exp(m - m_new) l / e + v exp(s - m_new) / e; m = m_new; l = e.
 * Written in double (the printed kernel uses half). Same shapes as
 * orc_attend_absorbed; lse = m + ln l at the end.
 */
void orc_attend_streaming(const double* q_abs, const float* kv, const int32_t* block_table, int mbps,
                          const int32_t* seqlens, int B, int s_q, int H, double scale, int causal,
                          double* o_lat, double* lse) {
    #pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < s_q; ++s)
            for (int h = 0; h < H; ++h) {
                int64_t row = ((int64_t)b * s_q + s) * H + h;
                const double* qa = q_abs + row * ORC_DQK;
                const int32_t* trow = block_table + (int64_t)b * mbps;
                int64_t n = visible_keys(seqlens[b], s_q, s, causal);
                double* acc = o_lat + row * ORC_DC;
                for (int c = 0; c < ORC_DC; ++c) acc[c] = 0.0;
                double m = -INFINITY, l = 0.0;
                for (int64_t t = 0; t < n; ++t) {
                    const float* k = kv_row(kv, trow, t);
                    double dot = 0.0;
                    for (int c = 0; c < ORC_DQK; ++c) dot += qa[c] * (double)k[c];
                    double sc = scale * dot;
                    double m_new = sc > m ? sc : m;
                    double keep = exp(m - m_new) * l;
                    double e = keep + exp(sc - m_new);
                    double a = keep / e, w = exp(sc - m_new) / e;
                    for (int c = 0; c < ORC_DC; ++c) acc[c] = acc[c] * a + (double)k[c] * w;
                    m = m_new;
                    l = e;
                }
                lse[row] = n > 0 ? m + log(l) : -INFINITY;
            }
}

/*
 * Split-KV combine of n partial results of one query row (pieces over
 * disjoint key ranges, each normalised by its own sum):
 * L = max_i lse_i; lse = L + ln sum_i exp(lse_i - L); o = sum_i exp(lse_i - lse) o_i.
 * o_parts [n, 512], lse_parts [n] -> o [512], *lse.
 */
void orc_combine(const double* o_parts, const double* lse_parts, int n, double* o, double* lse) {
    for (int c = 0; c < ORC_DC; ++c) o[c] = 0.0;
    double L = -INFINITY;
    for (int i = 0; i < n; ++i) if (lse_parts[i] > L) L = lse_parts[i];
    if (L == -INFINITY) { *lse = -INFINITY; return; }
    double sum = 0.0;
    for (int i = 0; i < n; ++i) sum += exp(lse_parts[i] - L);
    double total = L + log(sum);
    for (int i = 0; i < n; ++i) {
        double w = exp(lse_parts[i] - total);
        for (int c = 0; c < ORC_DC; ++c) o[c] += w * o_parts[(int64_t)i * ORC_DC + c];
    }
    *lse = total;
}

/*
 * Tile/split schedule. The pages fix only the call shape
 * [FM usage example: get_mla_metadata(cache_seqlens, ...) -> (tile_scheduler_metadata,
 * num_splits), computed once per decode step]; the rule below is this
 * project's own and is written out as the plainest walk over work units.
 *
 *  nblk_b  = ceil(seqlen_b / 64) pages (seqlen < 0 counts as 0).
 *  cost_b  = nblk_b + ovh if nblk_b > 0, else 0;  start_b = sum_{b' < b} cost_b'.
 *  total   = sum_b cost_b;  quota = max(1, ceil(total / num_parts)).
 *  Units are (b, page j) in order. Key of a unit: a short batch
 *  (nblk_b < min_split) puts every unit at key start_b, so it is never split;
 *  a long batch puts page 0 at start_b and page j >= 1 at start_b + ovh + j.
 *  A unit belongs to part floor(key / quota).
 *  A piece is a maximal run of one batch's units inside one part. Pieces are
 *  numbered in walk order (which is part order).
 *  tile_meta[p] = {begin_b, begin_page, end_b, end_page (exclusive),
 *                  first_piece, n_pieces, 0, 0}; an empty part is all zeros.
 *  num_splits[b] = index of batch b's first piece (exclusive prefix sum of the
 *  number of pieces per batch); num_splits[B] = total pieces.
 * Returns 0, or -1 on bad arguments.
 */
int orc_metadata(const int32_t* seqlens, int B, int num_parts, int ovh, int min_split,
                 int32_t* tile_meta, int32_t* num_splits) {
    if (B < 0 || num_parts <= 0 || ovh < 0 || min_split < 1) return -1;
    int64_t total = 0;
    for (int b = 0; b < B; ++b) {
        int64_t n = seqlens[b] > 0 ? ((int64_t)seqlens[b] + ORC_PAGE - 1) / ORC_PAGE : 0;
        if (n > 0) total += n + ovh;
    }
    int64_t quota = (total + num_parts - 1) / num_parts;
    if (quota < 1) quota = 1;
    memset(tile_meta, 0, sizeof(int32_t) * 8 * (size_t)num_parts);
    int32_t* pieces_of_batch = (int32_t*)calloc((size_t)(B > 0 ? B : 1), sizeof(int32_t));
    int64_t start = 0;
    int32_t piece_count = 0;
    int last_part = -1, last_batch = -1;
    for (int b = 0; b < B; ++b) {
        int64_t n = seqlens[b] > 0 ? ((int64_t)seqlens[b] + ORC_PAGE - 1) / ORC_PAGE : 0;
        if (n == 0) continue;
        int is_long = n >= min_split;
        for (int64_t j = 0; j < n; ++j) {
            int64_t key = (!is_long || j == 0) ? start : start + ovh + j;
            int p = (int)(key / quota);
            int32_t* row = tile_meta + (size_t)8 * p;
            if (p != last_part || b != last_batch) {
                /* a new piece starts here */
                if (row[5] == 0) {
                    row[0] = b;
                    row[1] = (int32_t)j;
                    row[4] = piece_count;
                }
                row[5] += 1;
                piece_count += 1;
                pieces_of_batch[b] += 1;
                last_part = p;
                last_batch = b;
            }
            row[2] = b;
            row[3] = (int32_t)(j + 1);
        }
        start += n + ovh;
    }
    num_splits[0] = 0;
    for (int b = 0; b < B; ++b) num_splits[b + 1] = num_splits[b] + pieces_of_batch[b];
    free(pieces_of_batch);
    return 0;
}

/*
 * Split-KV decode through a schedule: every piece of the schedule is attended
 * on its own (absorbed form over the piece's pages), then each query row of a
 * batch combines its pieces with orc_combine. Key ranges are clipped to the
 * row's visible keys, so a piece past a causal limit contributes lse = -inf.
 * Shapes as orc_attend_absorbed; tile_meta/num_splits from orc_metadata.
 * Also returns the per-piece partials when o_parts/lse_parts are non-NULL:
 * o_parts [total_pieces, s_q, H, 512], lse_parts [total_pieces, s_q, H].
 */
void orc_attend_split(const double* q_abs, const float* kv, const int32_t* block_table, int mbps,
                      const int32_t* seqlens, int B, int s_q, int H, double scale, int causal,
                      const int32_t* tile_meta, int num_parts, const int32_t* num_splits,
                      double* o_lat, double* lse, double* o_parts_out, double* lse_parts_out) {
    int total_pieces = num_splits[B];
    int64_t rows_per_piece = (int64_t)s_q * H;
    double* o_parts = o_parts_out ? o_parts_out
                                  : (double*)malloc(sizeof(double) * (size_t)(total_pieces > 0 ? total_pieces : 1) * rows_per_piece * ORC_DC);
    double* lse_parts = lse_parts_out ? lse_parts_out
                                      : (double*)malloc(sizeof(double) * (size_t)(total_pieces > 0 ? total_pieces : 1) * rows_per_piece);
    /* list the pieces: (batch, first page, end page) in piece order */
    int32_t* pb = (int32_t*)malloc(sizeof(int32_t) * (size_t)(total_pieces > 0 ? total_pieces : 1) * 3);
    for (int p = 0; p < num_parts; ++p) {
        const int32_t* row = tile_meta + (size_t)8 * p;
        if (row[5] == 0) continue;
        int k = 0;
        for (int b = row[0]; b <= row[2]; ++b) {
            int64_t n = seqlens[b] > 0 ? ((int64_t)seqlens[b] + ORC_PAGE - 1) / ORC_PAGE : 0;
            if (n == 0) continue;
            int lo = (b == row[0]) ? row[1] : 0;
            int hi = (b == row[2]) ? row[3] : (int)n;
            int idx = row[4] + k;
            pb[3 * idx + 0] = b;
            pb[3 * idx + 1] = lo;
            pb[3 * idx + 2] = hi;
            k += 1;
        }
    }
    #pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int i = 0; i < total_pieces; ++i)
        for (int s = 0; s < s_q; ++s)
            for (int h = 0; h < H; ++h) {
                int b = pb[3 * i];
                int64_t vis = visible_keys(seqlens[b], s_q, s, causal);
                int64_t t_lo = (int64_t)pb[3 * i + 1] * ORC_PAGE;
                int64_t t_hi = (int64_t)pb[3 * i + 2] * ORC_PAGE;
                if (t_hi > vis) t_hi = vis;
                int64_t row = ((int64_t)b * s_q + s) * H + h;
                int64_t prow = ((int64_t)i * s_q + s) * H + h;
                attend_absorbed_row(q_abs + row * ORC_DQK, kv, block_table + (int64_t)b * mbps, t_lo, t_hi,
                                    scale, o_parts + prow * ORC_DC, lse_parts + prow);
            }
    #pragma omp parallel for collapse(3) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < s_q; ++s)
            for (int h = 0; h < H; ++h) {
                int n = num_splits[b + 1] - num_splits[b];
                int64_t row = ((int64_t)b * s_q + s) * H + h;
                double* tmp_o = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * ORC_DC);
                double* tmp_l = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
                for (int i = 0; i < n; ++i) {
                    int64_t prow = ((int64_t)(num_splits[b] + i) * s_q + s) * H + h;
                    memcpy(tmp_o + (int64_t)i * ORC_DC, o_parts + prow * ORC_DC, sizeof(double) * ORC_DC);
                    tmp_l[i] = lse_parts[prow];
                }
                orc_combine(tmp_o, tmp_l, n, o_lat + row * ORC_DC, lse + row);
                free(tmp_o);
                free(tmp_l);
            }
    free(pb);
    if (!o_parts_out) free(o_parts);
    if (!lse_parts_out) free(lse_parts);
}

/*
 * Rotary position encoding of the decoupled rope parts [V3 sec. 3.1: RoPE(q_pos, t)
 * is a rotation that depends on the token position t; sec. 3.2: the position key
 * is RoPE applied per token]. The pages do not print the rotation itself; this
 * is the standard rotary encoding: the d-vector is read as d/2 adjacent pairs
 * (x[2i], x[2i+1]), and pair i is rotated by the angle t * theta_i with
 * theta_i = base^(-2i/d):
 *   y[2i]   = x[2i] cos(t theta_i) - x[2i+1] sin(t theta_i)
 *   y[2i+1] = x[2i] sin(t theta_i) + x[2i+1] cos(t theta_i)
 * x [rows, d] float, pos [rows] -> y [rows, d] double.
 */
void orc_rope(const float* x, int64_t rows, int d, const int64_t* pos, double base, double* y) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int i = 0; i < d / 2; ++i) {
            double theta = pow(base, -2.0 * i / d);
            double a = (double)pos[r] * theta;
            double c = cos(a), sn = sin(a);
            double x0 = x[r * d + 2 * i], x1 = x[r * d + 2 * i + 1];
            y[r * d + 2 * i] = x0 * c - x1 * sn;
            y[r * d + 2 * i + 1] = x0 * sn + x1 * c;
        }
    }
}

/*
 * Appending the s_q new tokens of each sequence to its paged cache [V3 sec. 4.3:
 * only the latent is stored, kv_cache.store(c_kv); sec. 3.2: the position key
 * is the rotary-encoded rope part]. Token s of sequence b sits at position
 * t = seqlen_b - s_q + s (the lengths already count the new tokens); its slot is
 * row t % 64 of block block_table[b][t / 64]. The slot receives
 * [c_KV (512, as given) | RoPE(k_rope (64), t)]. Tokens with t < 0 are skipped.
 * kv_new [B, s_q, 576] float (c_KV | un-rotated k_rope); kv [num_blocks, 64, 576]
 * double, updated in place (other slots untouched).
 */
void orc_cache_append(const float* kv_new, const int32_t* block_table, int mbps, const int32_t* seqlens, int B,
                      int s_q, double base, double* kv) {
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < s_q; ++s) {
            int64_t t = (int64_t)seqlens[b] - s_q + s;
            if (t < 0) continue;
            int64_t blk = block_table[(int64_t)b * mbps + t / ORC_PAGE];
            double* slot = kv + (blk * ORC_PAGE + t % ORC_PAGE) * ORC_DQK;
            const float* src = kv_new + ((int64_t)b * s_q + s) * ORC_DQK;
            for (int c = 0; c < ORC_DC; ++c) slot[c] = src[c];
            orc_rope(src + ORC_DC, 1, ORC_DR, &t, base, slot + ORC_DC);
        }
}

/*
 * Quantised latent cache [V3 sec. 7.2: the compressed latent is stored in 8
 * bits, c_t = Quantize(W_DKV h_t, bits = 8); DS1 sec. 3.1 names INT8 as the
 * representative KV quantisation]. The pages fix the width and nothing else.
 * Reading used here:
 *  - the quantised object is the per-token latent c_t (512 dims); the
 *    decoupled rope key is not part of c_KV and stays bf16;
 *  - symmetric INT8 codes in [-127, 127] with one scale per token;
 *  - the scale is the smallest power of two s with 127 s >= max_c |c_t[c]|
 *    (so c / s is exact and every code * s is exactly representable in bf16);
 *  - code = c / s rounded to the nearest integer, ties to even;
 *  - a token whose latent is all zero has s = 1 and all codes 0.
 * The smallest power of two: write amax = m 2^k with m in [0.5, 1) (frexp);
 * 127 * 2^(k-7) >= amax iff m <= 127/128, else 2^(k-6) is the smallest (64 m <=
 * 63.99 < 127 and 128 m > 127).
 * x [rows, 512] float -> codes [rows, 512] int8, scale [rows] float.
 */
void orc_quantize_latent(const float* x, int64_t rows, int8_t* codes, float* scale) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * ORC_DC;
        double amax = 0.0;
        for (int c = 0; c < ORC_DC; ++c) amax = fmax(amax, fabs((double)xr[c]));
        double s = 1.0;
        if (amax > 0.0) {
            int k;
            double m = frexp(amax, &k);
            s = ldexp(1.0, m <= 127.0 / 128.0 ? k - 7 : k - 6);
        }
        scale[r] = (float)s;
        for (int c = 0; c < ORC_DC; ++c) {
            double q = nearbyint((double)xr[c] / s);  /* default rounding: to nearest, ties to even */
            codes[r * ORC_DC + c] = (int8_t)q;
        }
    }
}

/*
 * The quantised cache as stored: one 640-byte record per token,
 *   bytes [0, 512)   the INT8 codes of c_KV (orc_quantize_latent),
 *   bytes [512, 640) k_rope as 64 bf16 values, little-endian, unchanged,
 * and the scales as a separate float array [tokens]. kv [tokens, 576] holds
 * values that are exact in bf16 (the rope part is copied bit for bit).
 */
void orc_quantize_cache(const float* kv, int64_t tokens, uint8_t* rec, float* scale) {
    float* lat = (float*)malloc(sizeof(float) * ORC_DC * (tokens > 0 ? tokens : 1));
    int8_t* codes = (int8_t*)malloc(ORC_DC * (tokens > 0 ? tokens : 1));
    for (int64_t t = 0; t < tokens; ++t)
        for (int c = 0; c < ORC_DC; ++c) lat[t * ORC_DC + c] = kv[t * ORC_DQK + c];
    orc_quantize_latent(lat, tokens, codes, scale);
    for (int64_t t = 0; t < tokens; ++t) {
        uint8_t* out = rec + t * 640;
        memcpy(out, codes + t * ORC_DC, ORC_DC);
        for (int d = 0; d < ORC_DR; ++d) {
            uint32_t bits;
            float v = kv[t * ORC_DQK + ORC_DC + d];
            memcpy(&bits, &v, 4);
            out[ORC_DC + 2 * d] = (uint8_t)((bits >> 16) & 0xFF);
            out[ORC_DC + 2 * d + 1] = (uint8_t)(bits >> 24);
        }
    }
    free(lat);
    free(codes);
}

/*
 * The cache the quantised records stand for: latent = code * scale (exact),
 * rope = the stored bf16 values. rec [tokens, 640] bytes, scale [tokens] ->
 * kv [tokens, 576] float. Attention over a quantised cache is attention over
 * this cache (orc_attend_absorbed).
 */
void orc_dequantize_cache(const uint8_t* rec, const float* scale, int64_t tokens, float* kv) {
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < tokens; ++t) {
        const uint8_t* in = rec + t * 640;
        for (int c = 0; c < ORC_DC; ++c) kv[t * ORC_DQK + c] = (float)((double)(int8_t)in[c] * (double)scale[t]);
        for (int d = 0; d < ORC_DR; ++d) {
            uint32_t bits = ((uint32_t)in[ORC_DC + 2 * d] << 16) | ((uint32_t)in[ORC_DC + 2 * d + 1] << 24);
            float v;
            memcpy(&v, &bits, 4);
            kv[t * ORC_DQK + ORC_DC + d] = v;
        }
    }
}

/* Threads the OpenMP runtime will use (1 when built without OpenMP). */
int orc_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
