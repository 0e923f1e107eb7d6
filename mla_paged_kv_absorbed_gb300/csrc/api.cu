// api.cu - the extern "C" boundary declared in include/mla.h: argument
// checks, TMA tensor-map construction, workspace layout and kernel launches.
// Nothing here computes any part of the method; every step runs on the GPU.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "mla.h"
#include "mla_internal.h"
#include "quant.cuh"

namespace mla {

WorkspaceLayout workspace_layout(int B, int s_q, int H, int num_parts) {
    WorkspaceLayout l;
    const size_t pieces = (size_t)B + (size_t)num_parts;
    const size_t rows = pieces * (size_t)s_q * (size_t)H;
    l.lse_offset = kWorkspaceHeader;
    l.o_offset = l.lse_offset + ((rows * sizeof(float) + 255) & ~size_t(255));
    l.total = l.o_offset + rows * kDLatent * sizeof(float);
    return l;
}

namespace {

std::atomic<long long> g_wait_ns{4000000000LL};
std::atomic<int> g_withhold{0};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor map with 128-byte swizzle (bf16 unless stated); dims[0] is the contiguous one.
bool make_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
               const uint32_t* box, CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base),
                    reinterpret_cast<const cuuint64_t*>(dims), reinterpret_cast<const cuuint64_t*>(strides_bytes),
                    reinterpret_cast<const cuuint32_t*>(box), elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The cache as a 3-D view {64 dims, num_blocks * 64 keys, 9 chunks} with
// strides {1152, 128} bytes, so that one box {64, 64, chunks} is a whole page
// (chunks = 9) or its 512 value columns (chunks = 8), landing in shared memory
// as [chunk][key][64 dims]. Used by the decode kernel and its gather test hook.
bool make_kv_page_map(CUtensorMap* map, const void* kv_cache, int num_blocks, int chunks) {
    const uint64_t dims[3] = {64, (uint64_t)num_blocks * kPage, (uint64_t)kDQK / 64};
    const uint64_t strides[2] = {(uint64_t)kDQK * 2, 128};
    const uint32_t box[3] = {64, (uint32_t)kPage, (uint32_t)chunks};
    return make_tmap(map, kv_cache, 3, dims, strides, box, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

struct DeviceInfo {
    int sm_count = 0, major = 0, minor = 0, max_clusters = -1;
};

bool device_info(DeviceInfo& info) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool valid[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lk(mu);
    if (!valid[dev]) {
        cudaDeviceProp p;
        if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) return false;
        cache[dev].sm_count = p.multiProcessorCount;
        cache[dev].major = p.major;
        cache[dev].minor = p.minor;
        valid[dev] = true;
    }
    info = cache[dev];
    return true;
}

}  // namespace

// SM count of the current device (cached per device ordinal), 0 on failure.
int device_sm_count() {
    DeviceInfo d;
    return device_info(d) ? d.sm_count : 0;
}

namespace {

int check_device() {
    DeviceInfo d;
    if (!device_info(d)) return MLA_ERR_CUDA;
    if (!(d.major == 10 && d.minor == 3)) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_heads(int H) { return H == 16 || H == 32 || H == 64 || H == 128; }
bool valid_sq(int s_q) { return s_q == 1 || s_q == 2; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

int head_gemm(const void* a, int a_row_elems, const void* w, int K, int N, int n_cta, void* out, int out_row_elems,
              const void* rope_src, int B, int s_q, int H, cudaStream_t stream) {
    const int R = B * s_q;
    // [64-column chunk][row] views (4-D, innermost first): one box is 128 rows
    // x several chunks of a head
    CUtensorMap tm_a, tm_b, tm_out;
    const uint64_t a_dims[4] = {64, (uint64_t)R, (uint64_t)a_row_elems / 64, (uint64_t)H};
    const uint64_t a_strides[3] = {(uint64_t)H * a_row_elems * 2, 128, (uint64_t)a_row_elems * 2};
    const uint32_t a_box[4] = {64, 128, 2, 1};
    const uint64_t b_dims[4] = {64, (uint64_t)K, (uint64_t)N / 64, (uint64_t)H};
    const uint64_t b_strides[3] = {(uint64_t)N * 2, 128, (uint64_t)K * N * 2};
    const uint32_t b_box[4] = {64, 128, (uint32_t)n_cta / 64, 1};
    const uint64_t o_dims[4] = {64, (uint64_t)R, (uint64_t)out_row_elems / 64, (uint64_t)H};
    const uint64_t o_strides[3] = {(uint64_t)H * out_row_elems * 2, 128, (uint64_t)out_row_elems * 2};
    const uint32_t o_box[4] = {64, 128, (uint32_t)n_cta / 64, 1};
    if (!make_tmap(&tm_a, a, 4, a_dims, a_strides, a_box)) return MLA_ERR_CUDA;
    if (!make_tmap(&tm_b, w, 4, b_dims, b_strides, b_box, CU_TENSOR_MAP_L2_PROMOTION_L2_256B)) return MLA_ERR_CUDA;
    if (!make_tmap(&tm_out, out, 4, o_dims, o_strides, o_box)) return MLA_ERR_CUDA;
    GemmArgs args;
    args.R = R;
    args.H = H;
    args.K = K;
    args.N = N;
    args.n_cta = n_cta;
    args.out = out;
    args.out_row_elems = out_row_elems;
    args.rope_src = rope_src;
    args.a_shared = 0;
    args.b_kmajor = 0;
    return cuda_status(launch_head_gemm(&tm_a, &tm_b, &tm_out, args, g_wait_ns.load(), stream));
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(int status) {
    switch (status) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: bad pointer, size, alignment or shape";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: device is not sm_103 or shape not supported";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call or kernel launch failed";
        case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded pipeline wait expired on the device";
        case MLA_ERR_BAD_BLOCK: return "MLA_ERR_BAD_BLOCK: block id outside the pool or seqlen past its table row";
        default: return "unknown mla status";
    }
}

int mla_version(void) { return 101; }

void mla_schedule_constants(int* piece_overhead, int* min_split_pages) {
    if (piece_overhead) *piece_overhead = kSchedOverhead;
    if (min_split_pages) *min_split_pages = kSchedMinSplitPages;
}

int mla_default_num_parts(int device, int s_q) {
    if (!valid_sq(s_q)) return -MLA_ERR_INVALID_ARG;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return -MLA_ERR_CUDA;
    if (device != prev && cudaSetDevice(device) != cudaSuccess) return -MLA_ERR_CUDA;
    DeviceInfo d;
    const bool ok = device_info(d);
    int clusters = ok ? decode_max_active_clusters(device) : 0;
    if (device != prev) cudaSetDevice(prev);
    if (!ok) return -MLA_ERR_CUDA;
    if (clusters <= 0) clusters = d.sm_count / 2;
    int parts = clusters / s_q;
    return parts > 0 ? parts : 1;
}

size_t mla_workspace_size(int B, int s_q, int H, int num_parts) {
    if (B <= 0 || !valid_sq(s_q) || !valid_heads(H) || num_parts <= 0) return 0;
    return workspace_layout(B, s_q, H, num_parts).total;
}

void mla_set_wait_limit_ns(long long ns) { g_wait_ns.store(ns > 0 ? ns : 4000000000LL); }

void mla_debug_withhold_value_load(int enable) { g_withhold.store(enable != 0 ? 1 : 0); }

int mla_get_metadata(const int32_t* cache_seqlens, int B, int s_q, int H, int h_kv, int num_parts,
                     int32_t* tile_meta, int32_t* num_splits, mla_stream_t stream) {
    if (!cache_seqlens || !tile_meta || !num_splits || B <= 0 || num_parts <= 0 || num_parts > 65536 || h_kv != 1 ||
        !valid_sq(s_q) || !valid_heads(H))
        return MLA_ERR_INVALID_ARG;
    int dev = check_device();
    if (dev != MLA_OK) return dev;
    return cuda_status(launch_metadata(cache_seqlens, B, num_parts, kSchedOverhead, kSchedMinSplitPages, tile_meta,
                                       num_splits, static_cast<cudaStream_t>(stream)));
}

int mla_absorb_q(const mla_bf16_t* q, const mla_bf16_t* w_uk, mla_bf16_t* q_abs, int B, int s_q, int H,
                 mla_stream_t stream) {
    if (!q || !w_uk || !q_abs || B <= 0 || !valid_sq(s_q) || !valid_heads(H)) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(w_uk) || !aligned16(q_abs)) return MLA_ERR_INVALID_ARG;
    int dev = check_device();
    if (dev != MLA_OK) return dev;
    return head_gemm(q, kDQ, w_uk, kDNope, kDLatent, 128, q_abs, kDQK, q, B, s_q, H,
                     static_cast<cudaStream_t>(stream));
}

int mla_out_proj(const mla_bf16_t* o_lat, const mla_bf16_t* w_uv, mla_bf16_t* out, int B, int s_q, int H,
                 mla_stream_t stream) {
    if (!o_lat || !w_uv || !out || B <= 0 || !valid_sq(s_q) || !valid_heads(H)) return MLA_ERR_INVALID_ARG;
    if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
    int dev = check_device();
    if (dev != MLA_OK) return dev;
    return head_gemm(o_lat, kDLatent, w_uv, kDLatent, kDV, 128, out, kDV, nullptr, B, s_q, H,
                     static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace mla {

// The decode entry points' host-side argument checks, apart from the
// workspace (no device call): MLA_OK or MLA_ERR_INVALID_ARG.
int decode_check_args(const void* q_abs, const void* kv_cache, const void* kv8, const float* kv_scale,
                      int num_blocks, const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens,
                      int B, int s_q, int H, const int32_t* tile_meta, const int32_t* num_splits, int num_parts,
                      float softmax_scale, int causal, const void* o_lat, const float* lse, const void* w_uv,
                      const void* out) {
    const bool q8 = kv8 != nullptr;
    if (w_uv != nullptr && (out == nullptr || !aligned16(w_uv) || !aligned16(out))) return MLA_ERR_INVALID_ARG;
    if (!q_abs || (q8 ? (!kv_scale || kv_cache) : !kv_cache) || !block_table || !cache_seqlens || !tile_meta ||
        !num_splits || !o_lat || !lse)
        return MLA_ERR_INVALID_ARG;
    if (q8 && (!aligned16(kv8) || !aligned16(kv_scale))) return MLA_ERR_INVALID_ARG;
    if (B <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || num_parts <= 0 || !valid_sq(s_q) || !valid_heads(H))
        return MLA_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || (causal != 0 && causal != 1)) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_abs) || (!q8 && !aligned16(kv_cache)) || !aligned16(o_lat) || !aligned16(lse))
        return MLA_ERR_INVALID_ARG;
    if ((uint64_t)num_blocks * kPage > 0xFFFFFFFFull) return MLA_ERR_INVALID_ARG;
    return MLA_OK;
}

namespace {
// The decode over either cache format: the bf16 cache (kv_cache, kv8 = NULL)
// or the INT8 records with their scales (kv8 and kv_scale, kv_cache = NULL).
// With w_uv = NULL the split pieces are merged into o_lat (combine kernel);
// otherwise the merge and the output projection run as one finalize kernel
// that writes out (o_lat then only holds the rows of unsplit sequences).
int decode_impl(const mla_bf16_t* q_abs, const void* kv_cache, const void* kv8, const float* kv_scale, int num_blocks,
                const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens, int B, int s_q,
                int H, const int32_t* tile_meta, const int32_t* num_splits, int num_parts, float softmax_scale,
                int causal, mla_bf16_t* o_lat, float* lse, void* workspace, size_t workspace_bytes,
                mla_stream_t stream, const mla_bf16_t* w_uv = nullptr, mla_bf16_t* out = nullptr) {
    const bool q8 = kv8 != nullptr;
    const int rc = decode_check_args(q_abs, kv_cache, kv8, kv_scale, num_blocks, block_table, max_blocks_per_seq,
                                     cache_seqlens, B, s_q, H, tile_meta, num_splits, num_parts, softmax_scale, causal,
                                     o_lat, lse, w_uv, out);
    if (rc != MLA_OK) return rc;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MLA_ERR_INVALID_ARG;
    const WorkspaceLayout wl = workspace_layout(B, s_q, H, num_parts);
    if (workspace_bytes < wl.total) return MLA_ERR_INVALID_ARG;
    int dev = check_device();
    if (dev != MLA_OK) return dev;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    DecodeMaps maps = {};
    CUtensorMap fin_w, fin_out;
    if (q8) {
        // the records as {128 code bytes, num_blocks * 64 keys, 4 planes}, strides
        // {640, 128}: one box is a page's 32 KB of codes as four [64 keys][128 B]
        // planes; the rope keys (bytes 512-639 of each record) as bf16 {64, keys}
        const uint64_t keys = (uint64_t)num_blocks * kPage;
        const uint64_t c_dims[3] = {128, keys, 4};
        const uint64_t c_strides[2] = {(uint64_t)kQ8Record, 128};
        const uint32_t c_box[3] = {128, (uint32_t)kPage, 4};
        if (!make_tmap(&maps.kv8, kv8, 3, c_dims, c_strides, c_box, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_DATA_TYPE_UINT8))
            return MLA_ERR_CUDA;
        const uint64_t r_dims[2] = {(uint64_t)kDRope, keys};
        const uint64_t r_strides[1] = {(uint64_t)kQ8Record};
        const uint32_t r_box[2] = {(uint32_t)kDRope, (uint32_t)kPage};
        if (!make_tmap(&maps.rope, static_cast<const uint8_t*>(kv8) + kDLatent, 2, r_dims, r_strides, r_box,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
            return MLA_ERR_CUDA;
    } else {
        // [dims, keys, chunk] views: one box per page (or per 64 query rows)
        if (!make_kv_page_map(&maps.kv, kv_cache, num_blocks, kDQK / 64)) return MLA_ERR_CUDA;
        if (!make_kv_page_map(&maps.v, kv_cache, num_blocks, kDLatent / 64)) return MLA_ERR_CUDA;
    }
    const uint64_t rows = (uint64_t)B * s_q;
    const uint64_t qrows_total = rows * (uint64_t)H;
    const uint32_t qrows = (uint32_t)(qrows_total < 64 ? qrows_total : 64);
    const uint64_t q_dims[3] = {64, qrows_total, (uint64_t)kDQK / 64};
    const uint64_t q_strides[2] = {(uint64_t)kDQK * 2, 128};
    const uint32_t q_box[3] = {64, qrows, (uint32_t)kDQK / 64};
    if (!make_tmap(&maps.q, q_abs, 3, q_dims, q_strides, q_box)) return MLA_ERR_CUDA;
    // outputs as {128-byte chunk, head row, chunk index, token}: one store box
    // covers four chunks of every head row of a token
    const uint32_t h_rows = (uint32_t)(H < 128 ? H : 128);
    const uint64_t o_dims[4] = {64, (uint64_t)H, (uint64_t)kDLatent / 64, rows};
    const uint64_t o_strides[3] = {(uint64_t)kDLatent * 2, 128, (uint64_t)H * kDLatent * 2};
    const uint32_t o_box[4] = {64, h_rows, 4, 1};
    if (!make_tmap(&maps.o, o_lat, 4, o_dims, o_strides, o_box)) return MLA_ERR_CUDA;
    const uint64_t pieces = ((uint64_t)B + (uint64_t)num_parts) * s_q;
    const uint64_t op_dims[4] = {64, (uint64_t)H, (uint64_t)kDLatent / 64, pieces};
    const uint64_t op_strides[3] = {(uint64_t)kDLatent * 2, 128, (uint64_t)H * kDLatent * 2};
    const uint32_t op_box[4] = {64, h_rows, 4, 1};
    if (!make_tmap(&maps.op, ws + wl.o_offset, 4, op_dims, op_strides, op_box, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
        return MLA_ERR_CUDA;

    DecodeArgs a = {};
    a.q_abs = q_abs;
    a.block_table = block_table;
    a.mbps = max_blocks_per_seq;
    a.seqlens = cache_seqlens;
    a.tile_meta = tile_meta;
    a.num_splits = num_splits;
    a.num_parts = num_parts;
    a.B = B;
    a.s_q = s_q;
    a.H = H;
    a.num_blocks = num_blocks;
    a.qrows = (int)qrows;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.causal = causal;
    a.o_lat = o_lat;
    a.lse = lse;
    a.lse_part = reinterpret_cast<float*>(ws + wl.lse_offset);
    a.o_part = ws + wl.o_offset;
    a.err = reinterpret_cast<int*>(ws);
    a.wait_ns = g_wait_ns.load();
    a.withhold = g_withhold.load();
    a.kv_scale = q8 ? kv_scale : nullptr;
    // a sequence is split only from kSchedMinSplitPages pages on: with a
    // narrower block table no piece needs merging, so the decode kernel also
    // writes the rows of empty sequences and the merge launch is left out
    // (the fused finalize merges and writes those rows itself)
    a.own_empty = (w_uv == nullptr && max_blocks_per_seq < kSchedMinSplitPages) ? 1 : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (w_uv != nullptr) {
        // the finalize kernel's maps: W_UV[h] as [2 column chunks][128 latent
        // rows][64] boxes (as the projection's), out as [2 chunks][128 rows][64]
        const uint64_t R = rows;
        const uint64_t w_dims[4] = {64, (uint64_t)kDLatent, (uint64_t)kDV / 64, (uint64_t)H};
        const uint64_t w_strides[3] = {(uint64_t)kDV * 2, 128, (uint64_t)kDLatent * kDV * 2};
        const uint32_t w_box[4] = {64, 128, (uint32_t)kDV / 64, 1};
        const uint64_t f_dims[4] = {64, R, (uint64_t)kDV / 64, (uint64_t)H};
        const uint64_t f_strides[3] = {(uint64_t)H * kDV * 2, 128, (uint64_t)kDV * 2};
        const uint32_t f_box[4] = {64, 128, (uint32_t)kDV / 64, 1};
        if (!make_tmap(&fin_w, w_uv, 4, w_dims, w_strides, w_box, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
            return MLA_ERR_CUDA;
        if (!make_tmap(&fin_out, out, 4, f_dims, f_strides, f_box)) return MLA_ERR_CUDA;
    }
    cudaError_t e = launch_decode(maps, a, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    if (w_uv != nullptr) {
        FinArgs f = {};
        f.num_splits = num_splits;
        f.R = B * s_q;
        f.s_q = s_q;
        f.H = H;
        f.o_part = a.o_part;
        f.lse_part = a.lse_part;
        f.o_lat = o_lat;
        f.lse = lse;
        f.err = a.err;
        f.wait_ns = a.wait_ns;
        return cuda_status(launch_finalize(&fin_w, &fin_out, f, st));
    }
    if (a.own_empty) return MLA_OK;
    e = launch_combine(num_splits, B, s_q, H, a.o_part, a.lse_part, o_lat, lse, st);
    return cuda_status(e);
}
}  // namespace
}  // namespace mla

extern "C" {

int mla_decode_paged(const mla_bf16_t* q_abs, const mla_bf16_t* kv_cache, int num_blocks, const int32_t* block_table,
                     int max_blocks_per_seq, const int32_t* cache_seqlens, int B, int s_q, int H,
                     const int32_t* tile_meta, const int32_t* num_splits, int num_parts, float softmax_scale,
                     int causal, mla_bf16_t* o_lat, float* lse, void* workspace, size_t workspace_bytes,
                     mla_stream_t stream) {
    if (!kv_cache) return MLA_ERR_INVALID_ARG;
    return mla::decode_impl(q_abs, kv_cache, nullptr, nullptr, num_blocks, block_table, max_blocks_per_seq,
                            cache_seqlens, B, s_q, H, tile_meta, num_splits, num_parts, softmax_scale, causal, o_lat,
                            lse, workspace, workspace_bytes, stream);
}

int mla_decode_out_proj(const mla_bf16_t* q_abs, const mla_bf16_t* kv_cache, int num_blocks,
                        const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens, int B,
                        int s_q, int H, const int32_t* tile_meta, const int32_t* num_splits, int num_parts,
                        float softmax_scale, int causal, const mla_bf16_t* w_uv, mla_bf16_t* o_lat, mla_bf16_t* out,
                        float* lse, void* workspace, size_t workspace_bytes, mla_stream_t stream) {
    if (!kv_cache || !w_uv || !out) return MLA_ERR_INVALID_ARG;
    return mla::decode_impl(q_abs, kv_cache, nullptr, nullptr, num_blocks, block_table, max_blocks_per_seq,
                            cache_seqlens, B, s_q, H, tile_meta, num_splits, num_parts, softmax_scale, causal, o_lat,
                            lse, workspace, workspace_bytes, stream, w_uv, out);
}

int mla_decode_paged_q8(const mla_bf16_t* q_abs, const uint8_t* kv8, const float* kv_scale, int num_blocks,
                        const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens, int B,
                        int s_q, int H, const int32_t* tile_meta, const int32_t* num_splits, int num_parts,
                        float softmax_scale, int causal, mla_bf16_t* o_lat, float* lse, void* workspace,
                        size_t workspace_bytes, mla_stream_t stream) {
    if (!kv8 || !kv_scale) return MLA_ERR_INVALID_ARG;
    return mla::decode_impl(q_abs, nullptr, kv8, kv_scale, num_blocks, block_table, max_blocks_per_seq, cache_seqlens,
                            B, s_q, H, tile_meta, num_splits, num_parts, softmax_scale, causal, o_lat, lse, workspace,
                            workspace_bytes, stream);
}

int mla_quantize_cache(const mla_bf16_t* kv, long long tokens, uint8_t* kv8, float* kv_scale, mla_stream_t stream) {
    if (!kv || !kv8 || !kv_scale || tokens <= 0) return MLA_ERR_INVALID_ARG;
    if (!aligned16(kv) || !aligned16(kv8) || !aligned16(kv_scale)) return MLA_ERR_INVALID_ARG;
    int dev = check_device();
    if (dev != MLA_OK) return dev;
    return cuda_status(launch_quantize(kv, tokens, kv8, kv_scale, static_cast<cudaStream_t>(stream)));
}



int mla_read_device_error(void* workspace, mla_stream_t stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int ws_err = 0, gemm_err = 0, rope_err = 0;
    if (workspace != nullptr) {
        if (cudaMemcpyAsync(&ws_err, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
            return MLA_ERR_CUDA;
        if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
    }
    int prefill_err = 0;
    if (gemm_error_fetch(&gemm_err, st) != cudaSuccess) return MLA_ERR_CUDA;
    if (rope_error_fetch(&rope_err, st) != cudaSuccess) return MLA_ERR_CUDA;
    if (prefill_error_fetch(&prefill_err, st) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
    return ws_err != 0 ? ws_err : (gemm_err != 0 ? gemm_err : (rope_err != 0 ? rope_err : prefill_err));
}

namespace {
// Prefill workspace: [256-byte header] [C: R x 512] [K: H x R x 192] [V: H x R x 128]
// bf16, R = B * max_blocks_per_seq * 64 rows, each region 1024-byte aligned.
struct PrefillLayout {
    size_t c, k, v, total, rows;
};
PrefillLayout prefill_layout(int B, int H, int mbps) {
    auto up = [](size_t x) { return (x + 1023) & ~size_t(1023); };
    PrefillLayout l;
    l.rows = (size_t)B * (size_t)mbps * kPage;
    l.c = 1024;
    l.k = up(l.c + l.rows * kDLatent * 2);
    l.v = up(l.k + (size_t)H * l.rows * kDQ * 2);
    l.total = up(l.v + (size_t)H * l.rows * kDV * 2);
    return l;
}
}  // namespace

size_t mla_prefill_workspace_size(int B, int H, int max_blocks_per_seq) {
    if (B <= 0 || !valid_heads(H) || max_blocks_per_seq <= 0) return 0;
    return prefill_layout(B, H, max_blocks_per_seq).total;
}

int mla_prefill_paged(const mla_bf16_t* q, const mla_bf16_t* kv_cache, int num_blocks, const int32_t* block_table,
                      int max_blocks_per_seq, const int32_t* cache_seqlens, int B, int s_q, int H,
                      const mla_bf16_t* w_uk, const mla_bf16_t* w_uv, float softmax_scale, int causal,
                      mla_bf16_t* out, float* lse, void* workspace, size_t workspace_bytes, mla_stream_t stream) {
    if (!q || !kv_cache || !block_table || !cache_seqlens || !w_uk || !w_uv || !out || !lse || !workspace)
        return MLA_ERR_INVALID_ARG;
    if (B <= 0 || s_q <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || !valid_heads(H)) return MLA_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || (causal != 0 && causal != 1)) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 1023u) != 0)
        return MLA_ERR_INVALID_ARG;
    const PrefillLayout pl = prefill_layout(B, H, max_blocks_per_seq);
    if (workspace_bytes < pl.total || (uint64_t)B * s_q > 0x7FFFFFFFull || pl.rows > 0x7FFFFFFFull)
        return MLA_ERR_INVALID_ARG;
    if (B > 65535) return MLA_ERR_INVALID_ARG;  // attention grid (query blocks, H, B)
    int dev = check_device();
    if (dev != MLA_OK) return dev;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* C = ws + pl.c;
    void* Kb = ws + pl.k;
    void* Vb = ws + pl.v;
    const uint64_t R = pl.rows;

    // 1. the latent rows and rope keys of every sequence, contiguous (zeros past seqlen)
    if (launch_prefill_gather(kv_cache, num_blocks, block_table, max_blocks_per_seq, cache_seqlens, B, H, C, Kb, st) !=
        cudaSuccess)
        return MLA_ERR_CUDA;

    // 2. K_nope[h] = C . W_UK[h]^T and V[h] = C . W_UV[h] as per-head GEMMs with a shared A
    CUtensorMap ta, tb, to;
    const uint64_t a_dims[4] = {64, R, (uint64_t)kDLatent / 64, 1};
    const uint64_t a_strides[3] = {(uint64_t)kDLatent * 2, 128, R * kDLatent * 2};
    const uint32_t box128[4] = {64, 128, 2, 1};
    if (!make_tmap(&ta, C, 4, a_dims, a_strides, box128)) return MLA_ERR_CUDA;
    GemmArgs g;
    g.R = (int)R;
    g.H = H;
    g.K = kDLatent;
    g.N = 128;
    g.n_cta = 128;
    g.rope_src = nullptr;
    g.a_shared = 1;
    {   // W_UK[h] is [128 (n) x 512 (k)]: a K-major B operand
        const uint64_t b_dims[4] = {64, (uint64_t)kDNope, (uint64_t)kDLatent / 64, (uint64_t)H};
        const uint64_t b_strides[3] = {(uint64_t)kDLatent * 2, 128, (uint64_t)kDNope * kDLatent * 2};
        const uint64_t o_dims[4] = {64, R, (uint64_t)kDQ / 64, (uint64_t)H};
        const uint64_t o_strides[3] = {(uint64_t)kDQ * 2, 128, R * kDQ * 2};
        if (!make_tmap(&tb, w_uk, 4, b_dims, b_strides, box128, CU_TENSOR_MAP_L2_PROMOTION_L2_256B)) return MLA_ERR_CUDA;
        if (!make_tmap(&to, Kb, 4, o_dims, o_strides, box128)) return MLA_ERR_CUDA;
        g.out = Kb;
        g.out_row_elems = kDQ;
        g.b_kmajor = 1;
        if (launch_head_gemm(&ta, &tb, &to, g, g_wait_ns.load(), st) != cudaSuccess) return MLA_ERR_CUDA;
    }
    {   // W_UV[h] is [512 (k) x 128 (n)]: an N-major B operand
        const uint64_t b_dims[4] = {64, (uint64_t)kDLatent, (uint64_t)kDV / 64, (uint64_t)H};
        const uint64_t b_strides[3] = {(uint64_t)kDV * 2, 128, (uint64_t)kDLatent * kDV * 2};
        const uint64_t o_dims[4] = {64, R, (uint64_t)kDV / 64, (uint64_t)H};
        const uint64_t o_strides[3] = {(uint64_t)kDV * 2, 128, R * kDV * 2};
        if (!make_tmap(&tb, w_uv, 4, b_dims, b_strides, box128, CU_TENSOR_MAP_L2_PROMOTION_L2_256B)) return MLA_ERR_CUDA;
        if (!make_tmap(&to, Vb, 4, o_dims, o_strides, box128)) return MLA_ERR_CUDA;
        g.out = Vb;
        g.out_row_elems = kDV;
        g.b_kmajor = 0;
        if (launch_head_gemm(&ta, &tb, &to, g, g_wait_ns.load(), st) != cudaSuccess) return MLA_ERR_CUDA;
    }

    // 3. causal attention per (sequence, head, 128-query tile)
    CUtensorMap tq, tk, tv;
    const uint64_t q_dims[4] = {64, (uint64_t)H, (uint64_t)B * s_q, (uint64_t)kDQ / 64};
    const uint64_t q_strides[3] = {(uint64_t)kDQ * 2, (uint64_t)H * kDQ * 2, 128};
    const uint32_t q_box[4] = {64, 1, 128, 3};
    if (!make_tmap(&tq, q, 4, q_dims, q_strides, q_box)) return MLA_ERR_CUDA;
    const uint64_t k_dims[4] = {64, R, (uint64_t)kDQ / 64, (uint64_t)H};
    const uint64_t k_strides[3] = {(uint64_t)kDQ * 2, 128, R * kDQ * 2};
    const uint32_t k_box[4] = {64, 64, 3, 1};
    if (!make_tmap(&tk, Kb, 4, k_dims, k_strides, k_box)) return MLA_ERR_CUDA;
    const uint64_t v_dims[4] = {64, R, (uint64_t)kDV / 64, (uint64_t)H};
    const uint64_t v_strides[3] = {(uint64_t)kDV * 2, 128, R * kDV * 2};
    const uint32_t v_box[4] = {64, 64, 2, 1};
    if (!make_tmap(&tv, Vb, 4, v_dims, v_strides, v_box)) return MLA_ERR_CUDA;
    return cuda_status(launch_prefill_attn(&tq, &tk, &tv, cache_seqlens, B, s_q, H, max_blocks_per_seq * kPage,
                                           softmax_scale, causal, out, lse, g_wait_ns.load(), st));
}

int mla_rope_append(mla_bf16_t* q, const mla_bf16_t* kv_new, const int32_t* cache_seqlens, const int32_t* block_table,
                    int max_blocks_per_seq, mla_bf16_t* kv_cache, int num_blocks, int B, int s_q, int H,
                    float rope_base, mla_stream_t stream) {
    if (!q || !kv_new || !cache_seqlens || !block_table || !kv_cache || B <= 0 || num_blocks <= 0 ||
        max_blocks_per_seq <= 0 || !valid_sq(s_q) || !valid_heads(H) || !(rope_base > 1.f))
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv_new) || !aligned16(kv_cache)) return MLA_ERR_INVALID_ARG;
    if ((int64_t)B * s_q > 0x7FFFFFFF) return MLA_ERR_INVALID_ARG;
    int dev = check_device();
    if (dev != MLA_OK) return dev;
    return cuda_status(launch_rope_append(q, kv_new, cache_seqlens, block_table, max_blocks_per_seq, kv_cache,
                                          nullptr, nullptr, num_blocks, B, s_q, H, (double)rope_base,
                                          static_cast<cudaStream_t>(stream)));
}

int mla_rope_append_q8(mla_bf16_t* q, const mla_bf16_t* kv_new, const int32_t* cache_seqlens,
                       const int32_t* block_table, int max_blocks_per_seq, uint8_t* kv8, float* kv_scale,
                       int num_blocks, int B, int s_q, int H, float rope_base, mla_stream_t stream) {
    if (!q || !kv_new || !cache_seqlens || !block_table || !kv8 || !kv_scale || B <= 0 || num_blocks <= 0 ||
        max_blocks_per_seq <= 0 || !valid_sq(s_q) || !valid_heads(H) || !(rope_base > 1.f))
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv_new) || !aligned16(kv8)) return MLA_ERR_INVALID_ARG;
    if ((int64_t)B * s_q > 0x7FFFFFFF) return MLA_ERR_INVALID_ARG;
    int dev = check_device();
    if (dev != MLA_OK) return dev;
    return cuda_status(launch_rope_append(q, kv_new, cache_seqlens, block_table, max_blocks_per_seq, nullptr, kv8,
                                          kv_scale, num_blocks, B, s_q, H, (double)rope_base,
                                          static_cast<cudaStream_t>(stream)));
}

int mla_debug_gather(const mla_bf16_t* kv_cache, int num_blocks, const int32_t* block_table, int max_blocks_per_seq,
                     const int32_t* cache_seqlens, int B, int max_tokens, mla_bf16_t* out, mla_stream_t stream) {
    if (!kv_cache || !block_table || !cache_seqlens || !out || num_blocks <= 0 || max_blocks_per_seq <= 0 || B <= 0 ||
        max_tokens <= 0 || !aligned16(kv_cache) || !aligned16(out))
        return MLA_ERR_INVALID_ARG;
    int dev = check_device();
    if (dev != MLA_OK) return dev;
    CUtensorMap tm_kv;
    if (!make_kv_page_map(&tm_kv, kv_cache, num_blocks, kDQK / 64)) return MLA_ERR_CUDA;
    return cuda_status(launch_debug_gather(&tm_kv, block_table, max_blocks_per_seq, cache_seqlens, B, max_tokens,
                                           num_blocks, out, static_cast<cudaStream_t>(stream)));
}

int mla_debug_mma(const mla_bf16_t* a, const mla_bf16_t* b, int K, int N, int b_kmajor, int a_tmem, float* d,
                  mla_stream_t stream) {
    if (!a || !b || !d || K <= 0 || K % 64 != 0 || K > 576 || !(N == 64 || N == 128 || N == 256) ||
        (b_kmajor != 0 && b_kmajor != 1) || (a_tmem < 0 || a_tmem > 2) || !aligned16(a) || !aligned16(b))
        return MLA_ERR_INVALID_ARG;
    int dev = check_device();
    if (dev != MLA_OK) return dev;
    CUtensorMap tm_a, tm_b;
    const uint64_t a_dims[2] = {(uint64_t)K, 128};
    const uint64_t a_strides[1] = {(uint64_t)K * 2};
    const uint32_t a_box[2] = {64, 128};
    if (!make_tmap(&tm_a, a, 2, a_dims, a_strides, a_box)) return MLA_ERR_CUDA;
    if (b_kmajor) {
        const uint64_t b_dims[2] = {(uint64_t)K, (uint64_t)N};
        const uint64_t b_strides[1] = {(uint64_t)K * 2};
        const uint32_t b_box[2] = {64, (uint32_t)N};
        if (!make_tmap(&tm_b, b, 2, b_dims, b_strides, b_box)) return MLA_ERR_CUDA;
    } else {
        const uint64_t b_dims[2] = {(uint64_t)N, (uint64_t)K};
        const uint64_t b_strides[1] = {(uint64_t)N * 2};
        const uint32_t b_box[2] = {64, 64};
        if (!make_tmap(&tm_b, b, 2, b_dims, b_strides, b_box)) return MLA_ERR_CUDA;
    }
    return cuda_status(launch_debug_mma(&tm_a, &tm_b, K, N, b_kmajor, a_tmem, a, d, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
