// C ABI of the library (include/gqa_attn.h): argument checks, launch
// planning, TMA tensor-map encoding and kernel launches.  No device memory is
// allocated and no device data is read back on the attention paths.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "gqa_attn.h"
#include "internal.h"

namespace {

using gqa::DecodeArgs;
using gqa::DecodePlan;
using gqa::PrefillArgs;

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

// [B, S, H, D] bf16, D contiguous, as a 4-D tensor map {D, S, H, B} with a
// {64, box_rows, 1, 1} box and 128-byte swizzle.  Rows past S read as zero.
// The tensor maps only move 16-bit elements; the type names the data.
CUtensorMapDataType elem_type(bool f16) {
    return f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

bool make_bshd_map(CUtensorMap* map, const void* ptr, int B, int S, int H, int D, bool f16, int box_rows = 128) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)H * D * 2, (cuuint64_t)D * 2, (cuuint64_t)S * H * D * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(map, elem_type(f16), 4, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Paged cache [pages * page_size, Hkv, D] bf16 as a 3-D map {D, Hkv, rows}
// with a {64, 1, box_tokens} box and 128-byte swizzle.
bool make_cache_map(CUtensorMap* map, const void* ptr, long rows, int Hkv, int D, int box_tokens, bool f16) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_tokens};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, elem_type(f16), 3, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Paged cache as a 5-D map {64, 8, D / 64, pages * page_size / 8, Hkv}: the
// token axis is split into 8-row groups, and the 64-column slices (128-byte
// stride) sit between the row-in-group and group axes.  A {64, 8, D / 64,
// box_tokens / 8, 1} box brings one page block of one head whole and lands in
// shared memory as [group][slice][8 rows][128 bytes] (128-byte swizzle), so
// consecutive boxes of a tile keep one uniform 8-row-group stride (D / 64 KB)
// for every slice, which lets one MMA descriptor span the tile's 64 keys.
bool make_cache_page_map(CUtensorMap* map, const void* ptr, long rows, int Hkv, int D, int box_tokens,
                         bool f16, int box_slices = 0) {
    auto fn = encode_fn();
    if (!fn || rows % 8 != 0 || box_tokens % 8 != 0) return false;
    const cuuint64_t row_bytes = (cuuint64_t)Hkv * D * 2;
    const cuuint64_t dims[5] = {64, 8, (cuuint64_t)(D / 64), (cuuint64_t)(rows / 8), (cuuint64_t)Hkv};
    const cuuint64_t strides[4] = {row_bytes, 128, 8 * row_bytes, (cuuint64_t)D * 2};
    const cuuint32_t box[5] = {64, 8, (cuuint32_t)(box_slices > 0 ? box_slices : D / 64), (cuuint32_t)(box_tokens / 8),
                               1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(map, elem_type(f16), 5, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Packed [total, H, D] rows (THD) as a 3-D map {D, H, total} with a
// {64, box_h, box_t} box and 128-byte swizzle: box_h heads of box_t
// consecutive tokens land as box_t * box_h rows of 128 bytes.
bool make_thd_map(CUtensorMap* map, const void* ptr, long total, int H, int D, int box_h, int box_t, bool f16) {
    auto fn = encode_fn();
    if (!fn || total <= 0) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)total};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_h, (cuuint32_t)box_t};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, elem_type(f16), 3, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int gcd_int(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static int cache[64] = {0};
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool head_dim_ok(int D) { return D == 64 || D == 128 || D == 256; }

constexpr long kMaxSeq = 1L << 30;

}  // namespace

extern "C" {

// Checks the optional terms and turns them into their kernel form.
static gqa_status make_extras(const gqa_options* op, float scale, gqa::Extras* x) {
    x->wl = x->wr = -1;
    x->cap_in = x->cap_out = 0.f;
    x->sinks = nullptr;
    if (!op) return GQA_OK;
    if (op->window_left < -1 || op->window_right < -1) return GQA_ERR_INVALID_ARG;
    if (!std::isfinite(op->softcap) || op->softcap < 0.f) return GQA_ERR_INVALID_ARG;
    if (op->sinks && !aligned4(op->sinks)) return GQA_ERR_MISALIGNED;
    if (op->dtype != GQA_BF16 && op->dtype != GQA_FP16) return GQA_ERR_INVALID_ARG;
    x->wl = op->window_left;
    x->wr = op->window_right;
    if (op->softcap > 0.f) {
        const double log2e = 1.4426950408889634074;
        x->cap_in = (float)(2.0 * log2e * (double)scale / (double)op->softcap);
        x->cap_out = (float)((double)op->softcap * log2e);
    }
    x->sinks = op->sinks;
    return GQA_OK;
}

gqa_status attn_fwd_dense(const void* q, const void* k, const void* v, const uint8_t* key_padding_mask,
                          void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                          float scale, gqa_stream_t stream) {
    return attn_fwd_dense_ex(q, k, v, key_padding_mask, o, lse, B, Hq, Hkv, Sq, Skv, D, causal, scale, nullptr,
                             stream);
}

gqa_status attn_fwd_dense_ex(const void* q, const void* k, const void* v, const uint8_t* key_padding_mask,
                             void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                             float scale, const gqa_options* opts, gqa_stream_t stream) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Sq < 0 || Skv < 0) return GQA_ERR_INVALID_ARG;
    if (Sq >= kMaxSeq || Skv >= kMaxSeq) return GQA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
    if (!head_dim_ok(D)) return GQA_ERR_UNSUPPORTED;
    if (Sq == 0) return GQA_OK;
    if (!q || !o || (Skv > 0 && (!k || !v))) return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o) || (Skv > 0 && (!aligned16(k) || !aligned16(v)))) return GQA_ERR_MISALIGNED;
    if (lse && !aligned4(lse)) return GQA_ERR_MISALIGNED;
    gqa::Extras ex;
    const gqa_status es = make_extras(opts, scale, &ex);
    if (es != GQA_OK) return es;
    const long n_qtiles = ((long)Sq + 127) / 128;
    if (n_qtiles * B * Hq >= (1L << 31)) return GQA_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    if (Skv == 0)
        return gqa::launch_empty_rows(o, lse, (long)B * Sq * Hq, D, st) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;

    CUtensorMap tq, tk, tv, to;
    const bool f16 = opts && opts->dtype == GQA_FP16;
    if (!make_bshd_map(&tq, q, B, Sq, Hq, D, f16) || !make_bshd_map(&tk, k, B, Skv, Hkv, D, f16) ||
        !make_bshd_map(&tv, v, B, Skv, Hkv, D, f16, D == 256 ? 64 : 128) || !make_bshd_map(&to, o, B, Sq, Hq, D, f16))
        return GQA_ERR_CUDA;
    PrefillArgs a{};
    a.mask = key_padding_mask;
    a.o = o;
    a.lse = lse;
    a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.Sq = Sq; a.Skv = Skv; a.D = D;
    a.causal = causal ? 1 : 0;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    a.num_sms = sm_count();
    a.f16 = f16 ? 1 : 0;
    a.x = ex;
    const cudaError_t e = D == 256 ? gqa::launch_prefill_d256(tq, tk, tv, to, a, st)
                                   : gqa::launch_prefill(tq, tk, tv, to, a, st);
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

size_t attn_decode_paged_workspace_size(int B, int Sq, int Hq, int Hkv, int D, int page_size, int max_pages) {
    if (!head_dim_ok(D)) return 0;
    DecodePlan p;
    if (!gqa::plan_decode(B, Sq, Hq, Hkv, D, page_size, max_pages, sm_count(), &p)) return 0;
    return p.workspace_bytes;
}

gqa_status attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* real_seqlen_kv,
                             const int32_t* block_table, int page_size, void* o, float* lse, int B, int Sq, int Hq,
                             int Hkv, int D, int num_pages, int max_pages, int causal, float scale,
                             void* workspace, size_t workspace_bytes, gqa_stream_t stream) {
    return attn_decode_paged_ex(q, k_cache, v_cache, real_seqlen_kv, block_table, page_size, o, lse, B, Sq, Hq, Hkv,
                                D, num_pages, max_pages, causal, scale, nullptr, workspace, workspace_bytes, stream);
}

gqa_status attn_decode_paged_ex(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* real_seqlen_kv, const int32_t* block_table, int page_size, void* o,
                                float* lse, int B, int Sq, int Hq, int Hkv, int D, int num_pages, int max_pages,
                                int causal, float scale, const gqa_options* opts, void* workspace,
                                size_t workspace_bytes, gqa_stream_t stream) {
    if (B <= 0 || Sq < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages < 0 || max_pages <= 0)
        return GQA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
    if ((long)max_pages * page_size >= kMaxSeq) return GQA_ERR_INVALID_ARG;
    if ((long)num_pages * page_size >= (1L << 31)) return GQA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
    if (!head_dim_ok(D)) return GQA_ERR_UNSUPPORTED;
    if (Sq == 0) return GQA_OK;
    if (!q || !k_cache || !v_cache || !real_seqlen_kv || !block_table || !o) return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o)) return GQA_ERR_MISALIGNED;
    if (!aligned4(real_seqlen_kv) || !aligned4(block_table) || (lse && !aligned4(lse))) return GQA_ERR_MISALIGNED;
    gqa::Extras ex;
    const gqa_status es = make_extras(opts, scale, &ex);
    if (es != GQA_OK) return es;
    DecodePlan p;
    if (!gqa::plan_decode(B, Sq, Hq, Hkv, D, page_size, max_pages, sm_count(), &p)) return GQA_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < p.workspace_bytes) return GQA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GQA_ERR_MISALIGNED;

    DecodeArgs a{};
    a.q = q; a.k_cache = k_cache; a.v_cache = v_cache;
    a.seqlens = real_seqlen_kv; a.table = block_table;
    a.o = o; a.lse = lse;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + (p.part_o_bytes + 255) / 256 * 256);
    a.B = B; a.Sq = Sq; a.Hq = Hq; a.Hkv = Hkv; a.D = D;
    a.page_size = page_size; a.max_pages = max_pages; a.num_pages = num_pages; a.causal = causal ? 1 : 0;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    a.chunk = p.chunk;
    a.max_splits = p.max_splits;
    a.seg_table = nullptr;
    a.n_part = 0;
    a.tc_grid = 0;
    a.f16 = opts && opts->dtype == GQA_FP16 ? 1 : 0;
    a.x = ex;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // KV groups of 32..128 query rows run on the balanced tensor-core decode
    // kernel, whose workspace holds per-piece partials and the segment table.
    if (num_pages > 0 && p.tc) {
        const int tbox = gqa::decode_tc_box_tokens(page_size);
        CUtensorMap tk, tv;
        if (make_cache_page_map(&tk, k_cache, (long)num_pages * page_size, Hkv, D, tbox, a.f16) &&
            make_cache_page_map(&tv, v_cache, (long)num_pages * page_size, Hkv, D, tbox, a.f16)) {
            char* ws = static_cast<char*>(workspace);
            const size_t o_bytes = (p.tc_part_o_bytes + 255) / 256 * 256;
            const size_t l_bytes = (p.tc_part_lse_bytes + 255) / 256 * 256;
            a.part_o = reinterpret_cast<float*>(ws);
            a.part_lse = reinterpret_cast<float*>(ws + o_bytes);
            a.seg_table = reinterpret_cast<int*>(ws + o_bytes + l_bytes);
            a.n_part = p.n_part;
            a.tc_grid = p.tc_grid;
            return gqa::launch_decode_tc(tk, tv, a, tbox, st) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
        }
    }
    // Pages that cut into 8-row multiples of the key tile are loaded by TMA;
    // other page sizes are gathered row by row.
    const int box = gqa::decode_box_tokens(D, page_size);
    CUtensorMap tk, tv;
    const bool use_tma = box > 0 && num_pages > 0 &&
                         make_cache_map(&tk, k_cache, (long)num_pages * page_size, Hkv, D, box, a.f16) &&
                         make_cache_map(&tv, v_cache, (long)num_pages * page_size, Hkv, D, box, a.f16);
    return gqa::launch_decode(a, use_tma ? &tk : nullptr, use_tma ? &tv : nullptr, box, st) == cudaSuccess
               ? GQA_OK
               : GQA_ERR_CUDA;
}

// Paged cache of e4m3fn bytes [pages * page_size, Hkv, D] as a 3-D byte map
// {D, Hkv, rows} with a {128, 1, box_tokens} box (128-byte rows, 128-byte swizzle).
static bool make_cache_map_fp8(CUtensorMap* map, const void* ptr, long rows, int Hkv, int D, int box_tokens) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)Hkv * D};
    const cuuint32_t box[3] = {128, 1, (cuuint32_t)box_tokens};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Paged cache of e4m3fn bytes as a 5-D map {128, 8, D / 128, pages * page_size / 8,
// Hkv}: a {128, 8, D / 128, box_tokens / 8, 1} box brings one page block of
// one head and lands as [8-row group][128-column half][8 rows][128 bytes].
static bool make_cache_page_map_fp8(CUtensorMap* map, const void* ptr, long rows, int Hkv, int D, int box_tokens) {
    auto fn = encode_fn();
    if (!fn || rows % 8 != 0 || box_tokens % 8 != 0) return false;
    const cuuint64_t row_bytes = (cuuint64_t)Hkv * D;
    const cuuint64_t dims[5] = {128, 8, (cuuint64_t)(D / 128), (cuuint64_t)(rows / 8), (cuuint64_t)Hkv};
    const cuuint64_t strides[4] = {row_bytes, 128, 8 * row_bytes, (cuuint64_t)D};
    const cuuint32_t box[5] = {128, 8, (cuuint32_t)(D / 128), (cuuint32_t)(box_tokens / 8), 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

gqa_status attn_decode_paged_fp8kv(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                                   const float* v_scale, const int32_t* real_seqlen_kv, const int32_t* block_table,
                                   int page_size, void* o, float* lse, int B, int Sq, int Hq, int Hkv, int D,
                                   int num_pages, int max_pages, int causal, float scale, const gqa_options* opts,
                                   void* workspace, size_t workspace_bytes, gqa_stream_t stream) {
    if (B <= 0 || Sq < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages < 0 || max_pages <= 0)
        return GQA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
    if ((long)max_pages * page_size >= kMaxSeq) return GQA_ERR_INVALID_ARG;
    if ((long)num_pages * page_size >= (1L << 31)) return GQA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
    if (D != 128 && D != 256) return GQA_ERR_UNSUPPORTED;
    // pages the byte boxes tile move by TMA; others are gathered row by row
    const int box = gqa::decode_box_tokens(D, page_size);
    if (Sq == 0) return GQA_OK;
    if (!q || !k_cache || !v_cache || !real_seqlen_kv || !block_table || !o) return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o)) return GQA_ERR_MISALIGNED;
    if (!aligned4(real_seqlen_kv) || !aligned4(block_table) || (lse && !aligned4(lse)) ||
        (k_scale && !aligned4(k_scale)) || (v_scale && !aligned4(v_scale)))
        return GQA_ERR_MISALIGNED;
    gqa::Extras ex;
    const gqa_status es = make_extras(opts, scale, &ex);
    if (es != GQA_OK) return es;
    DecodePlan p;
    if (!gqa::plan_decode(B, Sq, Hq, Hkv, D, page_size, max_pages, sm_count(), &p)) return GQA_ERR_UNSUPPORTED;
    // the partials of whichever path the sizes select (attn_decode_paged_workspace_size)
    if (!workspace || workspace_bytes < p.workspace_bytes) return GQA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GQA_ERR_MISALIGNED;

    DecodeArgs a{};
    a.q = q; a.k_cache = k_cache; a.v_cache = v_cache;
    a.seqlens = real_seqlen_kv; a.table = block_table;
    a.o = o; a.lse = lse;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + (p.part_o_bytes + 255) / 256 * 256);
    a.B = B; a.Sq = Sq; a.Hq = Hq; a.Hkv = Hkv; a.D = D;
    a.page_size = page_size; a.max_pages = max_pages; a.num_pages = num_pages; a.causal = causal ? 1 : 0;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    a.chunk = p.chunk;
    a.max_splits = p.max_splits;
    a.seg_table = nullptr;
    a.f16 = opts && opts->dtype == GQA_FP16 ? 1 : 0;
    a.x = ex;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    // with an empty pool no page is ever loaded; the maps then describe one page
    const long rows = (long)(num_pages > 0 ? num_pages : 1) * page_size;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap tk, tv;
    // KV groups of 32..128 query rows: the balanced tensor-core decode, its
    // byte tiles widened in shared memory
    if (p.tc) {
        const int tbox = gqa::decode_tc_box_tokens(page_size);
        if (!make_cache_page_map_fp8(&tk, k_cache, rows, Hkv, D, tbox) ||
            !make_cache_page_map_fp8(&tv, v_cache, rows, Hkv, D, tbox))
            return GQA_ERR_CUDA;
        char* ws = static_cast<char*>(workspace);
        const size_t o_bytes = (p.tc_part_o_bytes + 255) / 256 * 256;
        const size_t l_bytes = (p.tc_part_lse_bytes + 255) / 256 * 256;
        a.part_o = reinterpret_cast<float*>(ws);
        a.part_lse = reinterpret_cast<float*>(ws + o_bytes);
        a.seg_table = reinterpret_cast<int*>(ws + o_bytes + l_bytes);
        a.n_part = p.n_part;
        a.tc_grid = p.tc_grid;
        return gqa::launch_decode_tc_fp8(tk, tv, a, tbox, st) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
    }
    if (box > 0) {
        if (!make_cache_map_fp8(&tk, k_cache, rows, Hkv, D, box) ||
            !make_cache_map_fp8(&tv, v_cache, rows, Hkv, D, box))
            return GQA_ERR_CUDA;
    } else {
        tk = CUtensorMap{};                         // unused by the gather producer
        tv = CUtensorMap{};
    }
    return gqa::launch_decode_fp8(a, tk, tv, box, st) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

// ---------------------------------------------------------------- packed calls
// Workspace of a packed call: a 16-byte header holding the entry count, then
// two arrays of up to max_entries row-block entries of 32 bytes (as listed,
// and ordered by cost).
static int varlen_max_entries(int B, int total_q, int qpb) { return total_q / qpb + B + 1; }

static size_t varlen_ws_bytes(int B, int total_q, int Hq, int Hkv) {
    if (B <= 0 || total_q < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Hq / Hkv > 128) return 0;
    const int qpb = 128 / (Hq / Hkv);
    return 16 + 2 * (size_t)varlen_max_entries(B, total_q, qpb) * 32;
}

size_t attn_varlen_workspace_size(int B, int total_q, int Hq, int Hkv) {
    return varlen_ws_bytes(B, total_q, Hq, Hkv);
}

// Split-decode plan for the single-query requests of a paged call (B requests
// of one query each); false when the sizes leave them on the one-tile kernel
// (KV groups of 32 rows or more, whose decode runs on the tensor-core kernel).
static bool paged_decode_plan(int B, int Hq, int Hkv, int D, int page_size, int max_pages, DecodePlan* p) {
    if (!head_dim_ok(D) || page_size <= 0 || max_pages <= 0) return false;
    if (!gqa::plan_decode(B, 1, Hq, Hkv, D, page_size, max_pages, sm_count(), p)) return false;
    return !p->tc;
}

size_t attn_paged_workspace_size(int B, int total_q, int Hq, int Hkv, int D, int page_size, int max_pages) {
    const size_t v = varlen_ws_bytes(B, total_q, Hq, Hkv);
    DecodePlan p;
    if (v == 0 || !paged_decode_plan(B, Hq, Hkv, D, page_size, max_pages, &p)) return v;
    return (v + 255) / 256 * 256 + p.workspace_bytes;
}

// Shared checks and set-up of the two packed entry points.
static gqa_status varlen_common(const void* q, void* o, float* lse, const int32_t* cu_q, int B, int total_q,
                                int Hq, int Hkv, int D, int causal, float scale, const gqa_options* opts,
                                void* workspace, size_t workspace_bytes, PrefillArgs* a, CUtensorMap* tq,
                                CUtensorMap* to) {
    if (B <= 0 || total_q < 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return GQA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || total_q >= kMaxSeq) return GQA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
    if (!head_dim_ok(D) || Hq / Hkv > 128) return GQA_ERR_UNSUPPORTED;
    if (!q || !o || !cu_q) return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o)) return GQA_ERR_MISALIGNED;
    if (!aligned4(cu_q) || (lse && !aligned4(lse))) return GQA_ERR_MISALIGNED;
    gqa::Extras ex;
    const gqa_status es = make_extras(opts, scale, &ex);
    if (es != GQA_OK) return es;
    const size_t need = varlen_ws_bytes(B, total_q, Hq, Hkv);
    if (!workspace || workspace_bytes < need) return GQA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return GQA_ERR_MISALIGNED;
    const bool f16 = opts && opts->dtype == GQA_FP16;
    const int g = Hq / Hkv, qpb = 128 / g;
    if (total_q > 0 && (!make_thd_map(tq, q, total_q, Hq, D, g, qpb, f16) ||
                        !make_thd_map(to, o, total_q, Hq, D, g, qpb, f16)))
        return GQA_ERR_CUDA;
    a->mask = nullptr;
    a->o = o;
    a->lse = lse;
    a->B = B; a->Hq = Hq; a->Hkv = Hkv; a->Sq = 0; a->Skv = 0; a->D = D;
    a->causal = causal ? 1 : 0;
    a->scale_log2 = (float)((double)scale * 1.4426950408889634074);
    a->num_sms = sm_count();
    a->f16 = f16 ? 1 : 0;
    a->x = ex;
    a->n_entries = static_cast<const int32_t*>(workspace);
    a->work = static_cast<int32_t*>(workspace) + 1;
    a->entries = reinterpret_cast<const int32_t*>(static_cast<char*>(workspace) + 16);
    a->g = g;
    a->qpb = qpb;
    a->table = nullptr;
    a->page_size = a->max_pages = a->bt_k = a->bt_v = 0;
    return GQA_OK;
}

gqa_status attn_fwd_varlen(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                           const int32_t* cu_seqlens_kv, void* o, float* lse, int B, int total_q, int total_kv,
                           int Hq, int Hkv, int D, int causal, float scale, const gqa_options* opts,
                           void* workspace, size_t workspace_bytes, gqa_stream_t stream) {
    PrefillArgs a{};
    CUtensorMap tq, tk, tv, to;
    if (total_kv < 0 || total_kv >= kMaxSeq) return GQA_ERR_INVALID_ARG;
    gqa_status st = varlen_common(q, o, lse, cu_seqlens_q, B, total_q, Hq, Hkv, D, causal, scale, opts, workspace,
                                  workspace_bytes, &a, &tq, &to);
    if (st != GQA_OK) return st;
    if (!cu_seqlens_kv || (total_kv > 0 && (!k || !v))) return GQA_ERR_INVALID_ARG;
    if (!aligned4(cu_seqlens_kv) || (total_kv > 0 && (!aligned16(k) || !aligned16(v)))) return GQA_ERR_MISALIGNED;
    if (total_q == 0) return GQA_OK;
    // with no key at all the maps are never read; they then describe q
    const void* kb = total_kv > 0 ? k : q;
    const void* vb = total_kv > 0 ? v : q;
    const long kv_rows = total_kv > 0 ? total_kv : 1;
    if (!make_thd_map(&tk, kb, kv_rows, Hkv, D, 1, 128, a.f16) ||
        !make_thd_map(&tv, vb, kv_rows, Hkv, D, 1, D == 256 ? 64 : 128, a.f16))
        return GQA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int max_e = varlen_max_entries(B, total_q, a.qpb);
    int32_t* ws = static_cast<int32_t*>(workspace);
    // D = 64 and 128 run on the two-Q-tile kernel (items of two consecutive
    // row blocks sharing each K/V tile); D = 256 on the one-tile kernel
    const bool two = D <= 128;
    if (gqa::launch_varlen_plan(cu_seqlens_q, cu_seqlens_kv, false, B, a.qpb, a.g, a.causal, total_q, total_kv,
                                ws + 4 + (size_t)max_e * 8, ws + 4, ws, max_e, s, false, two) != cudaSuccess)
        return GQA_ERR_CUDA;
    const cudaError_t e = two ? gqa::launch_prefill_packed(tq, tk, tv, to, a, (long)max_e * Hkv, s)
                              : gqa::launch_varlen_packed(tq, tk, tv, to, a, (long)max_e * Hkv, s);
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

// A second stream per device and host thread, of the highest priority, with a
// fork and a join event.  The prefill chunks of a mixed paged call run on it
// beside the decode steps on the caller's stream: the chunks are tensor-bound
// and the decode steps memory-bound, so side by side on separate SMs they take
// less than one after the other.  Created on first use outside a stream
// capture and kept (a capture uses one created by an earlier call); nullptr if
// there is none (the call then runs everything on the caller's stream).
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

static SideStream* side_stream(cudaStream_t caller) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
    thread_local std::vector<SideStream> per_dev;
    if ((int)per_dev.size() <= dev) per_dev.resize(dev + 1);
    SideStream& ss = per_dev[dev];
    if (ss.s == nullptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(caller, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
        int least = 0, greatest = 0;
        cudaStream_t st = nullptr;
        cudaEvent_t f = nullptr, j = nullptr;
        if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
            cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking, greatest) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        if (cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
            if (f) cudaEventDestroy(f);
            cudaStreamDestroy(st);
            cudaGetLastError();
            return nullptr;
        }
        ss.s = st;
        ss.fork = f;
        ss.join = j;
    }
    return &ss;
}

gqa_status attn_fwd_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
                          const int32_t* cache_seqlens, const int32_t* block_table, int page_size, void* o,
                          float* lse, int B, int total_q, int Hq, int Hkv, int D, int num_pages, int max_pages,
                          int causal, float scale, const gqa_options* opts, void* workspace,
                          size_t workspace_bytes, gqa_stream_t stream) {
    PrefillArgs a{};
    CUtensorMap tq, tk, tv, to;
    if (page_size <= 0 || num_pages <= 0 || max_pages <= 0) return GQA_ERR_INVALID_ARG;
    if ((long)max_pages * page_size >= kMaxSeq) return GQA_ERR_INVALID_ARG;
    if ((long)num_pages * page_size >= (1L << 31)) return GQA_ERR_UNSUPPORTED;
    gqa_status st = varlen_common(q, o, lse, cu_seqlens_q, B, total_q, Hq, Hkv, D, causal, scale, opts, workspace,
                                  workspace_bytes, &a, &tq, &to);
    if (st != GQA_OK) return st;
    if (!k_cache || !v_cache || !cache_seqlens || !block_table) return GQA_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return GQA_ERR_MISALIGNED;
    if (!aligned4(cache_seqlens) || !aligned4(block_table)) return GQA_ERR_MISALIGNED;
    if (total_q == 0) return GQA_OK;
    a.table = block_table;
    a.page_size = page_size;
    a.max_pages = max_pages;
    const int vkeys = D == 256 ? 64 : 128;
    const long rows = (long)num_pages * page_size;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_pages = num_pages;
    if (page_size % 8 == 0) {
        // pages move as 8-row TMA blocks
        a.bt_k = gcd_int(page_size, 128);
        a.bt_v = gcd_int(page_size, vkeys);
        if (!make_cache_page_map(&tk, k_cache, rows, Hkv, D, a.bt_k, a.f16, D == 256 ? 2 : D / 64) ||
            !make_cache_page_map(&tv, v_cache, rows, Hkv, D, a.bt_v, a.f16))
            return GQA_ERR_CUDA;
    } else {
        // other page sizes: rows gathered with cp.async (the maps go unused)
        a.bt_k = a.bt_v = 0;
        tk = tq;
        tv = tq;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int max_e = varlen_max_entries(B, total_q, a.qpb);
    int32_t* ws = static_cast<int32_t*>(workspace);
    // Requests with exactly one query (decode steps) run on the split decode
    // kernel when the workspace also holds its partials: there all g heads of a
    // KV group share one MMA fragment and the keys stream at memory speed,
    // instead of g rows taking a 128-row tensor-core tile.  The prefill chunks
    // stay on the one-tile kernel; the two launches write disjoint rows.
    DecodePlan dp;
    char* wsc = static_cast<char*>(workspace);
    const size_t d_off = (varlen_ws_bytes(B, total_q, Hq, Hkv) + 255) / 256 * 256;
    const bool route = paged_decode_plan(B, Hq, Hkv, D, page_size, max_pages, &dp) &&
                       workspace_bytes >= d_off + dp.workspace_bytes &&
                       (reinterpret_cast<uintptr_t>(wsc + d_off) & 255u) == 0;
    // With decode steps routed, the chunks run on the side stream beside them,
    // keeping the share of the persistent CTAs the plan kernel computes (ws[2])
    SideStream* side = route ? side_stream(s) : nullptr;
    if (side) a.g_eff = ws + 2;
    if (gqa::launch_varlen_plan(cu_seqlens_q, cache_seqlens, true, B, a.qpb, a.g, a.causal, total_q,
                                (long)max_pages * page_size, ws + 4 + (size_t)max_e * 8, ws + 4, ws, max_e,
                                s, route, false, side ? a.num_sms : 0) != cudaSuccess)
        return GQA_ERR_CUDA;
    if (side) {
        // fork after the plan: the chunks (highest priority, so their CTAs
        // take their SMs first) and the decode steps become ready together
        if (cudaEventRecord(side->fork, s) != cudaSuccess || cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
            return GQA_ERR_CUDA;
        if (gqa::launch_varlen_paged(tq, tk, tv, to, a, (long)max_e * Hkv, side->s) != cudaSuccess ||
            cudaEventRecord(side->join, side->s) != cudaSuccess)
            return GQA_ERR_CUDA;
    }
    if (route) {
        DecodeArgs da{};
        da.q = q; da.k_cache = k_cache; da.v_cache = v_cache;
        da.seqlens = cache_seqlens; da.table = block_table;
        da.o = o; da.lse = lse;
        da.part_o = reinterpret_cast<float*>(wsc + d_off);
        da.part_lse = reinterpret_cast<float*>(wsc + d_off + (dp.part_o_bytes + 255) / 256 * 256);
        da.B = B; da.Sq = 1; da.Hq = Hq; da.Hkv = Hkv; da.D = D;
        da.page_size = page_size; da.max_pages = max_pages; da.num_pages = num_pages; da.causal = a.causal;
        da.scale_log2 = a.scale_log2;
        da.chunk = dp.chunk;
        da.max_splits = dp.max_splits;
        da.f16 = a.f16;
        da.x = a.x;
        da.q_rows = cu_seqlens_q;
        da.q_total = total_q;
        const int box = gqa::decode_box_tokens(D, page_size);
        CUtensorMap dk, dv;
        const bool use_tma = box > 0 && make_cache_map(&dk, k_cache, rows, Hkv, D, box, a.f16) &&
                             make_cache_map(&dv, v_cache, rows, Hkv, D, box, a.f16);
        if (gqa::launch_decode(da, use_tma ? &dk : nullptr, use_tma ? &dv : nullptr, box, s) != cudaSuccess)
            return GQA_ERR_CUDA;
    }
    if (side) return cudaStreamWaitEvent(s, side->join, 0) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;   // join
    return gqa::launch_varlen_paged(tq, tk, tv, to, a, (long)max_e * Hkv, s) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

gqa_status attn_validate_paged(const int32_t* real_seqlen_kv, const int32_t* block_table, int B, int Sq,
                               int page_size, int num_pages, int max_pages, int causal, gqa_stream_t stream) {
    (void)causal;
    if (B <= 0 || Sq < 0 || page_size <= 0 || num_pages < 0 || max_pages <= 0) return GQA_ERR_INVALID_ARG;
    if (!real_seqlen_kv || !block_table) return GQA_ERR_INVALID_ARG;
    std::vector<int32_t> lens(B), table((size_t)B * max_pages);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(lens.data(), real_seqlen_kv, sizeof(int32_t) * B, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(table.data(), block_table, sizeof(int32_t) * table.size(), cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return GQA_ERR_CUDA;
    for (int b = 0; b < B; ++b) {
        const long L = lens[b];
        if (L < 0 || L > (long)max_pages * page_size) return GQA_ERR_INVALID_ARG;
        const long need = (L + page_size - 1) / page_size;
        for (long p = 0; p < need; ++p) {
            const int32_t phys = table[(size_t)b * max_pages + p];
            if (phys < 0 || phys >= num_pages) return GQA_ERR_INVALID_ARG;
        }
    }
    return GQA_OK;
}

const char* gqa_status_string(gqa_status s) {
    switch (s) {
        case GQA_OK: return "ok";
        case GQA_ERR_INVALID_ARG: return "invalid argument";
        case GQA_ERR_UNSUPPORTED: return "unsupported combination";
        case GQA_ERR_MISALIGNED: return "pointer not aligned";
        case GQA_ERR_WORKSPACE: return "workspace missing or too small";
        case GQA_ERR_CUDA: return "CUDA error";
        case GQA_ERR_TIMEOUT: return "a kernel wait timed out";
    }
    return "unknown status";
}

gqa_status gqa_device_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GQA_ERR_CUDA;
    const int e = gqa::prefill_take_device_error();
    const int e2 = gqa::prefill_d256_take_device_error();
    const int v1 = gqa::varlen_packed_take_device_error();
    const int v2 = gqa::varlen_paged_take_device_error();
    const int d = gqa::decode_take_device_error();
    const int t = gqa::decode_tc_take_device_error();
    if (e < 0 || e2 < 0 || v1 < 0 || v2 < 0 || d < 0 || t < 0) return GQA_ERR_CUDA;
    return (e || e2 || v1 || v2 || d || t) ? GQA_ERR_TIMEOUT : GQA_OK;
}

const char* gqa_version(void) { return "gqa_attn 0.1 sm_103a"; }

}  // extern "C"
