// Internal interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace gqa {

// Optional terms of a call in kernel form (TileOPs "Attention Operators",
// GQADenseFwdOp stages 5-6; GQAPagedFwdOp sinks).
struct Extras {
    int wl, wr;             // window sizes; -1 = unlimited
    float cap_in;           // softcap c: 2 * log2(e) * scale / c, multiplying a raw score (0 = off)
    float cap_out;          // c * log2(e)
    const float* sinks;     // [Hq] natural-log logits joining the denominator only, or nullptr
};

struct PrefillArgs {
    const uint8_t* mask;  // [B, Skv] or nullptr
    void* o;              // [B, Sq, Hq, D] bf16
    float* lse;           // [B, Sq, Hq] or nullptr
    int B, Hq, Hkv, Sq, Skv, D;
    int causal;
    float scale_log2;     // scale * log2(e)
    int num_sms;          // persistent grid size
    int f16;              // inputs and output are float16 (else bfloat16)
    Extras x;
    // Packed calls (onetile.cuh): q / o [total_q, Hq, D]; row blocks listed by
    // the plan kernel.  Unused by the BSHD kernels.
    const int32_t* entries;   // [max_entries, 8]: b, q0, qs, sq, ks, L, -, -
    const int32_t* n_entries; // number of entries (device)
    int32_t* work;            // packed: item counter, zeroed by the plan kernel
    // paged calls whose decode steps run beside them on the split decode
    // kernel: CTAs at or past *g_eff exit at once, leaving their SMs to it
    // (written by the plan kernel); nullptr: every CTA works
    const int32_t* g_eff;
    int g;                    // query heads per KV head
    int qpb;                  // queries per row block: floor(128 / g)
    const int32_t* table;     // paged: block_table [B, max_pages]
    int page_size, max_pages;
    int bt_k, bt_v;           // paged: tokens per TMA box of a K / V chunk; 0: rows gathered with cp.async
    // paged, gathered rows (page sizes that are not a multiple of 8): the
    // caches [num_pages, page_size, Hkv, D] themselves
    const void* k_cache;
    const void* v_cache;
    int num_pages;
};

// Launches the tcgen05 prefill kernel.  The tensor maps describe q, k, v as
// 4-D [B, S, H, D] bf16 tensors with a {64, 128, 1, 1} box and 128-byte swizzle.
cudaError_t launch_prefill(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, const CUtensorMap& tm_o, const PrefillArgs& a,
                           cudaStream_t stream);
// The same two-Q-tile kernel over packed THD calls (D = 64 or 128): items are
// pairs of consecutive row blocks of one request, listed by the plan kernel
// with pairs set; tm_q / tm_o as for launch_varlen_packed, tm_k / tm_v
// {D, Hkv, total_kv} with {64, 1, 128} boxes.  max_items bounds pair entries
// * Hkv.
cudaError_t launch_prefill_packed(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                  const CUtensorMap& tm_o, const PrefillArgs& a, long max_items, cudaStream_t stream);
// Rows with no key at all (Skv == 0): O = 0, LSE = -inf.
cudaError_t launch_empty_rows(void* o, float* lse, long rows, int D, cudaStream_t stream);
int prefill_take_device_error();
// Head dim 256 (prefill_d256.cu): one query tile per CTA.  tm_q, tm_k, tm_o as
// above; tm_v with a {64, 64, 1, 1} box (64-key halves of a V tile).
cudaError_t launch_prefill_d256(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& tm_o, const PrefillArgs& a, cudaStream_t stream);
int prefill_d256_take_device_error();

// Packed calls (varlen_packed.cu, varlen_paged.cu; onetile.cuh).  The plan
// kernel lists the (request, row block) entries of a call into `tmp`, then
// into `entries` ([max_entries, 8] int32 each) ordered by estimated cost,
// heaviest first, and their count into *n_entries; kv holds cu_seqlens_kv
// [B + 1] (packed keys) or cache_seqlens [B] (paged), and kv_cap bounds a
// request's key count (total_kv, or max_pages * page_size).
// skip_single leaves requests with exactly one query out of the list (they
// run on the split decode kernel instead).
// pairs lists pairs of consecutive row blocks (q0 = 2k * qpb) for the
// two-Q-tile kernel.  With skip_single, n_entries[2] receives how many of
// `grid` persistent CTAs the listed blocks should keep so that they and the
// left-out decode steps, run at the same time, end together (grid when there
// is no decode step).
cudaError_t launch_varlen_plan(const int32_t* cu_q, const int32_t* kv, bool paged, int B, int qpb, int g, int causal,
                               int total_q, long kv_cap, int32_t* tmp, int32_t* entries, int32_t* n_entries,
                               int max_entries, cudaStream_t stream, bool skip_single = false, bool pairs = false,
                               int grid = 0);
// tm_q / tm_o: {D, Hq, total_q} with a {64, g, qpb} box.  Packed: tm_k / tm_v
// {D, Hkv, total_kv} with {64, 1, 128} and {64, 1, 128 or 64 (D = 256)} boxes.
// Paged: the caches as {64, 8, D / 64, pages * page_size / 8, Hkv} with
// {64, 8, D / 64 / (D == 256 ? 2 : 1), bt_k / 8, 1} (K) and
// {64, 8, D / 64, bt_v / 8, 1} (V) boxes.  max_items bounds entries * Hkv.
cudaError_t launch_varlen_packed(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                 const CUtensorMap& tm_o, const PrefillArgs& a, long max_items, cudaStream_t stream);
cudaError_t launch_varlen_paged(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& tm_o, const PrefillArgs& a, long max_items, cudaStream_t stream);
int varlen_packed_take_device_error();
int varlen_paged_take_device_error();

struct DecodeArgs {
    const void* q;          // [B, Sq, Hq, D]
    const void* k_cache;    // [P, ps, Hkv, D]
    const void* v_cache;
    const int32_t* seqlens; // [B]
    const int32_t* table;   // [B, max_pages]
    void* o;                // [B, Sq, Hq, D]
    float* lse;             // [B, Sq, Hq] or nullptr
    float* part_o;          // [B, Hkv, max_splits, R, D]
    float* part_lse;        // [B, Hkv, max_splits, R]  (log2 units)
    int B, Sq, Hq, Hkv, D, page_size, max_pages, num_pages, causal;
    float scale_log2;
    int chunk;              // tokens per split (multiple of the key tile)
    int max_splits;
    // Balanced tensor-core path: partials are indexed by piece id, and
    // seg_table[2s], seg_table[2s + 1] hold segment s's first id and piece
    // count; nullptr on the split path.
    int* seg_table;         // [B * Hkv, 2]
    int n_part;             // partial slots in part_o / part_lse
    int tc_grid;            // persistent CTAs (one per SM)
    int f16;                // q, caches and o are float16 (else bfloat16)
    Extras x;
    // float8_e4m3fn caches (attn_decode_paged_fp8kv): per-(request, KV head)
    // dequantization scales [B, Hkv], nullptr meaning 1
    const float* k_scale;
    const float* v_scale;
    // Packed queries (the single-query requests of attn_fwd_paged; split
    // kernels only): q_rows = cu_seqlens_q [B + 1] over q / o [q_total, Hq, D]
    // and lse [q_total, Hq]; with Sq = 1, request b takes part only when it
    // has exactly one query row, at row q_rows[b] (offsets clamped into
    // [0, q_total] as by the packed plan kernel).  nullptr: q, o and lse are
    // [B, Sq, Hq, ...].
    const int32_t* q_rows;
    int q_total;
};

struct DecodePlan {
    int chunk;
    int max_splits;
    int rows;               // g * Sq rows per KV head
    size_t part_o_bytes;
    size_t part_lse_bytes;
    size_t workspace_bytes; // enough for whichever path the sizes select
    // balanced tensor-core path (tc set when the sizes select it)
    bool tc;
    int tc_grid;
    int n_part;             // B * Hkv + tc_grid partial slots
    size_t tc_part_o_bytes, tc_part_lse_bytes, tc_table_bytes;
};

bool plan_decode(int B, int Sq, int Hq, int Hkv, int D, int page_size, int max_pages, int num_sms,
                 DecodePlan* plan);
// Tokens per TMA box for this page size (a multiple of 8 dividing both the
// page and the key tile), or 0 when pages must be gathered row by row.
int decode_box_tokens(int D, int page_size);
// tm_k / tm_v: 3-D maps {D, Hkv, pages * page_size} with a {64, 1, box_tokens}
// box, or nullptr for the cp.async gather kernel.
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap* tm_k, const CUtensorMap* tm_v, int box_tokens,
                          cudaStream_t stream);
int decode_take_device_error();
// Split decode over float8_e4m3fn caches (decode_fp8_kernel): tm_k / tm_v are
// 3-D byte maps {D, Hkv, pages * page_size} with a {128, 1, box_tokens} box;
// D is 128 or 256; the g * Sq rows of a KV group go in blocks of up to 64.
// Launches the combine as well.
cudaError_t launch_decode_fp8(const DecodeArgs& a, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                              int box_tokens, cudaStream_t stream);
// Merge of the split partials (decode_combine_kernel).
cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t stream);

// Tensor-core decode (decode_tc.cu) for 32..128 packed query rows per KV head.
bool decode_tc_eligible(int D, int R, int page_size);
int decode_tc_box_tokens(int page_size);
// tm_k / tm_v: the caches as {64, 8, D / 64, pages * page_size / 8, Hkv} with a
// {64, 8, D / 64, box_tokens / 8, 1} box (one page block of one head per box).
cudaError_t launch_decode_tc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const DecodeArgs& a,
                             int box_tokens, cudaStream_t stream);
// The same kernel over float8_e4m3fn caches (DecodeArgs k_scale / v_scale):
// tm_k / tm_v are 5-D byte maps {128, 8, D / 128, pages * page_size / 8, Hkv}
// with a {128, 8, D / 128, box_tokens / 8, 1} box (one page block of one head);
// warps widen each byte tile into the 16-bit rings.
cudaError_t launch_decode_tc_fp8(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const DecodeArgs& a,
                                 int box_tokens, cudaStream_t stream);
int decode_tc_take_device_error();

}  // namespace gqa
