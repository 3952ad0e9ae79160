// Packed queries over a paged cache (TileOPs "Attention Operators",
// GQAPagedFwdOp): q [total_q, Hq, D] with request b owning rows
// [cu_seqlens_q[b], cu_seqlens_q[b + 1]); its cache holds cache_seqlens[b]
// tokens, its query tokens included, in pages block_table[b, t / page_size].
// One launch serves any mix of prefill chunks and decode steps: every
// request's row blocks pack the g query heads of a KV group, so a decode step
// streams its cache once per KV head.  Pages move as 5-D TMA boxes of whole
// page blocks (page sizes that are multiples of 8).
#include "onetile.cuh"

namespace gqa {

cudaError_t launch_varlen_paged(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& tm_o, const PrefillArgs& a, long max_items, cudaStream_t stream) {
    switch (a.D * 2 + (a.f16 ? 1 : 0)) {
        case 64 * 2: return ot::launch_onetile<64, ot::kPaged, true, false>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        case 64 * 2 + 1: return ot::launch_onetile<64, ot::kPaged, true, true>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        case 128 * 2: return ot::launch_onetile<128, ot::kPaged, true, false>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        case 128 * 2 + 1: return ot::launch_onetile<128, ot::kPaged, true, true>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        case 256 * 2: return ot::launch_onetile<256, ot::kPaged, true, false>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        case 256 * 2 + 1: return ot::launch_onetile<256, ot::kPaged, true, true>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        default: return cudaErrorInvalidValue;
    }
}

int varlen_paged_take_device_error() { return ot::take_error(); }

}  // namespace gqa
