// Dense / chunked-prefill causal GQA attention forward for head dim 256: the
// one-query-tile kernel (onetile.cuh) on BSHD tensors.  With D = 256 one
// query tile's output accumulator takes 256 of the 512 TMEM columns, so a CTA
// owns one 128-row query tile and double-buffers its scores instead of
// running two query tiles as prefill.cu does; the 24/2/D256 geometry of MATE
// "QSA" is the case in point.
#include "onetile.cuh"

namespace gqa {

cudaError_t launch_prefill_d256(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& tm_o, const PrefillArgs& a, cudaStream_t stream) {
    if (a.D != 256) return cudaErrorInvalidValue;
    const int n_qtiles = (a.Sq + ot::BM - 1) / ot::BM;
    const long n_items = (long)n_qtiles * a.B * a.Hq;
    const bool opts = a.x.wl >= 0 || a.x.wr >= 0 || a.x.cap_out != 0.f || a.x.sinks != nullptr;
    switch ((opts ? 1 : 0) + (a.f16 ? 2 : 0)) {
        case 0: return ot::launch_onetile<256, ot::kBSHD, false, false>(tm_q, tm_k, tm_v, tm_o, a, n_items, n_qtiles,
                                                                      stream);
        case 1: return ot::launch_onetile<256, ot::kBSHD, true, false>(tm_q, tm_k, tm_v, tm_o, a, n_items, n_qtiles,
                                                                     stream);
        case 2: return ot::launch_onetile<256, ot::kBSHD, false, true>(tm_q, tm_k, tm_v, tm_o, a, n_items, n_qtiles,
                                                                     stream);
        default: return ot::launch_onetile<256, ot::kBSHD, true, true>(tm_q, tm_k, tm_v, tm_o, a, n_items, n_qtiles,
                                                                     stream);
    }
}

int prefill_d256_take_device_error() { return ot::take_error(); }

}  // namespace gqa
