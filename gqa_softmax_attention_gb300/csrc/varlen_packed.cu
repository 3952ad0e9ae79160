// Packed variable-length calls (TileOPs "Attention Operators",
// GQAVarlenFwdOp): q [total_q, Hq, D], k / v [total_kv, Hkv, D], request b
// owning query rows [cu_seqlens_q[b], cu_seqlens_q[b + 1]) and key rows
// [cu_seqlens_kv[b], cu_seqlens_kv[b + 1]).  Also the plan kernel shared with
// the paged calls: it lists the (request, row block) entries on the device,
// so the host never reads the offsets back.
#include "onetile.cuh"

namespace gqa {
namespace {

// One CTA of 1024 threads.  Request b gets ceil(Sq_b / qpb) entries
// {b, q0, qs, Sq_b, ks, L_b}.  Offsets are clamped into [0, total] and
// lengths into [0, kv_cap], so malformed metadata can give wrong results but
// no access out of range; entries past max_entries are dropped.  The
// requests are then ordered by estimated cost, heaviest first (a counting
// sort over NBUCKET cost buckets), each request's blocks together and its
// heaviest (last) block first.
constexpr int NBUCKET = 2048;
// SM time of one cached key of a decode step against one plan cost unit (see
// the end of varlen_plan_kernel), as the two kernels run side by side: the
// split decode kernel streams about 70 GB/s per SM on a share of the SMs, the
// one-tile kernel about 7.2 TFLOP/s per SM, so (4 bytes / 70 GB/s) / (2^15
// FLOP / 7.2 TFLOP/s) = 0.0126.  Set a little below: the chunks' persistent
// grid cannot grow into SMs the decode steps leave, while the decode CTAs do
// fill the SMs the chunks leave (measured on the mixed serving batch: 0.622,
// 0.606 and 0.683 ms at 0.009, 0.0126 and 0.016).
constexpr double kDecPerKey = 0.011;

__device__ __forceinline__ int entry_cost(const int4 e0, const int4 e1, int qpb, int g, int causal) {
    const int q0 = e0.y, sq = e0.w, L = e1.y;
    const int nq = min(qpb, sq - q0);
    const int last = q0 + nq - 1;                         // last query of the block
    const int keys = causal ? max(0, min(L, last + L - sq + 1)) : L;
    const int tiles = (keys + 127) / 128;
    // a block with few rows streams its keys at memory speed: weigh its tiles more
    return min(NBUCKET - 1, tiles * (nq * g >= 64 ? 2 : 3));
}

__global__ void __launch_bounds__(1024) varlen_plan_kernel(const int32_t* cu_q, const int32_t* kv, int paged,
                                                          int B, int qpb, int g, int causal, int total_q,
                                                          long kv_cap, int32_t* tmp, int32_t* entries,
                                                          int32_t* n_entries, int max_entries, int grid) {
    __shared__ int warp_sum[32];
    __shared__ unsigned long long pre_cost, dec_keys;   // listed blocks' cost; decode steps' cached keys
    __shared__ int base;
    __shared__ int bucket[NBUCKET];
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    // pairs (flag bit 2): an entry covers two consecutive row blocks
    const bool pairs = (paged & 4) != 0;
    const int span = pairs ? 2 * qpb : qpb;            // queries per entry
    auto cost_of = [&](int b, int q0, int qs, int sq, int ks, int L) {
        int c = entry_cost(make_int4(b, q0, qs, sq), make_int4(ks, L, 0, 0), qpb, g, causal);
        if (pairs && q0 + qpb < sq) c += entry_cost(make_int4(b, q0 + qpb, qs, sq), make_int4(ks, L, 0, 0), qpb, g, causal);
        return c;
    };
    if (threadIdx.x == 0) {
        base = 0;
        pre_cost = 0;
        dec_keys = 0;
    }
    for (int i = threadIdx.x; i < NBUCKET; i += 1024) bucket[i] = 0;
    __syncthreads();
    // 1. entries in request order
    for (int b0 = 0; b0 < B; b0 += 1024) {
        const int b = b0 + threadIdx.x;
        int qs = 0, sq = 0, ks = 0, L = 0, nrb = 0;
        if (b < B) {
            qs = min(max(cu_q[b], 0), total_q);
            sq = min(max(cu_q[b + 1], qs), total_q) - qs;
            if (paged & 1) {
                L = (int)min((long)max(kv[b], 0), kv_cap);
            } else {
                ks = (int)min((long)max(kv[b], 0), kv_cap);
                L = (int)min((long)max(kv[b + 1], ks), kv_cap) - ks;
            }
            nrb = (sq + span - 1) / span;
            if ((paged & 2) && sq == 1) nrb = 0;      // a decode step, run by the split decode kernel
        }
        int x = nrb;                                   // inclusive scan within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int s = warp_sum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            warp_sum[lane] = s;
        }
        __syncthreads();
        const int first = base + (warp > 0 ? warp_sum[warp - 1] : 0) + x - nrb;
        // the request's estimated cost: the sum of its blocks' costs
        int total = 0;
        for (int k = 0; k < nrb; ++k) total += cost_of(b, k * span, qs, sq, ks, L);
        if (total > 0) atomicAdd(&pre_cost, (unsigned long long)total);
        if ((paged & 2) && sq == 1 && b < B && L > 0) atomicAdd(&dec_keys, (unsigned long long)L);
        const int key = min(NBUCKET - 1, total / 16);
        for (int k = 0; k < nrb; ++k) {
            const int e = first + k;
            if (e >= max_entries) break;
            int4* dst = reinterpret_cast<int4*>(tmp + (size_t)e * ot::ENTRY_INTS);
            dst[0] = make_int4(b, k * span, qs, sq);
            dst[1] = make_int4(ks, L, key, 0);             // .w: the request's start once placed
        }
        __syncthreads();
        if (threadIdx.x == 1023) base = first + nrb;
        __syncthreads();
    }
    const int n = min(base, max_entries);
    // 2. requests ordered by estimated cost, heaviest first (a counting sort of
    // their total costs), each request's blocks kept together and placed from
    // its last block (the most keys under a causal mask) to its first: the
    // grid's snake order then works through one request's keys at a time,
    // which stay in L2 while its blocks need them.  A request's first entry
    // (q0 = 0) stands for the whole request.
    for (int e = threadIdx.x; e < n; e += 1024) {
        const int4* src = reinterpret_cast<const int4*>(tmp + (size_t)e * ot::ENTRY_INTS);
        const int4 e0 = src[0], e1 = src[1];
        // blocks of the request that made the list (all of them unless the
        // cap cut it short), so that the placed entries fill [0, n)
        if (e0.y == 0) atomicAdd(&bucket[e1.z], min((e0.w + span - 1) / span, n - e));
    }
    __syncthreads();
    {
        // bucket starts in descending cost order: thread t owns buckets
        // NBUCKET-1-2t and NBUCKET-2-2t; an exclusive block scan over threads
        static_assert(NBUCKET == 2 * 1024, "two buckets per thread");
        const int c1 = NBUCKET - 1 - 2 * threadIdx.x, c2 = c1 - 1;
        const int n1 = bucket[c1], n2 = bucket[c2];
        int x = n1 + n2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        __syncthreads();                               // warp_sum is free again
        if (lane == 31) warp_sum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int t = warp_sum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            warp_sum[lane] = t;
        }
        __syncthreads();
        const int start = (warp > 0 ? warp_sum[warp - 1] : 0) + x - n1 - n2;
        bucket[c1] = start;
        bucket[c2] = start + n1;
    }
    __syncthreads();
    // 3. each request reserves its range; then every block takes its place
    for (int e = threadIdx.x; e < n; e += 1024) {
        int4* src = reinterpret_cast<int4*>(tmp + (size_t)e * ot::ENTRY_INTS);
        const int4 e0 = src[0], e1 = src[1];
        if (e0.y == 0) src[1].w = atomicAdd(&bucket[e1.z], min((e0.w + span - 1) / span, n - e));
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n; e += 1024) {
        const int4* src = reinterpret_cast<const int4*>(tmp + (size_t)e * ot::ENTRY_INTS);
        const int4 e0 = src[0], e1 = src[1];
        const int k = e0.y / span;
        const int cnt = min((e0.w + span - 1) / span, n - (e - k));
        const int start = reinterpret_cast<const int4*>(tmp + (size_t)(e - k) * ot::ENTRY_INTS)[1].w;
        const int pos = start + cnt - 1 - k;
        if (pos < 0 || pos >= n) continue;
        int4* dst = reinterpret_cast<int4*>(entries + (size_t)pos * ot::ENTRY_INTS);
        dst[0] = e0;
        dst[1] = make_int4(e1.x, e1.y, 0, 0);
    }
    if (threadIdx.x == 0) {
        n_entries[0] = n;
        n_entries[1] = 0;                              // the attention kernel's item counter
        // The listed blocks' share of `grid` persistent CTAs when decode steps
        // run beside them: their estimated SM time against the decode steps',
        // so that both end together.  A cost unit is half a 128-key tile of a
        // full 128-row block (128 x 128 x D x 2 FLOP per KV head); a cached key
        // of a decode step is 4 D bytes per KV head (16-bit K and V); D and
        // Hkv cancel, and kDecPerKey converts the second into the first.
        int ge = grid;
        if (grid > 0 && pre_cost > 0 && dec_keys > 0) {
            const double tp = (double)pre_cost, td = (double)dec_keys * kDecPerKey;
            ge = (int)lrint((double)grid * tp / (tp + td));
            ge = min(grid, max(ge, min(grid, 8)));
        }
        n_entries[2] = ge;
    }
}

}  // namespace

cudaError_t launch_varlen_plan(const int32_t* cu_q, const int32_t* kv, bool paged, int B, int qpb, int g, int causal,
                               int total_q, long kv_cap, int32_t* tmp, int32_t* entries, int32_t* n_entries,
                               int max_entries, cudaStream_t stream, bool skip_single, bool pairs, int grid) {
    // flags: bit 0 paged (kv holds cache lengths), bit 1 skip single-query
    // requests, bit 2 pairs of row blocks
    const int flags = (paged ? 1 : 0) | (skip_single ? 2 : 0) | (pairs ? 4 : 0);
    varlen_plan_kernel<<<1, 1024, 0, stream>>>(cu_q, kv, flags, B, qpb, g, causal, total_q, kv_cap, tmp,
                                               entries, n_entries, max_entries, grid);
    return cudaGetLastError();
}

cudaError_t launch_varlen_packed(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                 const CUtensorMap& tm_o, const PrefillArgs& a, long max_items, cudaStream_t stream) {
    switch (a.D * 2 + (a.f16 ? 1 : 0)) {
        case 64 * 2: return ot::launch_onetile<64, ot::kPacked, true, false>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        case 64 * 2 + 1: return ot::launch_onetile<64, ot::kPacked, true, true>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        case 128 * 2: return ot::launch_onetile<128, ot::kPacked, true, false>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        case 128 * 2 + 1: return ot::launch_onetile<128, ot::kPacked, true, true>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        case 256 * 2: return ot::launch_onetile<256, ot::kPacked, true, false>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        case 256 * 2 + 1: return ot::launch_onetile<256, ot::kPacked, true, true>(tm_q, tm_k, tm_v, tm_o, a, max_items, 0, stream);
        default: return cudaErrorInvalidValue;
    }
}

int varlen_packed_take_device_error() { return ot::take_error(); }

}  // namespace gqa
