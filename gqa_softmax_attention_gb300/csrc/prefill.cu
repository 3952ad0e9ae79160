// Dense / chunked-prefill causal GQA attention forward on sm_103a.
//
// Computes, per (batch b, query head h, query row i), the softmax-weighted sum
// of the values of KV head r = h / (Hq/Hkv) over the visible keys
// j <= i + Skv - Sq that the padding mask keeps (TileOPs "Attention
// Operators", GQADenseFwdOp, stages 1, 4, 5, 7; RL-Kernel "Standard Softmax
// Attention", Tensor Contract).  The softmax is evaluated online over key
// tiles (running maximum and sum, FP32, base-2 exponent) so the score matrix is
// never stored, and the per-row log-sum-exp is returned in natural-log units
// (MATE "QSA", Core Attention).
//
// One CTA owns one 128-row query tile of one (b, h) and is warp-specialised:
//   warp 4     TMA producer: Q once, then K_j and V_j tiles through two
//              shared-memory rings (128-byte swizzle, 64-column boxes);
//   warp 5     MMA issuer (one thread): S_j = Q K_j^T into TMEM (two S
//              buffers), then O += P_j V_j with P read from TMEM;
//   warps 0-3  softmax: thread t owns query row t; it reads its S row from
//              TMEM, folds the causal / padding mask, updates the running
//              max and sum, writes P (bf16) back to TMEM, rescales O when the
//              max grows, and finally normalises O and writes O and LSE.
// Key tiles holding no visible key (beyond the causal bound or fully padded)
// are never loaded.  Every wait is bounded (ptx.cuh); on a timeout the CTA
// stops issuing work, drains what is in flight, frees TMEM and returns.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

__device__ int g_prefill_error;

constexpr int BM = 128;            // query rows per CTA (= TMEM lanes)
constexpr int BN = 128;            // keys per tile
constexpr int NUM_THREADS = 192;   // warps 0-3 softmax, 4 producer, 5 MMA
constexpr int WARP_LOAD = 4;
constexpr int WARP_MMA = 5;
constexpr float kLn2 = 0.693147180559945309f;

template <int D>
struct Cfg {
    static constexpr int KSUB = D / 64;                 // 64-column (128-byte) boxes per row
    static constexpr int SUB_BYTES = BN * 128;          // one box: 128 rows x 128 bytes
    static constexpr int TILE_BYTES = KSUB * SUB_BYTES; // one Q, K or V tile
    static constexpr int NK = D == 64 ? 3 : 2;          // K ring depth
    static constexpr int NV = D == 64 ? 3 : 2;          // V ring depth
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_V + NV * TILE_BYTES;
    // q_full, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_full[2], p_full[2], o_done, drain
    static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 + 2 + 1 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // 1 KB alignment slack; at least 120 KB so that one CTA holds an SM (it
    // takes all 512 TMEM columns).
    static constexpr int SMEM_BYTES = SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024;
    // TMEM columns (32-bit each): two S buffers, O, two P buffers (bf16 pairs).
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;
    static constexpr uint32_t COL_P0 = 256 + D, COL_P1 = 256 + D + 64;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t IDESC_QK = make_idesc_bf16(BM, BN, false, false);
    static constexpr uint32_t IDESC_PV = make_idesc_bf16(BM, D, false, true);
    static_assert(COL_P1 + 64 <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct TileInfo {
    int q0;          // first query row of the tile
    int rows_valid;  // rows of the tile that exist (ragged tail)
    int lim_first;   // keys [0, lim_first) are causally visible to every row of the tile
    int kv_end;      // no row of the tile sees a key >= kv_end
    int n_tiles;     // key tiles to visit
};

__device__ __forceinline__ TileInfo tile_info(int qtile, int Sq, int Skv, int causal) {
    TileInfo t;
    t.q0 = qtile * BM;
    t.rows_valid = min(BM, Sq - t.q0);
    const long p_first = (long)t.q0 + Skv - Sq;              // key position of the first row
    const long p_last = (long)t.q0 + t.rows_valid - 1 + Skv - Sq;
    if (causal) {
        t.kv_end = (int)max(0L, min((long)Skv, p_last + 1));
        t.lim_first = (int)max(0L, min((long)Skv, p_first + 1));
    } else {
        t.kv_end = Skv;
        t.lim_first = Skv;
    }
    t.n_tiles = (t.kv_end + BN - 1) / BN;
    return t;
}

// Bit `lane` of the result: key key0 + lane is below kv_end and kept by the
// padding mask.  Warp-collective.
__device__ __forceinline__ uint32_t mask_word(const uint8_t* mrow, int key0, int kv_end, int lane) {
    const int key = key0 + lane;
    const bool keep = key < kv_end && mrow[key] != 0;
    return __ballot_sync(0xffffffffu, keep);
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a, int n_qtiles) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw_base & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // Heaviest (last) query tiles first; adjacent CTAs share a KV head.
    const int bh = a.B * a.Hq;
    const int qtile = n_qtiles - 1 - (int)(blockIdx.x / bh);
    const int rem = (int)(blockIdx.x % bh);
    const int hq = rem % a.Hq;
    const int b = rem / a.Hq;
    const int hkv = hq / (a.Hq / a.Hkv);

    const uint32_t bar0 = sb + C::OFF_BAR;
    const uint32_t q_full = bar0;
    auto k_full = [&](int i) { return bar0 + 8u * (1 + i); };
    auto k_empty = [&](int i) { return bar0 + 8u * (1 + C::NK + i); };
    auto v_full = [&](int i) { return bar0 + 8u * (1 + 2 * C::NK + i); };
    auto v_empty = [&](int i) { return bar0 + 8u * (1 + 2 * C::NK + C::NV + i); };
    auto s_full = [&](int i) { return bar0 + 8u * (1 + 2 * C::NK + 2 * C::NV + i); };
    auto p_full = [&](int i) { return bar0 + 8u * (3 + 2 * C::NK + 2 * C::NV + i); };
    const uint32_t o_done = bar0 + 8u * (5 + 2 * C::NK + 2 * C::NV);
    const uint32_t drain = bar0 + 8u * (6 + 2 * C::NK + 2 * C::NV);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < C::NK; ++i) { mbar_init(k_full(i), 1); mbar_init(k_empty(i), 1); }
        for (int i = 0; i < C::NV; ++i) { mbar_init(v_full(i), 1); mbar_init(v_empty(i), 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(s_full(i), 1); mbar_init(p_full(i), BM); }
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const TileInfo ti = tile_info(qtile, a.Sq, a.Skv, a.causal);
    const uint8_t* mrow = a.mask ? a.mask + (size_t)b * a.Skv : nullptr;

    // Warp-collective: does key tile j hold no key the padding mask keeps?
    auto tile_empty = [&](int j) -> bool {
        if (!mrow) return false;
        uint32_t any = 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) any |= mask_word(mrow, j * BN + w * 32, ti.kv_end, lane);
        return any == 0;
    };

    if (warp == WARP_LOAD) {
        // ------------------------------------------------------------ producer
        if (ti.n_tiles > 0) {
            int nk = 0, nv = 0;   // K and V tile loads issued so far
            bool q_issued = false;
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                mbar_arrive_expect_tx(q_full, C::TILE_BYTES);
#pragma unroll
                for (int s = 0; s < C::KSUB; ++s)
                    tma_load_4d(sb + C::OFF_Q + s * C::SUB_BYTES, &tm_q, q_full, s * 64, ti.q0, hq, b);
                q_issued = true;
            }
            for (int j = 0; j < ti.n_tiles; ++j) {
                if (tile_empty(j)) continue;
                bool ok = true;
                if (lane == 0) {
                    const int ks = nk % C::NK;
                    ok = mbar_wait(k_empty(ks), ((nk / C::NK) & 1) ^ 1, abort_flag);
                    if (ok) {
                        mbar_arrive_expect_tx(k_full(ks), C::TILE_BYTES);
#pragma unroll
                        for (int s = 0; s < C::KSUB; ++s)
                            tma_load_4d(sb + C::OFF_K + ks * C::TILE_BYTES + s * C::SUB_BYTES, &tm_k,
                                        k_full(ks), s * 64, j * BN, hkv, b);
                        ++nk;
                        const int vs = nv % C::NV;
                        ok = mbar_wait(v_empty(vs), ((nv / C::NV) & 1) ^ 1, abort_flag);
                        if (ok) {
                            mbar_arrive_expect_tx(v_full(vs), C::TILE_BYTES);
#pragma unroll
                            for (int s = 0; s < C::KSUB; ++s)
                                tma_load_4d(sb + C::OFF_V + vs * C::TILE_BYTES + s * C::SUB_BYTES,
                                            &tm_v, v_full(vs), s * 64, j * BN, hkv, b);
                            ++nv;
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            if (lane == 0 && *abort_flag) {
                // Let copies already in flight land before the CTA goes away:
                // wait for the last load issued into each slot.
                if (q_issued) mbar_drain(q_full, 0);
                for (int s = 0; s < C::NK && s < nk; ++s) {
                    const int last = nk - 1 - ((nk - 1 - s) % C::NK);
                    mbar_drain(k_full(s), (last / C::NK) & 1);
                }
                for (int s = 0; s < C::NV && s < nv; ++s) {
                    const int last = nv - 1 - ((nv - 1 - s) % C::NV);
                    mbar_drain(v_full(s), (last / C::NV) & 1);
                }
            }
        }
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        if (ti.n_tiles > 0) {
            auto issue_pv = [&](int t) -> bool {
                const int pb = t & 1;
                if (!mbar_wait(p_full(pb), (t >> 1) & 1, abort_flag)) return false;
                const int vs = t % C::NV;
                if (!mbar_wait(v_full(vs), (t / C::NV) & 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t pcol = pb ? C::COL_P1 : C::COL_P0;
                const uint32_t vbase = sb + C::OFF_V + vs * C::TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // keys 16kk..16kk+15 of V: rows 16kk.. of every 64-column box
                    const uint64_t bdesc = make_sdesc_sw128(vbase + kk * 16 * 128, C::SUB_BYTES, 1024);
                    mma_bf16_ts(tmem + C::COL_O, tmem + pcol + kk * 8, bdesc, C::IDESC_PV,
                                (t > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(o_done);
                mma_commit(v_empty(vs));
                return true;
            };

            bool ok = true;
            if (lane == 0) ok = mbar_wait(q_full, 0, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            int it = 0;
            for (int j = 0; j < ti.n_tiles && ok; ++j) {
                if (tile_empty(j)) continue;
                if (lane == 0) {
                    const int ks = it % C::NK;
                    ok = mbar_wait(k_full(ks), (it / C::NK) & 1, abort_flag);
                    if (ok) {
                        tc_fence_after();
                        const uint32_t d = tmem + ((it & 1) ? C::COL_S1 : C::COL_S0);
                        const uint32_t kbase = sb + C::OFF_K + ks * C::TILE_BYTES;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t koff = (kk / 4) * C::SUB_BYTES + (kk % 4) * 32;
                            const uint64_t adesc = make_sdesc_sw128(sb + C::OFF_Q + koff, 16, 1024);
                            const uint64_t bdesc = make_sdesc_sw128(kbase + koff, 16, 1024);
                            mma_bf16_ss(d, adesc, bdesc, C::IDESC_QK, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(s_full(it & 1));
                        mma_commit(k_empty(ks));
                        if (it > 0) ok = issue_pv(it - 1);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                ++it;
            }
            if (ok && it > 0 && lane == 0) issue_pv(it - 1);
            __syncwarp();
            if (lane == 0) {
                // Every MMA issued above has completed once this arrives.
                mma_commit(drain);
                mbar_drain(drain, 0);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ softmax warps 0-3
        const int r = warp * 32 + lane;                       // row of the tile == TMEM lane
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        const int row_q = ti.q0 + r;
        const long p_row = (long)row_q + a.Skv - a.Sq;
        const int lim = a.causal ? (int)max(0L, min((long)a.Skv, p_row + 1)) : a.Skv;
        const float sl = a.scale_log2;
        float m_run = -INFINITY;
        float l_run = 0.f;
        bool ok = true;
        int it = 0;
        for (int j = 0; j < ti.n_tiles; ++j) {
            uint32_t mw[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
            bool all_kept = true;
            if (mrow) {
                uint32_t any = 0;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    mw[w] = mask_word(mrow, j * BN + w * 32, ti.kv_end, lane);
                    any |= mw[w];
                    all_kept = all_kept && (mw[w] == 0xffffffffu);
                }
                if (any == 0) continue;                         // skipped by every role
            }
            const int kbase = j * BN;
            const bool need_mask = (kbase + BN > ti.lim_first) || !all_kept;

            ok = __all_sync(0xffffffffu, mbar_wait(s_full(it & 1), (it >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const uint32_t scol = (it & 1) ? C::COL_S1 : C::COL_S0;
            float s[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(tmem + lane_addr + scol + 32 * c, s + 32 * c);

            float mx = -INFINITY;
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    const bool vis = (kbase + c < lim) && ((mw[c >> 5] >> (c & 31)) & 1u);
                    s[c] = vis ? s[c] * sl : -INFINITY;
                    mx = fmaxf(mx, s[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    s[c] *= sl;
                    mx = fmaxf(mx, s[c]);
                }
            }
            const float m_new = fmaxf(m_run, mx);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;   // no -inf - -inf
            const float alpha = fast_exp2(m_run - m_use);
            float rs = 0.f;
            uint32_t pk[BN / 2];
#pragma unroll
            for (int c = 0; c < BN / 2; ++c) {
                const float p0 = fast_exp2(s[2 * c] - m_use);
                const float p1 = fast_exp2(s[2 * c + 1] - m_use);
                rs += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
            }
            const uint32_t pcol = (it & 1) ? C::COL_P1 : C::COL_P0;
            tmem_st32(tmem + lane_addr + pcol, pk);
            tmem_st32(tmem + lane_addr + pcol + 32, pk + 32);
            l_run = l_run * alpha + rs;
            m_run = m_new;

            if (it > 0) {
                // O must hold P_{it-1} V_{it-1} before it is rescaled.
                ok = __all_sync(0xffffffffu, mbar_wait(o_done, (it - 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tmem + lane_addr + C::COL_O + 32 * c, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= alpha;
                        tmem_st32(tmem + lane_addr + C::COL_O + 32 * c, reinterpret_cast<uint32_t*>(o));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(p_full(it & 1));
            ++it;
        }

        if (ok && it > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(o_done, (it - 1) & 1, abort_flag));
            if (ok) tc_fence_after();
        }
        const bool row_ok = r < ti.rows_valid;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) +
                              (((size_t)b * a.Sq + row_q) * a.Hq + hq) * D;
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        if (ok && it > 0) {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tmem_ld32(tmem + lane_addr + C::COL_O + 32 * c, o);
                if (row_ok) {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(o[2 * e] * inv, o[2 * e + 1] * inv);
                    uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                }
            }
        } else if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
            for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (row_ok && a.lse)
            a.lse[((size_t)b * a.Sq + row_q) * a.Hq + hq] =
                l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(&g_prefill_error, (int)kErrPrefillWait);
}

__global__ void empty_rows_kernel(__nv_bfloat16* o, float* lse, long rows, int D) {
    const long n = rows * D;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        o[i] = __float2bfloat16_rn(0.f);
        if (lse && i % D == 0) lse[i / D] = -INFINITY;
    }
}

template <int D>
cudaError_t launch_prefill_t(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const PrefillArgs& a, cudaStream_t stream) {
    using C = Cfg<D>;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_qtiles = (a.Sq + BM - 1) / BM;
    const long grid = (long)n_qtiles * a.B * a.Hq;
    prefill_kernel<D><<<(unsigned)grid, NUM_THREADS, C::SMEM_BYTES, stream>>>(tm_q, tm_k, tm_v, a, n_qtiles);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const PrefillArgs& a, cudaStream_t stream) {
    switch (a.D) {
        case 64: return launch_prefill_t<64>(tm_q, tm_k, tm_v, a, stream);
        case 128: return launch_prefill_t<128>(tm_q, tm_k, tm_v, a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_empty_rows(void* o, float* lse, long rows, int D, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const long n = rows * D;
    const int threads = 256;
    const long blocks = (n + threads - 1) / threads < 4096 ? (n + threads - 1) / threads : 4096;
    empty_rows_kernel<<<(unsigned)blocks, threads, 0, stream>>>(reinterpret_cast<__nv_bfloat16*>(o), lse,
                                                                 rows, D);
    return cudaGetLastError();
}

int prefill_take_device_error() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof(int)) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace gqa
