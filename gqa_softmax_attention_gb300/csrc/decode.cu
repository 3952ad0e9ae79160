// Paged-KV decode: split-KV attention over a [pages, page_size, Hkv, D] cache,
// then an LSE-weighted combine of the splits.
//
// Request b's logical token t lives in slot t % page_size of physical page
// block_table[b, t / page_size]; query i of the request sits at key position
// i + L_b - Sq, so with the causal flag it sees keys t <= i + L_b - Sq
// (TileOPs "Attention Operators", MHADecodePagedWithKVCacheFwdOp and
// GQAPagedFwdOp).  The key axis of each request is cut into fixed-size splits
// whose partial results keep FP32 softmax statistics and are merged by their
// log-sum-exps without recomputing QK or PV (MATE "QSA", Core Attention,
// SplitKV).
//
// One CTA per (split, KV head, request, row block).  All g * Sq query rows
// that read this KV head are packed into the M dimension of m16n8k16
// tensor-core MMAs (rows padded to 16 * MF).  Keys are processed in tiles of
// TK tokens held in a multi-stage shared-memory ring laid out as 64-column
// sub-tiles with 128-byte rows (16-byte chunks XOR-swizzled by row % 8):
//   decode_tma_kernel     one producer warp fills the ring with TMA: each page
//                         of a KV head is a strided 3-D box {64 cols, 1 head,
//                         page tokens}; consumer warps only wait on mbarriers.
//                         Used when pages cut into 8-row multiples of the tile.
//   decode_gather_kernel  every thread gathers token rows with 16-byte
//                         cp.async copies (any page size).
// In both, consumer warps split the keys of a tile for S = Q K^T (each warp
// keeps its rows of Q in registers), rows are softmaxed by thread groups in
// shared memory (running max and sum, base 2), and the warps split the head
// dimension for O += P V.  Slots past the request's length never contribute:
// their scores are -inf and their value rows are zero in shared memory (never
// 0 * garbage).  Each split writes its normalised FP32 partial O and its base-2
// LSE to the workspace.
// decode_combine_kernel: one warp per output row; weights exp(lse_s - max),
//   normalised; a row no split saw gets O = 0 and LSE = -inf.
//
// The path is bound by HBM bandwidth; the MMAs are small and hidden under the
// loads, so warp-level mma.sync is used rather than tcgen05.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "gqa_attn.h"
#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

__device__ int g_decode_error;

constexpr float kLn2 = 0.693147180559945309f;

constexpr int key_tile(int D) { return D == 256 ? 32 : 64; }

template <int D, int MF, bool TMA, bool F16_ = false>
struct DCfg {
    static constexpr bool F16 = F16_;                        // float16 data (else bfloat16)
    static constexpr int TK = key_tile(D);                   // tokens per key tile
    static constexpr int KSPLIT = (MF == 1 && TK == 64) ? 4 : 2;   // consumer warps per 16-row fragment
    static constexpr int NC = MF * KSPLIT;                   // consumer warps
    static constexpr int NCT = NC * 32;                      // consumer threads
    static constexpr int NT = NCT + (TMA ? 32 : 0);          // + producer warp
    static constexpr int ROWS = 16 * MF;                     // padded rows per CTA
    static constexpr int NSUB = D / 64;                      // 64-column sub-tiles
    static constexpr int SUB_BYTES = TK * 128;               // one sub-tile of a K (or V) tile
    static constexpr int KV_TILE = NSUB * SUB_BYTES;
    static constexpr int KEYS_PER_WARP = TK / KSPLIT;
    static constexpr int NFK = KEYS_PER_WARP / 8;            // n8 fragments per warp in S = Q K^T
    static constexpr int DSL = D / KSPLIT;                   // head-dim slice per warp in O += P V
    static constexpr int NFD = DSL / 8;
    static constexpr int KSTEPS = D / 16;
    static constexpr int S_STRIDE = TK + 4;                  // floats per score row
    static constexpr int TPR = NCT / ROWS;                   // threads per row in the softmax
    static constexpr int KPT = TK / TPR;                     // keys per thread in the softmax
    static constexpr int Q_BYTES = ROWS * D * 2;
    static constexpr int FIXED = Q_BYTES + ROWS * S_STRIDE * 4 + ROWS * 128 + 3 * ROWS * 4 + 1024 + 256;
    // as many stages as fit next to the fixed part, capped
    static constexpr int NS_FIT = (227 * 1024 - FIXED) / (2 * KV_TILE);
    static constexpr int NS_CAP = D == 256 ? 4 : (D == 128 ? 3 : 6);
    static constexpr int NS = NS_FIT < NS_CAP ? NS_FIT : NS_CAP;
    static constexpr int OFF_KV = 0;                          // 1024-aligned stage ring first
    static constexpr int OFF_Q = OFF_KV + NS * 2 * KV_TILE;
    static constexpr int OFF_S = OFF_Q + Q_BYTES;
    static constexpr int OFF_P = OFF_S + ROWS * S_STRIDE * 4;
    static constexpr int OFF_A = OFF_P + ROWS * 128;
    static constexpr int OFF_L = OFF_A + ROWS * 4;
    static constexpr int OFF_M = OFF_L + ROWS * 4;
    static constexpr int OFF_BAR = OFF_M + ROWS * 4;         // full[NS], empty[NS]
    static constexpr int OFF_FLAG = OFF_BAR + 2 * NS * 8;
    static constexpr int SMEM = OFF_FLAG + 16 + 1024;        // + alignment slack
    static_assert(NS >= 2, "pipeline depth");
    static_assert(NFK % 2 == 0 && NFD % 2 == 0, "fragments are loaded in pairs");
    static_assert(KPT % 8 == 0 && TK * 2 <= 128, "softmax writes whole 16-byte chunks of a 128-byte P row");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Byte offset of 16-byte chunk c of row r in a [D/64][rows][128 B] tile.
__device__ __forceinline__ uint32_t sw_off(int r, int c, int sub_bytes) {
    return (uint32_t)((c >> 3) * sub_bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

struct Work {
    int split, hkv, b, rb, L, t_begin, t_end, n_tiles, row0, rows_here;
    long qrow0;     // row of query 0 of request b in q ([B * Sq] rows, or packed)
};

// Packed call (a.q_rows set): whether request b has exactly one query row, and
// that row (offsets clamped into [0, q_total] like the packed plan kernel's).
__device__ __forceinline__ bool packed_single(const DecodeArgs& a, int b, long& row) {
    const int qs = min(max(a.q_rows[b], 0), a.q_total);
    const int qe = min(max(a.q_rows[b + 1], qs), a.q_total);
    row = qs;
    return qe - qs == 1;
}

template <class C>
__device__ __forceinline__ bool work_of(const DecodeArgs& a, int R, int g, int n_rowblk, Work& w) {
    w.split = blockIdx.x;
    w.hkv = blockIdx.y;
    w.b = blockIdx.z / n_rowblk;
    w.rb = blockIdx.z % n_rowblk;
    w.qrow0 = (long)w.b * a.Sq;
    if (a.q_rows && !packed_single(a, w.b, w.qrow0)) return false;   // not a decode step: not ours
    // Lengths are clamped to the table's capacity so a bad length cannot send
    // a load past block_table.
    w.L = min(max(a.seqlens[w.b], 0), a.max_pages * a.page_size);
    w.row0 = w.rb * C::ROWS;
    w.rows_here = min(C::ROWS, R - w.row0);
    w.t_begin = w.split * a.chunk;
    if (w.t_begin >= w.L) return false;            // nothing here; the combine skips it
    w.t_end = min(w.L, w.t_begin + a.chunk);
    if (a.x.wl >= 0) {
        // keys left of every row's window are never read: start at the tile
        // holding the first row's lower bound (the combine reads no split
        // before the one holding a row's lower bound)
        const long lo = (long)(w.row0 / g) + w.L - a.Sq - a.x.wl;
        if (lo > w.t_begin) w.t_begin = (int)min((long)w.t_end, lo / C::TK * C::TK);
        if (w.t_begin >= w.t_end) return false;
    }
    w.n_tiles = (w.t_end - w.t_begin + C::TK - 1) / C::TK;
    return true;
}

// Consumer-side state and the per-tile steps shared by both kernels.
template <class C>
struct Consumer {
    static constexpr int CHUNKS = C::NSUB * 8;   // 16-byte chunks per row of D
    uint32_t sb;            // shared-memory base (1024-aligned)
    uint8_t* smem;
    int ctid, warp, lane, mf, wk, srow, ssub;
    int lim[2];             // exclusive visibility limit of the two fragment rows this lane holds
    int lo[2];              // their inclusive lower limit (left window)
    float cap_in, cap_out;  // softcap, or cap_out == 0
    float out_scale;        // multiplies the stored partial O (FP8 value scale; else 1)
    uint32_t qf[C::KSTEPS][4];
    float m_run, l_run;
    float acc[C::NFD][4];

    __device__ __forceinline__ void init(uint8_t* s, uint32_t base, const DecodeArgs& a, const Work& w, int g) {
        smem = s;
        sb = base;
        ctid = threadIdx.x;
        warp = ctid / 32;
        lane = ctid % 32;
        mf = warp / C::KSPLIT;
        wk = warp % C::KSPLIT;
        srow = ctid / C::TPR;
        ssub = ctid % C::TPR;
        m_run = -INFINITY;
        l_run = 0.f;
#pragma unroll
        for (int n = 0; n < C::NFD; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        cap_in = a.x.cap_in;
        cap_out = a.x.cap_out;
        out_scale = 1.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int rl = mf * 16 + (lane >> 2) + 8 * h;
            const int r = w.row0 + rl;
            lo[h] = 0;
            if (rl >= w.rows_here) {
                lim[h] = -1;
            } else {
                // keys [lo, lim) of query r / g at key position p (TileOPs
                // GQAPagedFwdOp: causal j <= p, window p - wL <= j <= p + wR)
                const long p = (long)(r / g) + w.L - a.Sq;
                long hi = w.t_end;
                if (a.causal) hi = min(hi, p + 1);
                if (a.x.wr >= 0) hi = min(hi, p + a.x.wr + 1);
                lim[h] = (int)max(-1L, hi);
                if (a.x.wl >= 0) lo[h] = (int)max(0L, min((long)w.L, p - a.x.wl));
            }
        }
    }

    // Q rows r = i * g + hl (query i, head hkv * g + hl) -> shared memory with
    // cp.async (padded rows zero), then into registers.  `bar` syncs consumers.
    template <class Bar>
    __device__ __forceinline__ void load_q(const DecodeArgs& a, const Work& w, int g, Bar bar) {
        const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(a.q);
        for (int idx = ctid; idx < C::ROWS * CHUNKS; idx += C::NCT) {
            const int rr = idx / CHUNKS, c = idx % CHUNKS;
            const uint32_t dst = sb + C::OFF_Q + sw_off(rr, c, C::ROWS * 128);
            if (rr < w.rows_here) {
                const int r = w.row0 + rr;
                const int i = r / g, hl = r % g;
                cp_async16(dst, qg + (((size_t)w.qrow0 + i) * a.Hq + w.hkv * g + hl) * (CHUNKS * 8) + c * 8, 16);
            } else {
                cp_async16(dst, qg, 0);
            }
        }
        cp_async_commit();
        cp_async_wait<0>();
        bar();
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            const int row = mf * 16 + (lane & 15);
            const int chunk = kk * 2 + (lane >> 4);
            ldsm_x4(sb + C::OFF_Q + sw_off(row, chunk, C::ROWS * 128), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
        }
    }

    // S = Q K^T for this warp's rows and keys, scaled and masked, into smem.
    __device__ __forceinline__ void qk(uint32_t sK, int t0, float sl) {
        float sacc[C::NFK][4];
#pragma unroll
        for (int n = 0; n < C::NFK; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
#pragma unroll
            for (int np = 0; np < C::NFK / 2; ++np) {
                const int key = wk * C::KEYS_PER_WARP + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int chunk = kk * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sK + sw_off(key, chunk, C::SUB_BYTES), b0, b1, b2, b3);
                mma16816<C::F16>(sacc[2 * np], qf[kk], b0, b1);
                mma16816<C::F16>(sacc[2 * np + 1], qf[kk], b2, b3);
            }
        }
        write_s(sacc, t0, sl);
    }

    // Scaled (or capped) and masked scores of this warp's keys into smem.
    __device__ __forceinline__ void write_s(const float (&sacc)[C::NFK][4], int t0, float sl) {
        float* sS = reinterpret_cast<float*>(smem + C::OFF_S);
#pragma unroll
        for (int n = 0; n < C::NFK; ++n) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rl = mf * 16 + (lane >> 2) + 8 * h;
                const int kl = wk * C::KEYS_PER_WARP + n * 8 + 2 * (lane & 3);
                const int t = t0 + kl;
                float x0 = sacc[n][2 * h] * sl, x1 = sacc[n][2 * h + 1] * sl;
                if (cap_out != 0.f) {
                    x0 = softcap_log2(sacc[n][2 * h], cap_in, cap_out);
                    x1 = softcap_log2(sacc[n][2 * h + 1], cap_in, cap_out);
                }
                float2 v;                                                 // the select drops stale rows
                v.x = t >= lo[h] && t < lim[h] ? x0 : -INFINITY;
                v.y = t + 1 >= lo[h] && t + 1 < lim[h] ? x1 : -INFINITY;
                *reinterpret_cast<float2*>(sS + rl * C::S_STRIDE + kl) = v;
            }
        }
    }

    // Online softmax over the tile, TPR threads per row; P (bf16) and the
    // rescale factor alpha go to smem.
    __device__ __forceinline__ void softmax() {
        const float* sS = reinterpret_cast<const float*>(smem + C::OFF_S);
        float* sAlpha = reinterpret_cast<float*>(smem + C::OFF_A);
        float x[C::KPT];
        const float* src = sS + srow * C::S_STRIDE + ssub * C::KPT;
#pragma unroll
        for (int e = 0; e < C::KPT; e += 4) {
            const float4 f = *reinterpret_cast<const float4*>(src + e);
            x[e] = f.x; x[e + 1] = f.y; x[e + 2] = f.z; x[e + 3] = f.w;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < C::KPT; ++e) mx = fmaxf(mx, x[e]);
#pragma unroll
        for (int o = C::TPR / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m_run, mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = fast_exp2(m_run - m_use);
        float sum = 0.f;
        uint32_t pk[C::KPT / 2];
#pragma unroll
        for (int e = 0; e < C::KPT / 2; ++e) {
            const float p0 = fast_exp2(x[2 * e] - m_use);
            const float p1 = fast_exp2(x[2 * e + 1] - m_use);
            sum += p0 + p1;
            pk[e] = pack2<C::F16>(p0, p1);
        }
#pragma unroll
        for (int o = C::TPR / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        l_run = l_run * alpha + sum;
        m_run = m_new;
#pragma unroll
        for (int q = 0; q < C::KPT / 8; ++q) {
            const int chunk = ssub * (C::KPT / 8) + q;
            *reinterpret_cast<uint4*>(smem + C::OFF_P + srow * 128 + ((chunk ^ (srow & 7)) << 4)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
        if (ssub == 0) sAlpha[srow] = alpha;
    }

    // O = O * alpha + P V for this warp's rows and head-dim slice.
    __device__ __forceinline__ void pv(uint32_t sV) {
        const float* sAlpha = reinterpret_cast<const float*>(smem + C::OFF_A);
        const float a0 = sAlpha[mf * 16 + (lane >> 2)];
        const float a1 = sAlpha[mf * 16 + (lane >> 2) + 8];
#pragma unroll
        for (int n = 0; n < C::NFD; ++n) {
            acc[n][0] *= a0; acc[n][1] *= a0;
            acc[n][2] *= a1; acc[n][3] *= a1;
        }
#pragma unroll
        for (int kk = 0; kk < C::TK / 16; ++kk) {
            uint32_t pa[4];
            {
                const int row = mf * 16 + (lane & 15);
                const int chunk = kk * 2 + (lane >> 4);
                ldsm_x4(sb + C::OFF_P + row * 128 + ((chunk ^ (row & 7)) << 4), pa[0], pa[1], pa[2], pa[3]);
            }
#pragma unroll
            for (int np = 0; np < C::NFD / 2; ++np) {
                const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int dchunk = (wk * C::DSL + np * 16) / 8 + (lane >> 4);
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(sV + sw_off(key, dchunk, C::SUB_BYTES), v0, v1, v2, v3);
                mma16816<C::F16>(acc[2 * np], pa, v0, v1);
                mma16816<C::F16>(acc[2 * np + 1], pa, v2, v3);
            }
        }
    }

    // Normalised partial O (FP32) and base-2 LSE of this split.  `bar` syncs consumers.
    template <class Bar>
    __device__ __forceinline__ void store(const DecodeArgs& a, const Work& w, int R, Bar bar) {
        float* sL = reinterpret_cast<float*>(smem + C::OFF_L);
        float* sM = reinterpret_cast<float*>(smem + C::OFF_M);
        if (ssub == 0) {
            sL[srow] = l_run;
            sM[srow] = m_run;
        }
        bar();
        const size_t part_row0 = ((size_t)(w.b * a.Hkv + w.hkv) * a.max_splits + w.split) * R + w.row0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int rl = mf * 16 + (lane >> 2) + 8 * h;
            if (rl < w.rows_here) {
                const float l = sL[rl];
                const float inv = l > 0.f ? out_scale / l : 0.f;
                float* dst = a.part_o + (part_row0 + rl) * (CHUNKS * 8) + wk * C::DSL + 2 * (lane & 3);
#pragma unroll
                for (int n = 0; n < C::NFD; ++n)
                    *reinterpret_cast<float2*>(dst + n * 8) =
                        make_float2(acc[n][2 * h] * inv, acc[n][2 * h + 1] * inv);
            }
        }
        if (ctid < w.rows_here) {
            const float l = sL[ctid];
            a.part_lse[part_row0 + ctid] = l > 0.f ? sM[ctid] + log2f(l) : -INFINITY;
        }
    }
};

template <int D, int MF, bool F16>
__global__ void __launch_bounds__(DCfg<D, MF, true, F16>::NT)
decode_tma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeArgs a, int R, int g, int n_rowblk, int box_tokens) {
    using C = DCfg<D, MF, true, F16>;
    griddep_launch_dependents();                 // the combine may be scheduled (it waits for this grid)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    Work w;
    if (!work_of<C>(a, R, g, n_rowblk, w)) return;

    const uint32_t bar0 = sb + C::OFF_BAR;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (C::NS + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), C::NC);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int warp = threadIdx.x / 32;
    if (warp == C::NC) {
        // ------------------------------------------------------------ TMA producer
        if ((threadIdx.x & 31) == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const int32_t* trow = a.table + (size_t)w.b * a.max_pages;
            const int nbox = C::TK / box_tokens;
            const uint32_t box_bytes = (uint32_t)box_tokens * 128;
            int issued = 0;
            for (int it = 0; it < w.n_tiles; ++it) {
                const int s = it % C::NS;
                if (!mbar_wait(empty(s), ((it / C::NS) & 1) ^ 1, abort_flag)) break;
                const int t0 = w.t_begin + it * C::TK;
                int rows[8];        // first cache row of each box, or -1
                int n = 0;
                for (int i = 0; i < nbox; ++i) {
                    const int t = t0 + i * box_tokens;
                    int row = -1;
                    if (t < w.t_end) {
                        const int page = trow[t / a.page_size];
                        // a page id outside the pool (a caller error) is not loaded
                        if (page >= 0 && page < a.num_pages) row = page * a.page_size + t % a.page_size;
                    }
                    rows[i] = row;
                    n += row >= 0;
                }
                mbar_arrive_expect_tx(full(s), (uint32_t)n * box_bytes * C::NSUB * 2);
                const uint32_t sK = sb + C::OFF_KV + s * 2 * C::KV_TILE;
                const uint32_t sV = sK + C::KV_TILE;
                for (int i = 0; i < nbox; ++i) {
                    if (rows[i] < 0) continue;
#pragma unroll
                    for (int sub = 0; sub < C::NSUB; ++sub) {
                        const uint32_t off = sub * C::SUB_BYTES + i * box_tokens * 128;
                        tma_load_3d(sK + off, &tm_k, full(s), sub * 64, w.hkv, rows[i]);
                        tma_load_3d(sV + off, &tm_v, full(s), sub * 64, w.hkv, rows[i]);
                    }
                }
                issued = it + 1;
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA goes away
                for (int it = issued - C::NS > 0 ? issued - C::NS : 0; it < issued; ++it)
                    mbar_drain(full(it % C::NS), (it / C::NS) & 1);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        Consumer<C> c;
        c.init(smem, sb, a, w, g);
        auto bar = [] { named_bar_sync(1, C::NCT); };
        c.load_q(a, w, g, bar);
        const float sl = a.scale_log2;
        for (int it = 0; it < w.n_tiles; ++it) {
            const int s = it % C::NS;
            const int t0 = w.t_begin + it * C::TK;
            const uint32_t sK = sb + C::OFF_KV + s * 2 * C::KV_TILE;
            const uint32_t sV = sK + C::KV_TILE;
            const bool ok = mbar_wait(full(s), (it / C::NS) & 1, abort_flag);
            if (ok) {
                const int nvalid = w.t_end - t0;
                if (nvalid < C::TK) {
                    // Value rows past the request's end hold stale data: zero them.
                    const int per_sub = (C::TK - nvalid) * 8;
                    for (int idx = c.ctid; idx < per_sub * C::NSUB; idx += C::NCT) {
                        const int sub = idx / per_sub;
                        const int rem = idx % per_sub;
                        *reinterpret_cast<uint4*>(smem + (sV - sb) + sub * C::SUB_BYTES +
                                                  (nvalid + rem / 8) * 128 + (rem % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                c.qk(sK, t0, sl);
            }
            if (!named_bar_and(1, C::NCT, ok)) break;   // every consumer leaves together
            c.softmax();
            named_bar_sync(1, C::NCT);
            c.pv(sV);
            __syncwarp();
            if (c.lane == 0) mbar_arrive(empty(s));
        }
        c.store(a, w, R, bar);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(&g_decode_error, (int)kErrDecodeWait);
}

template <int D, int MF, bool F16>
__global__ void __launch_bounds__(DCfg<D, MF, false, F16>::NT)
decode_gather_kernel(const DecodeArgs a, int R, int g, int n_rowblk) {
    using C = DCfg<D, MF, false, F16>;
    griddep_launch_dependents();                 // the combine may be scheduled (it waits for this grid)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    Work w;
    if (!work_of<C>(a, R, g, n_rowblk, w)) return;
    const __nv_bfloat16* kc = reinterpret_cast<const __nv_bfloat16*>(a.k_cache);
    const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(a.v_cache);
    const int32_t* trow = a.table + (size_t)w.b * a.max_pages;
    const int tid = threadIdx.x;

    auto load_tile = [&](int tile, int stage) {
        const int t0 = w.t_begin + tile * C::TK;
        const uint32_t sK = sb + C::OFF_KV + stage * 2 * C::KV_TILE;
        const uint32_t sV = sK + C::KV_TILE;
        constexpr int CH = C::NSUB * 8;
        for (int idx = tid; idx < C::TK * CH; idx += C::NT) {
            const int tok = idx / CH, ch = idx % CH;
            const int t = t0 + tok;
            const uint32_t off = sw_off(tok, ch, C::SUB_BYTES);
            const int page = t < w.t_end ? trow[t / a.page_size] : -1;
            // A page id outside the pool (a caller error) is read as zeros, never dereferenced.
            if (page >= 0 && page < a.num_pages) {
                const size_t e = (((size_t)page * a.page_size + t % a.page_size) * a.Hkv + w.hkv) * D + ch * 8;
                cp_async16(sK + off, kc + e, 16);
                cp_async16(sV + off, vc + e, 16);
            } else {
                cp_async16(sK + off, kc, 0);    // zero-fill: value rows past the end stay 0
                cp_async16(sV + off, vc, 0);
            }
        }
    };

    Consumer<C> c;
    c.init(smem, sb, a, w, g);
    auto bar = [] { __syncthreads(); };
    c.load_q(a, w, g, bar);
#pragma unroll
    for (int s = 0; s < C::NS - 1; ++s) {
        if (s < w.n_tiles) load_tile(s, s);
        cp_async_commit();
    }
    const float sl = a.scale_log2;
    for (int it = 0; it < w.n_tiles; ++it) {
        cp_async_wait<C::NS - 2>();
        __syncthreads();
        {
            const int nt = it + C::NS - 1;
            if (nt < w.n_tiles) load_tile(nt, nt % C::NS);
            cp_async_commit();
        }
        const int s = it % C::NS;
        const uint32_t sK = sb + C::OFF_KV + s * 2 * C::KV_TILE;
        c.qk(sK, w.t_begin + it * C::TK, sl);
        __syncthreads();
        c.softmax();
        __syncthreads();
        c.pv(sK + C::KV_TILE);
    }
    cp_async_wait<0>();
    c.store(a, w, R, bar);
}

// ---------------------------------------------------------------------------
// float8_e4m3fn caches (TileOPs "Attention Operators", GQADenseFwdOp stage 2:
// K^ = K * k_scale and V' = V * v_scale, one scale per request and KV head).
// One CTA per (split, KV head, request, row block), as in the 16-bit split
// path.  The producer brings the cache bytes in with TMA (128-byte rows,
// 128-byte swizzle).  Each consumer warp owns one 16-row fragment and a fixed
// share of every key tile (16 or 32 keys) and keeps its own online softmax
// over those keys, with scores, P and O in its registers: no barrier joins the
// warps while the tiles stream, and the warps sharing a fragment merge their
// (max, sum, O) once, through shared memory, after the last tile.  K and V
// fragments come straight from the e4m3 tiles by ldmatrix (two e4m3 per
// 16-bit element) and are widened to float16 in registers (exact: every e4m3fn
// value is a float16); the MMAs run in float16 with FP32 accumulation.  Q is
// rounded to float16 once (a bfloat16 Q keeps every bit for magnitudes in
// [2^-14, 65504]) and P is packed to float16; k_scale joins the softmax scale
// and the softcap's input, v_scale the stored partial O.
//   S = Q K^T: ldmatrix gives lane t four consecutive dims 4(t%4)..4(t%4)+3 of
//     a key in each 16-dim k-step; the first two serve as k = 2(t%4), 2(t%4)+1
//     of the m16n8k16 fragment and the last two as k = 2(t%4)+8, +9, and Q's
//     fragments are loaded under the same map, so every dot product is the
//     same sum in another order.
//   P: the score accumulators of key blocks 2j and 2j+1 are the A fragment of
//     P V's k-step j, packed in place.
//   O += P V: ldmatrix.trans gives lane t, for keys 2(t%4) and 2(t%4)+1, the
//     two dims 2(t/4), 2(t/4)+1 of a 16-dim chunk; a byte permute splits them
//     into an even-dim and an odd-dim n8 block, and the stored O interleaves
//     the two blocks back into dim order.
// SW: the swapped form for at most 8 query rows per KV head (one fragment):
// the keys and dims take the MMAs' M side and the rows their N = 8 side
// (fp8_swap_consumer).
template <int D, int MF, bool SW = false>
struct F8Cfg {
    static_assert(!SW || MF == 1, "the swapped form holds one block of 8 rows");
    static constexpr int TK = key_tile(D);                  // keys per tile (64, or 32 at D = 256)
    static constexpr int ROWS = SW ? 8 : 16 * MF;           // padded rows per CTA
    static constexpr int RW = SW ? 8 : 16;                  // rows of a warp's merge block
    static constexpr int KSPLIT = MF == 1 ? TK / 16 : TK / 32;   // warps per fragment, splitting each tile
    static constexpr int KPW = TK / KSPLIT;                 // keys of a tile per warp (16 or 32)
    static constexpr int NC = MF * KSPLIT;                  // consumer warps
    static constexpr int NCT = NC * 32;
    static constexpr int NT = NCT + 32;                     // + producer warp
    static constexpr int SUB8 = TK * 128;                   // 128 e4m3 columns of a tile
    static constexpr int NSUB8 = D / 128;
    static constexpr int TILE8 = NSUB8 * SUB8;              // one K or V tile of bytes
    static constexpr int KSTEPS = D / 16;
    static constexpr int NFK = KPW / 8;                     // key blocks of a warp's S
    static constexpr int NFD = D / 8;                       // dim blocks of O
    static constexpr int MROW = D + 4;                      // merge row: O, max, sum (16-byte rows)
    static constexpr int MERGE = KSPLIT > 1 ? NC * RW * MROW * 4 : 0;
    // byte ring: up to three CTAs per SM by shared memory at D = 128 with one
    // or two fragments, four in the swapped form (more bytes in flight per SM:
    // 4 x 3 stages measured 2.5 % faster than 3 x 4; 5 x 2 spilled)
    static constexpr int BUDGET = SW ? 56 * 1024 : (D == 128 && MF <= 2) ? 75 * 1024 : 113 * 1024;
    static constexpr int NS_FIT = (BUDGET - 2048) / (2 * TILE8);
    static constexpr int NS = NS_FIT < 6 ? NS_FIT : 6;
    static constexpr int RING = NS * 2 * TILE8;
    // CTAs per SM the registers must allow (the swapped form's accumulators
    // are half as large)
    static constexpr int MINB = SW ? 4 : (D == 128 && MF == 1) ? 2 : 1;
    static constexpr int OFF_KV = 0;                        // byte ring; the merge reuses it
    static constexpr int OFF_BAR = RING > MERGE ? RING : MERGE;   // full[NS], empty[NS]
    static constexpr int OFF_FLAG = OFF_BAR + 2 * NS * 8;
    static constexpr int SMEM = OFF_FLAG + 16 + 1024;
    static_assert(D == 128 || D == 256, "e4m3 rows of 128 or 256 bytes");
    static_assert(KPW % 16 == 0 && NFK % 2 == 0, "whole P V k-steps per warp");
    static_assert((MROW * 4) % 16 == 0, "float4 rows in the merge area");
    static_assert(NS >= 2 && SMEM <= 227 * 1024, "pipeline depth / shared memory budget");
};

// A bfloat16 pair -> a float16 pair (round to nearest even).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    const __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte offset of 16-byte chunk c (16 dims) of key row r in an e4m3 tile.
template <int SUB8>
__device__ __forceinline__ uint32_t off8(int r, int c) {
    return (uint32_t)((c >> 3) * SUB8 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// movmatrix: the transpose of an 8x8 matrix of 16-bit elements held one
// register per lane (lane l: row l / 4, columns 2 (l % 4), +1), same layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Consumer warps of the swapped form (at most 8 query rows per KV head, a
// whole row block per CTA).  With 4 rows, S = Q K^T and O += P V as m16n8k16
// MMAs with the rows on M would use 4 of 16 rows; here the transposes are
// computed instead, the keys (S) and the dims (O) on M and the rows on N = 8:
//   S^T = K Q^T: A = 16 keys x 16 dims of the e4m3 tile (ldmatrix, the four
//     bytes a lane receives widened as the k = 2t, 2t+1 and 2t+8, 2t+9 pairs,
//     t = lane % 4), B = Q^T under the same map of dims (a permutation of the
//     summation order); lane l holds keys l / 4 and l / 4 + 8 of rows 2t, 2t+1.
//   The online softmax runs per row over the keys of the warp's share: the
//     row max across the eight lanes of one t (shuffles), the lazy reference
//     max as elsewhere, each lane's partial row sums kept apart until the end.
//   O^T += V^T P^T: P^T (B, keys on k, rows on n) is the S^T accumulator
//     packed to float16 and transposed in registers (movmatrix); V^T (A) comes
//     from ldmatrix.trans of the value tile, whose 16-bit elements are dim
//     pairs: a byte permute splits them so that M row g takes dim 2g and row
//     g + 8 dim 2g + 1 of each 16-dim chunk.
// The warps of a CTA split each key tile and merge their (max, sum, O) once,
// as in the unswapped form.  Half the MMAs, and O takes 4 D / 16 registers.
template <int D, bool QBF, class C>
__device__ __forceinline__ void fp8_swap_consumer(const DecodeArgs& a, const Work& w, uint8_t* smem, uint32_t sb,
                                                  uint32_t bar0, volatile int* abort_flag, int warp, int lane, int R,
                                                  int g) {
    static_assert(C::KSPLIT > 1 && C::KPW == 16 && C::ROWS == 8 && C::NFD == D / 8,
                  "16 keys of each tile per warp, 8 rows, D / 16 accumulators of two dim blocks each");
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (C::NS + s); };
    const int wk = warp;                           // share of each key tile
    const int kw0 = wk * C::KPW;                   // this warp's first key of a tile
    const int gq = lane >> 2, t4 = lane & 3;
    const int kv = w.b * a.Hkv + w.hkv;
    const float ks = a.k_scale ? a.k_scale[kv] : 1.f;
    const float vs = a.v_scale ? a.v_scale[kv] : 1.f;
    const float sl = a.scale_log2 * ks;
    const float cap_in = a.x.cap_in * ks, cap_out = a.x.cap_out;
    // Q^T fragments: row gq of the block (zero past it), dims 16 kk + 4t .. +3
    uint32_t qf[C::KSTEPS][2];
    {
        const int r = w.row0 + gq;
        const bool valid = gq < w.rows_here;
        const uint16_t* qrow = reinterpret_cast<const uint16_t*>(a.q) +
                               (((size_t)w.qrow0 + r / g) * a.Hq + w.hkv * g + r % g) * D;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            uint2 v = make_uint2(0u, 0u);
            if (valid) v = *reinterpret_cast<const uint2*>(qrow + 16 * kk + 4 * t4);
            qf[kk][0] = QBF ? bf16x2_to_f16x2(v.x) : v.x;          // k = 2t, 2t+1
            qf[kk][1] = QBF ? bf16x2_to_f16x2(v.y) : v.y;          // k = 2t+8, 2t+9
        }
    }
    // rows 2t and 2t + 1 of the accumulators: key range [lo, lim)
    int lim[2], lo[2];
    int lim_min = INT_MAX, lo_max = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int rl = 2 * t4 + h;
        lo[h] = 0;
        lim[h] = -1;
        if (rl < w.rows_here) {
            // keys [lo, lim) of query r / g at key position p (TileOPs
            // GQAPagedFwdOp: causal j <= p, window p - wL <= j <= p + wR)
            const long p = (long)((w.row0 + rl) / g) + w.L - a.Sq;
            long hi = w.t_end;
            if (a.causal) hi = min(hi, p + 1);
            if (a.x.wr >= 0) hi = min(hi, p + a.x.wr + 1);
            lim[h] = (int)max(-1L, hi);
            if (a.x.wl >= 0) lo[h] = (int)max(0L, min((long)w.L, p - a.x.wl));
            lim_min = min(lim_min, lim[h]);
            lo_max = max(lo_max, lo[h]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lim_min = min(lim_min, __shfl_xor_sync(0xffffffffu, lim_min, o));
        lo_max = max(lo_max, __shfl_xor_sync(0xffffffffu, lo_max, o));
    }
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float acc[D / 16][4];                          // O^T: dims 16c + 2gq (+1), rows 2t, 2t+1
#pragma unroll
    for (int c = 0; c < D / 16; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
    const int m = lane >> 3;                       // ldmatrix: this lane addresses matrix m
    for (int it = 0; it < w.n_tiles; ++it) {
        const int s = it % C::NS;
        const int t0 = w.t_begin + it * C::TK;
        const uint32_t sK = sb + C::OFF_KV + s * 2 * C::TILE8;
        const uint32_t sV = sK + C::TILE8;
        if (!__all_sync(0xffffffffu, mbar_wait(full(s), (it / C::NS) & 1, abort_flag))) break;
        const int nvalid = w.t_end - t0;
        if (nvalid < kw0 + C::KPW) {
            // This warp's value rows past the request's end hold stale bytes:
            // zero them (no other warp reads them).
            const int r0 = nvalid > kw0 ? nvalid : kw0;
            const int per_sub = (kw0 + C::KPW - r0) * 8;
            for (int idx = lane; idx < per_sub * C::NSUB8; idx += 32)
                *reinterpret_cast<uint4*>(smem + (sV - sb) + (idx / per_sub) * C::SUB8 +
                                          (r0 + (idx % per_sub) / 8) * 128 + (idx % 8) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
            __syncwarp();
        }
        // ---- S^T = K Q^T over this warp's 16 keys (two accumulation chains)
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sz[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; kk += 2) {
            // matrices: (keys 0-7, chunk kk), (keys 8-15, kk), (keys 0-7, kk+1), (keys 8-15, kk+1)
            uint32_t r[4];
            ldsm_x4(sK + off8<C::SUB8>(kw0 + (m & 1) * 8 + (lane & 7), kk + (m >> 1)), r[0], r[1], r[2], r[3]);
            uint32_t a0[4], a1[4];
            e4m3x4_to_f16x4(r[0], a0[0], a0[2]);
            e4m3x4_to_f16x4(r[1], a0[1], a0[3]);
            e4m3x4_to_f16x4(r[2], a1[0], a1[2]);
            e4m3x4_to_f16x4(r[3], a1[1], a1[3]);
            mma16816<true>(sa, a0, qf[kk][0], qf[kk][1]);
            mma16816<true>(sz, a1, qf[kk + 1][0], qf[kk + 1][1]);
        }
        // element e: key gq + 8 (e >> 1) of the warp's share, row 2t + (e & 1)
        float sc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = sa[e] + sz[e];
        float mx[2] = {-INFINITY, -INFINITY};
        const bool unmasked = t0 + kw0 + C::KPW <= lim_min && t0 + kw0 >= lo_max && cap_out == 0.f;
        if (unmasked) {                             // every key of this warp's share is visible
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sc[e] *= sl;
                mx[e & 1] = fmaxf(mx[e & 1], sc[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = e & 1;
                const int t = t0 + kw0 + gq + 8 * (e >> 1);
                float x = cap_out != 0.f ? softcap_log2(sc[e], cap_in, cap_out) : sc[e] * sl;
                x = t >= lo[h] && t < lim[h] ? x : -INFINITY;       // the select drops stale keys
                sc[e] = x;
                mx[h] = fmaxf(mx[h], x);
            }
        }
        // Lazy rescale, as in the unswapped form (P stays below 2^8)
        float alpha[2], m_use[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 4));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 8));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 16));
            alpha[h] = 1.f;
            if (mx[h] > m_run[h] + 8.f) {
                alpha[h] = fast_exp2(m_run[h] - mx[h]);             // 0 while m_run is -inf
                m_run[h] = mx[h];
            }
            m_use[h] = m_run[h] == -INFINITY ? 0.f : m_run[h];      // no -inf - -inf
        }
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pv[e] = fast_exp2(sc[e] - m_use[e & 1]);
#pragma unroll
        for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * alpha[h] + (pv[h] + pv[h + 2]);
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                acc[c][0] *= alpha[0]; acc[c][1] *= alpha[1];
                acc[c][2] *= alpha[0]; acc[c][3] *= alpha[1];
            }
        }
        // P^T as the B fragments: keys 2t, 2t+1 (and + 8) of row gq
        const uint32_t pb0 = movmatrix_t(pack2<true>(pv[0], pv[1]));
        const uint32_t pb1 = movmatrix_t(pack2<true>(pv[2], pv[3]));
        // ---- O^T += V^T P^T, two 16-dim chunks per ldmatrix
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
            // matrices: (keys 0-7, chunk 2q), (keys 8-15, 2q), (keys 0-7, 2q+1), (keys 8-15, 2q+1)
            uint32_t r[4];
            ldsm_x4_t(sV + off8<C::SUB8>(kw0 + (m & 1) * 8 + (lane & 7), 2 * q + (m >> 1)), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                // bytes of r: V[k0][d], V[k0][d+1], V[k1][d], V[k1][d+1] (k0 = 2t, d = 2gq)
                uint32_t av[4];
                e4m3x4_dim_split(r[2 * i], av[0], av[1]);
                e4m3x4_dim_split(r[2 * i + 1], av[2], av[3]);
                mma16816<true>(acc[2 * q + i], av, pb0, pb1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));      // this warp is done with the stage
    }
    // ---- merge the warps and store the split's partial O (FP32, normalised) and base-2 LSE
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 4);
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 8);
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 16);
    }
    const size_t part_row0 = ((size_t)(w.b * a.Hkv + w.hkv) * a.max_splits + w.split) * R + w.row0;
    named_bar_sync(1, C::NCT);                     // every consumer warp is done with the ring
    float* mg = reinterpret_cast<float*>(smem + C::OFF_KV);
    float* mine = mg + (size_t)warp * C::RW * C::MROW;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float* row = mine + (2 * t4 + h) * C::MROW;
#pragma unroll
        for (int c = 0; c < D / 16; ++c)
            *reinterpret_cast<float2*>(row + 16 * c + 2 * gq) = make_float2(acc[c][h], acc[c][2 + h]);
        if (gq == 0) {
            row[D] = m_run[h];
            row[D + 1] = l_run[h];
        }
    }
    named_bar_sync(1, C::NCT);
    // warp wk merges dims [wk * D / KSPLIT, (wk + 1) * D / KSPLIT)
    constexpr int DW = D / C::KSPLIT;
    for (int rr = 0; rr < w.rows_here; ++rr) {
        float M = -INFINITY;
#pragma unroll
        for (int u = 0; u < C::KSPLIT; ++u) M = fmaxf(M, mg[(u * C::RW + rr) * C::MROW + D]);
        const float M_use = M == -INFINITY ? 0.f : M;
        float wgt[C::KSPLIT], L = 0.f;
#pragma unroll
        for (int u = 0; u < C::KSPLIT; ++u) {
            wgt[u] = fast_exp2(mg[(u * C::RW + rr) * C::MROW + D] - M_use);
            L += wgt[u] * mg[(u * C::RW + rr) * C::MROW + D + 1];
        }
        const float inv = L > 0.f ? vs / L : 0.f;
        for (int d = wk * DW + lane; d < (wk + 1) * DW; d += 32) {
            float o = 0.f;
#pragma unroll
            for (int u = 0; u < C::KSPLIT; ++u) o += wgt[u] * mg[(u * C::RW + rr) * C::MROW + d];
            a.part_o[(part_row0 + rr) * D + d] = o * inv;
        }
        if (wk == 0 && lane == 0) a.part_lse[part_row0 + rr] = L > 0.f ? M + log2f(L) : -INFINITY;
    }
}

template <int D, int MF, bool QBF, bool SW>
__global__ void __launch_bounds__(F8Cfg<D, MF, SW>::NT, F8Cfg<D, MF, SW>::MINB)
decode_fp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeArgs a, int R, int g, int n_rowblk, int box_tokens) {
    using C = F8Cfg<D, MF, SW>;
    griddep_launch_dependents();                 // the combine may be scheduled (it waits for this grid)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    Work w;
    if (!work_of<C>(a, R, g, n_rowblk, w)) return;

    const uint32_t bar0 = sb + C::OFF_BAR;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (C::NS + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), C::NC);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (warp == C::NC && box_tokens == 0) {
        // ------------------------------------------------------------ gather producer
        // Page sizes the byte boxes cannot tile: all 32 lanes copy each tile's
        // e4m3 rows with 16-byte cp.async into the same swizzled layout (rows
        // past the split's end are left to the consumers, a page id outside
        // the pool reads as zeros).  A slot's full barrier takes lane 0's
        // arrival once the slot's copies have landed; one slot stays in flight.
        const int32_t* trow = a.table + (size_t)w.b * a.max_pages;
        const uint8_t* kc = static_cast<const uint8_t*>(a.k_cache);
        const uint8_t* vc = static_cast<const uint8_t*>(a.v_cache);
        constexpr int CPR = D / 16;                 // 16-byte chunks per row
        int pend = -1;                              // slot whose copies are in flight
        bool good = true;
        for (int it = 0; it < w.n_tiles; ++it) {
            const int s = it % C::NS;
            if (lane == 0) good = mbar_wait(empty(s), ((it / C::NS) & 1) ^ 1, abort_flag);
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) break;
            const int t0 = w.t_begin + it * C::TK;
            const uint32_t sK = sb + C::OFF_KV + s * 2 * C::TILE8;
            const uint32_t sV = sK + C::TILE8;
            for (int idx = lane; idx < C::TK * CPR; idx += 32) {
                const int r = idx / CPR, c = idx % CPR;
                const int t = t0 + r;
                if (t >= w.t_end) continue;
                const int page = trow[t / a.page_size];
                const bool in_pool = page >= 0 && page < a.num_pages;
                const long row = in_pool ? (long)page * a.page_size + t % a.page_size : 0;
                const size_t src = ((size_t)row * a.Hkv + w.hkv) * D + c * 16;
                const uint32_t off = off8<C::SUB8>(r, c);
                cp_async16(sK + off, kc + src, in_pool ? 16u : 0u);
                cp_async16(sV + off, vc + src, in_pool ? 16u : 0u);
            }
            cp_async_commit();
            if (pend >= 0) {
                cp_async_wait<1>();
                __syncwarp();
                if (lane == 0) mbar_arrive(full(pend));
            }
            pend = s;
        }
        cp_async_wait<0>();                         // no copy outlives the CTA
        __syncwarp();
        if (good && pend >= 0 && lane == 0) mbar_arrive(full(pend));
    } else if (warp == C::NC) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const int32_t* trow = a.table + (size_t)w.b * a.max_pages;
            const int nbox = C::TK / box_tokens;
            const uint32_t box_bytes = (uint32_t)box_tokens * 128;
            int issued = 0;
            for (int it = 0; it < w.n_tiles; ++it) {
                const int s = it % C::NS;
                if (!mbar_wait(empty(s), ((it / C::NS) & 1) ^ 1, abort_flag)) break;
                const int t0 = w.t_begin + it * C::TK;
                int rows[8];        // first cache row of each box, or -1
                int n = 0;
                for (int i = 0; i < nbox; ++i) {
                    const int t = t0 + i * box_tokens;
                    int row = -1;
                    if (t < w.t_end) {
                        const int page = trow[t / a.page_size];
                        // a page id outside the pool (a caller error) is not loaded
                        if (page >= 0 && page < a.num_pages) row = page * a.page_size + t % a.page_size;
                    }
                    rows[i] = row;
                    n += row >= 0;
                }
                mbar_arrive_expect_tx(full(s), (uint32_t)n * box_bytes * C::NSUB8 * 2);
                const uint32_t sK = sb + C::OFF_KV + s * 2 * C::TILE8;
                const uint32_t sV = sK + C::TILE8;
                for (int i = 0; i < nbox; ++i) {
                    if (rows[i] < 0) continue;
#pragma unroll
                    for (int sub = 0; sub < C::NSUB8; ++sub) {
                        const uint32_t off = sub * C::SUB8 + i * box_tokens * 128;
                        tma_load_3d(sK + off, &tm_k, full(s), sub * 128, w.hkv, rows[i]);
                        tma_load_3d(sV + off, &tm_v, full(s), sub * 128, w.hkv, rows[i]);
                    }
                }
                issued = it + 1;
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA goes away
                for (int it = issued - C::NS > 0 ? issued - C::NS : 0; it < issued; ++it)
                    mbar_drain(full(it % C::NS), (it / C::NS) & 1);
            }
        }
    } else if constexpr (SW) {
        // ------------------------------------------------------------ consumer warps (swapped form)
        fp8_swap_consumer<D, QBF, C>(a, w, smem, sb, bar0, abort_flag, warp, lane, R, g);
    } else {
        // ------------------------------------------------------------ consumer warps
        const int mf = warp / C::KSPLIT;            // row fragment
        const int wk = warp % C::KSPLIT;            // share of each key tile
        const int kw0 = wk * C::KPW;                // this warp's first key of a tile
        const int t4 = lane & 3;
        const int kv = w.b * a.Hkv + w.hkv;
        const float ks = a.k_scale ? a.k_scale[kv] : 1.f;
        const float vs = a.v_scale ? a.v_scale[kv] : 1.f;
        const float sl = a.scale_log2 * ks;
        const float cap_in = a.x.cap_in * ks, cap_out = a.x.cap_out;
        // rows g and g + 8 of the fragment: key range [lo, lim) and Q fragments
        int lim[2], lo[2];
        uint32_t qf[C::KSTEPS][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int rl = mf * 16 + (lane >> 2) + 8 * h;
            const int r = w.row0 + rl;
            const bool valid = rl < w.rows_here;
            lo[h] = 0;
            lim[h] = -1;
            if (valid) {
                // keys [lo, lim) of query r / g at key position p (TileOPs
                // GQAPagedFwdOp: causal j <= p, window p - wL <= j <= p + wR)
                const long p = (long)(r / g) + w.L - a.Sq;
                long hi = w.t_end;
                if (a.causal) hi = min(hi, p + 1);
                if (a.x.wr >= 0) hi = min(hi, p + a.x.wr + 1);
                lim[h] = (int)max(-1L, hi);
                if (a.x.wl >= 0) lo[h] = (int)max(0L, min((long)w.L, p - a.x.wl));
            }
            const uint16_t* qrow = reinterpret_cast<const uint16_t*>(a.q) +
                                   (((size_t)w.qrow0 + r / g) * a.Hq + w.hkv * g + r % g) * D;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
                uint2 v = make_uint2(0u, 0u);
                if (valid) v = *reinterpret_cast<const uint2*>(qrow + 16 * kk + 4 * t4);
                qf[kk][h] = QBF ? bf16x2_to_f16x2(v.x) : v.x;          // k = 2(t%4), +1
                qf[kk][2 + h] = QBF ? bf16x2_to_f16x2(v.y) : v.y;      // k = 2(t%4) + 8, +9
            }
        }
        // keys every row of the fragment sees (rows past the block see all: their
        // Q is zero and their results are never stored)
        int lim_min = INT_MAX, lo_max = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (mf * 16 + (lane >> 2) + 8 * h < w.rows_here) {
                lim_min = min(lim_min, lim[h]);
                lo_max = max(lo_max, lo[h]);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lim_min = min(lim_min, __shfl_xor_sync(0xffffffffu, lim_min, o));
            lo_max = max(lo_max, __shfl_xor_sync(0xffffffffu, lo_max, o));
        }
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
        float acc[C::NFD][4];
#pragma unroll
        for (int n = 0; n < C::NFD; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        const int m = lane >> 3;                    // ldmatrix: this lane addresses matrix m
        for (int it = 0; it < w.n_tiles; ++it) {
            const int s = it % C::NS;
            const int t0 = w.t_begin + it * C::TK;
            const uint32_t sK = sb + C::OFF_KV + s * 2 * C::TILE8;
            const uint32_t sV = sK + C::TILE8;
            if (!__all_sync(0xffffffffu, mbar_wait(full(s), (it / C::NS) & 1, abort_flag))) break;
            const int nvalid = w.t_end - t0;
            if (nvalid < kw0 + C::KPW) {
                // This warp's value rows past the request's end hold stale bytes:
                // zero them (no other warp reads them).
                const int r0 = nvalid > kw0 ? nvalid : kw0;
                const int per_sub = (kw0 + C::KPW - r0) * 8;
                for (int idx = lane; idx < per_sub * C::NSUB8; idx += 32)
                    *reinterpret_cast<uint4*>(smem + (sV - sb) + (idx / per_sub) * C::SUB8 +
                                              (r0 + (idx % per_sub) / 8) * 128 + (idx % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- S = Q K^T over this warp's keys of the tile
            float sc[C::NFK][4];
#pragma unroll
            for (int n = 0; n < C::NFK; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; kk += 2) {
#pragma unroll
                for (int nb = 0; nb < C::NFK; nb += 2) {
                    // matrices: (block nb, step kk), (nb, kk+1), (nb+1, kk), (nb+1, kk+1)
                    uint32_t r[4];
                    ldsm_x4(sK + off8<C::SUB8>(kw0 + (nb + (m >> 1)) * 8 + (lane & 7), kk + (m & 1)), r[0], r[1],
                            r[2], r[3]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t b0, b1;
                        e4m3x4_to_f16x4(r[j], b0, b1);
                        mma16816<true>(sc[nb + (j >> 1)], qf[kk + (j & 1)], b0, b1);
                    }
                }
            }
            // ---- scaled, masked logits (log2 units) and the rows' maxima
            float mx[2] = {-INFINITY, -INFINITY};
            const bool unmasked = t0 + kw0 + C::KPW <= lim_min && t0 + kw0 >= lo_max && cap_out == 0.f;
            if (unmasked) {                             // every key of this warp's share is visible
#pragma unroll
                for (int n = 0; n < C::NFK; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        sc[n][e] *= sl;
                        mx[e >> 1] = fmaxf(mx[e >> 1], sc[n][e]);
                    }
            } else {
#pragma unroll
                for (int n = 0; n < C::NFK; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = e >> 1;
                        const int t = t0 + kw0 + 8 * n + 2 * t4 + (e & 1);
                        float x = cap_out != 0.f ? softcap_log2(sc[n][e], cap_in, cap_out) : sc[n][e] * sl;
                        x = t >= lo[h] && t < lim[h] ? x : -INFINITY;       // the select drops stale keys
                        sc[n][e] = x;
                        mx[h] = fmaxf(mx[h], x);
                    }
            }
            // Lazy rescale: the reference max moves only when the tile max exceeds
            // it by more than 2^8 (P stays below 2^8, far inside float16); O and
            // the sum share the reference, so the result is unchanged.
            float alpha[2], m_use[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
                alpha[h] = 1.f;
                if (mx[h] > m_run[h] + 8.f) {
                    alpha[h] = fast_exp2(m_run[h] - mx[h]);         // 0 while m_run is -inf
                    m_run[h] = mx[h];
                }
                m_use[h] = m_run[h] == -INFINITY ? 0.f : m_run[h];  // no -inf - -inf
            }
            // ---- P (float16) as P V's A fragments, this lane's share of the row sums
            uint32_t pa[C::KPW / 16][4];
            float rs[2] = {0.f, 0.f};
#pragma unroll
            for (int j = 0; j < C::KPW / 16; ++j)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const float* x = sc[2 * j + half];
                    const float p0 = fast_exp2(x[0] - m_use[0]), p1 = fast_exp2(x[1] - m_use[0]);
                    const float p2 = fast_exp2(x[2] - m_use[1]), p3 = fast_exp2(x[3] - m_use[1]);
                    rs[0] += p0 + p1;
                    rs[1] += p2 + p3;
                    pa[j][2 * half] = pack2<true>(p0, p1);         // row g, keys 16j + 8 half + 2(t%4), +1
                    pa[j][2 * half + 1] = pack2<true>(p2, p3);     // row g + 8
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * alpha[h] + rs[h];
            if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
                for (int n = 0; n < C::NFD; ++n) {
                    acc[n][0] *= alpha[0]; acc[n][1] *= alpha[0];
                    acc[n][2] *= alpha[1]; acc[n][3] *= alpha[1];
                }
            }
            // ---- O += P V over all dims; acc[4q + 2i + e]: chunk i of the 32-dim
            // group q, dims of parity e
#pragma unroll
            for (int kk = 0; kk < C::KPW / 16; ++kk) {
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    // matrices: (keys 0-7, chunk 2q), (keys 8-15, 2q), (keys 0-7, 2q+1), (keys 8-15, 2q+1)
                    uint32_t r[4];
                    ldsm_x4_t(sV + off8<C::SUB8>(kw0 + kk * 16 + (m & 1) * 8 + (lane & 7), 2 * q + (m >> 1)), r[0],
                              r[1], r[2], r[3]);
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        // bytes: V[k0][d], V[k0][d+1], V[k1][d], V[k1][d+1] (d even)
                        uint32_t e0, o0, e1, o1;
                        e4m3x4_dim_split(r[2 * i], e0, o0);
                        e4m3x4_dim_split(r[2 * i + 1], e1, o1);
                        mma16816<true>(acc[4 * q + 2 * i], pa[kk], e0, e1);
                        mma16816<true>(acc[4 * q + 2 * i + 1], pa[kk], o0, o1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));      // this warp is done with the stage
        }
        // ---- merge the warps of a fragment and store the split's partial O (FP32,
        // dims in order, normalised) and base-2 LSE
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
        }
        const size_t part_row0 = ((size_t)(w.b * a.Hkv + w.hkv) * a.max_splits + w.split) * R + w.row0;
        if constexpr (C::KSPLIT == 1) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rl = mf * 16 + (lane >> 2) + 8 * h;
                if (rl >= w.rows_here) continue;
                const float l = l_run[h];
                const float inv = l > 0.f ? vs / l : 0.f;
                float* dst = a.part_o + (part_row0 + rl) * D + 4 * t4;
#pragma unroll
                for (int q = 0; q < D / 32; ++q)
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const float* ev = acc[4 * q + 2 * i];
                        const float* od = acc[4 * q + 2 * i + 1];
                        *reinterpret_cast<float4*>(dst + 32 * q + 16 * i) =
                            make_float4(ev[2 * h] * inv, od[2 * h] * inv, ev[2 * h + 1] * inv, od[2 * h + 1] * inv);
                    }
                if (t4 == 0) a.part_lse[part_row0 + rl] = l > 0.f ? m_run[h] + log2f(l) : -INFINITY;
            }
        } else {
            named_bar_sync(1, C::NCT);                  // every consumer warp is done with the ring
            float* mg = reinterpret_cast<float*>(smem + C::OFF_KV);
            float* mine = mg + (size_t)warp * 16 * C::MROW;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rr = (lane >> 2) + 8 * h;     // row within the fragment
                float* row = mine + rr * C::MROW;
#pragma unroll
                for (int q = 0; q < D / 32; ++q)
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const float* ev = acc[4 * q + 2 * i];
                        const float* od = acc[4 * q + 2 * i + 1];
                        *reinterpret_cast<float4*>(row + 32 * q + 16 * i + 4 * t4) =
                            make_float4(ev[2 * h], od[2 * h], ev[2 * h + 1], od[2 * h + 1]);
                    }
                if (t4 == 0) {
                    row[D] = m_run[h];
                    row[D + 1] = l_run[h];
                }
            }
            named_bar_sync(1, C::NCT);
            // warp (mf, wk) merges dims [wk * D / KSPLIT, (wk + 1) * D / KSPLIT) of fragment mf
            const float* frag = mg + (size_t)(mf * C::KSPLIT) * 16 * C::MROW;
            constexpr int DW = D / C::KSPLIT;
            for (int rr = 0; rr < 16; ++rr) {
                const int rl = mf * 16 + rr;
                if (rl >= w.rows_here) break;
                float M = -INFINITY;
#pragma unroll
                for (int u = 0; u < C::KSPLIT; ++u) M = fmaxf(M, frag[(u * 16 + rr) * C::MROW + D]);
                const float M_use = M == -INFINITY ? 0.f : M;
                float wgt[C::KSPLIT], L = 0.f;
#pragma unroll
                for (int u = 0; u < C::KSPLIT; ++u) {
                    wgt[u] = fast_exp2(frag[(u * 16 + rr) * C::MROW + D] - M_use);
                    L += wgt[u] * frag[(u * 16 + rr) * C::MROW + D + 1];
                }
                const float inv = L > 0.f ? vs / L : 0.f;
                for (int d = wk * DW + lane; d < (wk + 1) * DW; d += 32) {
                    float o = 0.f;
#pragma unroll
                    for (int u = 0; u < C::KSPLIT; ++u) o += wgt[u] * frag[(u * 16 + rr) * C::MROW + d];
                    a.part_o[(part_row0 + rl) * D + d] = o * inv;
                }
                if (wk == 0 && lane == 0) a.part_lse[part_row0 + rl] = L > 0.f ? M + log2f(L) : -INFINITY;
            }
        }
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(&g_decode_error, (int)kErrDecodeWait);
}

template <int D, bool F16>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeArgs a, int R, int g) {
    // launched as a programmatic dependent of the split kernel: its partials
    // are complete and visible past this point
    griddep_wait();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const long row = (long)blockIdx.x * 4 + warp;
    const long total = (long)a.B * a.Sq * a.Hq;
    if (row >= total) return;
    const int h = (int)(row % a.Hq);
    const int i = (int)((row / a.Hq) % a.Sq);
    const int b = (int)(row / ((long)a.Hq * a.Sq));
    const int hkv = h / g, r = i * g + h % g;
    long orow = row;        // row of o [.., D] and lse
    if (a.q_rows) {
        long qr;
        if (!packed_single(a, b, qr)) return;       // rows of a prefill chunk are not ours
        orow = qr * a.Hq + h;
    }
    const int L = min(max(a.seqlens[b], 0), a.max_pages * a.page_size);
    int n;
    size_t base;
    if (a.seg_table) {
        // balanced path: the segment's pieces have consecutive ids (entries
        // outside the partial slots, possible only after a kernel gave up
        // waiting, read as no pieces)
        const int s = b * a.Hkv + hkv;
        int id0 = 0;
        n = 0;
        if (L > 0) {
            id0 = a.seg_table[2 * s];
            n = a.seg_table[2 * s + 1];
            if (id0 < 0 || n < 0 || (long)id0 + n > a.n_part) id0 = n = 0;
        }
        base = (size_t)id0 * R + r;
    } else {
        n = L > 0 ? (L + a.chunk - 1) / a.chunk : 0;
        base = (size_t)(b * a.Hkv + hkv) * a.max_splits * R + r;
        if (a.x.wl >= 0 && n > 0) {
            // splits wholly left of this row's window were not run
            const long lo = (long)i + L - a.Sq - a.x.wl;
            const int s0 = lo > 0 ? (int)min((long)n, lo / a.chunk) : 0;
            base += (size_t)s0 * R;
            n -= s0;
        }
    }

    float M = -INFINITY;
    for (int s = lane; s < n; s += 32) M = fmaxf(M, a.part_lse[base + (size_t)s * R]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.o) + (size_t)orow * D;
    constexpr int PER = D / 128 > 0 ? D / 128 : 1;     // float4 groups per lane
    // A sink joins the denominator once per row (GQAPagedFwdOp sinks): the
    // weights are taken against max(M, s); +inf zeroes the row.  A row no
    // split saw stays zero with LSE -inf.
    const float s2 = (a.x.sinks && M != -INFINITY) ? a.x.sinks[h] * 1.4426950408889634f : -INFINITY;
    if (s2 == INFINITY) {
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int d = (q * 32 + lane) * 4;
            if (d < D) *reinterpret_cast<uint2*>(out + d) = make_uint2(0u, 0u);
        }
        if (lane == 0 && a.lse) a.lse[orow] = INFINITY;
        return;
    }
    M = fmaxf(M, s2);
    if (M == -INFINITY) {
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int d = (q * 32 + lane) * 4;
            if (d < D) *reinterpret_cast<uint2*>(out + d) = make_uint2(0u, 0u);
        }
        if (lane == 0 && a.lse) a.lse[orow] = -INFINITY;
        return;
    }
    float accv[PER][4] = {};
    float den = s2 == -INFINITY ? 0.f : fast_exp2(s2 - M);
    // four pieces per pass so that their loads are in flight together
#pragma unroll 4
    for (int s = 0; s < n; ++s) {
        const size_t pr = base + (size_t)s * R;
        const float w = fast_exp2(a.part_lse[pr] - M);
        den += w;
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int d = (q * 32 + lane) * 4;
            if (d < D) {
                const float4 v = *reinterpret_cast<const float4*>(a.part_o + pr * D + d);
                accv[q][0] += w * v.x; accv[q][1] += w * v.y; accv[q][2] += w * v.z; accv[q][3] += w * v.w;
            }
        }
    }
    const float inv = 1.f / den;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        const int d = (q * 32 + lane) * 4;
        if (d < D)
            *reinterpret_cast<uint2*>(out + d) =
                make_uint2(pack2<F16>(accv[q][0] * inv, accv[q][1] * inv),
                           pack2<F16>(accv[q][2] * inv, accv[q][3] * inv));
    }
    if (lane == 0 && a.lse) a.lse[orow] = (M + log2f(den)) * kLn2;
}

int choose_mf(int R) {
    const int blocks16 = (R + 15) / 16;
    return blocks16 >= 4 ? 4 : blocks16;
}

template <int D, int MF, bool F16>
cudaError_t launch_split(const DecodeArgs& a, const CUtensorMap* tm_k, const CUtensorMap* tm_v, int box_tokens,
                         int R, int g, int n_rowblk, cudaStream_t stream) {
    dim3 grid(a.max_splits, a.Hkv, a.B * n_rowblk);
    if (tm_k) {
        using C = DCfg<D, MF, true, F16>;
        cudaError_t e = cudaFuncSetAttribute(decode_tma_kernel<D, MF, F16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        decode_tma_kernel<D, MF, F16><<<grid, C::NT, C::SMEM, stream>>>(*tm_k, *tm_v, a, R, g, n_rowblk, box_tokens);
    } else {
        using C = DCfg<D, MF, false, F16>;
        cudaError_t e = cudaFuncSetAttribute(decode_gather_kernel<D, MF, F16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        decode_gather_kernel<D, MF, F16><<<grid, C::NT, C::SMEM, stream>>>(a, R, g, n_rowblk);
    }
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, const CUtensorMap* tm_k, const CUtensorMap* tm_v, int box_tokens,
                     cudaStream_t stream) {
    const int g = a.Hq / a.Hkv;
    const int R = g * a.Sq;
    const int mf = choose_mf(R);
    const int n_rowblk = (R + 16 * mf - 1) / (16 * mf);
    cudaError_t e;
    switch (mf * 2 + (a.f16 ? 1 : 0)) {
        case 2: e = launch_split<D, 1, false>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream); break;
        case 3: e = launch_split<D, 1, true>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream); break;
        case 4: e = launch_split<D, 2, false>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream); break;
        case 5: e = launch_split<D, 2, true>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream); break;
        case 6: e = launch_split<D, 3, false>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream); break;
        case 7: e = launch_split<D, 3, true>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream); break;
        case 8: e = launch_split<D, 4, false>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream); break;
        default: e = launch_split<D, 4, true>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream); break;
    }
    if (e != cudaSuccess) return e;
    return launch_decode_combine(a, stream);
}

}  // namespace

int decode_box_tokens(int D, int page_size) {
    const int tk = key_tile(D);
    const int bt = page_size < tk ? page_size : tk;
    if (bt % 8 != 0 || page_size % bt != 0 || tk % bt != 0) return 0;
    return bt;
}

bool plan_decode(int B, int Sq, int Hq, int Hkv, int D, int page_size, int max_pages, int num_sms,
                 DecodePlan* plan) {
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || page_size <= 0 || max_pages <= 0)
        return false;
    // Splits start on multiples of 64 tokens for every head dimension, so the
    // 64-key tiles of decode_tc_kernel never straddle a page boundary.
    const int TK = 64;
    (void)D;
    const int g = Hq / Hkv;
    const long R = (long)g * Sq;
    const int mf = choose_mf((int)R);
    const long n_rowblk = (R + 16 * mf - 1) / (16 * mf);
    const long cap = (long)max_pages * page_size;
    // The host never reads the lengths: assume half the capacity on average and
    // aim for about four waves of CTAs so ragged lengths even out.
    const int ctas_per_sm = (D == 256 || mf >= 3) ? 1 : 2;
    const long units = (long)B * Hkv * n_rowblk;
    const long target = 4L * (num_sms > 0 ? num_sms : 148) * ctas_per_sm;
    long chunk = (units * ((cap + 1) / 2) + target - 1) / target;
    chunk = (chunk + TK - 1) / TK * TK;
    const long min_chunk = 4 * TK;
    const long cap_r = (cap + TK - 1) / TK * TK;
    if (chunk < min_chunk) chunk = min_chunk;
    if (chunk > cap_r) chunk = cap_r;
    if (chunk > (1L << 30)) return false;
    const long splits = (cap + chunk - 1) / chunk;
    if (splits > 65535 || (long)B * n_rowblk > 65535) return false;
    plan->chunk = (int)chunk;
    plan->max_splits = (int)(splits > 0 ? splits : 1);
    plan->rows = (int)R;
    plan->part_o_bytes = (size_t)B * Hkv * plan->max_splits * R * D * sizeof(float);
    plan->part_lse_bytes = (size_t)B * Hkv * plan->max_splits * R * sizeof(float);
    plan->workspace_bytes = (plan->part_o_bytes + 255) / 256 * 256 + (plan->part_lse_bytes + 255) / 256 * 256;
    // The balanced tensor-core path: one partial per (segment, CTA) piece, at
    // most B * Hkv + grid of them, and a 2-int entry per segment.
    plan->tc = decode_tc_eligible(D, (int)R, page_size) &&
               (long)B * Hkv * ((cap + 63) / 64) < (1L << 31) && (long)B * Hkv + num_sms < (1L << 24);
    if (plan->tc) {
        plan->tc_grid = num_sms > 0 ? num_sms : 148;
        plan->n_part = B * Hkv + plan->tc_grid;
        plan->tc_part_o_bytes = (size_t)plan->n_part * R * D * sizeof(float);
        plan->tc_part_lse_bytes = (size_t)plan->n_part * R * sizeof(float);
        plan->tc_table_bytes = (size_t)B * Hkv * 2 * sizeof(int);
        const size_t tc_bytes = (plan->tc_part_o_bytes + 255) / 256 * 256 +
                                (plan->tc_part_lse_bytes + 255) / 256 * 256 +
                                (plan->tc_table_bytes + 255) / 256 * 256;
        if (tc_bytes > plan->workspace_bytes) plan->workspace_bytes = tc_bytes;
    }
    return true;
}

namespace {
// The combine runs as a programmatic dependent launch of the split kernel:
// its blocks are scheduled while the split kernel finishes (every split kernel
// lets its dependents go at its start) and wait in griddep_wait(), so no launch
// gap separates the two.
template <int D, bool F16>
cudaError_t launch_combine_t(const DecodeArgs& a, int R, int g, unsigned blocks, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, F16>, a, R, g);
}
}  // namespace

cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t stream) {
    const int g = a.Hq / a.Hkv;
    const int R = g * a.Sq;
    const long rows = (long)a.B * a.Sq * a.Hq;
    const unsigned blocks = (unsigned)((rows + 3) / 4);
    switch (a.D * 2 + (a.f16 ? 1 : 0)) {
        case 64 * 2: return launch_combine_t<64, false>(a, R, g, blocks, stream);
        case 64 * 2 + 1: return launch_combine_t<64, true>(a, R, g, blocks, stream);
        case 128 * 2: return launch_combine_t<128, false>(a, R, g, blocks, stream);
        case 128 * 2 + 1: return launch_combine_t<128, true>(a, R, g, blocks, stream);
        case 256 * 2: return launch_combine_t<256, false>(a, R, g, blocks, stream);
        case 256 * 2 + 1: return launch_combine_t<256, true>(a, R, g, blocks, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap* tm_k, const CUtensorMap* tm_v, int box_tokens,
                          cudaStream_t stream) {
    switch (a.D) {
        case 64: return launch_d<64>(a, tm_k, tm_v, box_tokens, stream);
        case 128: return launch_d<128>(a, tm_k, tm_v, box_tokens, stream);
        case 256: return launch_d<256>(a, tm_k, tm_v, box_tokens, stream);
        default: return cudaErrorInvalidValue;
    }
}

namespace {
template <int D, int MF, bool QBF, bool SW = false>
cudaError_t launch_fp8_t(const DecodeArgs& a, const CUtensorMap& tm_k, const CUtensorMap& tm_v, int box_tokens,
                         int R, int g, int n_rowblk, cudaStream_t stream) {
    using C = F8Cfg<D, MF, SW>;
    cudaError_t e = cudaFuncSetAttribute(decode_fp8_kernel<D, MF, QBF, SW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid(a.max_splits, a.Hkv, a.B * n_rowblk);
    decode_fp8_kernel<D, MF, QBF, SW><<<grid, C::NT, C::SMEM, stream>>>(tm_k, tm_v, a, R, g, n_rowblk, box_tokens);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_fp8_d(const DecodeArgs& a, const CUtensorMap& tm_k, const CUtensorMap& tm_v, int box_tokens,
                         int R, int g, cudaStream_t stream) {
    const bool qbf = !a.f16;
    if (R <= 8) {
        // at most 8 rows per KV head: the swapped form (rows on the MMAs' N side)
        return qbf ? launch_fp8_t<D, 1, true, true>(a, tm_k, tm_v, box_tokens, R, g, 1, stream)
                   : launch_fp8_t<D, 1, false, true>(a, tm_k, tm_v, box_tokens, R, g, 1, stream);
    }
    const int mf = choose_mf(R);
    const int n_rowblk = (R + 16 * mf - 1) / (16 * mf);
    switch (mf * 2 + (qbf ? 1 : 0)) {
        case 2: return launch_fp8_t<D, 1, false>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream);
        case 3: return launch_fp8_t<D, 1, true>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream);
        case 4: return launch_fp8_t<D, 2, false>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream);
        case 5: return launch_fp8_t<D, 2, true>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream);
        case 6: return launch_fp8_t<D, 3, false>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream);
        case 7: return launch_fp8_t<D, 3, true>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream);
        case 8: return launch_fp8_t<D, 4, false>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream);
        default: return launch_fp8_t<D, 4, true>(a, tm_k, tm_v, box_tokens, R, g, n_rowblk, stream);
    }
}
}  // namespace

cudaError_t launch_decode_fp8(const DecodeArgs& a, const CUtensorMap& tm_k, const CUtensorMap& tm_v, int box_tokens,
                              cudaStream_t stream) {
    const int g = a.Hq / a.Hkv;
    const int R = g * a.Sq;
    cudaError_t e;
    switch (a.D) {
        case 128: e = launch_fp8_d<128>(a, tm_k, tm_v, box_tokens, R, g, stream); break;
        case 256: e = launch_fp8_d<256>(a, tm_k, tm_v, box_tokens, R, g, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    return launch_decode_combine(a, stream);
}

int decode_take_device_error() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(int)) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace gqa

// ---------------------------------------------------------------------------
// Paged decode for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: a serving
// engine whose device memory is entirely pre-reserved by its own pool, a
// plugin loaded into a host framework that forbids allocation while it
// executes, or a latency-critical loop that cannot pay for cudaMalloc's
// implicit synchronisation.  For them attn_decode_paged_noalloc keeps the
// split-KV partials in the fixed array below instead of a caller workspace.
//
// The array lives in this library's device image: every GPU that loads the
// library holds kStaticScratchBytes of it until the process exits.  Its
// device address is looked up once per device (the first call on a device,
// with that device current) and cached.  Every call shares the array and it
// keeps whatever the last call wrote; nothing in it needs to start at zero,
// because each call writes every partial it later reads.  Two calls whose
// kernels overlap on the GPU (for example on two streams) race on it.
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;   // 32 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_scratch_mu;
void* g_static_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_static_scratch on the current device, or nullptr.
void* static_scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    if (!g_static_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
        g_static_scratch_ptr[dev] = p;
    }
    return g_static_scratch_ptr[dev];
}

}  // namespace

extern "C" size_t attn_decode_paged_noalloc_max_workspace(void) { return kStaticScratchBytes; }

extern "C" gqa_status attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                const int32_t* real_seqlen_kv, const int32_t* block_table,
                                                int page_size, void* o, float* lse, int B, int Sq, int Hq, int Hkv,
                                                int D, int num_pages, int max_pages, int causal, float scale,
                                                gqa_stream_t stream) {
    void* scratch = static_scratch_address();
    if (!scratch) return GQA_ERR_CUDA;
    // Sizes whose partials exceed the array are refused with GQA_ERR_WORKSPACE
    // by the same check attn_decode_paged applies to a caller workspace.
    return attn_decode_paged(q, k_cache, v_cache, real_seqlen_kv, block_table, page_size, o, lse, B, Sq, Hq, Hkv,
                             D, num_pages, max_pages, causal, scale, scratch, kStaticScratchBytes, stream);
}
