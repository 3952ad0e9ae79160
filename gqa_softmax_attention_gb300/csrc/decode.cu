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
// decode_split_kernel: one CTA per (split, KV head, request, row block).  All
//   g * Sq query rows that read this KV head are packed into the M dimension
//   of m16n8k16 tensor-core MMAs (rows padded to 16 * MF).  Key/value rows of
//   64 tokens are gathered page by page with 16-byte cp.async copies (each
//   token row is D * 2 contiguous bytes) into a multi-stage shared-memory ring;
//   slots past the request's length are zero-filled, never read.  Warps split
//   the keys of a tile for S = Q K^T (each warp keeps its rows of Q in
//   registers), rows are softmaxed by thread groups in shared memory, and the
//   warps split the head dimension for O += P V.  Each split writes its
//   normalised FP32 partial O and its base-2 LSE to the workspace.
// decode_combine_kernel: one warp per output row; weights exp(lse_s - max),
//   normalised; a row no split saw gets O = 0 and LSE = -inf.
//
// This path is bound by HBM bandwidth; the MMAs are small and hidden under the
// gathers, so warp-level mma.sync is used rather than tcgen05.
#include <cmath>
#include <mutex>

#include "gqa_attn.h"
#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int TK = 64;   // tokens per key tile
constexpr float kLn2 = 0.693147180559945309f;

template <int D, int MF>
struct DCfg {
    static constexpr int KSPLIT = MF == 1 ? 4 : 2;           // warps per 16-row fragment
    static constexpr int NWARPS = MF * KSPLIT;
    static constexpr int NT = NWARPS * 32;
    static constexpr int ROWS = 16 * MF;                     // padded rows per CTA
    static constexpr int ROW_BYTES = D * 2;                  // one token's K (or V) row
    static constexpr int CHUNKS = D / 8;                     // 16-byte chunks per row
    static constexpr int NS = D == 64 ? 4 : (D == 128 ? 3 : 2);
    static constexpr int KV_TILE = TK * ROW_BYTES;
    static constexpr int KEYS_PER_WARP = TK / KSPLIT;
    static constexpr int NFK = KEYS_PER_WARP / 8;            // n8 fragments per warp in S = Q K^T
    static constexpr int DSL = D / KSPLIT;                   // head-dim slice per warp in O += P V
    static constexpr int NFD = DSL / 8;
    static constexpr int KSTEPS = D / 16;
    static constexpr int S_STRIDE = TK + 4;                  // floats per score row in smem
    static constexpr int TPR = NT / ROWS;                    // threads per row in the softmax
    static constexpr int KPT = TK / TPR;                     // keys per thread in the softmax
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + ROWS * ROW_BYTES;
    static constexpr int OFF_V = OFF_K + NS * KV_TILE;
    static constexpr int OFF_S = OFF_V + NS * KV_TILE;
    static constexpr int OFF_P = OFF_S + ROWS * S_STRIDE * 4;
    static constexpr int OFF_A = OFF_P + ROWS * TK * 2;
    static constexpr int OFF_L = OFF_A + ROWS * 4;
    static constexpr int OFF_M = OFF_L + ROWS * 4;
    static constexpr int SMEM = OFF_M + ROWS * 4;
    static_assert(NFK % 2 == 0 && NFD % 2 == 0, "fragments are loaded in pairs");
    static_assert(KPT % 8 == 0, "softmax writes whole 16-byte chunks of P");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

template <int D, int MF>
__global__ void __launch_bounds__(DCfg<D, MF>::NT)
decode_split_kernel(const DecodeArgs a, int R, int g, int n_rowblk) {
    using C = DCfg<D, MF>;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int split = blockIdx.x;
    const int hkv = blockIdx.y;
    const int b = blockIdx.z / n_rowblk;
    const int rb = blockIdx.z % n_rowblk;
    // Lengths are clamped to the table's capacity so a bad length cannot send
    // the gather past block_table.
    const int L = min(max(a.seqlens[b], 0), a.max_pages * a.page_size);
    const int t_begin = split * a.chunk;
    if (t_begin >= L) return;                      // nothing here; the combine skips it
    const int t_end = min(L, t_begin + a.chunk);
    const int n_tiles = (t_end - t_begin + TK - 1) / TK;
    const int row0 = rb * C::ROWS;
    const int rows_here = min(C::ROWS, R - row0);

    const int tid = threadIdx.x;
    const int warp = tid / 32;
    const int lane = tid % 32;
    const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* kc = reinterpret_cast<const __nv_bfloat16*>(a.k_cache);
    const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(a.v_cache);
    const int32_t* trow = a.table + (size_t)b * a.max_pages;

    // Q rows r = i * g + hl (query i, head hkv * g + hl); padded rows are zero.
    for (int idx = tid; idx < C::ROWS * C::CHUNKS; idx += C::NT) {
        const int rr = idx / C::CHUNKS, c = idx % C::CHUNKS;
        const uint32_t dst = sb + C::OFF_Q + rr * C::ROW_BYTES + ((c ^ (rr & 7)) << 4);
        if (rr < rows_here) {
            const int r = row0 + rr;
            const int i = r / g, hl = r % g;
            cp_async16(dst, qg + (((size_t)b * a.Sq + i) * a.Hq + hkv * g + hl) * D + c * 8, 16);
        } else {
            cp_async16(dst, qg, 0);
        }
    }
    cp_async_commit();

    auto load_tile = [&](int tile, int stage) {
        const int t0 = t_begin + tile * TK;
        for (int idx = tid; idx < TK * C::CHUNKS; idx += C::NT) {
            const int tok = idx / C::CHUNKS, c = idx % C::CHUNKS;
            const int t = t0 + tok;
            const uint32_t off = tok * C::ROW_BYTES + ((c ^ (tok & 7)) << 4);
            const uint32_t dk = sb + C::OFF_K + stage * C::KV_TILE + off;
            const uint32_t dv = sb + C::OFF_V + stage * C::KV_TILE + off;
            const int page = t < t_end ? trow[t / a.page_size] : -1;
            // A page id outside the pool (a caller error) is read as zeros, never dereferenced.
            if (page >= 0 && page < a.num_pages) {
                const size_t e = (((size_t)page * a.page_size + t % a.page_size) * a.Hkv + hkv) * D + c * 8;
                cp_async16(dk, kc + e, 16);
                cp_async16(dv, vc + e, 16);
            } else {
                cp_async16(dk, kc, 0);   // zero-fill: 0 * P stays 0 in O += P V
                cp_async16(dv, vc, 0);
            }
        }
    };

#pragma unroll
    for (int s = 0; s < C::NS - 1; ++s) {
        if (s < n_tiles) load_tile(s, s);
        cp_async_commit();
    }
    cp_async_wait<C::NS - 1>();                    // the Q group has landed
    __syncthreads();

    const int mf = warp / C::KSPLIT;               // this warp's 16-row fragment
    const int wk = warp % C::KSPLIT;               // key part (S) / head-dim part (PV)
    uint32_t qf[C::KSTEPS][4];
#pragma unroll
    for (int kk = 0; kk < C::KSTEPS; ++kk) {
        const int row = mf * 16 + (lane & 15);
        const int chunk = kk * 2 + (lane >> 4);
        ldsm_x4(sb + C::OFF_Q + row * C::ROW_BYTES + ((chunk ^ (row & 7)) << 4), qf[kk][0], qf[kk][1],
                qf[kk][2], qf[kk][3]);
    }

    // Visibility limit (exclusive) of the two rows this lane holds in S fragments.
    int lim[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int rl = mf * 16 + (lane >> 2) + 8 * h;
        const int r = row0 + rl;
        if (rl >= rows_here) {
            lim[h] = -1;
        } else if (a.causal) {
            const long p = (long)(r / g) + L - a.Sq;       // key position of query r / g
            lim[h] = (int)min((long)t_end, p + 1);
        } else {
            lim[h] = t_end;
        }
    }

    // Softmax row ownership: TPR consecutive threads share a row.
    const int srow = tid / C::TPR;
    const int ssub = tid % C::TPR;
    float m_run = -INFINITY, l_run = 0.f;
    float* sS = reinterpret_cast<float*>(smem + C::OFF_S);
    float* sAlpha = reinterpret_cast<float*>(smem + C::OFF_A);
    const float sl = a.scale_log2;

    float acc[C::NFD][4];
#pragma unroll
    for (int n = 0; n < C::NFD; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

    for (int it = 0; it < n_tiles; ++it) {
        cp_async_wait<C::NS - 2>();
        __syncthreads();
        {
            const int nt = it + C::NS - 1;
            if (nt < n_tiles) load_tile(nt, nt % C::NS);
            cp_async_commit();
        }
        const int stage = it % C::NS;
        const int t0 = t_begin + it * TK;
        const uint32_t sK = sb + C::OFF_K + stage * C::KV_TILE;
        const uint32_t sV = sb + C::OFF_V + stage * C::KV_TILE;

        // ---- S = Q K^T for this warp's rows and keys
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
                ldsm_x4(sK + key * C::ROW_BYTES + ((chunk ^ (key & 7)) << 4), b0, b1, b2, b3);
                mma_16816(sacc[2 * np], qf[kk], b0, b1);
                mma_16816(sacc[2 * np + 1], qf[kk], b2, b3);
            }
        }
#pragma unroll
        for (int n = 0; n < C::NFK; ++n) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rl = mf * 16 + (lane >> 2) + 8 * h;
                const int kl = wk * C::KEYS_PER_WARP + n * 8 + 2 * (lane & 3);
                const int t = t0 + kl;
                float2 v;
                v.x = t < lim[h] ? sacc[n][2 * h] * sl : -INFINITY;
                v.y = t + 1 < lim[h] ? sacc[n][2 * h + 1] * sl : -INFINITY;
                *reinterpret_cast<float2*>(sS + rl * C::S_STRIDE + kl) = v;
            }
        }
        __syncthreads();

        // ---- online softmax, TPR threads per row
        {
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
                pk[e] = pack_bf16x2(p0, p1);
            }
#pragma unroll
            for (int o = C::TPR / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            l_run = l_run * alpha + sum;
            m_run = m_new;
#pragma unroll
            for (int q = 0; q < C::KPT / 8; ++q) {
                const int chunk = ssub * (C::KPT / 8) + q;
                uint4* dst = reinterpret_cast<uint4*>(smem + C::OFF_P + srow * (TK * 2) +
                                                      ((chunk ^ (srow & 7)) << 4));
                *dst = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
            if (ssub == 0) sAlpha[srow] = alpha;
        }
        __syncthreads();

        // ---- O = O * alpha + P V for this warp's rows and head-dim slice
        {
            const float a0 = sAlpha[mf * 16 + (lane >> 2)];
            const float a1 = sAlpha[mf * 16 + (lane >> 2) + 8];
#pragma unroll
            for (int n = 0; n < C::NFD; ++n) {
                acc[n][0] *= a0; acc[n][1] *= a0;
                acc[n][2] *= a1; acc[n][3] *= a1;
            }
#pragma unroll
            for (int kk = 0; kk < TK / 16; ++kk) {
                uint32_t pa[4];
                {
                    const int row = mf * 16 + (lane & 15);
                    const int chunk = kk * 2 + (lane >> 4);
                    ldsm_x4(sb + C::OFF_P + row * (TK * 2) + ((chunk ^ (row & 7)) << 4), pa[0], pa[1],
                            pa[2], pa[3]);
                }
#pragma unroll
                for (int np = 0; np < C::NFD / 2; ++np) {
                    const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                    const int dchunk = (wk * C::DSL + np * 16) / 8 + (lane >> 4);
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(sV + key * C::ROW_BYTES + ((dchunk ^ (key & 7)) << 4), v0, v1, v2, v3);
                    mma_16816(acc[2 * np], pa, v0, v1);
                    mma_16816(acc[2 * np + 1], pa, v2, v3);
                }
            }
        }
    }
    cp_async_wait<0>();

    float* sL = reinterpret_cast<float*>(smem + C::OFF_L);
    float* sM = reinterpret_cast<float*>(smem + C::OFF_M);
    if (ssub == 0) {
        sL[srow] = l_run;
        sM[srow] = m_run;
    }
    __syncthreads();

    const size_t part_row0 = ((size_t)(b * a.Hkv + hkv) * a.max_splits + split) * R + row0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int rl = mf * 16 + (lane >> 2) + 8 * h;
        if (rl < rows_here) {
            const float l = sL[rl];
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float* dst = a.part_o + (part_row0 + rl) * D + wk * C::DSL + 2 * (lane & 3);
#pragma unroll
            for (int n = 0; n < C::NFD; ++n)
                *reinterpret_cast<float2*>(dst + n * 8) = make_float2(acc[n][2 * h] * inv, acc[n][2 * h + 1] * inv);
        }
    }
    if (tid < rows_here) {
        const float l = sL[tid];
        a.part_lse[part_row0 + tid] = l > 0.f ? sM[tid] + log2f(l) : -INFINITY;
    }
}

template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeArgs a, int R, int g) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const long row = (long)blockIdx.x * 4 + warp;
    const long total = (long)a.B * a.Sq * a.Hq;
    if (row >= total) return;
    const int h = (int)(row % a.Hq);
    const int i = (int)((row / a.Hq) % a.Sq);
    const int b = (int)(row / ((long)a.Hq * a.Sq));
    const int hkv = h / g, r = i * g + h % g;
    const int L = min(max(a.seqlens[b], 0), a.max_pages * a.page_size);
    const int n = L > 0 ? (L + a.chunk - 1) / a.chunk : 0;
    const size_t base = (size_t)(b * a.Hkv + hkv) * a.max_splits * R + r;

    float M = -INFINITY;
    for (int s = lane; s < n; s += 32) M = fmaxf(M, a.part_lse[base + (size_t)s * R]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.o) + (size_t)row * D;
    constexpr int PER = D / 128 > 0 ? D / 128 : 1;     // float4 groups per lane
    if (M == -INFINITY) {
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int d = (q * 32 + lane) * 4;
            if (d < D) *reinterpret_cast<uint2*>(out + d) = make_uint2(0u, 0u);
        }
        if (lane == 0 && a.lse) a.lse[row] = -INFINITY;
        return;
    }
    float accv[PER][4] = {};
    float den = 0.f;
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
                make_uint2(pack_bf16x2(accv[q][0] * inv, accv[q][1] * inv),
                           pack_bf16x2(accv[q][2] * inv, accv[q][3] * inv));
    }
    if (lane == 0 && a.lse) a.lse[row] = (M + log2f(den)) * kLn2;
}

int choose_mf(int R) {
    const int blocks16 = (R + 15) / 16;
    return blocks16 >= 4 ? 4 : blocks16;
}

template <int D, int MF>
cudaError_t launch_split(const DecodeArgs& a, int R, int g, int n_rowblk, cudaStream_t stream) {
    using C = DCfg<D, MF>;
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, MF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(a.max_splits, a.Hkv, a.B * n_rowblk);
    decode_split_kernel<D, MF><<<grid, C::NT, C::SMEM, stream>>>(a, R, g, n_rowblk);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t stream) {
    const int g = a.Hq / a.Hkv;
    const int R = g * a.Sq;
    const int mf = choose_mf(R);
    const int n_rowblk = (R + 16 * mf - 1) / (16 * mf);
    cudaError_t e;
    switch (mf) {
        case 1: e = launch_split<D, 1>(a, R, g, n_rowblk, stream); break;
        case 2: e = launch_split<D, 2>(a, R, g, n_rowblk, stream); break;
        case 3: e = launch_split<D, 3>(a, R, g, n_rowblk, stream); break;
        default: e = launch_split<D, 4>(a, R, g, n_rowblk, stream); break;
    }
    if (e != cudaSuccess) return e;
    const long rows = (long)a.B * a.Sq * a.Hq;
    decode_combine_kernel<D><<<(unsigned)((rows + 3) / 4), 128, 0, stream>>>(a, R, g);
    return cudaGetLastError();
}

}  // namespace

bool plan_decode(int B, int Sq, int Hq, int Hkv, int D, int page_size, int max_pages, int num_sms,
                 DecodePlan* plan) {
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || page_size <= 0 || max_pages <= 0)
        return false;
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
    return true;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.D) {
        case 64: return launch_d<64>(a, stream);
        case 128: return launch_d<128>(a, stream);
        case 256: return launch_d<256>(a, stream);
        default: return cudaErrorInvalidValue;
    }
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
