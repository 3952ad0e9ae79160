// Paged-KV decode on the 5th-generation tensor cores, for KV groups with many
// query rows (g * Sq from 32 to 128 rows per KV head, e.g. the 24/2/D256
// multi-query geometry of MATE "QSA").
//
// Contract as in decode.cu: request b's logical token t lives in slot
// t % page_size of page block_table[b, t / page_size]; query i sits at key
// position i + L_b - Sq (TileOPs "Attention Operators", GQAPagedFwdOp /
// MHADecodePagedWithKVCacheFwdOp).  Partial results are merged by their LSE
// as in MATE "QSA", Core Attention, SplitKV.
//
// Work is balanced, not split per request: the (request, KV head) segments,
// request-major, are laid end to end as one sequence of 64-key tiles, and a
// persistent grid of one CTA per SM takes equal contiguous ranges of it.  A
// CTA's range crosses segment boundaries; the K/V pipeline runs straight
// through them, and only the query rows, the running softmax state and the
// output accumulator change.  Each (segment, CTA) piece writes a normalised
// FP32 partial O and a base-2 LSE under partial id segment + CTA (unique: the
// pieces form a staircase), and the CTA that holds a segment's first tile
// records the segment's first id and piece count for decode_combine_kernel.
// One CTA per SM means no refill of the pipeline between work units and no
// partly filled last wave.
//
// With 48 query rows and D = 256, warp-level MMAs need Q in registers split by
// 16-row fragment, so every K and V element is read from shared memory once
// per fragment; here the tensor core reads each operand once instead:
//   warp 4     (before the main loop) sums the tiles of all segments and finds
//              where this CTA's range starts;
//   warps 0-3  copy the first piece's Q rows (packed i * g + hl, padding rows
//              zero) from global memory into TMEM, where they are the A
//              operand of S = Q K^T, so shared memory holds only the K/V rings;
//   warp 4     TMA producer: 64-key K and V tiles, one 5-D box per page
//              block (min(page tokens, 64) tokens, all D columns), each issued
//              by its own lane: a single thread issuing many small boxes is
//              the limit at small page sizes, and one box per block brings
//              D / 64 times fewer boxes than one per 64-column slice.  Tiles
//              are issued in the order the MMAs consume them (K0, K1, V0, K2,
//              V1, ...) through 3-4 deep K and 4-6 deep V rings (about 200 KB
//              in flight, which the memory latency at full bandwidth needs);
//              block-table entries are read 32 at a time by the warp.  With
//              float8_e4m3fn caches it loads byte tiles into byte rings instead,
//              K and V as two independent streams (each with its own cursor),
//              and warps 6-7 with the row-less warps of 0-3 widen them into the
//              16-bit rings as a K team and a V team;
//   warp 5     MMA issuer: S = Q K^T (M = 128 rows, N = 64 keys, Q from TMEM)
//              into one of two TMEM buffers, O += P V with P read from TMEM
//              (N = D, 16 keys per step, a fresh accumulator at each piece);
//              the descriptors are formed once per tile and stepped by
//              constants, so issuing keeps pace with the tensor pipe;
//   warps 0-3  softmax, one row per thread (only warps holding a query row):
//              running max and sum in base 2 with a lazy reference max (moved
//              only when a tile max exceeds it by more than 2^8), P written
//              over its S row, O rescaled when needed; at the end of a piece
//              the next piece's Q rows go into TMEM (prefetched to L2 one tile
//              earlier), then O / l and the LSE are written to the workspace.
// Rows past g * Sq in the 128-row M dimension are padding; their results are
// never stored.  Value rows past a request's end are zeroed in shared memory
// before P V reads them.  Every wait is bounded (ptx.cuh).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

__device__ int g_decode_tc_error;

constexpr int BM = 128;            // TMEM lanes = padded query rows
constexpr int BN = 64;             // keys per tile
constexpr int NUM_THREADS = 192;   // warps 0-3 softmax, 4 producer, 5 MMA
constexpr int WARP_LOAD = 4;
constexpr int WARP_MMA = 5;
// e4m3 caches: warps 6-7 widen each byte tile into the 16-bit rings
constexpr int WARP_W0 = 6;
constexpr int NUM_W = 2;
template <bool KV8>
constexpr int num_threads() { return NUM_THREADS + (KV8 ? 32 * NUM_W : 0); }
constexpr float kRescaleThreshold = 8.f;

template <int D, bool KV8 = false>
struct TCfg {
    static constexpr int NSUB = D / 64;
    // Shared-memory layout of a 64-key K or V tile: [8-key group][64-column
    // slice][8 keys][128 bytes] (128-byte swizzle), as the 5-D page-block
    // boxes land: the 8-row atoms of one slice are GROUP_STRIDE apart across
    // the whole tile, whatever the page size.
    static constexpr int GROUP_STRIDE = NSUB * 1024;
    static constexpr int KV_TILE = NSUB * BN * 128;
    // Q is held in TMEM, so shared memory is all K/V ring: about 200 KB in
    // flight per SM covers the memory latency at full bandwidth.  V tiles are
    // consumed about two tiles after their K (P V follows the softmax), so the
    // V ring is deeper.
    // With e4m3 caches the byte tiles (TMA, 5-D page-block boxes) come first
    // and the 16-bit rings the wideners fill are shallower.  At D = 256 the V
    // ring keeps three tiles (P V of a tile follows its K by two tiles: with
    // two, the 16-bit decode itself ran 35 % slower), the K ring two (so that
    // a tile is widened while S of the one before runs) and the byte rings two
    // each.  The K and V byte copies are issued as two independent streams
    // (see the producer): in one fixed order, a full V ring held back the next
    // K copy, and every split with a two-deep K ring lost (0.236 ms with one
    // K tile and three byte tiles a ring, 0.210 ms now, at B = 32).
    static constexpr int NK = KV8 ? (D == 256 ? 2 : 3) : (D == 256 ? 3 : 4);
    static constexpr int NV = KV8 ? (D == 256 ? 3 : 4) : (D == 256 ? 4 : 6);
    static constexpr int NSUB8 = D / 128;                  // 128-column halves of an e4m3 row
    // e4m3 tile: [8-key group][128-column half][8 keys][128 bytes], 128-byte swizzle
    static constexpr int GROUP8 = NSUB8 * 1024;
    static constexpr int TILE8 = KV8 ? NSUB8 * BN * 128 : 0;   // one K or V tile of bytes
    static constexpr int NK8 = KV8 ? (D == 256 ? 2 : 4) : 0;
    static constexpr int NV8 = NK8;
    static constexpr int OFF_K8 = 0;
    static constexpr int OFF_V8 = OFF_K8 + NK8 * TILE8;
    static constexpr int OFF_K = OFF_V8 + NV8 * TILE8;
    static constexpr int OFF_V = OFF_K + NK * KV_TILE;
    static constexpr int OFF_BAR = OFF_V + NV * KV_TILE;
    // q_ready, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_full[2],
    // p_full[2], o_done, drain, q_next, then k8_full[NK8], k8_empty[NK8],
    // v8_full[NV8], v8_empty[NV8]
    static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 + 2 + 1 + 1 + 1 + 2 * NK8 + 2 * NV8;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
    // TMEM: S0 | S1 | O | Q (Q rows as bf16 pairs, the A operand of S = Q K^T)
    static constexpr uint32_t COL_S0 = 0, COL_S1 = BN, COL_O = 2 * BN, COL_Q = 2 * BN + D;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(COL_Q + D / 2 <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// Where this CTA's range of the tile sequence starts and ends (shared memory).
struct Range {
    int g0, n;        // first global tile, tiles in the range
    int per;          // tiles per CTA
    int s0, lt0;      // segment and tile within it of the first tile
};

// First 64-key tile of request b that any query can see: with a left window
// the keys before the first query's lower bound L - Sq - wL are never read.
__device__ __forceinline__ int first_tile(const DecodeArgs& a, int L) {
    if (a.x.wl < 0 || L <= 0) return 0;
    const long lo = (long)L - a.Sq - a.x.wl;
    return lo > 0 ? (int)(lo / BN) : 0;
}

// A position in the tile sequence: segment s = b * Hkv + h holds the
// ceil(L_b / 64) - tf tiles from tile tf on; lt is the tile within the segment.
struct Cursor {
    int s, b, h, L, tf, nt, lt;
    __device__ __forceinline__ void set(const DecodeArgs& a, int seg) {
        s = seg;
        b = seg / a.Hkv;
        h = seg % a.Hkv;
        L = seg < a.B * a.Hkv ? min(max(a.seqlens[b], 0), a.max_pages * a.page_size) : 0;
        tf = first_tile(a, L);
        nt = (L + BN - 1) / BN - tf;
    }
    // The next tile, skipping empty segments (never past the last segment).
    __device__ __forceinline__ void next(const DecodeArgs& a) {
        if (++lt < nt) return;
        lt = 0;
        const int n_seg = a.B * a.Hkv;
        do {
            set(a, s + 1);
        } while (nt == 0 && s + 1 < n_seg);
    }
};

// One 64-column row per thread (two loads, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
    tmem_ld32(taddr, v);
    tmem_ld32(taddr + 32, v + 32);
}

__device__ __forceinline__ int request_tiles(const DecodeArgs& a, int b) {
    if (b >= a.B) return 0;
    const int L = min(max(a.seqlens[b], 0), a.max_pages * a.page_size);
    return (L + BN - 1) / BN - first_tile(a, L);
}

// Query row r of (b, h) (bf16 [B, Sq, Hq, D]) into this thread's TMEM lane,
// columns COL_Q.., zeros for padding rows; the whole warp calls it.
// to_f16: the row is bfloat16 and goes into TMEM as float16 (the e4m3 path's
// MMAs run in float16).
template <int D>
__device__ __forceinline__ void q_row_to_tmem(const DecodeArgs& a, uint32_t taddr, int r, int R, int g, int b,
                                              int h, bool to_f16) {
    const uint4* src = nullptr;
    if (r < R)
        src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                             (((size_t)b * a.Sq + r / g) * a.Hq + h * g + r % g) * D);
    uint32_t w[D / 2];
#pragma unroll
    for (int e = 0; e < D / 8; ++e) {
        const uint4 v = src ? __ldg(src + e) : make_uint4(0u, 0u, 0u, 0u);
        w[4 * e] = v.x; w[4 * e + 1] = v.y; w[4 * e + 2] = v.z; w[4 * e + 3] = v.w;
    }
    if (to_f16) {
#pragma unroll
        for (int e = 0; e < D / 2; ++e) {
            const __half2 hh = __floats2half2_rn(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
            w[e] = *reinterpret_cast<const uint32_t*>(&hh);
        }
    }
    __syncwarp();                                  // tcgen05.st is warp-collective
#pragma unroll
    for (int c = 0; c < D / 64; ++c) tmem_st32(taddr + 32 * c, w + 32 * c);
}

// F16: the MMA operand type (float16 for e4m3 caches, widened exactly).  KV8:
// float8_e4m3fn caches with per-(request, KV head) scales (a bfloat16 Q is
// then rounded to float16 once, when it goes into TMEM).
template <int D, bool F16, bool KV8>
__global__ void __launch_bounds__(num_threads<KV8>(), 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const DecodeArgs a, int R, int g, int box_tokens) {
    using C = TCfg<D, KV8>;
    // both MMA operands of the call's 16-bit type (P is packed to it as well)
    constexpr uint32_t IDESC_QK = make_idesc_16<F16>(BM, BN, false, false);
    constexpr uint32_t IDESC_PV = make_idesc_16<F16>(BM, D, false, true);
    const int cta = blockIdx.x;
    griddep_launch_dependents();                 // the combine may be scheduled (it waits for this grid)

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int n_sm_warps = (R + 31) / 32;          // softmax warps that hold a query row

    const uint32_t bar0 = sb + C::OFF_BAR;
    const uint32_t q_ready = bar0;
    auto k_full = [&](int i) { return bar0 + 8u * (1 + i); };
    auto k_empty = [&](int i) { return bar0 + 8u * (1 + C::NK + i); };
    auto v_full = [&](int i) { return bar0 + 8u * (1 + 2 * C::NK + i); };
    auto v_empty = [&](int i) { return bar0 + 8u * (1 + 2 * C::NK + C::NV + i); };
    auto s_full = [&](int i) { return bar0 + 8u * (1 + 2 * C::NK + 2 * C::NV + i); };
    auto p_full = [&](int i) { return bar0 + 8u * (3 + 2 * C::NK + 2 * C::NV + i); };
    const uint32_t o_done = bar0 + 8u * (5 + 2 * C::NK + 2 * C::NV);
    const uint32_t drain = bar0 + 8u * (6 + 2 * C::NK + 2 * C::NV);
    const uint32_t q_next = bar0 + 8u * (7 + 2 * C::NK + 2 * C::NV);
    const uint32_t bar8 = bar0 + 8u * (8 + 2 * C::NK + 2 * C::NV);
    auto k8_full = [&](int i) { return bar8 + 8u * i; };
    auto k8_empty = [&](int i) { return bar8 + 8u * (C::NK8 + i); };
    auto v8_full = [&](int i) { return bar8 + 8u * (2 * C::NK8 + i); };
    auto v8_empty = [&](int i) { return bar8 + 8u * (2 * C::NK8 + C::NV8 + i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    Range* range = reinterpret_cast<Range*>(smem + C::OFF_MISC + 16);

    if (threadIdx.x == 0) {
        mbar_init(q_ready, BM);
        // the 16-bit tiles land by TMA (one arrival with its bytes) or from the
        // wideners (one arrival per widener warp)
        const int nwt = NUM_W + (4 - n_sm_warps);
        int nwv = 0;                                  // widener positions in the V team (see team_of)
        for (int q = 0; q < nwt; ++q) nwv += (q + (q >> 1)) & 1;
        const int fill_k = KV8 ? nwt - nwv : 1, fill_v = KV8 ? nwv : 1;
        for (int i = 0; i < C::NK; ++i) { mbar_init(k_full(i), fill_k); mbar_init(k_empty(i), 1); }
        for (int i = 0; i < C::NV; ++i) { mbar_init(v_full(i), fill_v); mbar_init(v_empty(i), 1); }
        for (int i = 0; i < C::NK8; ++i) { mbar_init(k8_full(i), 1); mbar_init(k8_empty(i), fill_k); }
        for (int i = 0; i < C::NV8; ++i) { mbar_init(v8_full(i), 1); mbar_init(v8_empty(i), fill_v); }
        for (int i = 0; i < 2; ++i) { mbar_init(s_full(i), 1); mbar_init(p_full(i), 32 * n_sm_warps); }
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        mbar_init(q_next, 32 * n_sm_warps);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_LOAD) {
        // This CTA's range: tiles [cta * per, min((cta + 1) * per, T)) of the T
        // tiles of all segments, per = ceil(T / grid).
        long T = 0;
        for (int b0 = 0; b0 < a.B; b0 += 32) {
            int n = request_tiles(a, b0 + lane);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
            T += n;
        }
        T *= a.Hkv;
        const long per = (T + gridDim.x - 1) / gridDim.x;
        const long g0 = (long)cta * per;
        const long g1 = min(g0 + per, T);
        Range rg{(int)g0, (int)max(0L, g1 - g0), (int)per, 0, 0};
        if (g1 > g0) {
            long before = 0;   // tiles of the requests before b0, all heads
            for (int b0 = 0; b0 < a.B; b0 += 32) {
                const int n = request_tiles(a, b0 + lane);
                int incl = n;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                const unsigned hit = __ballot_sync(0xffffffffu, before + (long)incl * a.Hkv > g0);
                if (hit) {
                    const int l = __ffs(hit) - 1;
                    const int nb = __shfl_sync(0xffffffffu, n, l);
                    const long start = before + (long)(__shfl_sync(0xffffffffu, incl, l) - nb) * a.Hkv;
                    const int off = (int)(g0 - start);
                    rg.s0 = (b0 + l) * a.Hkv + off / nb;
                    rg.lt0 = off % nb;
                    break;
                }
                before += (long)__shfl_sync(0xffffffffu, incl, 31) * a.Hkv;
            }
        }
        if (lane == 0) *range = rg;
    }
    __syncthreads();
    const Range rg = *range;
    const int n = rg.n;
    if (n == 0) return;                            // nothing here (uniform)
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // ------------------------------------------------------------ wideners (e4m3 caches)
    // Each byte tile becomes the 16-bit tile the MMAs read, each team in its
    // own stream's tile order: rows [8-key group][64-
    // column slice][8 keys][128 bytes] with the 128-byte swizzle, exactly as the
    // 5-D page-block boxes land in the 16-bit path.  Warps 6-7 widen, and so do
    // the warps of 0-3 that hold no query row once their (zero) Q rows are in;
    // they form a K team and a V team, so a value tile waiting for its slot
    // never holds up the next key tile.
    const int n_w = NUM_W + (4 - n_sm_warps);
    // Team of widener position p: positions 0, 3, 4, 7, ... widen K and 1, 2, 5,
    // 6, ... V, so that with the row-less warps 2-3 and warps 6-7 each team
    // spans two SM sub-partitions (warp w issues on sub-partition w % 4): the
    // conversion pipe of one sub-partition does not carry a whole team.
    auto team_of = [](int p) { return ((p + (p >> 1)) & 1) != 0; };
    auto run_wideners = [&](int wpos) {             // position among the widener warps
        const bool team_v = team_of(wpos);
        int team_n = 0, rank = 0;
        for (int q = 0; q < n_w; ++q) {
            if (team_of(q) != team_v) continue;
            if (q < wpos) ++rank;
            ++team_n;
        }
        const int wt = rank * 32 + lane;
        int nk = 0, nv = 0;
        auto widen = [&](bool is_v) -> bool {
            const int cnt = is_v ? nv : nk;
            const int r8 = is_v ? C::NV8 : C::NK8, r16 = is_v ? C::NV : C::NK;
            const int s8 = cnt % r8, s16 = cnt % r16;
            if (!__all_sync(0xffffffffu, mbar_wait(is_v ? v8_full(s8) : k8_full(s8), (cnt / r8) & 1, abort_flag)))
                return false;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(is_v ? v_empty(s16) : k_empty(s16), ((cnt / r16) & 1) ^ 1, abort_flag)))
                return false;
            const uint8_t* src = smem + (is_v ? C::OFF_V8 : C::OFF_K8) + s8 * C::TILE8;
            uint8_t* dst = smem + (is_v ? C::OFF_V : C::OFF_K) + s16 * C::KV_TILE;
            constexpr int CH8 = D / 16;            // 16-byte e4m3 chunks of a row
            constexpr int U = 2;                   // chunks loaded before any is stored
            const int step = 32 * team_n;
            for (int base = wt; base < BN * CH8; base += U * step) {
                // The loads of a batch are issued together: the stores cannot
                // be proven apart from the next loads, so a one-chunk loop
                // would wait out the shared-memory latency once per chunk.
                uint4 x[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int idx = base + u * step;
                    const int k = idx % BN, c8 = idx / BN;   // 8-lane phases: eight keys, one chunk (no bank conflict)
                    if (idx < BN * CH8)
                        x[u] = *reinterpret_cast<const uint4*>(src + (k >> 3) * C::GROUP8 + (c8 >> 3) * 1024 +
                                                               (k & 7) * 128 + (((c8 & 7) ^ (k & 7)) << 4));
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int idx = base + u * step;
                    if (idx >= BN * CH8) break;
                    const int k = idx % BN, c16 = 2 * (idx / BN);   // two 8-dim chunks share one 64-column slice
                    uint8_t* row = dst + (k >> 3) * C::GROUP_STRIDE + (c16 >> 3) * 1024 + (k & 7) * 128;
                    uint32_t h[8];
                    e4m3x4_to_f16x4(x[u].x, h[0], h[1]);
                    e4m3x4_to_f16x4(x[u].y, h[2], h[3]);
                    e4m3x4_to_f16x4(x[u].z, h[4], h[5]);
                    e4m3x4_to_f16x4(x[u].w, h[6], h[7]);
                    *reinterpret_cast<uint4*>(row + (((c16 & 7) ^ (k & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4*>(row + ((((c16 + 1) & 7) ^ (k & 7)) << 4)) =
                        make_uint4(h[4], h[5], h[6], h[7]);
                }
            }
            fence_proxy_async_smem();              // the tensor core reads what the warp wrote
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(is_v ? v8_empty(s8) : k8_empty(s8));
                mbar_arrive(is_v ? v_full(s16) : k_full(s16));
            }
            __syncwarp();
            if (is_v) ++nv; else ++nk;
            return true;
        };
        for (int it = 0; it < n; ++it)
            if (!widen(team_v)) break;
    };
    if (warp == WARP_LOAD) {
        // ------------------------------------------------------------ producer
        const int nbox = BN / box_tokens;          // page blocks per tile; lane i loads block i
        const uint32_t blk_bytes = (uint32_t)box_tokens * 128 * C::NSUB;
        int win = -(1 << 30), pid = -1, win_b = -1;   // block-table window of request win_b
        int nk = 0, nv = 0;
        bool ok = true;
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        Cursor cur;
        cur.set(a, rg.s0);
        cur.lt = rg.lt0;
        // 16-bit caches: loads are issued in the order the MMAs consume them: K0,
        // K1, V0, K2, V1, ...  Lane i finds the first cache row of page block i of a tile
        // when the tile's K is issued (-1: not loaded) and keeps it, for two
        // tiles, for the tile's V, with the tile's KV head.
        int row_ring0 = -1, row_ring1 = -1, n_ring0 = 0, n_ring1 = 0, h_ring0 = 0, h_ring1 = 0;
        auto find_rows = [&](int it) {             // tile `it` is at `cur`
            if (cur.b != win_b) {
                win_b = cur.b;
                win = -(1 << 30);
            }
            const int32_t* trow = a.table + (size_t)cur.b * a.max_pages;
            const int t = (cur.tf + cur.lt) * BN + lane * box_tokens;
            const int lp = t / a.page_size;
            const int lp_first = __shfl_sync(0xffffffffu, lp, 0);
            const int lp_last = __shfl_sync(0xffffffffu, lp, nbox - 1);
            if (lp_last - win >= 32 || lp_first < win) {   // warp-uniform refill of the window
                win = lp_first;
                pid = win + lane < a.max_pages ? trow[win + lane] : -1;
            }
            const int page = __shfl_sync(0xffffffffu, pid, (lp - win) & 31);
            int row = -1;
            // a page id outside the pool (a caller error) is not loaded
            if (lane < nbox && t < cur.L && page >= 0 && page < a.num_pages)
                row = page * a.page_size + t % a.page_size;
            const int cnt = __popc(__ballot_sync(0xffffffffu, row >= 0));
            if (it & 1) { row_ring1 = row; n_ring1 = cnt; h_ring1 = cur.h; }
            else { row_ring0 = row; n_ring0 = cnt; h_ring0 = cur.h; }
            if (it + 1 < n) cur.next(a);
        };
        auto load = [&](int it, bool is_v) -> bool {   // whole warp; 16-bit caches
            const int row = (it & 1) ? row_ring1 : row_ring0;
            const int cnt_rows = (it & 1) ? n_ring1 : n_ring0;
            const int h = (it & 1) ? h_ring1 : h_ring0;
            const int cnt = is_v ? nv : nk;
            const int ring = is_v ? C::NV : C::NK;
            const int slot = cnt % ring;
            const uint32_t empty_bar = is_v ? v_empty(slot) : k_empty(slot);
            const uint32_t full_bar = is_v ? v_full(slot) : k_full(slot);
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait(empty_bar, ((cnt / ring) & 1) ^ 1, abort_flag);
                if (ok) mbar_arrive_expect_tx(full_bar, (uint32_t)cnt_rows * blk_bytes);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
            __syncwarp();                          // the expect-tx precedes every lane's copy
            const void* map = is_v ? (const void*)&tm_v : (const void*)&tm_k;
            const uint32_t dst = sb + (is_v ? C::OFF_V : C::OFF_K) + slot * C::KV_TILE + lane * blk_bytes;
            if (row >= 0) tma_load_5d(dst, map, full_bar, 0, 0, 0, row / 8, h);
            if (is_v) ++nv; else ++nk;
            return true;
        };
        if constexpr (KV8) {
            // e4m3 caches: K and V as two streams, each with its own cursor and
            // block-table window, a stream's next copy issued as soon as its byte
            // slot is free (polled without suspending), V(i) never before K(i).
            // The wideners drain the two byte rings independently, so neither
            // stream waits behind the other's full ring.
            struct Stream { Cursor cur; int win, pid, win_b, it, cnt, row, rows, h; bool found; };
            auto init = [&](Stream& S) {
                S.cur.set(a, rg.s0);
                S.cur.lt = rg.lt0;
                S.win = -(1 << 30); S.pid = -1; S.win_b = -1; S.it = 0; S.cnt = 0; S.found = false;
            };
            auto find = [&](Stream& S) {           // the stream's next tile: rows as find_rows gives them
                Cursor& c = S.cur;
                if (c.b != S.win_b) { S.win_b = c.b; S.win = -(1 << 30); }
                const int32_t* trow = a.table + (size_t)c.b * a.max_pages;
                const int t = (c.tf + c.lt) * BN + lane * box_tokens;
                const int lp = t / a.page_size;
                const int lp_first = __shfl_sync(0xffffffffu, lp, 0);
                const int lp_last = __shfl_sync(0xffffffffu, lp, nbox - 1);
                if (lp_last - S.win >= 32 || lp_first < S.win) {
                    S.win = lp_first;
                    S.pid = S.win + lane < a.max_pages ? trow[S.win + lane] : -1;
                }
                const int page = __shfl_sync(0xffffffffu, S.pid, (lp - S.win) & 31);
                int row = -1;
                if (lane < nbox && t < c.L && page >= 0 && page < a.num_pages) row = page * a.page_size + t % a.page_size;
                S.row = row;
                S.rows = __popc(__ballot_sync(0xffffffffu, row >= 0));
                S.h = c.h;
                S.found = true;
                if (S.it + 1 < n) c.next(a);
            };
            auto try_issue = [&](Stream& S, bool is_v) -> bool {   // whole warp; false: slot still busy
                const int ring = is_v ? C::NV8 : C::NK8;
                const int slot = S.cnt % ring;
                const uint32_t empty_bar = is_v ? v8_empty(slot) : k8_empty(slot);
                const uint32_t full_bar = is_v ? v8_full(slot) : k8_full(slot);
                int free_slot = 0;
                if (lane == 0) free_slot = mbar_test_wait(empty_bar, ((S.cnt / ring) & 1) ^ 1) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, free_slot, 0)) return false;
                if (lane == 0) mbar_arrive_expect_tx(full_bar, (uint32_t)S.rows * box_tokens * 128 * C::NSUB8);
                __syncwarp();                      // the expect-tx precedes every lane's copy
                // one {128, 8, D / 128, box_tokens / 8, 1} byte box per page block
                const uint32_t dst = sb + (is_v ? C::OFF_V8 : C::OFF_K8) + slot * C::TILE8 +
                                     lane * box_tokens * 128 * C::NSUB8;
                if (S.row >= 0)
                    tma_load_5d(dst, is_v ? (const void*)&tm_v : (const void*)&tm_k, full_bar, 0, 0, 0, S.row / 8, S.h);
                ++S.cnt;
                ++S.it;
                S.found = false;
                return true;
            };
            Stream sk, sv;
            init(sk);
            init(sv);
            unsigned long long idle_since = 0;
            while (sk.it < n || sv.it < n) {
                bool did = false;
                if (sk.it < n) {
                    if (!sk.found) find(sk);
                    did |= try_issue(sk, false);
                }
                if (sv.it < n && sv.it < sk.it) {
                    if (!sv.found) find(sv);
                    did |= try_issue(sv, true);
                }
                if (did) {
                    idle_since = 0;
                    continue;
                }
                // neither slot free: poll again shortly, within the wait limit
                int stop = 0;
                if (lane == 0) {
                    const unsigned long long now = globaltimer_ns();
                    if (idle_since == 0) idle_since = now;
                    if (*abort_flag) stop = 1;
                    else if (now - idle_since > kWaitTimeoutNs) { *abort_flag = 1; stop = 1; }
                }
                if (__shfl_sync(0xffffffffu, stop, 0)) break;
                __nanosleep(64);
            }
            nk = sk.cnt;
            nv = sv.cnt;
        } else {
            find_rows(0);
            ok = load(0, false);
            for (int it = 0; it < n && ok; ++it) {
                if (it + 1 < n) {
                    find_rows(it + 1);
                    ok = load(it + 1, false);
                    if (!ok) break;
                }
                ok = load(it, true);
            }
        }
        if (lane == 0) {
            if (*abort_flag) {
                // let the copies in flight land: the last load of each slot
                constexpr int RK = KV8 ? C::NK8 : C::NK, RV = KV8 ? C::NV8 : C::NV;
                for (int s = 0; s < RK && s < nk; ++s) {
                    const int last = nk - 1 - ((nk - 1 - s) % RK);
                    mbar_drain(KV8 ? k8_full(s) : k_full(s), (last / RK) & 1);
                }
                for (int s = 0; s < RV && s < nv; ++s) {
                    const int last = nv - 1 - ((nv - 1 - s) % RV);
                    mbar_drain(KV8 ? v8_full(s) : v_full(s), (last / RV) & 1);
                }
            }
        }
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer (lane 0 issues)
        Cursor cq, cp;                             // tiles of the next S = Q K^T and the next P V
        cq.set(a, rg.s0);
        cq.lt = rg.lt0;
        cp = cq;
        int q_pieces = 0;                          // later pieces whose Q has been waited for
        auto issue_qk = [&](int i) -> bool {       // tile i is at cq
            if (i > 0 && cq.lt == 0) {
                // first tile of a later piece: its Q rows replace the previous ones
                if (!__all_sync(0xffffffffu, mbar_wait(q_next, q_pieces & 1, abort_flag))) return false;
                ++q_pieces;
            }
            const int ks = i % C::NK;
            if (!__all_sync(0xffffffffu, mbar_wait(k_full(ks), (i / C::NK) & 1, abort_flag))) return false;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t d = tmem + ((i & 1) ? C::COL_S1 : C::COL_S0);
                // K-major B: 8-key atoms GROUP_STRIDE apart; step kk moves 32 bytes
                // within a slice, every fourth step to the next slice (1 KB on)
                const uint64_t kdesc = make_sdesc_sw128(sb + C::OFF_K + ks * C::KV_TILE, 16, C::GROUP_STRIDE);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ts(d, tmem + C::COL_Q + kk * 8,
                                kdesc + (uint64_t)((((kk / 4) * 1024 + (kk % 4) * 32)) >> 4), IDESC_QK,
                                kk > 0 ? 1u : 0u);
                mma_commit(s_full(i & 1));
                mma_commit(k_empty(ks));
            }
            __syncwarp();
            if (i + 1 < n) cq.next(a);
            return true;
        };
        bool ok = __all_sync(0xffffffffu, mbar_wait(q_ready, 0, abort_flag));
        if (ok) tc_fence_after();
        if (ok) ok = issue_qk(0);
        if (ok && n > 1) ok = issue_qk(1);
        for (int i = 0; i < n && ok; ++i) {
            ok = __all_sync(0xffffffffu, mbar_wait(p_full(i & 1), (i >> 1) & 1, abort_flag));
            if (!ok) break;
            const int vs = i % C::NV;
            ok = __all_sync(0xffffffffu, mbar_wait(v_full(vs), (i / C::NV) & 1, abort_flag));
            if (!ok) break;
            const uint32_t vb = sb + C::OFF_V + vs * C::KV_TILE;
            const bool fresh = i == 0 || cp.lt == 0;   // first tile of a piece: O starts over
            const int nvalid = min(BN, cp.L - (cp.tf + cp.lt) * BN);
            if (nvalid < BN) {
                // Value rows past the request's end hold stale data: zero them
                // before the tensor core reads the tile.
                for (int idx = lane; idx < (BN - nvalid) * 8 * C::NSUB; idx += 32) {
                    const int key = nvalid + idx / (8 * C::NSUB);
                    const int s = (idx / 8) % C::NSUB, chunk = idx % 8;
                    *reinterpret_cast<uint4*>(smem + (vb - sb) + (key / 8) * C::GROUP_STRIDE + s * 1024 +
                                              (key % 8) * 128 + chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t pcol = (i & 1) ? C::COL_S1 : C::COL_S0;
                // MN-major B: 64-column slices 1 KB apart, 8-key atoms GROUP_STRIDE
                // apart; step kk takes keys 16kk..16kk+15 (two atoms)
                const uint64_t vdesc = make_sdesc_sw128(vb, 1024, C::GROUP_STRIDE);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_bf16_ts(tmem + C::COL_O, tmem + pcol + kk * 8,
                                vdesc + (uint64_t)((2 * kk * C::GROUP_STRIDE) >> 4), IDESC_PV,
                                (!fresh || kk > 0) ? 1u : 0u);
                mma_commit(o_done);
                mma_commit(v_empty(vs));
            }
            __syncwarp();
            if (i + 1 < n) cp.next(a);
            // S of tile i+2 overwrites P of tile i: issued after its P V.
            if (i + 2 < n) ok = issue_qk(i + 2);
        }
        if (lane == 0) {
            mma_commit(drain);                    // every MMA issued above has completed once this arrives
            mbar_drain(drain, 0);
        }
        __syncwarp();
    } else if (KV8 && warp >= WARP_W0) {
        run_wideners((4 - n_sm_warps) + (warp - WARP_W0));
    } else {
        // ------------------------------------------------------------ warps 0-3: first Q rows into TMEM
        // Row r = i * g + hl is query i of head h * g + hl; rows past g * Sq are zero.
        Cursor c0;
        c0.set(a, rg.s0);
        q_row_to_tmem<D>(a, tmem + ((uint32_t)(warp * 32) << 16) + C::COL_Q, warp * 32 + lane, R, g, c0.b, c0.h,
                         KV8 && !a.f16);
        tc_fence_before();
        mbar_arrive(q_ready);
    }
    if (KV8 && warp < 4 && warp >= n_sm_warps) run_wideners(warp - n_sm_warps);
    if (warp < n_sm_warps) {
        // ------------------------------------------------------------ softmax warps
        const int r = warp * 32 + lane;            // padded row == TMEM lane
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        const bool row_ok = r < R;
        // softmax scale and softcap input of the piece (times its k_scale with
        // e4m3 caches), and the factor of its stored O (its v_scale)
        float sl = a.scale_log2, cap_in = a.x.cap_in, o_scale = 1.f;
        Cursor c;
        c.set(a, rg.s0);
        c.lt = rg.lt0;
        // visible keys of this row: [lo, lim); lim_first / lo_last bound every row's
        int lim = 0, lo = 0, lim_first = 0, lo_last = 0;
        auto key_hi = [&](long p, int L) {
            long hi = L;
            if (a.causal) hi = min(hi, p + 1);
            if (a.x.wr >= 0) hi = min(hi, p + a.x.wr + 1);
            return (int)max(0L, hi);
        };
        auto key_lo = [&](long p, int L) { return a.x.wl >= 0 ? (int)max(0L, min((long)L, p - a.x.wl)) : 0; };
        auto piece_setup = [&]() {
            if constexpr (KV8) {
                const int kv = c.b * a.Hkv + c.h;
                const float ks = a.k_scale ? a.k_scale[kv] : 1.f;
                sl = a.scale_log2 * ks;
                cap_in = a.x.cap_in * ks;
                o_scale = a.v_scale ? a.v_scale[kv] : 1.f;
            }
            const int L = c.L;
            const long p = (long)(r / g) + L - a.Sq;       // key position of this row's query
            lim = row_ok ? key_hi(p, L) : 0;
            lo = row_ok ? key_lo(p, L) : 0;
            lim_first = key_hi((long)L - a.Sq, L);
            lo_last = key_lo((long)L - 1, L);
        };
        piece_setup();
        int piece_lt0 = rg.lt0;                    // tile of the segment the piece starts at
        float m_ref = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int it = 0; it < n; ++it) {
            const int t0 = (c.tf + c.lt) * BN;
            const bool first = it == 0 || c.lt == 0;
            const bool last = c.lt == c.nt - 1 || it == n - 1;
            Cursor nx = c;
            if (last && it + 1 < n) {
                // the next piece's Q row: into L2 now, into TMEM after this tile
                nx.next(a);
                if (row_ok) {
                    const char* p = reinterpret_cast<const char*>(a.q) +
                                    (((size_t)nx.b * a.Sq + r / g) * a.Hq + nx.h * g + r % g) * D * 2;
#pragma unroll
                    for (int e = 0; e < D * 2 / 128; ++e)
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(p + 128 * e));
                }
            }
            ok = __all_sync(0xffffffffu, mbar_wait(s_full(it & 1), (it >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const uint32_t scol = (it & 1) ? C::COL_S1 : C::COL_S0;
            float s[BN];
            tmem_ld64(tmem + lane_addr + scol, s);
            const bool capped = a.x.cap_out != 0.f;
            const bool fast = t0 + BN <= lim_first && t0 >= lo_last && sl > 0.f && !capped;
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
            if (fast) {
#pragma unroll
                for (int cc = 0; cc < BN; cc += 2) mx8[(cc >> 1) & 7] = fmax3(mx8[(cc >> 1) & 7], s[cc], s[cc + 1]);
            } else {
#pragma unroll
                for (int cc = 0; cc < BN; ++cc) {
                    const float lg = capped ? softcap_log2(s[cc], cap_in, a.x.cap_out) : s[cc] * sl;
                    const float x = t0 + cc >= lo && t0 + cc < lim ? lg : -INFINITY;   // the select drops stale rows
                    s[cc] = x;
                    mx8[cc & 7] = fmaxf(mx8[cc & 7], x);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) mx8[e] = fmaxf(mx8[e], mx8[e + 4]);
            const float mx_raw = fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3]));
            const float mx = fast ? mx_raw * sl : mx_raw;
            float alpha = 1.f;
            if (mx > m_ref + kRescaleThreshold) {
                alpha = fast_exp2(m_ref - mx);
                m_ref = mx;
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
            const uint64_t fa2 = f32x2(fast ? sl : 1.f, fast ? sl : 1.f);
            const uint64_t nm2 = f32x2(-m_use, -m_use);
            uint64_t rs4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) rs4[e] = f32x2(0.f, 0.f);
            uint32_t pk[BN / 2];
#pragma unroll
            for (int cc = 0; cc < BN / 2; ++cc) {
                float x0, x1;
                f32x2_split(ffma2(f32x2(s[2 * cc], s[2 * cc + 1]), fa2, nm2), x0, x1);
                const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                rs4[cc & 3] = fadd2(rs4[cc & 3], f32x2(p0, p1));
                pk[cc] = pack2<F16>(p0, p1);
            }
            rs4[0] = fadd2(rs4[0], rs4[2]);
            rs4[1] = fadd2(rs4[1], rs4[3]);
            float r0, r1, r2, r3;
            f32x2_split(rs4[0], r0, r1);
            f32x2_split(rs4[1], r2, r3);
            l_run = l_run * alpha + ((r0 + r1) + (r2 + r3));
            tmem_st32(tmem + lane_addr + scol, pk);          // P over the first 32 columns of S
            if (!first) {
                // O must hold P V of the previous tile before it is rescaled (the
                // first tile of a piece starts a fresh O)
                ok = __all_sync(0xffffffffu, mbar_wait(o_done, (it - 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        float o[32];
                        tmem_ld32(tmem + lane_addr + C::COL_O + 32 * cc, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= alpha;
                        tmem_st32(tmem + lane_addr + C::COL_O + 32 * cc, reinterpret_cast<uint32_t*>(o));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(p_full(it & 1));
            if (last) {
                if (it + 1 < n) {
                    // S of this tile is done, so Q is free: the next piece's rows
                    q_row_to_tmem<D>(a, tmem + lane_addr + C::COL_Q, r, R, g, nx.b, nx.h, KV8 && !a.f16);
                    tc_fence_before();
                    mbar_arrive(q_next);
                }
                // ---- epilogue of the piece: O / l and the LSE
                ok = __all_sync(0xffffffffu, mbar_wait(o_done, it & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const int id = c.s + cta;                  // partial id of this piece
                const size_t part_row = (size_t)id * R + r;
                const float inv = l_run > 0.f ? o_scale / l_run : 0.f;
#pragma unroll 1
                for (int cc = 0; cc < D / 32; cc += 2) {
                    float o[64];
                    __syncwarp();                          // tcgen05.ld is warp-collective: reconverge (two loads per pass)
                    tmem_ld32(tmem + lane_addr + C::COL_O + 32 * cc, o);
                    tmem_ld32(tmem + lane_addr + C::COL_O + 32 * cc + 32, o + 32);
                    if (row_ok) {
                        float4* dst = reinterpret_cast<float4*>(a.part_o + part_row * D + 32 * cc);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            dst[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv,
                                                 o[4 * e + 3] * inv);
                    }
                }
                if (row_ok) a.part_lse[part_row] = l_run > 0.f ? m_ref + log2f(l_run) : -INFINITY;
                if (piece_lt0 == 0 && r == 0) {
                    // this CTA holds the segment's first tile: record its pieces
                    const long seg_start = (long)rg.g0 + it - c.lt;
                    const int c_last = (int)((seg_start + c.nt - 1) / rg.per);
                    a.seg_table[2 * c.s] = id;
                    a.seg_table[2 * c.s + 1] = c_last - cta + 1;
                }
                m_ref = -INFINITY;
                l_run = 0.f;
                tc_fence_before();
            }
            if (it + 1 < n) {
                c.next(a);
                if (c.lt == 0) {
                    piece_setup();
                    piece_lt0 = 0;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(&g_decode_tc_error, (int)kErrDecodeWait);
}

template <int D, bool F16, bool KV8 = false>
cudaError_t launch_t(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const DecodeArgs& a,
                     int box_tokens, cudaStream_t stream) {
    using C = TCfg<D, KV8>;
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<D, F16, KV8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int g = a.Hq / a.Hkv;
    const int R = g * a.Sq;
    decode_tc_kernel<D, F16, KV8><<<a.tc_grid, num_threads<KV8>(), C::SMEM_BYTES, stream>>>(tm_k, tm_v, a, R, g,
                                                                                           box_tokens);
    return cudaGetLastError();
}

}  // namespace

bool decode_tc_eligible(int D, int R, int page_size) {
    return (D == 128 || D == 256) && R >= 32 && R <= BM && decode_tc_box_tokens(page_size) > 0;
}

int decode_tc_box_tokens(int page_size) {
    // page blocks of 8..64 tokens (whole 8-row groups) that tile both a page
    // and a 64-key tile
    const int bt = page_size < BN ? page_size : BN;
    if (bt % 8 != 0 || page_size % bt != 0 || BN % bt != 0) return 0;
    return bt;
}

cudaError_t launch_decode_tc(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const DecodeArgs& a, int box_tokens, cudaStream_t stream) {
    cudaError_t e;
    switch (a.D) {
        case 128: e = a.f16 ? launch_t<128, true>(tm_k, tm_v, a, box_tokens, stream)
                            : launch_t<128, false>(tm_k, tm_v, a, box_tokens, stream); break;
        case 256: e = a.f16 ? launch_t<256, true>(tm_k, tm_v, a, box_tokens, stream)
                            : launch_t<256, false>(tm_k, tm_v, a, box_tokens, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    return launch_decode_combine(a, stream);
}

cudaError_t launch_decode_tc_fp8(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const DecodeArgs& a,
                                 int box_tokens, cudaStream_t stream) {
    cudaError_t e;
    switch (a.D) {
        case 128: e = launch_t<128, true, true>(tm_k, tm_v, a, box_tokens, stream); break;
        case 256: e = launch_t<256, true, true>(tm_k, tm_v, a, box_tokens, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    return launch_decode_combine(a, stream);
}

int decode_tc_take_device_error() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_decode_tc_error, sizeof(int)) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_decode_tc_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace gqa
