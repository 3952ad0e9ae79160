// Dense / chunked-prefill causal GQA attention forward for head dim 256 on
// sm_103a.
//
// Same computation as prefill.cu (TileOPs "Attention Operators",
// GQADenseFwdOp stages 1-7; RL-Kernel "Standard Softmax Attention", Tensor
// Contract; natural-log LSE per MATE "QSA", Core Attention), for the 24/2/D256
// geometry of MATE "QSA".  With D = 256 one query tile's output accumulator
// takes 256 of the 512 TMEM columns, so a CTA owns ONE 128-row query tile and
// double-buffers its scores instead: TMEM = S0 | S1 (128 columns each) | O.
// The tensor core computes S of key tile i+1 while the softmax warps work on
// tile i, and O += P V of tile i follows.
//
// Warp roles (384 threads, one CTA per SM, persistent over work items):
//   warps 0-3   softmax: thread t owns query row t; reads its S row from
//               TMEM, folds the causal / window / padding mask, keeps the
//               running max and sum, writes P (16-bit) over its S row, and
//               rescales its O row when the reference max moves;
//   warps 4-7   epilogue: once an item's last P V has completed, reads O,
//               frees it for the next item, and stores O / l (TMA, two
//               alternating 64-column staging boxes) and the LSE, while the
//               next item's first tiles already run;
//   warp 8      TMA producer: the Q tile, then K and V through one ring of
//               32 KB slots, in the order the MMAs consume them: K of a tile
//               as two 128-column halves (QK^T has N = 128 keys, K = 256 split
//               in two), V as two 64-key halves of all 256 columns;
//   warp 9      MMA issuer (one thread): QK(0), QK(1), PV(0), QK(2), PV(1), ...
//   warps 10-11 complete the third warpgroup (register limits are per
//               warpgroup).
// The MMA shapes stay at M128 x N128 (QK) and M128 x N256 (PV): the tensor
// core takes about the same time for an N = 64 MMA as for N = 128, so halving
// a tile along the keys would halve the QK rate; splitting K along its head
// dimension and V along its keys keeps both at full rate with 32 KB slots.
//
// The lazy rescale is the one of prefill.cu: O is touched only when the
// reference max moves by more than kRescaleThreshold.  Rescaling O before PV
// of tile i needs PV of tile i-1 complete (o_ready); S of tile i having landed
// already implies PV of tile i-2, so the phase waited for is never more than
// one behind the barrier.  Every wait is bounded; on a timeout the CTA stops
// issuing work, drains what is in flight, frees TMEM and returns.
#include <cmath>

#include "internal.h"
#include "prefill_tiles.cuh"
#include "ptx.cuh"

namespace gqa {
namespace {

__device__ int g_prefill256_error;

using namespace pf;
constexpr int D = 256;
constexpr int NUM_THREADS = 384;
constexpr int WARP_EPI0 = 4;
constexpr int WARP_LOAD = 8;
constexpr int WARP_MMA = 9;
// Registers: 168 per thread at launch (64,512 in all); the softmax warpgroup
// takes 208, the epilogue warpgroup (half a packed O row at a time) 152 and the
// producer/MMA warpgroup 144: (208 + 152 + 144) * 128.
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 208;
constexpr int kRegsEpi = 152;
constexpr int kRegsOther = 144;
static_assert((kRegsSoftmax + kRegsEpi + kRegsOther) * 128 <= kRegsLaunch * NUM_THREADS, "register split");

constexpr int BOX = BM * 128;             // one 64-column box of 128 rows (16 KB)
constexpr int VBOX = 64 * 128;            // one 64-column box of 64 rows (8 KB)
constexpr int CHUNK = 2 * BOX;            // one ring slot: half of a K or V tile (32 KB)
constexpr int NS = 4;                     // ring slots
constexpr int OFF_Q = 0;                  // 4 boxes
constexpr int OFF_RING = OFF_Q + 4 * BOX;
constexpr int OFF_STAGE = OFF_RING + NS * CHUNK;   // 2 output boxes
constexpr int OFF_STATS = OFF_STAGE + 2 * BOX;     // m[128], l[128] (floats), visited-tile count
constexpr int OFF_BAR = OFF_STATS + 2 * BM * 4 + 16;
// q_full, q_empty, r_full[NS], r_empty[NS], s_full[2], p_full[2], o_ready,
// o_final, o_empty, stats_full, stats_empty, drain
constexpr int NBAR = 2 + 2 * NS + 4 + 6;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;       // 1 KB alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
constexpr uint32_t COL_S0 = 0, COL_O = 256, TMEM_COLS = 512;

template <bool OPTS, bool F16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
prefill_d256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const PrefillArgs a, int n_qtiles) {
    constexpr uint32_t IDESC_QK = make_idesc_16<F16>(BM, BN, false, false);
    constexpr uint32_t IDESC_PV = make_idesc_16<F16>(BM, D, false, true);
    const int wl = OPTS ? a.x.wl : -1;
    const int wr = OPTS ? a.x.wr : -1;
    const float cap_in = OPTS ? a.x.cap_in : 0.f;
    const float cap_out = OPTS ? a.x.cap_out : 0.f;
    const float* sinks = OPTS ? a.x.sinks : nullptr;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw_base & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // Work items: heaviest (last) query tiles first, adjacent items on one KV
    // head; round r takes item r * G + cta (even r) or r * G + G - 1 - cta.
    const int bh = a.B * a.Hq;
    const int n_items = n_qtiles * bh;
    const int G = gridDim.x;
    const int cta = blockIdx.x;
    auto item_of = [&](int r) -> int {
        const long w = (long)r * G + ((r & 1) ? G - 1 - cta : cta);
        return w < n_items ? (int)w : -1;
    };
    struct Item {
        int b, hq, hkv, first;
        TileInfo t;
        const uint8_t* mrow;
    };
    auto describe = [&](int w) {
        Item it;
        const int qt = n_qtiles - 1 - w / bh;
        const int rem = w % bh;
        it.hq = rem % a.Hq;
        it.b = rem / a.Hq;
        it.hkv = it.hq / (a.Hq / a.Hkv);
        it.t = tile_info(qt * BM, a.Sq, a.Skv, a.causal, wl, wr);
        it.first = it.t.kv_begin / BN;
        it.mrow = a.mask ? a.mask + (size_t)it.b * a.Skv : nullptr;
        return it;
    };
    // Visited key tiles of an item (non-empty, in [first, n_tiles)).  Warp-collective.
    auto count_tiles = [&](const Item& it) {
        int c = 0;
        for (int chunk = it.first / 32; chunk * 32 < it.t.n_tiles; ++chunk)
            c += __popc(tile_flags(it.mrow, chunk, it.first, it.t.n_tiles, it.t.kv_end, lane));
        return c;
    };

    const uint32_t bar0 = sb + OFF_BAR;
    const uint32_t q_full = bar0, q_empty = bar0 + 8;
    auto r_full = [&](int s) { return bar0 + 8u * (2 + s); };
    auto r_empty = [&](int s) { return bar0 + 8u * (2 + NS + s); };
    auto s_full = [&](int k) { return bar0 + 8u * (2 + 2 * NS + k); };
    auto p_full = [&](int k) { return bar0 + 8u * (4 + 2 * NS + k); };
    const uint32_t o_ready = bar0 + 8u * (6 + 2 * NS);
    const uint32_t o_final = o_ready + 8, o_empty = o_ready + 16;
    const uint32_t stats_full = o_ready + 24, stats_empty = o_ready + 32, drain = o_ready + 40;
    float* st_m = reinterpret_cast<float*>(smem + OFF_STATS);
    float* st_l = st_m + BM;
    volatile int* st_cnt = reinterpret_cast<volatile int*>(st_l + BM);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < NS; ++s) { mbar_init(r_full(s), 1); mbar_init(r_empty(s), 1); }
        for (int k = 0; k < 2; ++k) { mbar_init(s_full(k), 1); mbar_init(p_full(k), BM); }
        mbar_init(o_ready, 1);
        mbar_init(o_final, 1);
        mbar_init(o_empty, BM);
        mbar_init(stats_full, BM);
        mbar_init(stats_empty, BM);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= WARP_LOAD) {
        regs_dec<kRegsOther>();
        if (warp == WARP_LOAD) {
            // ------------------------------------------------------------ producer
            int nc = 0, nq = 0;                     // ring chunks and Q tiles issued
            bool ok = true;
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
            }
            // one ring slot: its barrier armed for 32 KB, then the boxes
            auto take_slot = [&](uint32_t& dst, uint32_t& full) -> bool {
                const int s = nc % NS;
                if (!mbar_wait(r_empty(s), ((nc / NS) & 1) ^ 1, abort_flag)) return false;
                full = r_full(s);
                dst = sb + OFF_RING + s * CHUNK;
                mbar_arrive_expect_tx(full, CHUNK);
                ++nc;
                return true;
            };
            auto load_k = [&](const Item& it, int j) -> bool {   // columns 128h .. 128h + 127, keys of tile j
                for (int h = 0; h < 2; ++h) {
                    uint32_t dst, full;
                    if (!take_slot(dst, full)) return false;
                    tma_load_4d(dst, &tm_k, full, 128 * h, j * BN, it.hkv, it.b);
                    tma_load_4d(dst + BOX, &tm_k, full, 128 * h + 64, j * BN, it.hkv, it.b);
                }
                return true;
            };
            auto load_v = [&](const Item& it, int j) -> bool {   // keys 64h .. 64h + 63 of tile j, all columns
                for (int h = 0; h < 2; ++h) {
                    uint32_t dst, full;
                    if (!take_slot(dst, full)) return false;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        tma_load_4d(dst + s * VBOX, &tm_v, full, 64 * s, j * BN + 64 * h, it.hkv, it.b);
                }
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int w = item_of(r);
                if (w < 0) break;
                const Item it = describe(w);
                const int c = count_tiles(it);
                if (c == 0) continue;
                if (lane == 0) {
                    ok = mbar_wait(q_empty, (nq & 1) ^ 1, abort_flag);
                    if (ok) {
                        mbar_arrive_expect_tx(q_full, 4 * BOX);
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            tma_load_4d(sb + OFF_Q + s * BOX, &tm_q, q_full, 64 * s, it.t.q0, it.hq, it.b);
                        ++nq;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                // K of tile 0, then (K of tile i+1, V of tile i) for each tile i
                TileIter tiles(it.mrow, it.first, it.t.n_tiles, it.t.kv_end, lane);
                int j = tiles.next();
                if (lane == 0) ok = load_k(it, j);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                while (ok && j >= 0) {
                    const int jn = tiles.next();
                    if (lane == 0) {
                        if (jn >= 0) ok = load_k(it, jn);
                        if (ok) ok = load_v(it, j);
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    j = jn;
                }
            }
            nc = __shfl_sync(0xffffffffu, nc, 0);
            nq = __shfl_sync(0xffffffffu, nq, 0);
            if (lane == 0 && *abort_flag) {
                // let the copies in flight land: the last load of each slot
                for (int s = 0; s < NS && s < nc; ++s) {
                    const int last = nc - 1 - ((nc - 1 - s) % NS);
                    mbar_drain(r_full(s), (last / NS) & 1);
                }
                if (nq > 0) mbar_drain(q_full, (nq - 1) & 1);
            }
        } else if (warp == WARP_MMA) {
            // ------------------------------------------------------------ MMA issuer
            int nc = 0, nq = 0;     // ring chunks and Q tiles consumed
            int g = 0;              // visited tiles of earlier items (S buffer / p_full parity)
            int oe = 0;             // o_empty phases waited
            bool ok = true;
            // waits for the two ring slots of the next chunk pair; returns the first slot
            auto take_pair = [&](int& s0) -> bool {
                s0 = nc % NS;
                if (!mbar_wait(r_full(s0), (nc / NS) & 1, abort_flag)) return false;
                if (!mbar_wait(r_full((nc + 1) % NS), ((nc + 1) / NS) & 1, abort_flag)) return false;
                tc_fence_after();
                return true;
            };
            auto release_pair = [&](int s0) {
                mma_commit(r_empty(s0));
                mma_commit(r_empty((s0 + 1) % NS));
                nc += 2;
            };
            // S of visited tile gi (global count) = Q K^T: K = 256 in 16 steps,
            // the first 8 from the first K half (columns 0-127), the rest from the second
            auto issue_qk = [&](int gi) -> bool {
                int s0;
                if (!take_pair(s0)) return false;
                const uint32_t k0 = sb + OFF_RING + s0 * CHUNK;
                const uint32_t k1 = sb + OFF_RING + ((s0 + 1) % NS) * CHUNK;
                const uint32_t d = tmem + COL_S0 + (gi & 1) * BN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qoff = (kk / 4) * BOX + (kk % 4) * 32;
                    const uint32_t koff = ((kk % 8) / 4) * BOX + (kk % 4) * 32;
                    mma_bf16_ss(d, make_sdesc_sw128(sb + OFF_Q + qoff, 16, 1024),
                                make_sdesc_sw128((kk < 8 ? k0 : k1) + koff, 16, 1024), IDESC_QK, kk > 0 ? 1u : 0u);
                }
                mma_commit(s_full(gi & 1));
                release_pair(s0);
                return true;
            };
            // O (+)= P V of visited tile gi: 8 steps of 16 keys, 4 from each V half;
            // the V boxes (64 columns x 64 keys) are MN-major operands spaced 8 KB apart
            auto issue_pv = [&](int gi, bool fresh) -> bool {
                if (!mbar_wait(p_full(gi & 1), (gi >> 1) & 1, abort_flag)) return false;
                int s0;
                if (!take_pair(s0)) return false;
                const uint32_t v0 = sb + OFF_RING + s0 * CHUNK;
                const uint32_t v1 = sb + OFF_RING + ((s0 + 1) % NS) * CHUNK;
                const uint32_t p = tmem + COL_S0 + (gi & 1) * BN;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t bdesc = make_sdesc_sw128((kk < 4 ? v0 : v1) + (kk % 4) * 16 * 128, VBOX, 1024);
                    mma_bf16_ts(tmem + COL_O, p + kk * 8, bdesc, IDESC_PV, (!fresh || kk > 0) ? 1u : 0u);
                }
                release_pair(s0);
                mma_commit(o_ready);
                return true;
            };
            // the epilogue of every earlier item has read O
            auto wait_o_empty = [&](int n_item) -> bool {
                for (; oe < n_item; ++oe)
                    if (!mbar_wait(o_empty, oe & 1, abort_flag)) return false;
                return true;
            };
            for (int r = 0, n_item = 0; ok; ++r, ++n_item) {
                const int w = item_of(r);
                if (w < 0) break;
                const Item it = describe(w);
                const int c = count_tiles(it);
                if (lane == 0) {
                    if (c > 0) {
                        ok = mbar_wait(q_full, nq++ & 1, abort_flag);
                        if (ok) ok = issue_qk(g);
                        if (ok && c > 1) ok = issue_qk(g + 1);
                        if (ok) ok = wait_o_empty(n_item);
                        if (ok) ok = issue_pv(g, true);
                        for (int i = 1; i + 1 < c && ok; ++i) {
                            ok = issue_qk(g + i + 1);
                            if (ok) ok = issue_pv(g + i, false);
                        }
                        if (ok) mma_commit(q_empty);        // every S of the item is issued
                        if (ok && c > 1) ok = issue_pv(g + c - 1, false);
                        g += c;
                    } else {
                        ok = wait_o_empty(n_item);
                    }
                    // one phase per item: every MMA of the item has completed
                    if (ok) mma_commit(o_final);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
            if (lane == 0) {
                mma_commit(drain);
                mbar_drain(drain, 0);
            }
            __syncwarp();
            named_bar_sync(2, 8 * 32 + 32);          // softmax and epilogue warps are done with TMEM
            tc_fence_after();
            tmem_dealloc(tmem, TMEM_COLS);
        }
    } else if (warp < WARP_EPI0) {
        regs_inc<kRegsSoftmax>();
        // ------------------------------------------------------------ softmax warps 0-3
        const int r = warp * 32 + lane;                        // row of the tile == TMEM lane
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        const float sl = a.scale_log2;
        int g = 0;                   // visited tiles so far
        int n = 0;                   // items finished
        bool ok = true;
        for (int rr = 0; ok; ++rr) {
            const int w = item_of(rr);
            if (w < 0) break;
            const Item itm = describe(w);
            const TileInfo ti = itm.t;
            const uint8_t* mrow = itm.mrow;
            const long p_row = (long)ti.q0 + r + a.Skv - a.Sq;
            const int lim = (int)key_hi(p_row, a.Skv, a.causal, wr);   // visible keys: [lo, lim)
            const int lo = (int)key_lo(p_row, a.Skv, wl);
            float m_ref = -INFINITY;
            float l_run = 0.f;
            int it = 0;
            TileIter tiles(mrow, itm.first, ti.n_tiles, ti.kv_end, lane);
            auto fetch = [&](int j, uint8_t* mb) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int key = j * BN + q * 32 + lane;
                    mb[q] = (mrow && j >= 0 && key < ti.kv_end) ? mrow[key] : (uint8_t)(mrow ? 0 : 1);
                }
            };
            int j = tiles.next();
            uint8_t mb[4];
            fetch(j, mb);
            while (j >= 0) {
                const int jn = tiles.next();
                uint8_t mbn[4];
                fetch(jn, mbn);
                uint32_t mw[4];
                bool all_kept = true;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    mw[q] = __ballot_sync(0xffffffffu, mb[q] != 0);
                    all_kept = all_kept && (mw[q] == 0xffffffffu);
                }
                const int kbase = j * BN;
                const bool need_mask = (kbase + BN > ti.lim_first) || kbase < ti.lo_last || !all_kept;
                const uint32_t col_s = COL_S0 + (g & 1) * BN;

                ok = __all_sync(0xffffffffu, mbar_wait(s_full(g & 1), (g >> 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                uint32_t sr[BN];
                tmem_ld128(tmem + lane_addr + col_s, sr);
                float* s = reinterpret_cast<float*>(sr);

                const bool capped = cap_out != 0.f;
                const bool fast = !need_mask && sl > 0.f && !capped;
                float mx8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
                if (fast) {
#pragma unroll
                    for (int c = 0; c < BN; c += 2) mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], s[c], s[c + 1]);
                } else {
                    uint32_t vis[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int rel = lim - (kbase + 32 * q);
                        const uint32_t below = rel >= 32 ? 0xffffffffu : (rel <= 0 ? 0u : ((1u << rel) - 1u));
                        const int rlo = lo - (kbase + 32 * q);
                        const uint32_t above = rlo <= 0 ? 0xffffffffu : (rlo >= 32 ? 0u : ~((1u << rlo) - 1u));
                        vis[q] = mw[q] & below & above;
                    }
                    if (capped) {
#pragma unroll
                        for (int c = 0; c < BN; ++c) {
                            const float x = ((vis[c / 32] >> (c % 32)) & 1u)
                                                ? softcap_log2(s[c], cap_in, cap_out) : -INFINITY;
                            s[c] = x;
                            mx8[c & 7] = fmaxf(mx8[c & 7], x);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < BN; ++c) {
                            const float x = ((vis[c / 32] >> (c % 32)) & 1u) ? s[c] * sl : -INFINITY;
                            s[c] = x;
                            mx8[c & 7] = fmaxf(mx8[c & 7], x);
                        }
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
                const float fa = fast ? sl : 1.f;
                uint32_t pk[BN / 2];
                const float rs = exp_row<0, F16>(s, fa, m_use, pk);
                tmem_st64(tmem + lane_addr + col_s, pk);          // P over the first 64 columns of S
                l_run = l_run * alpha + rs;

                if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // PV of the previous tile must have completed before O is rescaled
                    ok = __all_sync(0xffffffffu, mbar_wait(o_ready, (g - 1) & 1, abort_flag));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tmem + lane_addr + COL_O + 32 * c, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= alpha;
                        tmem_st32(tmem + lane_addr + COL_O + 32 * c, reinterpret_cast<uint32_t*>(o));
                    }
                }
                tc_fence_before();
                mbar_arrive(p_full(g & 1));
                ++it;
                ++g;
                j = jn;
#pragma unroll
                for (int q = 0; q < 4; ++q) mb[q] = mbn[q];
            }
            if (!ok) break;
            // hand the row statistics to the epilogue once it has read the previous ones
            if (n > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(stats_empty, (n - 1) & 1, abort_flag));
                if (!ok) break;
            }
            st_m[r] = m_ref;
            st_l[r] = l_run;
            if (r == 0) *st_cnt = it;
            mbar_arrive(stats_full);
            ++n;
        }
        named_bar_arrive(2, 8 * 32 + 32);
    } else {
        regs_dec<kRegsEpi>();
        // ------------------------------------------------------------ epilogue warps 4-7
        const int r = (warp - WARP_EPI0) * 32 + lane;
        const uint32_t lane_addr = (uint32_t)((warp % 4) * 32) << 16;
        int n = 0;                   // items finished
        int nb = 0;                  // output boxes stored (staging buffer alternation)
        bool ok = true;
        for (int rr = 0;; ++rr) {
            const int w = item_of(rr);
            if (w < 0) break;
            const Item itm = describe(w);
            const TileInfo ti = itm.t;
            ok = mbar_wait(stats_full, n & 1, abort_flag) && mbar_wait(o_final, n & 1, abort_flag);
            if (!named_bar_and(3, BM, ok)) break;     // the whole warpgroup stops together
            tc_fence_after();
            const int cnt = *st_cnt;
            const float m_ref = st_m[r];
            const float l_run = st_l[r];
            const int row_q = ti.q0 + r;
            const bool row_ok = r < ti.rows_valid;
            float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            float lse2 = l_run > 0.f ? m_ref + log2f(l_run) : -INFINITY;
            if (sinks && l_run > 0.f) {
                const float s2 = sinks[itm.hq] * 1.4426950408889634f;
                if (s2 == INFINITY) {
                    inv = 0.f;
                    lse2 = INFINITY;
                } else {
                    const float M = fmaxf(m_ref, s2);
                    const float keep = fast_exp2(m_ref - M);
                    const float l_tot = l_run * keep + fast_exp2(s2 - M);
                    inv = keep / l_tot;
                    lse2 = M + log2f(l_tot);
                }
            }
            if (cnt > 0) {
                // O / l packed to 16 bits, 128 columns at a time; O is free once
                // the second half is read
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t ow[64];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float f[32];
                        tmem_ld32(tmem + lane_addr + COL_O + 128 * half + 32 * c, f);
#pragma unroll
                        for (int e = 0; e < 16; ++e) ow[16 * c + e] = pack2<F16>(f[2 * e] * inv, f[2 * e + 1] * inv);
                    }
                    if (half == 1) {
                        tc_fence_before();
                        mbar_arrive(stats_empty);
                        mbar_arrive(o_empty);
                    }
                    // two 64-column boxes through the alternating staging buffers
#pragma unroll
                    for (int sub = 0; sub < 2; ++sub, ++nb) {
                        const uint32_t stage = sb + OFF_STAGE + (nb & 1) * BOX;
                        if (r == 0) bulk_wait_read_1();       // the store two boxes back has read this buffer
                        named_bar_sync(3, BM);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint32_t* u = ow + 32 * sub + 4 * q;
                            st_shared_v4(stage + r * 128 + ((q ^ (r & 7)) << 4), u[0], u[1], u[2], u[3]);
                        }
                        fence_proxy_async_smem();
                        named_bar_sync(3, BM);
                        if (r == 0) {
                            tma_store_4d(&tm_o, stage, 128 * half + 64 * sub, ti.q0, itm.hq, itm.b);
                            bulk_commit_group();
                        }
                    }
                }
            } else {
                mbar_arrive(stats_empty);
                mbar_arrive(o_empty);
                if (row_ok) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) +
                                                          (((size_t)itm.b * a.Sq + row_q) * a.Hq + itm.hq) * D);
#pragma unroll
                    for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (row_ok && a.lse) a.lse[((size_t)itm.b * a.Sq + row_q) * a.Hq + itm.hq] = lse2 * kLn2;
            ++n;
        }
        if (r == 0) bulk_wait_read_all();
        tc_fence_before();
        named_bar_arrive(2, 8 * 32 + 32);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(&g_prefill256_error, (int)kErrPrefillWait);
}

template <bool OPTS, bool F16>
cudaError_t launch_t(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                     const CUtensorMap& tm_o, const PrefillArgs& a, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(prefill_d256_kernel<OPTS, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_qtiles = (a.Sq + BM - 1) / BM;
    const long n_items = (long)n_qtiles * a.B * a.Hq;
    const long sms = a.num_sms > 0 ? a.num_sms : 148;
    const long grid = n_items < sms ? n_items : sms;    // persistent: one CTA per SM
    prefill_d256_kernel<OPTS, F16><<<(unsigned)grid, NUM_THREADS, SMEM_BYTES, stream>>>(tm_q, tm_k, tm_v, tm_o, a,
                                                                                       n_qtiles);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_d256(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& tm_o, const PrefillArgs& a, cudaStream_t stream) {
    if (a.D != D) return cudaErrorInvalidValue;
    const bool opts = a.x.wl >= 0 || a.x.wr >= 0 || a.x.cap_out != 0.f || a.x.sinks != nullptr;
    switch ((opts ? 1 : 0) + (a.f16 ? 2 : 0)) {
        case 0: return launch_t<false, false>(tm_q, tm_k, tm_v, tm_o, a, stream);
        case 1: return launch_t<true, false>(tm_q, tm_k, tm_v, tm_o, a, stream);
        case 2: return launch_t<false, true>(tm_q, tm_k, tm_v, tm_o, a, stream);
        default: return launch_t<true, true>(tm_q, tm_k, tm_v, tm_o, a, stream);
    }
}

int prefill_d256_take_device_error() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_prefill256_error, sizeof(int)) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_prefill256_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace gqa
