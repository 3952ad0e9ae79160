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
// One CTA owns two 128-row query tiles (Q0, Q1) of one (b, h); both read the
// same K/V tiles.  The same kernel serves packed THD calls (variable-length
// requests laid end to end): there a query tile holds the g query heads of one
// KV head for 128 / g consecutive queries of one request, the two tiles are
// consecutive row blocks of that request, and the CTAs claim such items from a
// counter in the call's workspace in the order a plan kernel wrote.  Warp roles:
//   warp 8     TMA producer: Q0 and Q1 once, then K_j and V_j tiles through two
//              shared-memory rings (128-byte swizzle, 64-column boxes);
//   warp 9     MMA issuer (one thread): S_k = Q_k K_j^T into TMEM, then
//              O_k += P_k V_j with P_k read from TMEM, alternating k = 0, 1 so
//              the tensor core works on one tile while the other is softmaxed;
//   warps 0-3  softmax of Q0, warps 4-7 softmax of Q1: thread t owns row t; it
//              reads its S row from TMEM, folds the causal / padding mask,
//              updates the running max and sum, writes P (bf16) back over its
//              S row, rescales its O row when needed, and finally normalises O
//              into its Q tile's shared-memory buffer, from which one thread
//              stores the tile with TMA, and writes the LSE.
// Warps 10-11 complete the third warpgroup (register rebalancing works per
// warpgroup); in packed calls they zero the value rows past a request's end in
// its last key tile before that tile's P V.  TMEM (512 columns): S0 | S1 |
// O0 | O1; P_k occupies the first 64 columns of S_k.
//
// The O rescale is lazy: the reference max of a row only moves when the tile
// max exceeds it by more than kRescaleThreshold (log2 units), so most tiles
// touch no O at all.  Once every row of a warp has a reference, a tile is
// exponentiated against it without taking its row max; only a row sum above
// kSumLimit (2^32) sends the warp back to the scores in TMEM for the max.  The
// result is exact either way: O and l are accumulated against the same
// reference.  A rescale of O_k before PV of tile i needs PV of tile i-1
// complete; that is implied by S_k of tile i having landed, since its commit
// follows that PV in the MMA thread's order.
//
// Key tiles holding no visible key (beyond the causal bound or fully padded)
// are never loaded, and tiles past Q0's causal bound are skipped for Q0.
// Every wait is bounded (ptx.cuh); on a timeout the CTA stops issuing work,
// drains what is in flight, frees TMEM and returns.
#include <cmath>

#include "internal.h"
#include "prefill_tiles.cuh"
#include "ptx.cuh"

namespace gqa {
namespace {

__device__ int g_prefill_error;

using namespace pf;
// Layouts: dense BSHD calls (attn_fwd_dense) and packed THD rows
// (attn_fwd_varlen).
constexpr int kModeDense = 0, kModePacked = 1;
constexpr int NQ = 2;              // Q tiles per CTA
constexpr int NUM_THREADS = 384;   // warps 0-7 softmax, 8 producer, 9 MMA, 10-11 idle
constexpr int WARP_LOAD = 8;
constexpr int WARP_MMA = 9;
// Registers per thread: the launch gives 168 to all 384 threads (64,512); the
// two softmax warpgroups take 192 each and the producer/MMA warpgroup keeps
// 120 (its peeled issue loop needs them; measured best of 208/88 ... 176/152):
// 192 * 256 + 120 * 128 = 64,512, the launch total.
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 192;
constexpr int kRegsOther = 120;
static_assert(kRegsSoftmax * 256 + kRegsOther * 128 <= kRegsLaunch * NUM_THREADS, "register split");

template <int D>
struct Cfg {
    static constexpr int KSUB = D / 64;                 // 64-column (128-byte) boxes per row
    static constexpr int SUB_BYTES = BN * 128;          // one box: 128 rows x 128 bytes
    static constexpr int TILE_BYTES = KSUB * SUB_BYTES; // one Q, K or V tile
    static constexpr int NK = D == 64 ? 4 : 2;          // K ring depth
    static constexpr int NV = D == 64 ? 4 : 2;          // V ring depth
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NQ * TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
    static constexpr int OFF_STAGE = OFF_V + NV * TILE_BYTES;   // one 64-column output box per Q tile
    static constexpr int OFF_BAR = OFF_STAGE + NQ * SUB_BYTES;
    // q_full[2], q_empty[2], k_full[NK], k_empty[NK], v_full[NV], v_empty[NV],
    // s_full[2], p_full[2], o_final[2], drain, info_full[2], info_empty[2],
    // v_landed, v_fixed
    static constexpr int NBAR = 4 + 2 * NK + 2 * NV + 6 + 1 + 4 + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    // two 64-byte item records (tile counts, first flag word, first tile's mask
    // words, the item's index)
    static constexpr int OFF_INFO = OFF_MISC + 16;
    static constexpr int SMEM_USED = OFF_INFO + 2 * 64;
    // 1 KB alignment slack; at least 120 KB so that one CTA holds an SM (it
    // takes all 512 TMEM columns).
    static constexpr int SMEM_BYTES = SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024;
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128;
    static constexpr uint32_t COL_O0 = 256, COL_O1 = 256 + D;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(COL_O1 + D <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// OPTS: the call has a window, a softcap or sinks.  Without them every option
// term is a compile-time constant and the code is the plain causal / padded
// kernel.
template <int D, int MODE, bool OPTS, bool F16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const PrefillArgs a, int n_qpairs) {
    using C = Cfg<D>;
    constexpr bool PACKED = MODE != kModeDense;
    // both MMA operands of the call's 16-bit type (P is packed to it as well)
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

    // Work items.  Dense: w = 0 .. n_items-1, heaviest (last) query tiles
    // first and adjacent items on one KV head; round r of this persistent CTA
    // takes item r * G + cta (even r) or r * G + G - 1 - cta (odd r), so heavy
    // and light items alternate across rounds.  Packed: item w = (pair entry
    // w / Hkv of the plan, KV head w % Hkv), two consecutive row blocks of one
    // request, claimed in the plan's order from the workspace's counter.  The
    // producer hands every item's index to the other roles in its record.
    const int bh = a.B * a.Hq;
    const int g = PACKED ? a.g : 1;              // query rows per query (heads of a KV group)
    const int qpb = PACKED ? a.qpb : BM;         // queries per Q tile
    const int n_items = PACKED ? *a.n_entries * a.Hkv : n_qpairs * bh;
    const int G = gridDim.x;
    const int cta = blockIdx.x;
    auto item_of = [&](int r) -> int {
        const long w = (long)r * G + ((r & 1) ? G - 1 - cta : cta);
        return w < n_items ? (int)w : -1;
    };
    struct Item {
        int b, hq, hkv, q0, first, n_all, kv_end_all;
        int qs, ks, sq, skv;    // packed: first query / key row of the request, its queries and keys
        TileInfo t0, t1;        // t_k.q0: first query of Q tile k (within the request)
        const uint8_t* mrow;
    };
    auto describe = [&](int w) {
        Item it;
        if constexpr (PACKED) {
            const int4* e = reinterpret_cast<const int4*>(a.entries + (size_t)(w / a.Hkv) * 8);
            const int4 e0 = e[0], e1 = e[1];
            it.b = e0.x;
            it.hkv = w % a.Hkv;
            it.hq = it.hkv * g;
            it.q0 = e0.y;
            it.qs = e0.z;
            it.sq = e0.w;
            it.ks = e1.x;
            it.skv = e1.y;
            it.t0 = tile_info_n(it.q0, qpb, it.sq, it.skv, a.causal, wl, wr);
            it.t1 = tile_info_n(it.q0 + qpb, qpb, it.sq, it.skv, a.causal, wl, wr);
        } else {
            const int qp = n_qpairs - 1 - w / bh;
            const int rem = w % bh;
            it.hq = rem % a.Hq;
            it.b = rem / a.Hq;
            it.hkv = it.hq / (a.Hq / a.Hkv);
            it.q0 = qp * (NQ * BM);
            it.qs = it.ks = 0;
            it.sq = a.Sq;
            it.skv = a.Skv;
            it.t0 = tile_info(it.q0, a.Sq, a.Skv, a.causal, wl, wr);
            it.t1 = tile_info(it.q0 + BM, a.Sq, a.Skv, a.causal, wl, wr);
        }
        it.n_all = max(it.t0.n_tiles, it.t1.n_tiles);
        it.kv_end_all = max(it.t0.kv_end, it.t1.kv_end);
        // both Q tiles walk the tiles from the first one either needs (Q1's
        // window starts later: its extra leading tiles are fully masked)
        it.first = (it.t0.n_tiles > 0 ? it.t0.kv_begin : it.t1.kv_begin) / BN;
        it.mrow = (!PACKED && a.mask) ? a.mask + (size_t)it.b * a.Skv : nullptr;
        return it;
    };
    // Visited key tiles of an item (non-empty, from its first tile to kv_end of
    // either Q tile) are numbered i = 0, 1, ...; Q_k takes part in the first c_k
    // of them.  Warp-collective.
    auto count_tiles = [&](const Item& it, int& c0, int& c1, int& c_all, uint32_t& f0) {
        c0 = c1 = c_all = 0;
        f0 = 0;
        for (int chunk = it.first / 32; chunk * 32 < it.n_all; ++chunk) {
            const uint32_t f = tile_flags(it.mrow, chunk, it.first, it.n_all, it.kv_end_all, lane);
            if (chunk == it.first / 32) f0 = f;
            c_all += __popc(f);
            c0 += __popc(f & below_bits(it.t0.n_tiles, chunk));
            c1 += __popc(f & below_bits(it.t1.n_tiles, chunk));
        }
    };

    const uint32_t bar0 = sb + C::OFF_BAR;
    auto q_full = [&](int k) { return bar0 + 8u * k; };
    auto q_empty = [&](int k) { return bar0 + 8u * (2 + k); };
    auto k_full = [&](int i) { return bar0 + 8u * (4 + i); };
    auto k_empty = [&](int i) { return bar0 + 8u * (4 + C::NK + i); };
    auto v_full = [&](int i) { return bar0 + 8u * (4 + 2 * C::NK + i); };
    auto v_empty = [&](int i) { return bar0 + 8u * (4 + 2 * C::NK + C::NV + i); };
    auto s_full = [&](int k) { return bar0 + 8u * (4 + 2 * C::NK + 2 * C::NV + k); };
    auto p_full = [&](int k) { return bar0 + 8u * (6 + 2 * C::NK + 2 * C::NV + k); };
    auto o_final = [&](int k) { return bar0 + 8u * (8 + 2 * C::NK + 2 * C::NV + k); };
    const uint32_t drain = bar0 + 8u * (10 + 2 * C::NK + 2 * C::NV);
    auto info_full = [&](int i) { return bar0 + 8u * (11 + 2 * C::NK + 2 * C::NV + i); };
    auto info_empty = [&](int i) { return bar0 + 8u * (13 + 2 * C::NK + 2 * C::NV + i); };
    // packed: the value rows past the request's end in an item's last tile are
    // zeroed (warps 10-11) before its P V: the MMA thread, which takes the
    // tiles in order, signals v_landed once that tile is in and waits for
    // v_fixed
    const uint32_t v_landed = bar0 + 8u * (15 + 2 * C::NK + 2 * C::NV);
    const uint32_t v_fixed = bar0 + 8u * (16 + 2 * C::NK + 2 * C::NV);
    // Item records, written by the producer one item ahead of its consumers:
    // c0, c1, c_all, the flag word of the first 32-tile chunk and the mask
    // words of the first visited tile, so that no consumer scans the padding
    // mask in global memory at an item boundary.
    uint32_t* info = reinterpret_cast<uint32_t*>(smem + C::OFF_INFO);
    constexpr int REC = PACKED ? 16 : 8;   // words per record (packed: the item's index in word 8)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    if (threadIdx.x == 0) {
        for (int k = 0; k < NQ; ++k) {
            mbar_init(q_full(k), 1);
            mbar_init(q_empty(k), 1);
            mbar_init(s_full(k), 1);
            mbar_init(p_full(k), BM);
            mbar_init(o_final(k), 1);
        }
        for (int i = 0; i < C::NK; ++i) { mbar_init(k_full(i), 1); mbar_init(k_empty(i), 1); }
        for (int i = 0; i < C::NV; ++i) { mbar_init(v_full(i), 1); mbar_init(v_empty(i), 1); }
        mbar_init(drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(info_full(i), 1);
            // the MMA thread and the eight softmax warps (packed: and warps 10-11)
            mbar_init(info_empty(i), PACKED ? 1 + 8 + 2 : 1 + 8);
        }
        mbar_init(v_landed, 1);
        mbar_init(v_fixed, 2);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if constexpr (PACKED) {
        // Q rows past g * qpb are never loaded: zero them once (finite rows,
        // whose results are never stored)
        const int rows = g * qpb;
        const int per = (BM - rows) * 8 * C::KSUB;   // 16-byte chunks per Q tile
        for (int x = threadIdx.x; x < NQ * per; x += NUM_THREADS) {
            const int kq = x / per, y = x % per;
            const int row = rows + y / (8 * C::KSUB), sl = (y / 8) % C::KSUB, q = y % 8;
            *reinterpret_cast<uint4*>(smem + C::OFF_Q + kq * C::TILE_BYTES + sl * C::SUB_BYTES + row * 128 + q * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Each role ends on its own (no shared tail), so register limits apply per
    // role: the MMA warp frees TMEM once the softmax warps have arrived on
    // barrier 2 after their last TMEM access.
    if (warp >= 8) {
        regs_dec<kRegsOther>();
        if (warp == WARP_LOAD) {
            // ------------------------------------------------------------ producer
            int nk = 0, nv = 0, nq0 = 0, nq1 = 0;   // loads issued so far
            bool ok = true;
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
            }
            for (int r = 0; ok; ++r) {
                int w;
                if constexpr (PACKED) {
                    w = -1;
                    if (lane == 0) {
                        w = atomicAdd(a.work, 1);
                        if (w >= n_items) w = -1;
                    }
                    w = __shfl_sync(0xffffffffu, w, 0);
                } else {
                    w = item_of(r);
                }
                if (w < 0) {
                    // packed: a last record with no item (dense consumers
                    // know the item count)
                    if (PACKED && lane == 0) {
                        const int slot = r & 1;
                        if (mbar_wait(info_empty(slot), ((r >> 1) & 1) ^ 1, abort_flag)) {
                            info[REC * slot + 8] = 0xffffffffu;
                            mbar_arrive(info_full(slot));
                        }
                    }
                    break;
                }
                const Item it = describe(w);
                int c0, c1, c_all;
                uint32_t f0;
                count_tiles(it, c0, c1, c_all, f0);
                TileIter tiles(it.mrow, it.first, it.n_all, it.kv_end_all, lane, f0);
                int j = tiles.next();                  // first visited tile, -1 if none
                uint32_t mw0[4];                       // its kept keys, as the softmax forms them
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int key = j * BN + q * 32 + lane;
                    const bool keep = it.mrow ? (j >= 0 && key < it.kv_end_all && it.mrow[key] != 0) : true;
                    mw0[q] = __ballot_sync(0xffffffffu, keep);
                }
                if (lane == 0) {
                    const int slot = r & 1;
                    ok = mbar_wait(info_empty(slot), ((r >> 1) & 1) ^ 1, abort_flag);
                    if (ok) {
                        uint32_t* rec = info + REC * slot;
                        if constexpr (PACKED) rec[8] = (uint32_t)w;
                        rec[0] = (uint32_t)c0;
                        rec[1] = (uint32_t)c1;
                        rec[2] = (uint32_t)c_all;
                        rec[3] = f0;
#pragma unroll
                        for (int q = 0; q < 4; ++q) rec[4 + q] = mw0[q];
                        mbar_arrive(info_full(slot));
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok || c_all == 0) continue;
                // Load order Q0, K(first), Q1, V(first), K, V, ...: S0 of the first
                // tile can start before Q1 has landed.  Q_k is loaded once the last
                // S of the previous Q_k is done.
                auto load_q = [&](int k) -> bool {   // lane 0
                    const int nq = k == 0 ? nq0 : nq1;
                    if (!mbar_wait(q_empty(k), (nq & 1) ^ 1, abort_flag)) return false;
                    if constexpr (PACKED) {
                        // {64, g, qpb} boxes: row q * g + h of the tile is query q, head hq + h
                        mbar_arrive_expect_tx(q_full(k), (uint32_t)(C::KSUB * g * qpb * 128));
#pragma unroll
                        for (int s = 0; s < C::KSUB; ++s)
                            tma_load_3d(sb + C::OFF_Q + k * C::TILE_BYTES + s * C::SUB_BYTES, &tm_q, q_full(k),
                                        s * 64, it.hq, it.qs + it.q0 + k * qpb);
                    } else {
                        mbar_arrive_expect_tx(q_full(k), C::TILE_BYTES);
#pragma unroll
                        for (int s = 0; s < C::KSUB; ++s)
                            tma_load_4d(sb + C::OFF_Q + k * C::TILE_BYTES + s * C::SUB_BYTES, &tm_q, q_full(k),
                                        s * 64, it.q0 + k * BM, it.hq, it.b);
                    }
                    if (k == 0) ++nq0; else ++nq1;
                    return true;
                };
                if (lane == 0 && c0 > 0) ok = load_q(0);
                bool q1_due = c1 > 0;
                for (; j >= 0 && __shfl_sync(0xffffffffu, ok, 0); j = tiles.next()) {
                    if (lane == 0) {
                        const int ks = nk % C::NK;
                        ok = mbar_wait(k_empty(ks), ((nk / C::NK) & 1) ^ 1, abort_flag);
                        if (ok) {
                            mbar_arrive_expect_tx(k_full(ks), C::TILE_BYTES);
#pragma unroll
                            for (int s = 0; s < C::KSUB; ++s) {
                                const uint32_t dst = sb + C::OFF_K + ks * C::TILE_BYTES + s * C::SUB_BYTES;
                                if constexpr (PACKED)
                                    tma_load_3d(dst, &tm_k, k_full(ks), s * 64, it.hkv, it.ks + j * BN);
                                else
                                    tma_load_4d(dst, &tm_k, k_full(ks), s * 64, j * BN, it.hkv, it.b);
                            }
                            ++nk;
                        }
                        if (ok && q1_due) ok = load_q(1);
                        if (ok) {
                            const int vs = nv % C::NV;
                            ok = mbar_wait(v_empty(vs), ((nv / C::NV) & 1) ^ 1, abort_flag);
                            if (ok) {
                                mbar_arrive_expect_tx(v_full(vs), C::TILE_BYTES);
#pragma unroll
                                for (int s = 0; s < C::KSUB; ++s) {
                                    const uint32_t dst = sb + C::OFF_V + vs * C::TILE_BYTES + s * C::SUB_BYTES;
                                    if constexpr (PACKED)
                                        tma_load_3d(dst, &tm_v, v_full(vs), s * 64, it.hkv, it.ks + j * BN);
                                    else
                                        tma_load_4d(dst, &tm_v, v_full(vs), s * 64, j * BN, it.hkv, it.b);
                                }
                                ++nv;
                            }
                        }
                    }
                    q1_due = false;
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
            if (lane == 0 && *abort_flag) {
                // Let copies already in flight land before the CTA goes away:
                // wait for the last load issued into each slot.
                for (int s = 0; s < C::NK && s < nk; ++s) {
                    const int last = nk - 1 - ((nk - 1 - s) % C::NK);
                    mbar_drain(k_full(s), (last / C::NK) & 1);
                }
                for (int s = 0; s < C::NV && s < nv; ++s) {
                    const int last = nv - 1 - ((nv - 1 - s) % C::NV);
                    mbar_drain(v_full(s), (last / C::NV) & 1);
                }
                if (nq0 > 0) mbar_drain(q_full(0), (nq0 - 1) & 1);
                if (nq1 > 0) mbar_drain(q_full(1), (nq1 - 1) & 1);
            }
        } else if (warp == WARP_MMA) {
            // ------------------------------------------------------------ MMA issuer
            int kt = 0, vt = 0;                    // K and V tiles consumed by earlier items
            int nq0 = 0, nq1 = 0, pc0 = 0, pc1 = 0;   // Q loads consumed, P tiles taken
            int nfix = 0;                          // v_fixed phases waited (packed)
            bool ok = true;
            for (int r = 0; ok; ++r) {
                if (!PACKED && item_of(r) < 0) break;  // dense: no record past the last item
                int c0 = 0, c1 = 0, c_all = 0;         // lane 0 holds the item's tile counts
                int w = 0;
                if (lane == 0) {
                    const int slot = r & 1;
                    ok = mbar_wait(info_full(slot), (r >> 1) & 1, abort_flag);
                    if (ok) {
                        if constexpr (PACKED) w = (int)info[REC * slot + 8];
                        c0 = (int)info[REC * slot];
                        c1 = (int)info[REC * slot + 1];
                        c_all = (int)info[REC * slot + 2];
                        mbar_arrive(info_empty(slot));
                    }
                }
                if constexpr (PACKED) {
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (__shfl_sync(0xffffffffu, w, 0) < 0) break;  // the last record (or a wait gave up)
                }
                if (lane == 0 && ok && c_all > 0) {
                    auto issue_s = [&](int k, int slot) {
                        const uint32_t kbase = sb + C::OFF_K + slot * C::TILE_BYTES;
                        const uint32_t qbase = sb + C::OFF_Q + k * C::TILE_BYTES;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t koff = (kk / 4) * C::SUB_BYTES + (kk % 4) * 32;
                            mma_bf16_ss(tmem + (k == 0 ? C::COL_S0 : C::COL_S1),
                                        make_sdesc_sw128(qbase + koff, 16, 1024),
                                        make_sdesc_sw128(kbase + koff, 16, 1024), IDESC_QK, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(s_full(k));
                    };
                    auto issue_pv = [&](int k, int slot, int i) {
                        const uint32_t vbase = sb + C::OFF_V + slot * C::TILE_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            // keys 16kk..16kk+15 of V: rows 16kk.. of every 64-column box
                            const uint64_t bdesc = make_sdesc_sw128(vbase + kk * 16 * 128, C::SUB_BYTES, 1024);
                            mma_bf16_ts(tmem + (k == 0 ? C::COL_O0 : C::COL_O1),
                                        tmem + (k == 0 ? C::COL_S0 : C::COL_S1) + kk * 8, bdesc, IDESC_PV,
                                        (i > 0 || kk > 0) ? 1u : 0u);
                        }
                    };
                    // V of visited tile i (ring slot vs); packed: the item's last tile
                    // also waits for its value rows past the request's end to be zeroed
                    auto wait_v = [&](int i, int vs) -> bool {
                        if (!mbar_wait(v_full(vs), ((vt + i) / C::NV) & 1, abort_flag)) return false;
                        if (PACKED && i == c_all - 1) {
                            mbar_arrive(v_landed);
                            if (!mbar_wait(v_fixed, nfix & 1, abort_flag)) return false;
                            ++nfix;
                        }
                        return true;
                    };
                    // first tile: S0 once Q0 and K are in, S1 once Q1 is (loaded after K)
                    if (c0 > 0) ok = mbar_wait(q_full(0), nq0++ & 1, abort_flag);
                    if (ok) ok = mbar_wait(k_full(kt % C::NK), (kt / C::NK) & 1, abort_flag);
                    if (ok) {
                        tc_fence_after();
                        if (c0 > 0) issue_s(0, kt % C::NK);
                    }
                    if (ok && c1 > 0) {
                        ok = mbar_wait(q_full(1), nq1++ & 1, abort_flag);
                        if (ok) {
                            tc_fence_after();
                            issue_s(1, kt % C::NK);
                        }
                    }
                    if (ok) mma_commit(k_empty(kt % C::NK));
                    // Common causal case (Q1 sees Q0's tiles, plus at most one more):
                    // the loop is peeled where Q0 ends, so that o_final(0) is
                    // committed right after Q0's last P V and Q0's epilogue
                    // overlaps Q1's last tile, with no conditional in the loop.
                    const bool peel = c0 >= 1 && c1 == c_all && (c1 == c0 || c1 == c0 + 1);
                    if (peel && ok) {
                        auto pv = [&](int k, int vs, int i) -> bool {
                            const int pc = k == 0 ? pc0++ : pc1++;
                            if (!mbar_wait(p_full(k), pc & 1, abort_flag)) return false;
                            tc_fence_after();
                            issue_pv(k, vs, i);
                            return true;
                        };
                        auto wait_k = [&](int kn) -> bool {
                            if (!mbar_wait(k_full(kn % C::NK), (kn / C::NK) & 1, abort_flag)) return false;
                            tc_fence_after();
                            return true;
                        };
                        // tiles 0 .. c0-2: both Q tiles take P V of tile i and S of tile i+1
                        for (int i = 0; i + 1 < c0 && ok; ++i) {
                            const int vs = (vt + i) % C::NV;
                            const int kn = kt + i + 1;
                            ok = wait_v(i, vs);
                            if (ok) ok = pv(0, vs, i);
                            if (ok) ok = wait_k(kn);
                            if (!ok) break;
                            issue_s(0, kn % C::NK);
                            if (!pv(1, vs, i)) { ok = false; break; }
                            issue_s(1, kn % C::NK);
                            mma_commit(v_empty(vs));
                            mma_commit(k_empty(kn % C::NK));
                        }
                        // every S0 of the item is issued: Q0 may be replaced
                        if (ok) mma_commit(q_empty(0));
                        // tile c0-1: Q0's last P V, then its epilogue may start
                        const int i = c0 - 1;
                        const int vs = (vt + i) % C::NV;
                        if (ok) ok = wait_v(i, vs);
                        if (ok) ok = pv(0, vs, i);
                        if (ok) mma_commit(o_final(0));
                        if (ok && c1 == c0 + 1) {
                            const int kn = kt + c0;
                            ok = wait_k(kn);
                            if (ok) ok = pv(1, vs, i);
                            if (ok) {
                                issue_s(1, kn % C::NK);
                                mma_commit(v_empty(vs));
                                mma_commit(k_empty(kn % C::NK));
                                mma_commit(q_empty(1));
                                const int vs2 = (vt + c0) % C::NV;
                                ok = wait_v(c0, vs2);
                                if (ok) ok = pv(1, vs2, c0);
                                if (ok) mma_commit(v_empty(vs2));
                            }
                        } else if (ok) {
                            mma_commit(q_empty(1));
                            ok = pv(1, vs, i);
                            if (ok) mma_commit(v_empty(vs));
                        }
                        if (ok) mma_commit(o_final(1));
                        kt += c_all;
                        vt += c_all;
                    }
                    // Visited tiles 0 .. c_all-2: P V of tile i, then S of tile i+1.
                    // The item's commits of q_empty / o_final come after the loop:
                    // conditional commits inside it slowed the steady state.
                    for (int i = 0; !peel && i + 1 < c_all && ok; ++i) {
                        const int vs = (vt + i) % C::NV;
                        ok = wait_v(i, vs);
                        if (!ok) break;
                        const int kn = kt + i + 1;     // K tile of visited tile i+1
                        for (int k = 0; k < NQ && ok; ++k) {
                            const int cnt = k == 0 ? c0 : c1;
                            if (i < cnt) {
                                const int pc = k == 0 ? pc0++ : pc1++;
                                ok = mbar_wait(p_full(k), pc & 1, abort_flag);
                                if (!ok) break;
                                tc_fence_after();
                                issue_pv(k, vs, i);
                            }
                            if (k == 0) {
                                ok = mbar_wait(k_full(kn % C::NK), (kn / C::NK) & 1, abort_flag);
                                if (!ok) break;
                                tc_fence_after();
                            }
                            // S_k of tile i+1 overwrites P_k of tile i: issued after its PV.
                            if (i + 1 < cnt) issue_s(k, kn % C::NK);
                        }
                        if (!ok) break;
                        mma_commit(v_empty(vs));
                        mma_commit(k_empty(kn % C::NK));
                    }
                    // every S of the item is issued: its Q tiles may be replaced
                    if (!peel && ok) {
                        if (c0 > 0) mma_commit(q_empty(0));
                        if (c1 > 0) mma_commit(q_empty(1));
                    }
                    // the last visited tile: P V only
                    if (!peel && ok) {
                        const int i = c_all - 1;
                        const int vs = (vt + i) % C::NV;
                        ok = wait_v(i, vs);
                        for (int k = 0; k < NQ && ok; ++k) {
                            const int cnt = k == 0 ? c0 : c1;
                            if (i < cnt) {
                                const int pc = k == 0 ? pc0++ : pc1++;
                                ok = mbar_wait(p_full(k), pc & 1, abort_flag);
                                if (!ok) break;
                                tc_fence_after();
                                issue_pv(k, vs, i);
                            }
                        }
                        if (ok) mma_commit(v_empty(vs));
                        kt += c_all;
                        vt += c_all;
                        if (ok) {
                            mma_commit(o_final(0));
                            mma_commit(o_final(1));
                        }
                    }
                }
                // one o_final phase per Q tile and item (also for a tile with no key):
                // arrives when every MMA of the item has completed
                if (lane == 0 && ok && c_all == 0) {
                    mma_commit(o_final(0));
                    mma_commit(o_final(1));
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
            if (lane == 0) {
                mma_commit(drain);                // every MMA issued above has completed once this arrives
                mbar_drain(drain, 0);
            }
            __syncwarp();
            named_bar_sync(2, 8 * 32 + 32);          // softmax warps are done with TMEM
            tc_fence_after();
            tmem_dealloc(tmem, C::TMEM_COLS);
        } else if constexpr (PACKED) {
            // ------------------------------------------------------------ warps 10-11
            // In an item's last visited tile, the value rows past the request's
            // end hold the next request's rows, where 0 * NaN would not vanish: zero them once the tile
            // has landed, before its P V (the MMA thread waits on v_fixed).
            const int t = (warp - 10) * 32 + lane;     // 0 .. 63
            int vt = 0;                                // V tiles of earlier items
            int nl = 0;                                // v_landed phases waited
            for (int r = 0;; ++r) {
                const int slot = r & 1;
                const bool got = __all_sync(0xffffffffu, mbar_wait(info_full(slot), (r >> 1) & 1, abort_flag));
                const int w = got ? (int)info[REC * slot + 8] : -1;
                const int c_all = got ? (int)info[REC * slot + 2] : 0;
                __syncwarp();
                if (lane == 0) mbar_arrive(info_empty(slot));
                if (w < 0) break;
                if (c_all == 0) continue;
                const Item it = describe(w);
                // packed items visit the tiles [first, n_all) without gaps
                const int jl = it.n_all - 1;
                const int i = vt + c_all - 1;
                vt += c_all;
                // v_landed first (one phase per item, in order): the slot's phase
                // for this tile is then the current one and stays so until the
                // MMA thread has seen v_fixed
                if (!__all_sync(0xffffffffu, mbar_wait(v_landed, nl & 1, abort_flag))) break;
                ++nl;
                if (!__all_sync(0xffffffffu, mbar_wait(v_full(i % C::NV), (i / C::NV) & 1, abort_flag))) break;
                const int r0 = it.skv - jl * BN;           // first row past the request's end (> 0)
                if (r0 < BN) {
                    const uint32_t base = C::OFF_V + (i % C::NV) * C::TILE_BYTES;
                    const int n = (BN - r0) * C::KSUB * 8;  // 16-byte chunks
                    for (int x = t; x < n; x += 64) {
                        const int row = r0 + x / (C::KSUB * 8), sl = (x / 8) % C::KSUB, q = x % 8;
                        *reinterpret_cast<uint4*>(smem + base + sl * C::SUB_BYTES + row * 128 + q * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();       // generic writes, read by the tensor core
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(v_fixed);
            }
        }
    } else {
        regs_inc<kRegsSoftmax>();
        // ------------------------------------------------------------ softmax warps 0-7
        const int k = warp / 4;                                // Q tile of this warpgroup
        const int r = (warp % 4) * 32 + lane;                  // row of the tile == TMEM lane
        const uint32_t lane_addr = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t col_s = k == 0 ? C::COL_S0 : C::COL_S1;
        const uint32_t col_o = k == 0 ? C::COL_O0 : C::COL_O1;
        const uint32_t stage = sb + C::OFF_STAGE + k * C::SUB_BYTES;   // this warpgroup's output box
        const float sl = a.scale_log2;
        int sf = 0;                  // S tiles taken so far (s_full parity)
        int n_done = 0;              // items finished (o_final parity)
        bool ok = true;
        for (int rr = 0;; ++rr) {
            // The item record: the first chunk's tile flags, the first visited
            // tile's kept keys (the mask bytes of each later tile are fetched one
            // tile ahead) and, for packed calls, the claimed item's index.  A
            // dense item is known before its record arrives; a packed one only
            // from it, and the warpgroup agrees that the record arrived before
            // anything is taken from it.
            Item itm;
            if constexpr (!PACKED) {
                const int wd = item_of(rr);
                if (wd < 0) break;
                itm = describe(wd);
            }
            const int slot = rr & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(info_full(slot), (rr >> 1) & 1, abort_flag));
            uint32_t mw[4];              // kept keys of the current tile, 32 per word
            uint32_t f0 = 0;
            int w = -1;
#pragma unroll
            for (int q = 0; q < 4; ++q) mw[q] = ok ? info[REC * slot + 4 + q] : 0u;
            if (ok) {
                f0 = info[REC * slot + 3];
                if constexpr (PACKED) w = (int)info[REC * slot + 8];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(info_empty(slot));
            __syncwarp();
            if constexpr (PACKED) {
                if (!named_bar_and(3 + k, BM, ok) || w < 0) break;
                itm = describe(w);
            }
            const TileInfo ti = k == 0 ? itm.t0 : itm.t1;
            const uint8_t* mrow = itm.mrow;
            const int row_q = ti.q0 + r / g;             // this row's query (within the request)
            const int skv = PACKED ? itm.skv : a.Skv, sq = PACKED ? itm.sq : a.Sq;
            const long p_row = (long)row_q + skv - sq;
            const int lim = (int)key_hi(p_row, skv, a.causal, wr);   // visible keys: [lo, lim)
            const int lo = (int)key_lo(p_row, skv, wl);
            float m_ref = -INFINITY;     // reference max (log2 units, scaled)
            float l_run = 0.f;
            int it = 0;
            TileIter tiles(mrow, itm.first, itm.n_all, itm.kv_end_all, lane, f0);
            auto fetch = [&](int j, uint8_t* mb) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int key = j * BN + q * 32 + lane;
                    mb[q] = (mrow && j >= 0 && key < itm.kv_end_all) ? mrow[key] : (uint8_t)(mrow ? 0 : 1);
                }
            };
            int j = ok ? tiles.next() : -1;
            for (; j >= 0 && j < ti.n_tiles;) {
                const int jn = tiles.next();
                uint8_t mbn[4];
                fetch(jn, mbn);
                bool all_kept = true;
#pragma unroll
                for (int q = 0; q < 4; ++q) all_kept = all_kept && (mw[q] == 0xffffffffu);
                const int kbase = j * BN;
                const bool need_mask = (kbase + BN > ti.lim_first) || kbase < ti.lo_last || !all_kept;

                ok = __all_sync(0xffffffffu, mbar_wait(s_full(k), sf & 1, abort_flag));
                ++sf;
                if (!ok) break;
                tc_fence_after();
                uint32_t sr[BN];
                tmem_ld128(tmem + lane_addr + col_s, sr);
                float* s = reinterpret_cast<float*>(sr);

                // Scores to exp2 arguments.  Fast path (no mask in this tile,
                // positive scale, no cap): raw scores, the scale folded into the
                // exp2 argument; otherwise scores become logits (log2 units,
                // capped when a softcap is set) and masked ones -inf.
                const bool capped = cap_out != 0.f;
                const bool fast = !need_mask && sl > 0.f && !capped;
                auto to_logits = [&]() {
                    if (fast) return;
                    uint32_t vis[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        // keys of this 32-column group inside the row's [lo, lim)
                        const int rel = lim - (kbase + 32 * q);
                        const uint32_t below = rel >= 32 ? 0xffffffffu : (rel <= 0 ? 0u : ((1u << rel) - 1u));
                        const int rlo = lo - (kbase + 32 * q);
                        const uint32_t above = rlo <= 0 ? 0xffffffffu : (rlo >= 32 ? 0u : ~((1u << rlo) - 1u));
                        vis[q] = mw[q] & below & above;
                    }
                    if (capped) {
#pragma unroll
                        for (int c = 0; c < BN; ++c)
                            s[c] = ((vis[c / 32] >> (c % 32)) & 1u) ? softcap_log2(s[c], cap_in, cap_out) : -INFINITY;
                    } else {
#pragma unroll
                        for (int c = 0; c < BN; ++c) s[c] = ((vis[c / 32] >> (c % 32)) & 1u) ? s[c] * sl : -INFINITY;
                    }
                };
                to_logits();
                // exp2 argument: s * fa - m (fa = scale on the fast path, 1 otherwise)
                const float fa = fast ? sl : 1.f;
                float alpha = 1.f;
                float rs = 0.f;
                // Once every row of the warp has a reference max, the tile is
                // exponentiated against it directly, with no row max: P and l
                // stay exact relative to the reference, and fp32 / 16-bit P hold
                // values up to the row-sum limit.  A row whose sum passes the
                // limit (or is not finite) sends the warp to the path below.
                bool done = false;
                if (__all_sync(0xffffffffu, m_ref != -INFINITY)) {
                    uint32_t pk[BN / 2];
                    rs = exp_row<F16>(s, fa, m_ref, pk);
                    if (!__any_sync(0xffffffffu, !(rs <= kSumLimit))) {
                        tmem_st64(tmem + lane_addr + col_s, pk);   // P over the first 64 columns of S
                        done = true;
                    }
                }
                if (!done) {
                    // The tile's row max, from the scores still in TMEM (P is not
                    // written yet), over 8 independent chains; the reference max
                    // moves only when the tile max exceeds it by more than the
                    // rescale threshold (lazy rescale).
                    tmem_ld128(tmem + lane_addr + col_s, sr);
                    to_logits();
                    float mx8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
                    for (int c = 0; c < BN; c += 2) mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], s[c], s[c + 1]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) mx8[e] = fmaxf(mx8[e], mx8[e + 4]);
                    const float mx_raw = fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3]));
                    const float mx = fast ? mx_raw * sl : mx_raw;      // scaled (log2 units)
                    if (mx > m_ref + kRescaleThreshold) {
                        alpha = fast_exp2(m_ref - mx);              // 0 when m_ref is -inf
                        m_ref = mx;
                    }
                    const float m_use = m_ref == -INFINITY ? 0.f : m_ref;   // no -inf - -inf
                    uint32_t pk[BN / 2];
                    rs = exp_row<F16>(s, fa, m_use, pk);
                    tmem_st64(tmem + lane_addr + col_s, pk);       // P over the first 64 columns of S
                }
                l_run = l_run * alpha + rs;

                // PV of the previous tile is complete (S of this tile landed after
                // it), so O may be rescaled here, before PV of this tile.
                if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tmem + lane_addr + col_o + 32 * c, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= alpha;
                        tmem_st32(tmem + lane_addr + col_o + 32 * c, reinterpret_cast<uint32_t*>(o));
                    }
                }
                tc_fence_before();
                mbar_arrive(p_full(k));
                ++it;
                j = jn;
#pragma unroll
                for (int q = 0; q < 4; ++q) mw[q] = __ballot_sync(0xffffffffu, mbn[q] != 0);
            }
            // ---- epilogue of this Q tile: the last P V done.  It runs even after
            // a wait gave up, so that the warpgroup's named barriers below see
            // all four warps.
            if (ok) {
                ok = __all_sync(0xffffffffu, mbar_wait(o_final(k), n_done & 1, abort_flag));
                if (ok) tc_fence_after();
            }
            ++n_done;
            const bool row_ok = PACKED ? (r < g * qpb && r / g < ti.rows_valid) : r < ti.rows_valid;
            // this row's place in o [.., D] and lse
            const size_t orow = PACKED ? (size_t)(itm.qs + row_q) * a.Hq + itm.hq + r % g
                                       : ((size_t)itm.b * a.Sq + row_q) * a.Hq + itm.hq;
            // O / l, and the LSE in log2 units; a sink adds exp(s) to l only
            // (GQAPagedFwdOp sinks), taken against max(m_ref, s) so nothing
            // overflows; +inf zeroes the row
            float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            float lse2 = l_run > 0.f ? m_ref + log2f(l_run) : -INFINITY;
            if (sinks && l_run > 0.f) {
                const float s2 = sinks[itm.hq + r % g] * 1.4426950408889634f;
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
            // O / l as bf16 goes, one 64-column box at a time, into this
            // warpgroup's staging buffer in the 128-byte-swizzled box layout of
            // the output map, and one thread stores each box with TMA: whole
            // 128-byte rows instead of 16-byte pieces strided by Hq * D.  Rows
            // past Sq lie outside the map and are not written.  A tile with no
            // visited key, or a wait that gave up, writes zeros directly.  The
            // last box of an item is left reading while the warpgroup moves on;
            // the storing thread waits for it before the buffer is written again.
            // A packed block that the request's end cuts short is stored row by
            // row (its box would reach the next request's rows).
            const bool whole = !PACKED || ti.rows_valid == qpb;
            if (r == 0) bulk_wait_read_all();
            __syncwarp();
            const bool staged = named_bar_and(3 + k, BM, ok && it > 0 && whole);
            if (staged) {
                uint32_t ow[D];
                if constexpr (D == 128) {
                    tmem_ld128(tmem + lane_addr + col_o, ow);
                } else {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c)
                        tmem_ld32(tmem + lane_addr + col_o + 32 * c, reinterpret_cast<float*>(ow + 32 * c));
                }
#pragma unroll
                for (int sub = 0; sub < C::KSUB; ++sub) {
                    __syncwarp();                              // converged at the .aligned barriers
                    if (sub > 0) named_bar_sync(3 + k, BM);   // the previous box has been read out
#pragma unroll
                    for (int q = 0; q < 8; ++q) {              // 16-byte chunk q of the box row
                        const float* f = reinterpret_cast<const float*>(ow + 64 * sub + 8 * q);
                        st_shared_v4(stage + r * 128 + ((q ^ (r & 7)) << 4), pack2<F16>(f[0] * inv, f[1] * inv),
                                     pack2<F16>(f[2] * inv, f[3] * inv), pack2<F16>(f[4] * inv, f[5] * inv),
                                     pack2<F16>(f[6] * inv, f[7] * inv));
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(3 + k, BM);
                    if (r == 0) {
                        if constexpr (PACKED)
                            tma_store_3d(&tm_o, stage, sub * 64, itm.hq, itm.qs + ti.q0);
                        else
                            tma_store_4d(&tm_o, stage, sub * 64, ti.q0, itm.hq, itm.b);
                        bulk_commit_group();
                        if (sub + 1 < C::KSUB) bulk_wait_read_all();
                    }
                }
            } else if (PACKED && !whole && ok && it > 0) {
                // the rows of a cut block, 16 bytes at a time
                uint32_t ow[D];
                if constexpr (D == 128) {
                    tmem_ld128(tmem + lane_addr + col_o, ow);
                } else {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c)
                        tmem_ld32(tmem + lane_addr + col_o + 32 * c, reinterpret_cast<float*>(ow + 32 * c));
                }
                if (row_ok) {
                    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) + orow * D);
#pragma unroll
                    for (int e = 0; e < D / 8; ++e) {
                        const float* f = reinterpret_cast<const float*>(ow + 8 * e);
                        dst[e] = make_uint4(pack2<F16>(f[0] * inv, f[1] * inv), pack2<F16>(f[2] * inv, f[3] * inv),
                                            pack2<F16>(f[4] * inv, f[5] * inv), pack2<F16>(f[6] * inv, f[7] * inv));
                    }
                }
            } else if (row_ok) {
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) + orow * D);
#pragma unroll
                for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (row_ok && a.lse) a.lse[orow] = lse2 * kLn2;
            tc_fence_before();
            if (!named_bar_and(3 + k, BM, ok)) break;     // the whole warpgroup stops together
        }
        if (r == 0) bulk_wait_all();                    // the last stores are done before the CTA ends
        __syncwarp();
        named_bar_arrive(2, 8 * 32 + 32);
        if (threadIdx.x == 0 && *abort_flag) atomicExch(&g_prefill_error, (int)kErrPrefillWait);
    }
}

__global__ void empty_rows_kernel(__nv_bfloat16* o, float* lse, long rows, int D) {
    const long n = rows * D;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        o[i] = __float2bfloat16_rn(0.f);
        if (lse && i % D == 0) lse[i / D] = -INFINITY;
    }
}

template <int D, int MODE, bool OPTS, bool F16>
cudaError_t launch_prefill_t(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const CUtensorMap& tm_o, const PrefillArgs& a, long max_items, cudaStream_t stream) {
    using C = Cfg<D>;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, MODE, OPTS, F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_qpairs = MODE == kModeDense ? (a.Sq + NQ * BM - 1) / (NQ * BM) : 0;
    const long n_items = MODE == kModeDense ? (long)n_qpairs * a.B * a.Hq : max_items;
    const long sms = a.num_sms > 0 ? a.num_sms : 148;
    const long grid = n_items < sms ? n_items : sms;    // persistent: one CTA per SM
    if (grid <= 0) return cudaSuccess;
    prefill_kernel<D, MODE, OPTS, F16><<<(unsigned)grid, NUM_THREADS, C::SMEM_BYTES, stream>>>(tm_q, tm_k, tm_v,
                                                                                              tm_o, a, n_qpairs);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_prefill_mode(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& tm_o, const PrefillArgs& a, long max_items, cudaStream_t stream) {
    const bool opts = a.x.wl >= 0 || a.x.wr >= 0 || a.x.cap_out != 0.f || a.x.sinks != nullptr;
    const int sel = (opts ? 1 : 0) + (a.f16 ? 2 : 0);
    switch (a.D * 4 + sel) {
        case 64 * 4 + 0: return launch_prefill_t<64, MODE, false, false>(tm_q, tm_k, tm_v, tm_o, a, max_items, stream);
        case 64 * 4 + 1: return launch_prefill_t<64, MODE, true, false>(tm_q, tm_k, tm_v, tm_o, a, max_items, stream);
        case 64 * 4 + 2: return launch_prefill_t<64, MODE, false, true>(tm_q, tm_k, tm_v, tm_o, a, max_items, stream);
        case 64 * 4 + 3: return launch_prefill_t<64, MODE, true, true>(tm_q, tm_k, tm_v, tm_o, a, max_items, stream);
        case 128 * 4 + 0: return launch_prefill_t<128, MODE, false, false>(tm_q, tm_k, tm_v, tm_o, a, max_items, stream);
        case 128 * 4 + 1: return launch_prefill_t<128, MODE, true, false>(tm_q, tm_k, tm_v, tm_o, a, max_items, stream);
        case 128 * 4 + 2: return launch_prefill_t<128, MODE, false, true>(tm_q, tm_k, tm_v, tm_o, a, max_items, stream);
        case 128 * 4 + 3: return launch_prefill_t<128, MODE, true, true>(tm_q, tm_k, tm_v, tm_o, a, max_items, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const CUtensorMap& tm_o, const PrefillArgs& a, cudaStream_t stream) {
    return launch_prefill_mode<kModeDense>(tm_q, tm_k, tm_v, tm_o, a, 0, stream);
}

cudaError_t launch_prefill_packed(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                  const CUtensorMap& tm_o, const PrefillArgs& a, long max_items, cudaStream_t stream) {
    return launch_prefill_mode<kModePacked>(tm_q, tm_k, tm_v, tm_o, a, max_items, stream);
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
