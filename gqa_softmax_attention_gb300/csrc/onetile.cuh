// One-query-tile causal GQA attention forward on sm_103a: the kernel behind
// dense prefill at head dim 256 and behind every packed variable-length call.
//
// Computes what prefill.cu computes (TileOPs "Attention Operators",
// GQADenseFwdOp stages 1-7; RL-Kernel "Standard Softmax Attention", Tensor
// Contract; natural-log LSE per MATE "QSA", Core Attention) for three input
// layouts:
//   kBSHD    q [B, Sq, Hq, D], k / v [B, Skv, Hkv, D]; one item = one 128-row
//            query tile of one (b, h);
//   kPacked  packed rows (TileOPs GQAVarlenFwdOp): q [total_q, Hq, D],
//            k / v [total_kv, Hkv, D], request b owning the rows its
//            cu_seqlens name;
//   kPaged   packed queries over a paged cache (TileOPs GQAPagedFwdOp):
//            k / v [pages, page_size, Hkv, D] read through block_table, the
//            cache length of a request counting its query tokens.
// In the two packed layouts an item is a row block of one (request, KV
// head): the g = Hq / Hkv query heads of the group are packed into the tile
// rows (row r = query q0 + r / g, head hkv * g + r % g; floor(128 / g)
// queries per block), so every key and value a request reads serves all g
// heads at once: a decode request streams its cache once per KV head.
//
// TMEM holds S0 | S1 (128 columns each) | O (D columns): the tensor core
// computes S of key tile i+1 while the softmax warps work on tile i.
// Warp roles (384 threads, one CTA per SM, persistent over the items):
//   warps 0-3   softmax: thread t owns tile row t; reads its S row from TMEM,
//               folds the causal / window / padding mask, keeps the running
//               max and sum, writes P (16-bit) over its S row and rescales
//               its O row when the reference max moves;
//   warps 4-7   epilogue: once an item's last P V has completed, reads O,
//               frees it for the next item, and stores O / l and the LSE
//               (TMA through two alternating staging boxes for whole
//               blocks, row by row for a block cut by its request's end),
//               while the next item's first tiles already run;
//   warp 8      TMA producer: the Q block, then K and V through one ring of
//               32 KB slots in the order the MMAs consume them;
//   warp 9      MMA issuer: QK(0), QK(1), PV(0), QK(2), PV(1), ...; it also
//               zeroes the value rows of an item's last key tile that lie
//               past the request's end before P V reads them (packed and
//               paged layouts: those rows hold other requests' values or
//               stale cache slots, and 0 * NaN would not vanish);
//   warps 10-11 complete the third warpgroup (register limits are per
//               warpgroup).
// The MMA shapes stay M128 x N128 (QK) and M128 x N(D) (PV); at D = 256 K is
// split into two 128-column halves and V into two 64-key halves so that each
// half fills one ring slot.  Shared-memory operand layouts:
//   slice-major  (kBSHD, kPacked): a {64, rows} box per 64-column slice,
//                8-row atoms 1 KB apart, slices rows * 128 bytes apart;
//   group-major  (kPaged): one 5-D box per page block lands as
//                [8-key group][slice][8 keys][128 bytes], slices 1 KB apart.
// Both are described by a slice stride and an 8-key-group stride, which is
// all the MMA descriptors need.
//
// The lazy rescale is that of prefill.cu.  Rescaling O before PV of tile i
// needs PV of tile i-1 complete (o_ready, waited for only by a warp that
// rescales): S of tile i having landed implies PV of tile i-2, so the phase
// waited for is never more than one behind.  Every wait is bounded; on a
// timeout the CTA stops issuing work, drains what is in flight, frees TMEM
// and returns.
#pragma once
#include <cmath>

#include "internal.h"
#include "prefill_tiles.cuh"
#include "ptx.cuh"

namespace gqa {
namespace {

__device__ int g_onetile_error;

namespace ot {

using namespace pf;

enum Mode : int { kBSHD = 0, kPacked = 1, kPaged = 2 };

constexpr int NUM_THREADS = 384;
constexpr int WARP_EPI0 = 4;
constexpr int WARP_LOAD = 8;
constexpr int WARP_MMA = 9;
// Registers: 168 per thread at launch (64,512 in all); the softmax warpgroup
// takes 208, the epilogue warpgroup (half a packed O row at a time) 152 and
// the producer/MMA warpgroup 144: (208 + 152 + 144) * 128.
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 208;
constexpr int kRegsEpi = 152;
constexpr int kRegsOther = 144;
static_assert((kRegsSoftmax + kRegsEpi + kRegsOther) * 128 <= kRegsLaunch * NUM_THREADS, "register split");

constexpr int BOX = BM * 128;      // one 64-column box of 128 rows (16 KB)
constexpr int SLOT = 32768;        // one ring slot
constexpr int ENTRY_INTS = 8;      // a row block of a packed call: b, q0, qs, sq, ks, L, -, -

template <int D, int MODE>
struct Cfg {
    static constexpr int KSL = D / 64;                  // 64-column slices per row
    static constexpr int CK = D == 256 ? 2 : 1;         // ring chunks per K tile (halves along D)
    static constexpr int CV = D == 256 ? 2 : 1;         // ring chunks per V tile (halves along the keys)
    static constexpr int KSL_C = KSL / CK;              // slices per K chunk
    static constexpr int VKEYS = BN / CV;               // keys per V chunk
    static constexpr int K_CHUNK = BN * 128 * KSL_C;    // bytes
    static constexpr int V_CHUNK = VKEYS * 128 * KSL;
    static constexpr bool GROUPED = MODE == kPaged;
    static constexpr int K_SLICE = GROUPED ? 1024 : BN * 128;
    static constexpr int K_GROUP = GROUPED ? KSL_C * 1024 : 1024;
    static constexpr int V_SLICE = GROUPED ? 1024 : VKEYS * 128;
    static constexpr int V_GROUP = GROUPED ? KSL * 1024 : 1024;
    static constexpr int NS = D == 256 ? 4 : 5;         // ring slots
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = OFF_Q + KSL * BOX;
    static constexpr int OFF_STAGE = OFF_RING + NS * SLOT;   // 2 output boxes
    static constexpr int OFF_STATS = OFF_STAGE + 2 * BOX;    // m[128], l[128], visited-tile count
    static constexpr int OFF_BAR = OFF_STATS + 2 * BM * 4 + 16;
    // q_full, q_empty, r_full[NS], r_empty[NS], s_full[2], p_full[2], o_ready,
    // o_final, o_empty, stats_full, stats_empty, drain, item_full[2], item_empty[2]
    static constexpr int NBAR = 2 + 2 * NS + 4 + 6 + 4;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;        // 1 KB alignment slack
    static_assert(K_CHUNK <= SLOT && V_CHUNK <= SLOT, "ring slot");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};
constexpr uint32_t COL_S0 = 0, COL_O = 256, TMEM_COLS = 512;

template <int D, int MODE, bool OPTS, bool F16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
onetile_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const PrefillArgs a, int n_qtiles) {
    // CTAs past the share the plan gave this launch leave their SMs to the
    // decode steps running beside it (uniform per CTA, before any set-up)
    if (a.g_eff != nullptr && (int)blockIdx.x >= *a.g_eff) return;
    using C = Cfg<D, MODE>;
    constexpr bool PACKED = MODE != kBSHD;
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

    // rows per query in a tile (1, or the group size when heads are packed)
    const int g = PACKED ? a.g : 1;
    const int qpb = PACKED ? a.qpb : BM;         // queries per block
    const int n_e = PACKED ? *a.n_entries : 0;
    // Work items.  kBSHD: heaviest (last) query tiles first, adjacent items on
    // one KV head; round r takes item r * G + cta (even r) or r * G + G - 1 -
    // cta (odd r).  Packed: item w = (row block w / Hkv, KV head w % Hkv), the
    // requests ordered by estimated cost, heaviest first; items are claimed
    // in that order from a counter in the workspace (the plan kernel zeroes
    // it), so that a CTA whose items ran long takes fewer of them.
    const int n_items = PACKED ? n_e * a.Hkv : n_qtiles * a.B * a.Hq;
    const int G = gridDim.x;
    const int cta = blockIdx.x;
    auto item_of = [&](int r) -> int {
        const long w = (long)r * G + ((r & 1) ? G - 1 - cta : cta);
        return w < n_items ? (int)w : -1;
    };
    struct Item {
        int b, hq, hkv;     // hq: the query head (kBSHD) or the group's first head
        int qs, ks;         // packed row of the request's first query / key
        int sq, skv;        // the request's queries and keys
        int first;          // first visited key tile
        TileInfo t;         // t.q0: first query of the block (within the request)
        const uint8_t* mrow;
    };
    auto describe = [&](int w) {
        Item it;
        if constexpr (PACKED) {
            const int4* e = reinterpret_cast<const int4*>(a.entries + (size_t)(w / a.Hkv) * ENTRY_INTS);
            const int4 e0 = e[0], e1 = e[1];
            it.b = e0.x;
            it.hkv = w % a.Hkv;
            it.hq = it.hkv * g;
            it.qs = e0.z;
            it.sq = e0.w;
            it.ks = e1.x;
            it.skv = e1.y;
            it.t = tile_info_n(e0.y, qpb, it.sq, it.skv, a.causal, wl, wr);
            it.mrow = nullptr;
        } else {
            const int bh = a.B * a.Hq;
            const int qt = n_qtiles - 1 - w / bh;
            const int rem = w % bh;
            it.hq = rem % a.Hq;
            it.b = rem / a.Hq;
            it.hkv = it.hq / (a.Hq / a.Hkv);
            it.qs = it.ks = 0;
            it.sq = a.Sq;
            it.skv = a.Skv;
            it.t = tile_info(qt * BM, a.Sq, a.Skv, a.causal, wl, wr);
            it.mrow = a.mask ? a.mask + (size_t)it.b * a.Skv : nullptr;
        }
        it.first = it.t.kv_begin / BN;
        return it;
    };
    // Visited key tiles of an item (non-empty, in [first, n_tiles)).  Warp-collective.
    auto count_tiles = [&](const Item& it) {
        if (!it.mrow) return it.t.n_tiles - it.first;
        int c = 0;
        for (int chunk = it.first / 32; chunk * 32 < it.t.n_tiles; ++chunk)
            c += __popc(tile_flags(it.mrow, chunk, it.first, it.t.n_tiles, it.t.kv_end, lane));
        return c;
    };

    const uint32_t bar0 = sb + C::OFF_BAR;
    const uint32_t q_full = bar0, q_empty = bar0 + 8;
    auto r_full = [&](int s) { return bar0 + 8u * (2 + s); };
    auto r_empty = [&](int s) { return bar0 + 8u * (2 + C::NS + s); };
    auto s_full = [&](int k) { return bar0 + 8u * (2 + 2 * C::NS + k); };
    auto p_full = [&](int k) { return bar0 + 8u * (4 + 2 * C::NS + k); };
    const uint32_t o_ready = bar0 + 8u * (6 + 2 * C::NS);
    const uint32_t o_final = o_ready + 8, o_empty = o_ready + 16;
    const uint32_t stats_full = o_ready + 24, stats_empty = o_ready + 32, drain = o_ready + 40;
    auto item_full = [&](int k) { return o_ready + 48u + 8u * k; };
    auto item_empty = [&](int k) { return o_ready + 64u + 8u * k; };
    float* st_m = reinterpret_cast<float*>(smem + C::OFF_STATS);
    float* st_l = st_m + BM;
    volatile int* st_cnt = reinterpret_cast<volatile int*>(st_l + BM);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* item_rec = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);   // two claimed items
    // Packed: the producer claims items and hands each one's index to the
    // MMA warp and the eight softmax / epilogue warps through a two-slot
    // record; the last record it writes is -1.  Warp-collective.
    auto claim_item = [&](int r) -> int {
        if constexpr (!PACKED) {
            return item_of(r);
        } else {
            int w = -1;
            if (lane == 0) {
                const int slot = r & 1;
                if (mbar_wait(item_empty(slot), ((r >> 1) & 1) ^ 1, abort_flag)) {
                    w = atomicAdd(a.work, 1);
                    if (w >= n_items) w = -1;
                    item_rec[slot] = w;
                    mbar_arrive(item_full(slot));
                }
            }
            return __shfl_sync(0xffffffffu, w, 0);
        }
    };
    auto next_item = [&](int r) -> int {
        if constexpr (!PACKED) {
            return item_of(r);
        } else {
            const int slot = r & 1;
            const bool got = __all_sync(0xffffffffu, mbar_wait(item_full(slot), (r >> 1) & 1, abort_flag));
            const int w = got ? item_rec[slot] : -1;
            __syncwarp();
            if (lane == 0) mbar_arrive(item_empty(slot));
            return w;
        }
    };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < C::NS; ++s) { mbar_init(r_full(s), 1); mbar_init(r_empty(s), 1); }
        for (int k = 0; k < 2; ++k) { mbar_init(s_full(k), 1); mbar_init(p_full(k), BM); }
        mbar_init(o_ready, 1);
        mbar_init(o_final, 1);
        mbar_init(o_empty, BM);
        mbar_init(stats_full, BM);
        mbar_init(stats_empty, BM);
        mbar_init(drain, 1);
        for (int k = 0; k < 2; ++k) {
            mbar_init(item_full(k), 1);
            mbar_init(item_empty(k), 1 + 8);   // the MMA warp and the eight softmax / epilogue warps
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if constexpr (PACKED) {
        // Q rows past g * qpb are never loaded: zero them once (finite rows,
        // their results are never stored)
        const int rows = a.g * a.qpb;
        for (int idx = threadIdx.x; idx < (BM - rows) * 8 * C::KSL; idx += NUM_THREADS) {
            const int row = rows + idx / (8 * C::KSL), s = (idx / 8) % C::KSL, q = idx % 8;
            *reinterpret_cast<uint4*>(smem + C::OFF_Q + s * BOX + row * 128 + q * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
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
            int nc = 0, nq = 0;                     // ring chunks and Q blocks issued (lane 0's count)
            bool ok = true;
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
            }
            // Waits for the next ring slot and arms its barrier for `bytes`.
            // TMA-tensor layouts: lane 0 alone (it issues every copy).  Paged:
            // warp-collective, every lane learning the slot (lanes copy one
            // page block each).
            // Paged caches whose page size is not a multiple of 8 are gathered
            // row by row with cp.async into the same layout the page-block
            // boxes give; a slot's full barrier then takes lane 0's plain
            // arrival once that slot's copies have landed.
            const bool gather = MODE == kPaged && a.bt_k == 0;
            auto take_slot = [&](uint32_t& dst, uint32_t& full, uint32_t bytes) -> bool {
                const int s = nc % C::NS;
                bool good = true;
                if (MODE != kPaged || lane == 0) {
                    good = mbar_wait(r_empty(s), ((nc / C::NS) & 1) ^ 1, abort_flag);
                    if (good && !gather) mbar_arrive_expect_tx(r_full(s), bytes);
                }
                if constexpr (MODE == kPaged) {
                    good = __shfl_sync(0xffffffffu, good, 0);
                    __syncwarp();                    // the expect-tx precedes every lane's copy
                }
                full = r_full(s);
                dst = sb + C::OFF_RING + s * SLOT;
                if (good) ++nc;
                return good;
            };
            // Paged: lane l < n copies block l (bt keys from key0 + l * bt) if it
            // starts below the request's end; returns the bytes of those copies.
            auto paged_blocks = [&](const Item& it, int key0, int bt, int n) -> int {
                const int key = key0 + lane * bt;
                return __popc(__ballot_sync(0xffffffffu, lane < n && key < it.skv)) * bt;
            };
            auto paged_copy = [&](const Item& it, const CUtensorMap* map, uint32_t dst, uint32_t full, int key0,
                                  int bt, int n, int group_stride, int slice0) {
                const int key = key0 + lane * bt;
                if (lane < n && key < it.skv) {
                    const int page = __ldg(a.table + (size_t)it.b * a.max_pages + key / a.page_size);
                    const long row = (long)page * a.page_size + key % a.page_size;
                    // a page id outside the pool reads as zeros (the coordinate is out of range)
                    tma_load_5d(dst + (lane * bt / 8) * group_stride, map, full, 0, 0, slice0, (int)(row / 8),
                                it.hkv);
                }
            };
            // Gathered rows: keys key0 .. key0 + nkeys - 1 (those below the
            // request's end), 64-column slices slice0 .. slice0 + nsl - 1, as
            // [8-key group][slice][8 keys][128 B] with the 128-byte swizzle; a
            // page id outside the pool reads as zeros.  The copies are
            // committed as one group; the previous slot's barrier is then
            // released once its group has landed (one slot stays in flight).
            uint32_t pend = 0;                      // full barrier of the slot still in flight
            auto release = [&](int keep) {
                if (pend == 0) return;
                if (keep) cp_async_wait<1>(); else cp_async_wait<0>();
                fence_proxy_async_smem();           // cp.async writes, read by the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(pend);
                pend = 0;
            };
            auto gather_copy = [&](const Item& it, const void* cache, uint32_t dst, uint32_t full, int key0,
                                   int nkeys, int slice0, int nsl, int group_stride) {
                const uint16_t* base = static_cast<const uint16_t*>(cache);
                for (int idx = lane; idx < nkeys * nsl * 8; idx += 32) {
                    const int r = idx / (nsl * 8), s = (idx / 8) % nsl, q = idx % 8;
                    const int key = key0 + r;
                    if (key >= it.skv) continue;
                    const int page = __ldg(a.table + (size_t)it.b * a.max_pages + key / a.page_size);
                    const bool in_pool = page >= 0 && page < a.num_pages;
                    const long row = in_pool ? (long)page * a.page_size + key % a.page_size : 0;
                    const uint16_t* src = base + (row * a.Hkv + it.hkv) * D + 64 * (slice0 + s) + 8 * q;
                    cp_async16(dst + (r / 8) * group_stride + s * 1024 + (r % 8) * 128 + ((q ^ (r % 8)) << 4), src,
                               in_pool ? 16u : 0u);
                }
                cp_async_commit();
                release(1);
                pend = full;
            };
            auto load_k = [&](const Item& it, int j) -> bool {
                for (int c = 0; c < C::CK; ++c) {
                    uint32_t dst, full;
                    if (gather) {
                        if (!take_slot(dst, full, 0)) return false;
                        gather_copy(it, a.k_cache, dst, full, j * BN, BN, c * C::KSL_C, C::KSL_C, C::K_GROUP);
                    } else if constexpr (MODE == kPaged) {
                        const int n = BN / a.bt_k;
                        const int rows = paged_blocks(it, j * BN, a.bt_k, n);
                        if (!take_slot(dst, full, (uint32_t)(rows * 128 * C::KSL_C))) return false;
                        paged_copy(it, &tm_k, dst, full, j * BN, a.bt_k, n, C::K_GROUP, c * C::KSL_C);
                    } else {                        // lane 0 only
                        if (!take_slot(dst, full, C::K_CHUNK)) return false;
#pragma unroll
                        for (int s = 0; s < C::KSL_C; ++s) {
                            const int col = 64 * (c * C::KSL_C + s);
                            if constexpr (MODE == kPacked)
                                tma_load_3d(dst + s * C::K_SLICE, &tm_k, full, col, it.hkv, it.ks + j * BN);
                            else
                                tma_load_4d(dst + s * C::K_SLICE, &tm_k, full, col, j * BN, it.hkv, it.b);
                        }
                    }
                }
                return true;
            };
            auto load_v = [&](const Item& it, int j) -> bool {
                for (int c = 0; c < C::CV; ++c) {
                    uint32_t dst, full;
                    const int key0 = j * BN + c * C::VKEYS;
                    if (gather) {
                        if (!take_slot(dst, full, 0)) return false;
                        gather_copy(it, a.v_cache, dst, full, key0, C::VKEYS, 0, C::KSL, C::V_GROUP);
                    } else if constexpr (MODE == kPaged) {
                        const int n = C::VKEYS / a.bt_v;
                        const int rows = paged_blocks(it, key0, a.bt_v, n);
                        if (!take_slot(dst, full, (uint32_t)(rows * 128 * C::KSL))) return false;
                        paged_copy(it, &tm_v, dst, full, key0, a.bt_v, n, C::V_GROUP, 0);
                    } else {                        // lane 0 only
                        if (!take_slot(dst, full, C::V_CHUNK)) return false;
#pragma unroll
                        for (int s = 0; s < C::KSL; ++s) {
                            if constexpr (MODE == kPacked)
                                tma_load_3d(dst + s * C::V_SLICE, &tm_v, full, 64 * s, it.hkv, it.ks + key0);
                            else
                                tma_load_4d(dst + s * C::V_SLICE, &tm_v, full, 64 * s, key0, it.hkv, it.b);
                        }
                    }
                }
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int w = claim_item(r);
                if (w < 0) break;
                const Item it = describe(w);
                const int c = count_tiles(it);
                if (c == 0) continue;
                if (lane == 0) {
                    ok = mbar_wait(q_empty, (nq & 1) ^ 1, abort_flag);
                    if (ok) {
                        if constexpr (PACKED) {
                            // {64, g, qpb} boxes: rows q * g + head of queries q0.. of the group
                            mbar_arrive_expect_tx(q_full, (uint32_t)(C::KSL * g * qpb * 128));
#pragma unroll
                            for (int s = 0; s < C::KSL; ++s)
                                tma_load_3d(sb + C::OFF_Q + s * BOX, &tm_q, q_full, 64 * s, it.hq, it.qs + it.t.q0);
                        } else {
                            mbar_arrive_expect_tx(q_full, C::KSL * BOX);
#pragma unroll
                            for (int s = 0; s < C::KSL; ++s)
                                tma_load_4d(sb + C::OFF_Q + s * BOX, &tm_q, q_full, 64 * s, it.t.q0, it.hq, it.b);
                        }
                        ++nq;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                // K of tile 0, then (K of tile i+1, V of tile i) for each tile i
                TileIter tiles(it.mrow, it.first, it.t.n_tiles, it.t.kv_end, lane);
                int j = tiles.next();
                if (MODE == kPaged || lane == 0) ok = load_k(it, j);
                if (MODE != kPaged) ok = __shfl_sync(0xffffffffu, ok, 0);
                while (ok && j >= 0) {
                    const int jn = tiles.next();
                    if (MODE == kPaged || lane == 0) {
                        if (jn >= 0) ok = load_k(it, jn);
                        if (ok) ok = load_v(it, j);
                    }
                    if (MODE != kPaged) ok = __shfl_sync(0xffffffffu, ok, 0);
                    j = jn;
                }
                // the item's last gathered slot, before the next item's waits
                // (its Q slot frees only once this item's MMAs have run)
                if (gather) release(0);
            }
            if (gather) cp_async_wait<0>();         // no copy outlives the loop
            if (lane == 0 && *abort_flag && !gather) {
                // let the copies in flight land: the last load of each slot
                for (int s = 0; s < C::NS && s < nc; ++s) {
                    const int last = nc - 1 - ((nc - 1 - s) % C::NS);
                    mbar_drain(r_full(s), (last / C::NS) & 1);
                }
                if (nq > 0) mbar_drain(q_full, (nq - 1) & 1);
            }
        } else if (warp == WARP_MMA) {
            // ------------------------------------------------------------ MMA issuer
            // Lane 0 alone issues every MMA of an item but its last P V (a
            // single polling lane keeps the issue loop short); the whole warp
            // takes the last P V, whose value rows past the request's end it
            // zeroes first (packed layouts).
            int nc = 0, nq = 0;     // ring chunks and Q blocks consumed
            int g_t = 0;            // visited tiles of earlier items (S buffer / p_full parity)
            int oe = 0;             // o_empty phases waited
            bool ok = true;
            auto chunk_addr = [&](int k) { return sb + C::OFF_RING + ((nc + k) % C::NS) * SLOT; };
            auto take = [&](int n) -> bool {        // lane 0: the next n ring chunks have landed
                for (int k = 0; k < n; ++k)
                    if (!mbar_wait(r_full((nc + k) % C::NS), ((nc + k) / C::NS) & 1, abort_flag)) return false;
                tc_fence_after();
                return true;
            };
            auto release = [&](int n) {             // lane 0
                for (int k = 0; k < n; ++k) mma_commit(r_empty((nc + k) % C::NS));
                nc += n;
            };
            // S of visited tile gi = Q K^T over D / 16 steps of 16 columns (lane 0)
            auto issue_qk = [&](int gi) -> bool {
                if (!take(C::CK)) return false;
                const uint32_t d = tmem + COL_S0 + (gi & 1) * BN;
                // descriptors of the Q tile and of each K chunk, advanced by
                // constant offsets (>> 4) per step
                const uint64_t qdesc = make_sdesc_sw128(sb + C::OFF_Q, 16, 1024);
                uint64_t kdesc[C::CK];
#pragma unroll
                for (int c = 0; c < C::CK; ++c) kdesc[c] = make_sdesc_sw128(chunk_addr(c), 16, C::K_GROUP);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    constexpr int PER = D / 16 / C::CK;       // steps per K chunk
                    const int kl = kk % PER;
                    const uint32_t qoff = (kk / 4) * BOX + (kk % 4) * 32;
                    const uint32_t koff = (kl / 4) * C::K_SLICE + (kl % 4) * 32;
                    mma_bf16_ss(d, qdesc + (qoff >> 4), kdesc[kk / PER] + (koff >> 4), IDESC_QK, kk > 0 ? 1u : 0u);
                }
                mma_commit(s_full(gi & 1));
                release(C::CK);
                return true;
            };
            // O (+)= P V of visited tile gi: 8 steps of 16 keys (lane 0)
            auto mma_pv = [&](int gi, bool fresh) {
                const uint32_t p = tmem + COL_S0 + (gi & 1) * BN;
                uint64_t vdesc[C::CV];
#pragma unroll
                for (int c = 0; c < C::CV; ++c) vdesc[c] = make_sdesc_sw128(chunk_addr(c), C::V_SLICE, C::V_GROUP);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    constexpr int PER = BN / 16 / C::CV;       // steps per V chunk
                    const int kc = (kk % PER) * 16;
                    mma_bf16_ts(tmem + COL_O, p + kk * 8, vdesc[kk / PER] + (((kc / 8) * C::V_GROUP) >> 4), IDESC_PV,
                                (!fresh || kk > 0) ? 1u : 0u);
                }
                release(C::CV);
                mma_commit(o_ready);
            };
            auto issue_pv = [&](int gi, bool fresh) -> bool {      // lane 0
                if (!mbar_wait(p_full(gi & 1), (gi >> 1) & 1, abort_flag)) return false;
                if (!take(C::CV)) return false;
                mma_pv(gi, fresh);
                return true;
            };
            // lane 0: the epilogue of every earlier item has read O
            auto wait_o_empty = [&](int n_item) -> bool {
                for (; oe < n_item; ++oe)
                    if (!mbar_wait(o_empty, oe & 1, abort_flag)) return false;
                return true;
            };
            for (int r = 0, n_item = 0; ok; ++r, ++n_item) {
                const int w = next_item(r);
                if (w < 0) break;
                const Item it = describe(w);
                const int c = count_tiles(it);
                if (lane == 0) {
                    if (c > 0) {
                        ok = mbar_wait(q_full, nq++ & 1, abort_flag);
                        if (ok) ok = issue_qk(g_t);
                        if (ok && c > 1) ok = issue_qk(g_t + 1);
                        if (ok) ok = wait_o_empty(n_item);
                        if (ok && c > 1) ok = issue_pv(g_t, true);
                        for (int i = 1; i + 1 < c && ok; ++i) {
                            ok = issue_qk(g_t + i + 1);
                            if (ok) ok = issue_pv(g_t + i, false);
                        }
                        if (ok) mma_commit(q_empty);               // every S of the item is issued
                        // BSHD: no value row to zero, lane 0 issues the last P V too
                        if (!PACKED && ok) ok = issue_pv(g_t + c - 1, c == 1);
                    } else {
                        ok = wait_o_empty(n_item);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                nc = __shfl_sync(0xffffffffu, nc, 0);
                nq = __shfl_sync(0xffffffffu, nq, 0);
                oe = __shfl_sync(0xffffffffu, oe, 0);
                if (PACKED && ok && c > 0) {
                    // the item's last P V, by the whole warp
                    const int gi = g_t + c - 1;
                    ok = __all_sync(0xffffffffu, mbar_wait(p_full(gi & 1), (gi >> 1) & 1, abort_flag));
                    for (int k = 0; k < C::CV && ok; ++k)
                        ok = __all_sync(0xffffffffu,
                                        mbar_wait(r_full((nc + k) % C::NS), ((nc + k) / C::NS) & 1, abort_flag));
                    if (ok) {
                        tc_fence_after();
                        const int nvalid = PACKED ? min(BN, it.skv - (it.t.n_tiles - 1) * BN) : BN;
                        if (PACKED && nvalid < BN) {
                            for (int idx = lane; idx < (BN - nvalid) * 8 * C::KSL; idx += 32) {
                                const int key = nvalid + idx / (8 * C::KSL);
                                const int s = (idx / 8) % C::KSL, q = idx % 8;
                                const int kc = key % C::VKEYS;
                                const uint32_t off = chunk_addr(key / C::VKEYS) - sb + s * C::V_SLICE +
                                                     (kc / 8) * C::V_GROUP + (kc % 8) * 128 + q * 16;
                                *reinterpret_cast<uint4*>(smem + off) = make_uint4(0u, 0u, 0u, 0u);
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            tc_fence_after();
                        }
                        if (lane == 0) mma_pv(gi, c == 1);
                        nc = __shfl_sync(0xffffffffu, nc, 0);
                    }
                }
                g_t += c;
                // one phase per item: every MMA of the item has completed
                if (ok && lane == 0) mma_commit(o_final);
                __syncwarp();
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
        const int rq = r / g;                                  // query of this row within the block
        int gt = 0;                  // visited tiles so far
        int n = 0;                   // items finished
        bool ok = true;
        for (int rr = 0; ok; ++rr) {
            const int w = next_item(rr);
            if (w < 0) break;
            const Item itm = describe(w);
            const TileInfo ti = itm.t;
            const uint8_t* mrow = itm.mrow;
            const long p_row = (long)ti.q0 + rq + itm.skv - itm.sq;
            const int lim = (int)key_hi(p_row, itm.skv, a.causal, wr);   // visible keys: [lo, lim)
            const int lo = (int)key_lo(p_row, itm.skv, wl);
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
                const uint32_t col_s = COL_S0 + (gt & 1) * BN;

                ok = __all_sync(0xffffffffu, mbar_wait(s_full(gt & 1), (gt >> 1) & 1, abort_flag));
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
                const float rs = exp_row<F16>(s, fa, m_use, pk);
                tmem_st64(tmem + lane_addr + col_s, pk);          // P over the first 64 columns of S
                l_run = l_run * alpha + rs;

                if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // PV of the previous tile must have completed before O is rescaled
                    ok = __all_sync(0xffffffffu, mbar_wait(o_ready, (gt - 1) & 1, abort_flag));
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
                mbar_arrive(p_full(gt & 1));
                ++it;
                ++gt;
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
        const int rq = r / g, rh = r % g;           // query and head of this row within the block
        int n = 0;                   // items finished
        int nb = 0;                  // output boxes stored (staging buffer alternation)
        bool ok = true;
        for (int rr = 0;; ++rr) {
            const int w = next_item(rr);
            if (w < 0) break;
            const Item itm = describe(w);
            const TileInfo ti = itm.t;
            // warp-collective waits: the warp must be converged at the
            // .aligned barrier below and at every tcgen05.ld
            ok = __all_sync(0xffffffffu, mbar_wait(stats_full, n & 1, abort_flag));
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_final, n & 1, abort_flag));
            if (!named_bar_and(3, BM, ok)) break;     // the whole warpgroup stops together
            tc_fence_after();
            const int cnt = *st_cnt;
            const float m_ref = st_m[r];
            const float l_run = st_l[r];
            const int head = itm.hq + (PACKED ? rh : 0);
            const bool row_ok = (PACKED ? r < g * qpb : true) && rq < ti.rows_valid;
            // output row: [B, Sq, Hq] (kBSHD) or [total_q, Hq] (packed)
            const size_t orow = PACKED ? ((size_t)itm.qs + ti.q0 + rq) * a.Hq + head
                                       : ((size_t)itm.b * a.Sq + ti.q0 + rq) * a.Hq + head;
            float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            float lse2 = l_run > 0.f ? m_ref + log2f(l_run) : -INFINITY;
            if (sinks && l_run > 0.f) {
                const float s2 = sinks[head] * 1.4426950408889634f;
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
            // Whole blocks go out with TMA; a packed block cut by its request's
            // end is written row by row (its box would reach the next request).
            // The choice is the same for every thread of the item.
            const bool boxed = !PACKED || ti.rows_valid == qpb;
            constexpr int HALF = D < 128 ? D : 128;     // O columns read per pass
            // O / l packed to 16 bits, HALF columns at a time; O is free once the
            // last columns are read
            auto read_o = [&](int half, uint32_t* ow) {
                // tcgen05.ld is warp-collective (.sync.aligned): reconverge first
                __syncwarp();
#pragma unroll
                for (int c = 0; c < HALF / 32; ++c) {
                    float f[32];
                    tmem_ld32(tmem + lane_addr + COL_O + HALF * half + 32 * c, f);
#pragma unroll
                    for (int e = 0; e < 16; ++e) ow[16 * c + e] = pack2<F16>(f[2 * e] * inv, f[2 * e + 1] * inv);
                }
                if (half == D / HALF - 1) {
                    tc_fence_before();
                    mbar_arrive(stats_empty);
                    mbar_arrive(o_empty);
                }
            };
            if (cnt > 0 && boxed) {
#pragma unroll
                for (int half = 0; half < D / HALF; ++half) {
                    uint32_t ow[HALF / 2];
                    read_o(half, ow);
                    // 64-column boxes through the alternating staging buffers
#pragma unroll
                    for (int sub = 0; sub < HALF / 64; ++sub, ++nb) {
                        const uint32_t stage = sb + C::OFF_STAGE + (nb & 1) * BOX;
                        if (r == 0) bulk_wait_read_1();       // the store two boxes back has read this buffer
                        __syncwarp();
                        named_bar_sync(3, BM);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint32_t* u = ow + 32 * sub + 4 * q;
                            st_shared_v4(stage + r * 128 + ((q ^ (r & 7)) << 4), u[0], u[1], u[2], u[3]);
                        }
                        fence_proxy_async_smem();
                        named_bar_sync(3, BM);
                        if (r == 0) {
                            const int col = HALF * half + 64 * sub;
                            if constexpr (PACKED)
                                tma_store_3d(&tm_o, stage, col, itm.hq, itm.qs + ti.q0);
                            else
                                tma_store_4d(&tm_o, stage, col, ti.q0, itm.hq, itm.b);
                            bulk_commit_group();
                        }
                    }
                }
            } else if (cnt > 0) {
#pragma unroll
                for (int half = 0; half < D / HALF; ++half) {
                    uint32_t ow[HALF / 2];
                    read_o(half, ow);
                    if (row_ok) {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + orow * D + HALF * half);
#pragma unroll
                        for (int e = 0; e < HALF / 8; ++e)
                            dst[e] = make_uint4(ow[4 * e], ow[4 * e + 1], ow[4 * e + 2], ow[4 * e + 3]);
                    }
                }
            } else {
                mbar_arrive(stats_empty);
                mbar_arrive(o_empty);
                if (row_ok) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + orow * D);
#pragma unroll
                    for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (row_ok && a.lse) a.lse[orow] = lse2 * kLn2;
            ++n;
        }
        if (r == 0) bulk_wait_read_all();
        tc_fence_before();
        named_bar_arrive(2, 8 * 32 + 32);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(&g_onetile_error, (int)kErrPrefillWait);
}

template <int D, int MODE, bool OPTS, bool F16>
cudaError_t launch_onetile(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const CUtensorMap& tm_o, const PrefillArgs& a, long max_items, int n_qtiles,
                           cudaStream_t stream) {
    using C = Cfg<D, MODE>;
    cudaError_t e = cudaFuncSetAttribute(onetile_kernel<D, MODE, OPTS, F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long sms = a.num_sms > 0 ? a.num_sms : 148;
    const long grid = max_items < sms ? max_items : sms;    // persistent: one CTA per SM
    if (grid <= 0) return cudaSuccess;
    onetile_kernel<D, MODE, OPTS, F16><<<(unsigned)grid, NUM_THREADS, C::SMEM_BYTES, stream>>>(tm_q, tm_k, tm_v,
                                                                                              tm_o, a, n_qtiles);
    return cudaGetLastError();
}

int take_error() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_onetile_error, sizeof(int)) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_onetile_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace ot
}  // namespace
}  // namespace gqa
