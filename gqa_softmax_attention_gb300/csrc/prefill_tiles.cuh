// Key-tile bookkeeping and the row exponential shared by the dense prefill
// kernels (prefill.cu: D = 64 / 128, two query tiles per CTA; prefill_d256.cu:
// D = 256, one query tile per CTA).
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace gqa {
namespace pf {

constexpr int BM = 128;            // query rows per Q tile (= TMEM lanes)
constexpr int BN = 128;            // keys per tile
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.f;   // log2 units: P <= 256 between rescales
// Row-sum limit of a tile exponentiated against a stale reference max (no
// row max taken): 2^32.  A row's sum stays below tiles x 2^32, far from the
// fp32 range, and its P values below 2^32 (16-bit P holds them).
constexpr float kSumLimit = 4294967296.f;

struct TileInfo {
    int q0;          // first query row of the tile
    int rows_valid;  // rows of the tile that exist (ragged tail; may be 0)
    int lim_first;   // keys below lim_first are inside every row's upper bound
    int lo_last;     // keys from lo_last on are inside every row's lower (window) bound
    int kv_begin;    // no row of the tile sees a key < kv_begin
    int kv_end;      // no row of the tile sees a key >= kv_end
    int n_tiles;     // key tiles in [0, kv_end)
};

// Visible keys of the query at key position p: [lo, hi) (TileOPs "Attention
// Operators", GQADenseFwdOp stage 5: causal j <= p, window p - wL <= j <= p + wR).
__device__ __forceinline__ long key_hi(long p, int Skv, int causal, int wr) {
    long hi = Skv;
    if (causal) hi = min(hi, p + 1);
    if (wr >= 0) hi = min(hi, p + wr + 1);
    return max(0L, hi);
}
__device__ __forceinline__ long key_lo(long p, int Skv, int wl) {
    return wl >= 0 ? min((long)Skv, max(0L, p - wl)) : 0L;
}

// Bounds of a block of up to nq queries starting at query q0 (rows_valid
// counts the queries of the block that exist).
__device__ __forceinline__ TileInfo tile_info_n(int q0, int nq, int Sq, int Skv, int causal, int wl, int wr) {
    TileInfo t;
    t.q0 = q0;
    t.rows_valid = max(0, min(nq, Sq - q0));
    if (t.rows_valid == 0) {
        t.kv_begin = t.kv_end = t.lim_first = t.lo_last = 0;
    } else {
        const long p_first = (long)q0 + Skv - Sq;        // key position of the first row
        const long p_last = p_first + t.rows_valid - 1;
        t.kv_end = (int)key_hi(p_last, Skv, causal, wr);
        t.lim_first = (int)key_hi(p_first, Skv, causal, wr);
        t.kv_begin = (int)key_lo(p_first, Skv, wl);
        t.lo_last = (int)key_lo(p_last, Skv, wl);
        if (t.kv_begin >= t.kv_end) t.kv_begin = t.kv_end = t.lim_first = t.lo_last = 0;
    }
    t.n_tiles = (t.kv_end + BN - 1) / BN;
    return t;
}

__device__ __forceinline__ TileInfo tile_info(int q0, int Sq, int Skv, int causal, int wl, int wr) {
    return tile_info_n(q0, BM, Sq, Skv, causal, wl, wr);
}

// Warp-collective.  Bit l of the result is set when key tile 32 * chunk + l
// (in [first, n_tiles)) holds a key below kv_end that the padding mask keeps; lane l
// scans that tile, so 32 tiles cost one pass.  Without a mask every tile
// below n_tiles counts.
__device__ __forceinline__ uint32_t tile_flags(const uint8_t* mrow, int chunk, int first, int n_tiles, int kv_end,
                                               int lane) {
    const int j = chunk * 32 + lane;
    bool any = j >= first && j < n_tiles;
    if (mrow && any) {
        const int k0 = j * BN, k1 = min(k0 + BN, kv_end);
        const uint8_t* p = mrow + k0;
        any = false;
        if (k1 - k0 == BN && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
            const uint4* q = reinterpret_cast<const uint4*>(p);
            uint32_t acc = 0;
#pragma unroll
            for (int e = 0; e < BN / 16; ++e) {
                const uint4 v = __ldg(q + e);
                acc |= v.x | v.y | v.z | v.w;
            }
            any = acc != 0;
        } else {
            for (int k = 0; k < k1 - k0 && !any; ++k) any = p[k] != 0;
        }
    }
    return __ballot_sync(0xffffffffu, any);
}

// Walks the visited key tiles (non-empty ones in [first, n_tiles)) in increasing
// order, 32 tiles per scan.  Warp-collective; every lane sees the same tiles.
struct TileIter {
    const uint8_t* mrow;
    int first, n_tiles, kv_end, lane, chunk;
    uint32_t f;
    __device__ __forceinline__ TileIter(const uint8_t* m, int fst, int n, int e, int l)
        : mrow(m), first(fst), n_tiles(n), kv_end(e), lane(l), chunk(fst / 32 - 1), f(0) {}
    // Primed with the flag word of the first chunk (fst / 32), already scanned.
    __device__ __forceinline__ TileIter(const uint8_t* m, int fst, int n, int e, int l, uint32_t f_first)
        : mrow(m), first(fst), n_tiles(n), kv_end(e), lane(l), chunk(fst / 32), f(f_first) {}
    __device__ __forceinline__ int next() {   // next visited tile, or -1
        while (f == 0) {
            ++chunk;
            if (chunk * 32 >= n_tiles) return -1;
            f = tile_flags(mrow, chunk, first, n_tiles, kv_end, lane);
        }
        const int l = __ffs(f) - 1;
        f &= f - 1;
        return chunk * 32 + l;
    }
};

// Bits of the tiles of chunk `chunk` whose index is below n.
__device__ __forceinline__ uint32_t below_bits(int n, int chunk) {
    const int rel = n - chunk * 32;
    return rel >= 32 ? 0xffffffffu : (rel <= 0 ? 0u : ((1u << rel) - 1u));
}

// p[c] = 2^(s[c] * fa - m_use) for NCOL (default 128) columns of a row: P packed to bf16x2 in
// pk, the row sum returned.  Two columns per paired FMA / add.
template <bool F16, int NCOL = BN>
__device__ __forceinline__ float exp_row(const float* s, float fa, float m_use, uint32_t* pk) {
    const uint64_t fa2 = f32x2(fa, fa);
    const uint64_t nm2 = f32x2(-m_use, -m_use);
    uint64_t rs4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) rs4[e] = f32x2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < NCOL / 2; ++c) {
        float x0, x1, p0, p1;
        f32x2_split(ffma2(f32x2(s[2 * c], s[2 * c + 1]), fa2, nm2), x0, x1);
        p0 = fast_exp2(x0);
        p1 = fast_exp2(x1);
        rs4[c & 3] = fadd2(rs4[c & 3], f32x2(p0, p1));
        pk[c] = pack2<F16>(p0, p1);
    }
    rs4[0] = fadd2(rs4[0], rs4[2]);
    rs4[1] = fadd2(rs4[1], rs4[3]);
    float r0, r1, r2, r3;
    f32x2_split(rs4[0], r0, r1);
    f32x2_split(rs4[1], r2, r3);
    return (r0 + r1) + (r2 + r3);
}

}  // namespace pf
}  // namespace gqa
