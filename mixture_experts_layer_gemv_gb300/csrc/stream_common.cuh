// Device building blocks of the weight-streaming expert kernels (expert_stream.cu):
// unit/tile decomposition, launch plans, TMA-box dot products and the A/B partial-sum
// buffers.
//
// The unit and tile arithmetic runs at the start of every CTA, on the critical path of
// a decode step, so it is 32-bit (the host refuses stages of kMaxStreamUnits units or
// more) and takes each part's K range from a table instead of dividing again: a 64-bit
// division is a long dependent chain of instructions, and a tile decoded with them took
// thousands of cycles.
#pragma once

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {
namespace stream {

constexpr int kCons = 8;                    // consumer warps: 8 x 16 rows = one tile
constexpr int kThreads = (kCons + 1) * 32;  // + one producer warp
constexpr int kConsThreads = kCons * 32;
constexpr int kTile = 128;
constexpr int kBox = kTile * kBlk;          // 16 KB: 128 rows x 128 bytes
// Activation rows of a unit sit kRowPitch bytes apart: 16 bytes more than a K block, so
// that the 8 rows of an mma B fragment fall in different shared-memory banks.
constexpr int kRowPitch = kBlk + 16;
constexpr int kBRows = 2048;                // the unit's activation rows (8 x kRowPitch, 1 KB-rounded)
constexpr int kStagesGU = 5;
constexpr int kMaxStagesD = 10;

constexpr int kMaxParts = 4;

// The unit sequence of a stage. Output rows come in "rows" of 128 (row group x 128-row
// slice): n_r routed rows with kc_r K blocks each, then n_s shared rows with kc_s.
// Each row's K blocks are split into P contiguous parts, part p holding blocks
// [lo[p], lo[p+1]) with lo[p] = p * kc / P; a tile is one (row, part) and a unit one
// (tile, K block). Units are ordered row-major, K block fastest.
struct TileSpace {
    int n_r, kc_r, n_s, kc_s, P;
    int lo_r[kMaxParts + 1], lo_s[kMaxParts + 1];
    __device__ int total() const { return n_r * kc_r + n_s * kc_s; }
    // lo[p] of the routed (shared = 0) or shared rows, p <= P
    __device__ __forceinline__ int lo(int shared, int p) const {
        int v = 0;
#pragma unroll
        for (int q = 0; q <= kMaxParts; ++q)
            if (q == p) v = shared ? lo_s[q] : lo_r[q];
        return v;
    }
    // tile of unit u; *kb receives its K block within the row
    __device__ int tile_of(int u, int* kb) const {
        const int shared = u >= n_r * kc_r;
        const int v = shared ? u - n_r * kc_r : u;
        const int kc = shared ? kc_s : kc_r;
        const int row = v / kc, kin = v - row * kc;
        int p = 0;
#pragma unroll
        for (int q = 1; q < kMaxParts; ++q)
            if (q < P && kin >= lo(shared, q)) p = q;
        *kb = kin;
        return (shared ? n_r * P : 0) + row * P + p;
    }
};

__device__ __forceinline__ TileSpace make_space(int n_r, int kc_r, int n_s, int kc_s, int P) {
    TileSpace t;
    t.n_r = n_r;
    t.kc_r = kc_r;
    t.n_s = n_s;
    t.kc_s = kc_s;
    t.P = P;
#pragma unroll
    for (int q = 0; q <= kMaxParts; ++q) {
        t.lo_r[q] = q * kc_r / P;
        t.lo_s[q] = q * kc_s / P;
    }
    return t;
}

// Launch plan shared by a streaming kernel and the kernels that read its tiles: the
// number of active CTAs and the K-part count P, so that every part fits in a range.
struct Plan {
    int nb, P;
};
__device__ __forceinline__ Plan make_plan(int n_r, int kc_r, int n_s, int kc_s, int grid, int max_parts) {
    const int U = n_r * kc_r + n_s * kc_s;
    Plan pl;
    pl.nb = max(1, min(grid, U));
    int kcmax = 0, kcmin = INT_MAX;  // over the kinds that have rows
    if (n_r > 0) kcmax = kcmin = kc_r;
    if (n_s > 0) {
        kcmax = max(kcmax, kc_s);
        kcmin = min(kcmin, kc_s);
    }
    if (kcmax == 0) kcmax = kcmin = 1;
    const int L = max(1, U / pl.nb);
    int P = (kcmax + L - 1) / L;
    P = max(1, min(P, min(max_parts, kcmin)));
    const int need = (kcmax + P - 1) / P;  // longest part
    if (need > L) pl.nb = max(1, U / need);
    pl.P = P;
    return pl;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// Lane (g, t4)'s A fragment pair (rows r and r+8, 16-byte chunk c) from a
// 128-byte-swizzled box: chunk c of row r sits at chunk position c ^ (r % 8).
__device__ __forceinline__ void load_a(const uint8_t* box, int r, int g, int c, uint4& lo, uint4& hi) {
    const int sw = (c ^ g) << 4;
    lo = lds128(box + r * kBlk + sw);
    hi = lds128(box + (r + 8) * kBlk + sw);
}

__device__ __forceinline__ void mma_step64(float (&c)[4], const uint4& ar, const uint4& ar8, const uint4& b, int half) {
    if (half == 0)
        mma_e4m3_16832(c, ar.x, ar8.x, ar.y, ar8.y, b.x, b.y);
    else
        mma_e4m3_16832(c, ar.z, ar8.z, ar.w, ar8.w, b.z, b.w);
}

// One 128 x 128-byte box times 8 activation rows (brow: this lane's row g, 128 bytes
// of K; bvalid: row g exists): the fp32 16x8 partial of this warp (rows 16w..16w+15).
// Columns of missing rows are zero and are not read from shared memory.
__device__ __forceinline__ void box_dot(float (&c)[4], const uint8_t* box, const uint8_t* brow, bool bvalid, int warp,
                                        int g, int t4) {
    const int r = warp * 16 + g;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        uint4 lo, hi;
        load_a(box, r, g, 4 * s + t4, lo, hi);
        const uint4 b = bvalid ? lds128(brow + s * 64 + 16 * t4) : make_uint4(0, 0, 0, 0);
        mma_step64(c, lo, hi, b, 0);
        mma_step64(c, lo, hi, b, 1);
    }
}

// MXFP8: the same box times 8 activation rows, one fp32 16x8 partial per 32-wide K block
// (c[q], q = 0..3), so that each block's E8M0 scales can be applied to its own partial.
// Lane (g, t4) supplies bytes [32q + 8t4, 32q + 8t4 + 8) of its A rows and B column for
// the MMA of block q; the MMA pairs A's and B's K slots the same way, so the products
// match and the sum runs over exactly that block.
__device__ __forceinline__ void box_dot_mx(float (&c)[4][4], const uint8_t* box, const uint8_t* brow, bool bvalid,
                                           int warp, int g, int t4) {
    const int r = warp * 16 + g;  // rows r and r + 8 share the swizzle phase r % 8
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int off = (((2 * q + (t4 >> 1)) ^ (r & 7)) << 4) + 8 * (t4 & 1);
        const uint2 lo = *reinterpret_cast<const uint2*>(box + r * kBlk + off);
        const uint2 hi = *reinterpret_cast<const uint2*>(box + (r + 8) * kBlk + off);
        const uint2 b = bvalid ? *reinterpret_cast<const uint2*>(brow + 32 * q + 8 * t4) : make_uint2(0, 0);
        mma_e4m3_16832(c[q], lo.x, hi.x, lo.y, hi.y, b.x, b.y);
    }
}

// A CTA's contiguous share [u0, u1) of the units: CTA b of nb takes U / nb units, one
// more for the first U % nb.
struct Range {
    int U, u0, u1, first_tile;
    int nb, b, kb0;
};

__device__ __forceinline__ Range make_range(const TileSpace& ts, int nb, int b) {
    Range r;
    r.U = ts.total();
    r.nb = nb;
    r.b = b;
    const int q = r.U / nb, rem = r.U - q * nb;
    r.u0 = b < nb ? b * q + min(b, rem) : 0;
    r.u1 = b < nb ? r.u0 + q + (b < rem ? 1 : 0) : 0;
    r.kb0 = 0;
    r.first_tile = (b < nb && r.u1 > r.u0) ? ts.tile_of(r.u0, &r.kb0) : 0;
    return r;
}

// One tile of a CTA's unit range, decoded once before the streaming loops so that
// neither the producer nor the consumers stall on descriptor loads or index
// arithmetic at tile boundaries.
struct TileRec {
    int shared, expert, group, row_begin, nrows, slice, part;
    int kb0;  // absolute K block of this range's first unit of the tile
    int n;    // units of the tile in this range
    int hs;   // 1: the range holds the tile's first unit
    int he;   // 1: the range holds the tile's last unit
    int pad;
    union {
        int tok[kGroupRows];  // gate/up: token of each activation row, -1 if none
        float w[kGroupRows];  // down: routing weight of each row (1 for the shared experts)
    };
};
constexpr int kMaxTab = 96;
constexpr size_t kTabBytes = (size_t)kMaxTab * sizeof(TileRec);

// Tile t of range rg: its row group (routed rows: groups[gi] for row gi * slices_r +
// slice; shared rows: tokens 8 sg .. 8 sg + 7 for row sg * slices_s + slice), its K part
// and the part's units inside the range.
__device__ inline TileRec make_rec(const TileSpace& ts, const Range& rg, int t, int slices_r, int slices_s,
                                   const RowGroup* groups, int T, int k, const int32_t* perm_src,
                                   const float* topk_w) {
    TileRec r;
    const int shared = t >= ts.n_r * ts.P;
    const int v = shared ? t - ts.n_r * ts.P : t;
    const int row = v / ts.P, p = v - row * ts.P;
    const int slices = shared ? slices_s : slices_r;
    const int gi = row / slices;
    r.shared = shared;
    r.slice = row - gi * slices;
    r.part = p;
    if (shared) {
        r.expert = -1;
        r.group = -1;
        r.row_begin = gi * kGroupRows;
        r.nrows = min(kGroupRows, T - r.row_begin);
    } else {
        const RowGroup g = groups[gi];
        r.expert = g.expert;
        r.group = gi;
        r.row_begin = g.row_begin;
        r.nrows = g.nrows;
    }
    const int kc = shared ? ts.kc_s : ts.kc_r;
    const int plo = ts.lo(shared, p), phi = ts.lo(shared, p + 1);
    const int st = (shared ? ts.n_r * ts.kc_r : 0) + row * kc + plo;  // the tile's first unit
    const int len = phi - plo;
    const int lo = st > rg.u0 ? st : rg.u0, hi = st + len < rg.u1 ? st + len : rg.u1;
    r.kb0 = plo + (lo - st);
    r.n = hi - lo;
    r.hs = st >= rg.u0;
    r.he = st + len <= rg.u1;
    r.pad = 0;
    const int Tk = T * k;
    int f[kGroupRows];
#pragma unroll
    for (int c = 0; c < kGroupRows; ++c) f[c] = (c < r.nrows && !shared) ? perm_src[r.row_begin + c] : -1;
#pragma unroll
    for (int c = 0; c < kGroupRows; ++c) {
        if (topk_w) {
            r.w[c] = c >= r.nrows ? 0.f : shared ? 1.f : ((unsigned)f[c] < (unsigned)Tk ? topk_w[f[c]] : 0.f);
        } else {
            r.tok[c] = c >= r.nrows ? -1 : shared ? r.row_begin + c : ((unsigned)f[c] < (unsigned)Tk ? f[c] / k : -1);
        }
    }
    return r;
}

// Decode the tiles of range rg into tab (cooperatively, threads tid of nthreads); the
// first kMaxTab are stored, the rest are decoded when reached. Returns the tile count.
__device__ inline int build_table(TileRec* tab, const TileSpace& ts, const Range& rg, int slices_r, int slices_s,
                                  const RowGroup* groups, int T, int k, const int32_t* perm_src, const float* topk_w,
                                  int tid, int nthreads) {
    int kbl;
    const int last = ts.tile_of(rg.u1 - 1, &kbl);
    const int n = last - rg.first_tile + 1;
    for (int i = tid; i < n && i < kMaxTab; i += nthreads)
        tab[i] = make_rec(ts, rg, rg.first_tile + i, slices_r, slices_s, groups, T, k, perm_src, topk_w);
    return n;
}

// Partial results of a stage: dense buffers A[m] and B[m], both [P][rows][N] with the
// output's row order (permuted rows for routed experts, tokens for the shared ones).
struct Partials {
    float* A[2];
    float* B[2];
    long rows;  // rows per part
    int N;      // row length
};

// Store this warp's share of a tile: vals[m][i] is row warp*16 + g + 8*(i>=2),
// column 2*t4 + (i&1) of matrix m. The CTA holding the tile's first unit writes A (and
// zeros to B when it also holds the last); a CTA holding the rest writes B.
template <int NMAT>
__device__ __forceinline__ void store_rec(const float (&vals)[NMAT][4], const TileRec& r, const Partials& pt) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int col = 2 * t4 + (i & 1);
        if (col >= r.nrows) continue;
        const int row = warp * 16 + g + (i >= 2 ? 8 : 0);
        const size_t o = ((size_t)r.part * pt.rows + r.row_begin + col) * pt.N + r.slice * kTile + row;
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            if (r.hs) {
                pt.A[m][o] = vals[m][i];
                if (r.he) pt.B[m][o] = 0.f;
            } else {
                pt.B[m][o] = vals[m][i];
            }
        }
    }
}

// Sum over the P parts of A + B at four consecutive channels col4.. of output row
// `orow` of matrix m.
__device__ __forceinline__ float4 read4(const Partials& pt, int P, int m, long orow, int col4) {
    // all 2P loads first, then the sums in part order: one memory round trip
    float4 a[kMaxParts], b[kMaxParts];
#pragma unroll
    for (int p = 0; p < kMaxParts; ++p)
        if (p < P) {
            const size_t o = ((size_t)p * pt.rows + orow) * pt.N + col4;
            a[p] = __ldcg(reinterpret_cast<const float4*>(pt.A[m] + o));
            b[p] = __ldcg(reinterpret_cast<const float4*>(pt.B[m] + o));
        }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int p = 0; p < kMaxParts; ++p)
        if (p < P) {
            acc.x += a[p].x + b[p].x;
            acc.y += a[p].y + b[p].y;
            acc.z += a[p].z + b[p].z;
            acc.w += a[p].w + b[p].w;
        }
    return acc;
}

}  // namespace stream
}  // namespace moe
