// Device building blocks of the weight-streaming expert kernels (expert_stream.cu)
// and the fused small-T layer kernel (moe_fused.cu): unit/tile decomposition,
// launch plans, TMA-box dot products and the A/B partial-sum buffers.
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

// The unit sequence of a stage. Output rows come in "rows" of 128 (row group x 128-row
// slice): n_r routed rows with kc_r K blocks each, then n_s shared rows with kc_s.
// Each row's K blocks are split into P contiguous parts; a tile is one (row, part) and
// a unit one (tile, K block). Units are ordered row-major, K block fastest.
struct TileSpace {
    int n_r, kc_r, n_s, kc_s, P;
    __device__ long total() const { return (long)n_r * kc_r + (long)n_s * kc_s; }
    __device__ int kc_of(long t) const { return t < (long)n_r * P ? kc_r : kc_s; }
    // first K block of part p of a row with kc blocks
    __device__ int part_lo(int kc, int p) const { return (int)((long)p * kc / P); }
    __device__ long start(long t) const {
        if (t < (long)n_r * P) return (t / P) * kc_r + part_lo(kc_r, (int)(t % P));
        const long v = t - (long)n_r * P;
        return (long)n_r * kc_r + (v / P) * kc_s + part_lo(kc_s, (int)(v % P));
    }
    __device__ int len(long t) const {
        const int kc = kc_of(t), p = (int)(t % P);
        return part_lo(kc, p + 1) - part_lo(kc, p);
    }
    // tile of unit u; *kb receives its absolute K block
    __device__ long tile_of(long u, int* kb) const {
        long row, base_t;
        int kc, kin;
        if (u < (long)n_r * kc_r) {
            row = u / kc_r;
            kin = (int)(u % kc_r);
            kc = kc_r;
            base_t = 0;
        } else {
            const long v = u - (long)n_r * kc_r;
            row = v / kc_s;
            kin = (int)(v % kc_s);
            kc = kc_s;
            base_t = (long)n_r * P;
        }
        *kb = kin;
        const int p = (int)(((long)(kin + 1) * P - 1) / kc);  // part whose range holds kin
        return base_t + row * P + p;
    }
};

// Launch plan shared by a streaming kernel and the kernels that read its tiles: the
// number of active CTAs and the K-part count P, so that every part fits in a range.
struct Plan {
    int nb, P;
};
constexpr int kMaxParts = 4;
__device__ __forceinline__ Plan make_plan(int n_r, int kc_r, int n_s, int kc_s, int grid, int max_parts) {
    const long U = (long)n_r * kc_r + (long)n_s * kc_s;
    Plan pl;
    pl.nb = (int)std::max<long>(1, std::min<long>(grid, U));
    int kcmax = 0, kcmin = INT_MAX;  // over the kinds that have rows
    if (n_r > 0) kcmax = kcmin = kc_r;
    if (n_s > 0) {
        kcmax = std::max(kcmax, kc_s);
        kcmin = std::min(kcmin, kc_s);
    }
    if (kcmax == 0) kcmax = kcmin = 1;
    const long L = std::max<long>(1, U / pl.nb);
    int P = (int)((kcmax + L - 1) / L);
    P = std::max(1, std::min(P, std::min(max_parts, kcmin)));
    const long need = (kcmax + P - 1) / P;  // longest part
    if (need > L) pl.nb = (int)std::max<long>(1, U / need);
    pl.P = P;
    return pl;
}

// The routing data the tile decoders read (the work list, perm_src, topk_w, the group
// count) is written by the router kernel. The down kernel decodes its tiles before its own
// dependency wait: the router had completed, its writes visible, before the gate/up
// kernel's wait returned, and the down kernel is launched only after every gate/up CTA
// has passed that wait.
__device__ __forceinline__ int routed_groups(const Ctrl* c) { return c->n_routed_groups; }

// A tile decoded: which row group, which 128-row slice of the output, which K part.
struct TileInfo {
    int shared;     // 1: shared experts
    int expert;     // routed expert id (routed tiles)
    int group;      // routed row-group index (routed tiles)
    int row_begin;  // permuted row (routed) or token (shared) of column 0
    int nrows;      // activation columns, <= 8
    int slice;      // 128-row slice index within the matrix
    int part;       // K part
};

__device__ __forceinline__ TileInfo decode_tile(const TileSpace& ts, long t, int slices_r, int slices_s,
                                                const RowGroup* groups, int T) {
    TileInfo ti;
    ti.part = (int)(t % ts.P);
    if (t < (long)ts.n_r * ts.P) {
        const long row = t / ts.P;
        const int gi = (int)(row / slices_r);
        const RowGroup rg = groups[gi];
        ti.shared = 0;
        ti.expert = rg.expert;
        ti.group = gi;
        ti.row_begin = rg.row_begin;
        ti.nrows = rg.nrows;
        ti.slice = (int)(row % slices_r);
    } else {
        const long row = (t - (long)ts.n_r * ts.P) / ts.P;
        ti.shared = 1;
        ti.expert = -1;
        ti.group = -1;
        ti.row_begin = (int)(row / slices_s) * kGroupRows;
        ti.nrows = min(kGroupRows, T - ti.row_begin);
        ti.slice = (int)(row % slices_s);
    }
    return ti;
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

struct Range {
    long U, u0, u1, first_tile;
    int nb, b, kb0;
};

__device__ __forceinline__ Range make_range(const TileSpace& ts, int nb, int b) {
    Range r;
    r.U = ts.total();
    r.nb = nb;
    r.b = b;
    r.u0 = b < nb ? (long)b * r.U / nb : 0;
    r.u1 = b < nb ? (long)(b + 1) * r.U / nb : 0;
    r.kb0 = 0;
    r.first_tile = (b < nb && r.u1 > r.u0) ? ts.tile_of(r.u0, &r.kb0) : 0;
    return r;
}

// One tile of a CTA's unit range, decoded once before the streaming loops so that
// neither the producer nor the consumers stall on descriptor loads or 64-bit index
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

__device__ inline TileRec make_rec(const TileSpace& ts, const Range& rg, long t, int slices_r, int slices_s,
                                   const RowGroup* groups, int T, int k, const int32_t* perm_src,
                                   const float* topk_w) {
    TileRec r;
    const TileInfo ti = decode_tile(ts, t, slices_r, slices_s, groups, T);
    r.shared = ti.shared;
    r.expert = ti.expert;
    r.group = ti.group;
    r.row_begin = ti.row_begin;
    r.nrows = ti.nrows;
    r.slice = ti.slice;
    r.part = ti.part;
    const long st = ts.start(t), len = ts.len(t);
    const long lo = st > rg.u0 ? st : rg.u0, hi = st + len < rg.u1 ? st + len : rg.u1;
    int kbs;
    ts.tile_of(st, &kbs);
    r.kb0 = kbs + (int)(lo - st);
    r.n = (int)(hi - lo);
    r.hs = st >= rg.u0;
    r.he = st + len <= rg.u1;
    r.pad = 0;
    const int Tk = T * k;
    int f[kGroupRows];
#pragma unroll
    for (int c = 0; c < kGroupRows; ++c)
        f[c] = (c < ti.nrows && !ti.shared) ? perm_src[ti.row_begin + c] : -1;
#pragma unroll
    for (int c = 0; c < kGroupRows; ++c) {
        if (topk_w) {
            r.w[c] = c >= ti.nrows ? 0.f : ti.shared ? 1.f : ((unsigned)f[c] < (unsigned)Tk ? topk_w[f[c]] : 0.f);
        } else {
            r.tok[c] = c >= ti.nrows ? -1 : ti.shared ? ti.row_begin + c : ((unsigned)f[c] < (unsigned)Tk ? f[c] / k : -1);
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
    const long last = ts.tile_of(rg.u1 - 1, &kbl);
    const int n = (int)(last - rg.first_tile + 1);
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
// column 2*t4 + (i&1) of matrix m.
template <int NMAT>
__device__ __forceinline__ void store_tile(const float (&vals)[NMAT][4], const TileSpace& ts, const Range& rg, long t,
                                           const TileInfo& ti, const Partials& pt) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t4 = lane & 3;
    const long st = ts.start(t);
    const bool holds_start = st >= rg.u0;
    const bool holds_end = st + ts.len(t) <= rg.u1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int col = 2 * t4 + (i & 1);
        if (col >= ti.nrows) continue;
        const int row = warp * 16 + g + (i >= 2 ? 8 : 0);
        const size_t o = ((size_t)ti.part * pt.rows + ti.row_begin + col) * pt.N + ti.slice * kTile + row;
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            if (holds_start) {
                pt.A[m][o] = vals[m][i];
                if (holds_end) pt.B[m][o] = 0.f;
            } else {
                pt.B[m][o] = vals[m][i];
            }
        }
    }
}

// Sum over the P parts of A + B at four consecutive channels col4.. of output row
// `orow` of matrix m.
// store_tile with the tile described by a TileRec
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
