// Device building blocks of the weight-streaming expert kernels (expert_stream.cu):
// unit/tile decomposition, launch plans, the routing data in shared memory, TMA-box dot
// products and the A/B partial-sum buffers.
#pragma once

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "moe_internal.h"
#include "route_common.cuh"

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
// a unit one (tile, K block). Units are ordered row-major, K block fastest. Ix is the
// index type of units and tiles: int whenever the host has bounded the unit count
// below 2^31 (every decode shape), long long otherwise.
template <typename Ix>
struct TileSpace {
    Ix n_r;
    int kc_r;
    Ix n_s;
    int kc_s, P;
    __device__ Ix total() const { return n_r * kc_r + n_s * kc_s; }
    __device__ int kc_of(Ix t) const { return t < n_r * P ? kc_r : kc_s; }
    // first K block of part p of a row with kc blocks
    __device__ int part_lo(int kc, int p) const { return p * kc / P; }
    __device__ Ix start(Ix t) const {
        if (t < n_r * P) return (t / P) * kc_r + part_lo(kc_r, (int)(t % P));
        const Ix v = t - n_r * P;
        return n_r * kc_r + (v / P) * kc_s + part_lo(kc_s, (int)(v % P));
    }
    __device__ int len(Ix t) const {
        const int kc = kc_of(t), p = (int)(t % P);
        return part_lo(kc, p + 1) - part_lo(kc, p);
    }
    // tile of unit u; *kb receives its absolute K block
    __device__ Ix tile_of(Ix u, int* kb) const {
        Ix row, base_t;
        int kc, kin;
        if (u < n_r * kc_r) {
            row = u / kc_r;
            kin = (int)(u % kc_r);
            kc = kc_r;
            base_t = 0;
        } else {
            const Ix v = u - n_r * kc_r;
            row = v / kc_s;
            kin = (int)(v % kc_s);
            kc = kc_s;
            base_t = n_r * P;
        }
        *kb = kin;
        const int p = ((kin + 1) * P - 1) / kc;  // part whose range holds kin
        return base_t + row * P + p;
    }
};

// Launch plan shared by a streaming kernel and the kernels that read its tiles: the
// number of active CTAs and the K-part count P, so that every part fits in a range.
struct Plan {
    int nb, P;
};
constexpr int kMaxParts = 4;
template <typename Ix>
__device__ __forceinline__ Plan make_plan(Ix n_r, int kc_r, Ix n_s, int kc_s, int grid, int max_parts) {
    const Ix U = n_r * kc_r + n_s * kc_s;
    Plan pl;
    pl.nb = (int)(U < (Ix)grid ? U : (Ix)grid);
    if (pl.nb < 1) pl.nb = 1;
    int kcmax = 0, kcmin = INT_MAX;  // over the kinds that have rows
    if (n_r > 0) kcmax = kcmin = kc_r;
    if (n_s > 0) {
        kcmax = std::max(kcmax, kc_s);
        kcmin = std::min(kcmin, kc_s);
    }
    if (kcmax == 0) kcmax = kcmin = 1;
    const Ix L = std::max<Ix>(1, U / pl.nb);
    int P = (int)((kcmax + L - 1) / L);
    P = std::max(1, std::min(P, std::min(max_parts, kcmin)));
    const int need = (kcmax + P - 1) / P;  // longest part
    if (need > L) pl.nb = (int)std::max<Ix>(1, U / need);
    pl.P = P;
    return pl;
}

// The routing data the tile decoders read (the row groups, perm_src, topk_w and the group
// count), written by the router kernel (or the row-group kernel of the stage API) two or
// more kernels before the streaming kernels. The down kernel decodes its tiles before its
// own dependency wait: the router had completed, its writes performed at device scope,
// before the gate/up kernel's wait returned, and the down kernel is launched only after
// every gate/up CTA has passed that wait. Those reads go through L2 (ld.global.cg), the
// device's point of coherence, so no line an earlier kernel left in this SM's L1 can
// answer them.
constexpr int kMaxGroupsSmem = 256;  // row groups copied into shared memory
constexpr int kMaxRowsSmem = 512;    // routed rows (T*k) whose source slot and weight are copied

// 16-byte aligned: the row groups are copied with 16-byte vector stores.
struct alignas(16) RouteSmem {
    RowGroup groups[kMaxGroupsSmem];
    int32_t perm[kMaxRowsSmem];
    float w[kMaxRowsSmem];
    int n_groups;
};

// Where a decoder finds the routing data: shared-memory copies (smem = 1), or the
// workspace itself when it does not fit (read through L2).
struct RouteView {
    const RowGroup* groups;
    const int32_t* perm;
    const float* w;  // null: token ids wanted (gate/up); else routing weights (down)
    int n_groups;
    int smem;
    int E, R;     // routed experts, routed rows (T*k): the bounds of a valid record
    int* status;  // device status word (kStatusBadId for a record out of bounds)
};

// A row group as the decoders use it. A record outside the routing's bounds (an expert
// id outside [0, E), rows outside [0, T*k), none or more than kGroupRows of them) is read
// as an empty group of expert 0 and reported, so that no weight, scale or partial-sum
// address is ever formed from it.
__device__ __forceinline__ RowGroup route_group(const RouteView& v, int gi) {
    RowGroup g;
    if (v.smem) {
        g = v.groups[gi];
    } else {
        const int4 q = __ldcg(reinterpret_cast<const int4*>(v.groups) + gi);
        g = RowGroup{q.x, q.y, q.z, q.w};
    }
    if ((unsigned)g.expert >= (unsigned)v.E || g.nrows < 1 || g.nrows > kGroupRows || g.row_begin < 0 ||
        g.row_begin > v.R - g.nrows) {
        set_status(v.status, kStatusBadId);
        g = RowGroup{0, 0, 0, 0};
    }
    return g;
}
__device__ __forceinline__ int route_perm(const RouteView& v, int r) { return v.smem ? v.perm[r] : __ldcg(v.perm + r); }
__device__ __forceinline__ float route_w(const RouteView& v, int f) { return v.smem ? v.w[f] : __ldcg(v.w + f); }

// Gather the routing data into s with one round of loads (all threads tid < nthreads;
// ends with __syncthreads). max_groups: the workspace's row-group capacity.
__device__ inline RouteView load_route(RouteSmem* s, const Ctrl* ctrl, const RowGroup* groups, int max_groups,
                                       const int32_t* perm_src, const float* topk_w, int R, int E, int* status,
                                       int tid, int nthreads) {
    // every load is issued before any store (one memory round trip): with nthreads >= 256
    // a thread copies at most one row group and two rows
    const bool fits = max_groups <= kMaxGroupsSmem && R <= kMaxRowsSmem && 2 * nthreads >= kMaxRowsSmem &&
                      nthreads >= kMaxGroupsSmem;
    if (tid == 0) s->n_groups = min(max(__ldcg(&ctrl->n_routed_groups), 0), max_groups);
    if (fits) {
        const int i1 = tid + nthreads;
        const bool hg = tid < max_groups, h0 = tid < R, h1 = i1 < R;
        const int4 g = hg ? __ldcg(reinterpret_cast<const int4*>(groups) + tid) : make_int4(0, 0, 0, 0);
        const int p0 = h0 ? __ldcg(perm_src + tid) : 0, p1 = h1 ? __ldcg(perm_src + i1) : 0;
        const float w0 = topk_w && h0 ? __ldcg(topk_w + tid) : 0.f, w1 = topk_w && h1 ? __ldcg(topk_w + i1) : 0.f;
        if (hg) reinterpret_cast<int4*>(s->groups)[tid] = g;
        if (h0) {
            s->perm[tid] = p0;
            s->w[tid] = w0;
        }
        if (h1) {
            s->perm[i1] = p1;
            s->w[i1] = w1;
        }
    }
    __syncthreads();
    RouteView v;
    v.n_groups = s->n_groups;
    v.smem = fits ? 1 : 0;
    v.groups = fits ? s->groups : groups;
    v.perm = fits ? s->perm : perm_src;
    v.w = topk_w ? (fits ? s->w : topk_w) : nullptr;
    v.E = E;
    v.R = R;
    v.status = status;
    return v;
}

// Scratch of local_route: the CTA-wide top-k's keys, group keys and partial sums, the T*k
// selected ids, inverse positions, the counting sort's ranks and per-expert counts,
// offsets and group offsets.
constexpr int kLocalRows = kLocalT * 16;  // T*k slots (top_k <= 16)
struct alignas(16) LocalRouteSmem {
    unsigned key[routing::kMaxE];  // first: read as uint4
    unsigned gkey[32];
    float part[32];
    int32_t ids[kLocalRows];
    int32_t inv[kLocalRows];
    int32_t rank[kLocalRows];
    int32_t gor[kLocalRows];
    int32_t cnt[routing::kMaxE], gcnt[routing::kMaxE], goff[routing::kMaxE];
    int32_t off[routing::kMaxE + 1];
    int32_t offsets[routing::kMaxE + 1];
};

// The routing of T <= kLocalT tokens derived by one CTA from the router's logits (read
// through L2): softmax and group-limited top-k of each token by one warp (the router's own
// function, so every CTA makes the same selection), then the stable counting sort of the
// T*k slots and the row groups, in shared memory. publish (gate/up CTA 0): the result is
// also written to the workspace for the combine kernel and the caller. All nthreads
// threads call it; it ends with __syncthreads. want_w: the view carries the routing
// weights (down) rather than token ids (gate/up).
__device__ inline RouteView local_route(RouteSmem* s, LocalRouteSmem* L, const StreamArgs& a, bool publish,
                                        bool want_w, int tid, int nthreads) {
    using namespace routing;
    const int warp = tid >> 5, lane = tid & 31, T = a.T, k = a.k, E = a.E, n = T * k;
    if (T == 1 && E <= nthreads) {
        // one token: the whole CTA ranks the experts (the router's one-token selection)
        cta_topk1(a.logits, E, a.G, a.Gk, k, a.scale, L->key, L->gkey, L->part, L->ids, s->w, nullptr);
    } else if (warp < T) {
        float lg[kMaxE / 32];
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i) {
            const int e = lane + 32 * i;
            lg[i] = e < E ? __ldcg(a.logits + (size_t)warp * E + e) : -INFINITY;
        }
        topk_warp(lg, E, a.G, a.Gk, k, a.scale, nullptr, L->ids + warp * k, s->w + warp * k, nullptr);
    }
    __syncthreads();
    small_permute(L->ids, n, E, L->cnt, L->off, L->gcnt, L->goff, L->rank, L->offsets, s->perm, L->inv, s->groups,
                  L->gor, &s->n_groups);
    __syncthreads();
    if (publish) {
        for (int i = tid; i < n; i += nthreads) {
            a.pub_ids[i] = L->ids[i];
            a.pub_w[i] = s->w[i];
            a.pub_perm[i] = s->perm[i];
            a.pub_inv[i] = L->inv[i];
            a.pub_group_of_row[i] = L->gor[i];
        }
        for (int e = tid; e <= E; e += nthreads) a.pub_offsets[e] = L->offsets[e];
        for (int g = tid; g < s->n_groups; g += nthreads) a.pub_groups[g] = s->groups[g];
        if (tid == 0) *a.pub_n_groups = s->n_groups;
    }
    RouteView v;
    v.n_groups = s->n_groups;
    v.smem = 1;
    v.groups = s->groups;
    v.perm = s->perm;
    v.w = want_w ? s->w : nullptr;
    v.E = E;
    v.R = n;
    v.status = a.status;
    return v;
}

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

template <typename Ix>
__device__ __forceinline__ TileInfo decode_tile(const TileSpace<Ix>& ts, Ix t, int slices_r, int slices_s,
                                                const RouteView& rv, int T) {
    TileInfo ti;
    ti.part = (int)(t % ts.P);
    if (t < ts.n_r * ts.P) {
        const Ix row = t / ts.P;
        const int gi = (int)(row / slices_r);
        const RowGroup rg = route_group(rv, gi);
        ti.shared = 0;
        ti.expert = rg.expert;
        ti.group = gi;
        ti.row_begin = rg.row_begin;
        ti.nrows = rg.nrows;
        ti.slice = (int)(row % slices_r);
    } else {
        const Ix row = (t - ts.n_r * ts.P) / ts.P;
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

template <typename Ix>
struct Range {
    Ix U, u0, u1, first_tile;
    int nb, b, kb0;
};

template <typename Ix>
__device__ __forceinline__ Range<Ix> make_range(const TileSpace<Ix>& ts, int nb, int b) {
    Range<Ix> r;
    r.U = ts.total();
    r.nb = nb;
    r.b = b;
    // b * U fits the index type (the host bounds units x CTAs for int indices)
    r.u0 = b < nb ? (Ix)b * r.U / nb : 0;
    r.u1 = b < nb ? (Ix)(b + 1) * r.U / nb : 0;
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

template <typename Ix>
__device__ inline TileRec make_rec(const TileSpace<Ix>& ts, const Range<Ix>& rg, Ix t, int slices_r, int slices_s,
                                   const RouteView& rv, int T, int k) {
    TileRec r;
    const TileInfo ti = decode_tile(ts, t, slices_r, slices_s, rv, T);
    r.shared = ti.shared;
    r.expert = ti.expert;
    r.group = ti.group;
    r.row_begin = ti.row_begin;
    r.nrows = ti.nrows;
    r.slice = ti.slice;
    r.part = ti.part;
    const Ix st = ts.start(t);
    const int len = ts.len(t);
    const Ix lo = st > rg.u0 ? st : rg.u0, hi = st + len < rg.u1 ? st + len : rg.u1;
    int kbs;
    ts.tile_of(st, &kbs);
    r.kb0 = kbs + (int)(lo - st);
    r.n = (int)(hi - lo);
    r.hs = st >= rg.u0;
    r.he = st + len <= rg.u1;
    r.pad = 0;
    const int Tk = T * k;
#ifdef MOE_DEBUG
    // debug builds: the decomposition's invariants for every tile (a tile that breaks one
    // is reported and streams nothing)
    {
        const int kc = ts.kc_of(t), slices = ti.shared ? slices_s : slices_r;
        const bool ok = r.n >= 1 && r.kb0 >= 0 && r.kb0 + r.n <= kc && r.part >= 0 && r.part < ts.P &&
                        r.slice >= 0 && r.slice < slices && r.row_begin >= 0 && r.nrows >= 0 &&
                        r.nrows <= kGroupRows && r.row_begin + r.nrows <= (ti.shared ? T : Tk);
        if (!ok) {
            set_status(rv.status, kStatusBadId);
            r.n = 0;
            r.nrows = 0;
            r.row_begin = 0;
            r.expert = ti.shared ? -1 : 0;
        }
    }
#endif
    int f[kGroupRows];
#pragma unroll
    for (int c = 0; c < kGroupRows; ++c) f[c] = (c < r.nrows && !r.shared) ? route_perm(rv, r.row_begin + c) : -1;
#pragma unroll
    for (int c = 0; c < kGroupRows; ++c) {
        if (rv.w) {
            r.w[c] = c >= r.nrows ? 0.f : r.shared ? 1.f : ((unsigned)f[c] < (unsigned)Tk ? route_w(rv, f[c]) : 0.f);
        } else {
            r.tok[c] = c >= r.nrows ? -1 : r.shared ? r.row_begin + c : ((unsigned)f[c] < (unsigned)Tk ? f[c] / k : -1);
        }
    }
    return r;
}

// make_rec kept out of line, for tiles beyond the table (decoded when reached): keeps the
// streaming loops' register footprint that of a table lookup.
template <typename Ix>
__device__ __noinline__ TileRec make_rec_far(const TileSpace<Ix>& ts, const Range<Ix>& rg, Ix t, int slices_r,
                                             int slices_s, const RouteView& rv, int T, int k) {
    return make_rec(ts, rg, t, slices_r, slices_s, rv, T, k);
}

// Decode the tiles of range rg into tab (cooperatively, threads tid of nthreads); the
// first kMaxTab are stored, the rest are decoded when reached. Returns the tile count.
template <typename Ix>
__device__ inline int build_table(TileRec* tab, const TileSpace<Ix>& ts, const Range<Ix>& rg, int slices_r,
                                  int slices_s, const RouteView& rv, int T, int k, int tid, int nthreads) {
    int kbl;
    const Ix last = ts.tile_of(rg.u1 - 1, &kbl);
    const int n = (int)(last - rg.first_tile + 1);
    for (int i = tid; i < n && i < kMaxTab; i += nthreads)
        tab[i] = make_rec(ts, rg, rg.first_tile + (Ix)i, slices_r, slices_s, rv, T, k);
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

// Store this warp's share of the tile described by r: vals[m][i] is row warp*16 + g +
// 8*(i>=2), column 2*t4 + (i&1) of matrix m. The range holding the tile's first unit
// writes A (and zeros into B when it also holds the last unit); the other writes B.
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
