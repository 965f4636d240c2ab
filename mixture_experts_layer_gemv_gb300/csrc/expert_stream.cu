// Stages P1/P2 and Q1/Q2 of the DeepSeek-V2 MoE layer ("DSV2-236B-MegaKernel",
// README stage flowchart, MoE subgraph) in the weight-streaming regime, where each
// expert sees at most a few tokens and every FP8 weight byte is used by at most 8
// activation rows: bound by HBM bandwidth (decode is a matrix-vector product: the
// DeepSeek-V4.1 Flash Kernel Journey lecture, "Skill 5").
//
// Work decomposition (stream-K). A tile is 128 output rows of one matrix (gate and up
// together for P1/Q1) for one row group of <= 8 activation rows; a unit is one tile
// times one 128-wide K block (one FP8 scale block). All units of a stage are laid out
// in one sequence and every CTA (one per SM) takes an equal contiguous range of it, so
// every SM streams the same number of bytes whatever the routing.
//
// No CTA waits for another. The K range of every output row block is split into P
// parts, P just large enough that no part (a tile) is longer than a CTA's range, so a
// tile has at most two contributors. Partial sums go to two dense fp32 buffers with
// the layout of the output: the CTA holding a tile's first unit stores into A (and, if
// it also holds the last unit, zeros into B); when the tile is cut by a range boundary
// the next CTA stores the rest into B. A reader adds A + B over the P parts in a fixed
// order: deterministic, with no fence, atomic, spin, counter or zero-initialisation.
//
// Data movement. One producer thread streams weight boxes of 128 rows x 128 bytes with
// 2-D TMA (128-byte swizzle) into a ring of shared-memory stages guarded by mbarriers;
// eight consumer warps each own 16 rows of the tile and run mma.m16n8k32
// (E4M3 x E4M3 -> fp32) as a dequantising dot-product engine. Block scales are applied
// once per unit: acc += partial * s_w[rowblock][kblock] * s_x[token][kblock].
//
// The down kernel builds its FP8 operand itself: for each row group it sums the gate/up
// tiles, forms a = SiLU(g) * u and quantises every 128 values (one gate/up tile, one
// down K block) to E4M3 with a power-of-two scale, in shared memory, while its producer
// is already streaming down weights (which depend only on the routing).
//
// Launch chaining. The kernels are launched with programmatic stream serialisation.
// The gate/up kernel prefetches the shared experts' weights (independent of the
// routing) into L2 before it waits for the router.
#include "stream_common.cuh"

namespace moe {

namespace {

using namespace stream;

template <typename Ix>
__device__ __forceinline__ TileSpace<Ix> gateup_space(const StreamArgs& a, int ng, int P) {
    return TileSpace<Ix>{(Ix)ng * (a.I / kTile), a.H / kBlk, (Ix)a.n_shared_groups * (a.Is / kTile), a.H / kBlk, P};
}
template <typename Ix>
__device__ __forceinline__ Plan gateup_plan(const StreamArgs& a, int ng) {
    return make_plan<Ix>((Ix)ng * (a.I / kTile), a.H / kBlk, (Ix)a.n_shared_groups * (a.Is / kTile), a.H / kBlk,
                         a.grid_gu, a.max_parts);
}
template <typename Ix>
__device__ __forceinline__ TileSpace<Ix> down_space(const StreamArgs& a, int ng, int P) {
    const int slices = a.H / kTile;
    return TileSpace<Ix>{(Ix)ng * slices, a.I / kBlk, (Ix)a.n_shared_groups * slices, a.Is / kBlk, P};
}
template <typename Ix>
__device__ __forceinline__ Plan down_plan(const StreamArgs& a, int ng) {
    const int slices = a.H / kTile;
    return make_plan<Ix>((Ix)ng * slices, a.I / kBlk, (Ix)a.n_shared_groups * slices, a.Is / kBlk, a.grid_d,
                         a.max_parts);
}

__device__ __forceinline__ uint32_t ldg32(const uint8_t* p) { return __ldg(reinterpret_cast<const uint32_t*>(p)); }

// ================================================================== gate / up
// kMX: MXFP8 weights and activations (E8M0 scales per row / token and 32 K)
// kLocal: the routing is derived here from the router's logits (local_route); only the
// int-indexed instantiations have it
template <bool kMX, typename Ix, bool kLocal>
__global__ void __launch_bounds__(kThreads, 1)
    gateup_stream_kernel(const StreamArgs a, const __grid_constant__ TmaMap tm_g, const __grid_constant__ TmaMap tm_u,
                         const __grid_constant__ TmaMap tm_sg, const __grid_constant__ TmaMap tm_su) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int S = kStagesGU;
    constexpr int SB = 2 * kBox + kBRows;
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * SB);
    uint64_t* empty = full + S;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int H = a.H, Hb = H / kBlk;
    if (tid == 0) trace_stamp(a.trace, 1, 0);

    // the fault-injection word the host wrote before the call (read while the router runs)
    __shared__ unsigned s_inject;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCons);
        }
        fence_mbar_init();
        s_inject = __ldcg(&a.ctrl->inject);
    }
    for (int s = 0; s < S; ++s)  // activation rows beyond a group's size are read but masked
        for (int i = tid; i < kBRows / 16; i += kThreads)
            reinterpret_cast<uint4*>(smem + s * SB + 2 * kBox)[i] = make_uint4(0, 0, 0, 0);
    if (warp == kCons && lane == 0) {
        prefetch_tmap(&tm_g);
        prefetch_tmap(&tm_u);
        if (a.Is > 0) {
            prefetch_tmap(&tm_sg);
            prefetch_tmap(&tm_su);
            // the shared experts' gate/up weights do not depend on the routing:
            // pull this CTA's slice of them into L2 while the router runs
            const size_t bytes = (size_t)a.Is * H;
            const size_t per = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~size_t(15);
            const size_t lo = std::min(bytes, per * blockIdx.x), hi = std::min(bytes, lo + per);
            for (size_t o = lo; o < hi; o += 65536) {
                const uint32_t n = (uint32_t)std::min<size_t>(65536, hi - o);
                bulk_prefetch_l2(a.ws_gate + o, n);
                bulk_prefetch_l2(a.ws_up + o, n);
            }
        }
    }
    __syncthreads();
    pdl_wait();  // routing, activation codes and the work list are complete
    pdl_launch_dependents();
    if (tid == 0) trace_stamp(a.trace, 1, 1);

    // the routing data in one round of loads, then the plan and this CTA's tiles, with
    // the token of every activation row, from shared memory
    __shared__ RouteSmem s_route;
    RouteView rv;
    if constexpr (kLocal) {
        __shared__ LocalRouteSmem s_local;
        rv = local_route(&s_route, &s_local, a, blockIdx.x == 0, false, tid, kThreads);
    } else {
        rv = load_route(&s_route, a.ctrl, a.groups, a.max_groups, a.perm_src, nullptr, a.T * a.k, a.E, a.status, tid,
                        kThreads);
    }
    const int slices_r = a.I / kTile, slices_s = a.Is / kTile;
    const Plan pl = gateup_plan<Ix>(a, rv.n_groups);
    const TileSpace<Ix> ts = gateup_space<Ix>(a, rv.n_groups, pl.P);
    const Range<Ix> rg = make_range(ts, pl.nb, blockIdx.x);
    if (blockIdx.x >= pl.nb || rg.u1 <= rg.u0) return;
    const Partials pt{{a.g_r, a.u_r}, {a.gb_r, a.ub_r}, (long)a.T * a.k, a.I};
    const Partials pts{{a.g_s, a.u_s}, {a.gb_s, a.ub_s}, (long)a.T, a.Is};
    __shared__ TileRec s_tab[kMaxTab];
    const int ntiles = build_table(s_tab, ts, rg, slices_r, slices_s, rv, a.T, a.k, tid, kThreads);
    __syncthreads();
    auto rec = [&](int i) {
        return i < kMaxTab ? s_tab[i] : make_rec_far(ts, rg, rg.first_tile + (Ix)i, slices_r, slices_s, rv, a.T, a.k);
    };

    if (warp == kCons) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        // failure-detection tests: issue nothing, so that every consumer wait runs out
        if (s_inject & kInjectSkipGateupLoads) return;
        // Evict-first: the routed experts' weights always (a row group's pass over them is
        // not followed by another soon enough to hit in L2, and the partial sums that the
        // down kernel and the combine read back should outlive them), the shared experts'
        // only when no other row group reads them again (up to 8 tokens).
        const uint64_t wpol = l2_policy_evict_first();
        int s = 0, ph = 0;
        long q = 0;  // units issued
        bool stop = false;
        for (int i = 0; i < ntiles && !stop; ++i) {
            const TileRec r = rec(i);
            const uint8_t* xrow[kGroupRows];
            int nrow = 0;
#pragma unroll
            for (int c = 0; c < kGroupRows; ++c) {
                xrow[c] = r.tok[c] >= 0 ? a.xq + (size_t)r.tok[c] * H : nullptr;
                nrow += xrow[c] != nullptr;
            }
            const int y = r.shared ? r.slice * kTile : r.expert * a.I + r.slice * kTile;
            const void* mg = r.shared ? (const void*)&tm_sg : (const void*)&tm_g;
            const void* mu = r.shared ? (const void*)&tm_su : (const void*)&tm_u;
            for (int j = 0; j < r.n; ++j, ++q) {
                if (q >= S && !mbar_wait_bounded(&empty[s], ph ^ 1)) {
                    set_status(a.status, kStatusTimeout);
                    stop = true;
                    break;
                }
                const int kb = r.kb0 + j;
                uint8_t* st = smem + s * SB;
                mbar_arrive_expect_tx(&full[s], 2 * kBox + nrow * kBlk);
                if (a.stream_once || !r.shared) {
                    tma_load_2d_hint(st, mg, kb * kBlk, y, &full[s], wpol);
                    tma_load_2d_hint(st + kBox, mu, kb * kBlk, y, &full[s], wpol);
                } else {
                    tma_load_2d(st, mg, kb * kBlk, y, &full[s]);
                    tma_load_2d(st + kBox, mu, kb * kBlk, y, &full[s]);
                }
#pragma unroll
                for (int c = 0; c < kGroupRows; ++c)
                    if (xrow[c]) bulk_load(st + 2 * kBox + c * kRowPitch, xrow[c] + kb * kBlk, kBlk, &full[s]);
                if (++s == S) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        return;  // the consumers wait for every copy issued here before the CTA exits
    }

    // ---------------------------------------------------------------- consumers
    bool failed = false;
    int s = 0, ph = 0;
    for (int i = 0; i < ntiles; ++i) {
        const TileRec r = rec(i);
        const float *sgr = nullptr, *sur = nullptr;
        if constexpr (!kMX) {
            if (r.shared) {
                sgr = a.ss_gate + (size_t)r.slice * Hb;
                sur = a.ss_up + (size_t)r.slice * Hb;
            } else {
                const size_t e = (size_t)r.expert;
                sgr = a.s_gate + (e * (a.I / kBlk) + r.slice) * Hb;
                sur = a.s_up + (e * (a.I / kBlk) + r.slice) * Hb;
            }
        }
        const int tok0 = r.tok[2 * t4], tok1 = r.tok[2 * t4 + 1];
        const float* xs0 = !kMX && tok0 >= 0 ? a.xs + (size_t)tok0 * Hb : nullptr;
        const float* xs1 = !kMX && tok1 >= 0 ? a.xs + (size_t)tok1 * Hb : nullptr;
        // MXFP8: E8M0 scale rows of this lane's two weight rows (tile rows warp*16 + g and
        // + 8) and of its two tokens; 4 bytes (the 4 blocks of 32) per 128-wide K block
        const int Hs = H / 32;
        const uint8_t *wg8 = nullptr, *wu8 = nullptr, *x80 = nullptr, *x81 = nullptr;
        if constexpr (kMX) {
            const size_t row = (r.shared ? 0 : (size_t)r.expert * a.I) + (size_t)r.slice * kTile + warp * 16 + g;
            wg8 = (r.shared ? a.ss_gate8 : a.s_gate8) + row * Hs;
            wu8 = (r.shared ? a.ss_up8 : a.s_up8) + row * Hs;
            x80 = tok0 >= 0 ? a.xs8 + (size_t)tok0 * Hs : nullptr;
            x81 = tok1 >= 0 ? a.xs8 + (size_t)tok1 * Hs : nullptr;
        }
        int tokg = -1;  // this lane's B column: activation row g
#pragma unroll
        for (int c = 0; c < kGroupRows; ++c)
            if (c == g) tokg = r.tok[c];
        const bool bv = tokg >= 0;
        float acc[2][4] = {};
        for (int j = 0; j < r.n; ++j) {
            const int kb = r.kb0 + j;
            if constexpr (kMX) {
                const uint32_t g0 = ldg32(wg8 + kb * 4), g1 = ldg32(wg8 + 8 * Hs + kb * 4);
                const uint32_t u0 = ldg32(wu8 + kb * 4), u1 = ldg32(wu8 + 8 * Hs + kb * 4);
                const uint32_t s0 = x80 ? ldg32(x80 + kb * 4) : 0u, s1 = x81 ? ldg32(x81 + kb * 4) : 0u;
                if (!failed && !mbar_wait_bounded(&full[s], ph)) {
                    set_status(a.status, kStatusTimeout);
                    failed = true;
                }
                const uint8_t* st = smem + s * SB;
                float cg[4][4] = {}, cu[4][4] = {};
                if (!failed) {
                    box_dot_mx(cg, st, st + 2 * kBox + g * kRowPitch, bv, warp, g, t4);
                    box_dot_mx(cu, st + kBox, st + 2 * kBox + g * kRowPitch, bv, warp, g, t4);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float a0 = x80 ? e8m0_to_float((s0 >> (8 * q)) & 0xFF) : 0.f;
                    const float a1 = x81 ? e8m0_to_float((s1 >> (8 * q)) & 0xFF) : 0.f;
                    const float gs0 = e8m0_to_float((g0 >> (8 * q)) & 0xFF), gs1 = e8m0_to_float((g1 >> (8 * q)) & 0xFF);
                    const float us0 = e8m0_to_float((u0 >> (8 * q)) & 0xFF), us1 = e8m0_to_float((u1 >> (8 * q)) & 0xFF);
                    acc[0][0] = fmaf(cg[q][0], gs0 * a0, acc[0][0]);
                    acc[0][1] = fmaf(cg[q][1], gs0 * a1, acc[0][1]);
                    acc[0][2] = fmaf(cg[q][2], gs1 * a0, acc[0][2]);
                    acc[0][3] = fmaf(cg[q][3], gs1 * a1, acc[0][3]);
                    acc[1][0] = fmaf(cu[q][0], us0 * a0, acc[1][0]);
                    acc[1][1] = fmaf(cu[q][1], us0 * a1, acc[1][1]);
                    acc[1][2] = fmaf(cu[q][2], us1 * a0, acc[1][2]);
                    acc[1][3] = fmaf(cu[q][3], us1 * a1, acc[1][3]);
                }
            } else {
                const float swg = __ldg(sgr + kb), swu = __ldg(sur + kb);
                const float sx0 = xs0 ? __ldg(xs0 + kb) : 0.f;
                const float sx1 = xs1 ? __ldg(xs1 + kb) : 0.f;
                // after a timed-out wait this warp keeps walking the units (so its control flow
                // matches its siblings') but waits for and computes nothing more
                if (!failed && !mbar_wait_bounded(&full[s], ph)) {
                    set_status(a.status, kStatusTimeout);
                    failed = true;
                }
                const uint8_t* st = smem + s * SB;
                float cg[4] = {0.f, 0.f, 0.f, 0.f}, cu[4] = {0.f, 0.f, 0.f, 0.f};
                if (!failed) {
                    box_dot(cg, st, st + 2 * kBox + g * kRowPitch, bv, warp, g, t4);
                    box_dot(cu, st + kBox, st + 2 * kBox + g * kRowPitch, bv, warp, g, t4);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    if (tid == 0 && i == 0 && j == 0) trace_stamp(a.trace, 1, 2);
                }
                acc[0][0] = fmaf(cg[0], swg * sx0, acc[0][0]);
                acc[0][1] = fmaf(cg[1], swg * sx1, acc[0][1]);
                acc[0][2] = fmaf(cg[2], swg * sx0, acc[0][2]);
                acc[0][3] = fmaf(cg[3], swg * sx1, acc[0][3]);
                acc[1][0] = fmaf(cu[0], swu * sx0, acc[1][0]);
                acc[1][1] = fmaf(cu[1], swu * sx1, acc[1][1]);
                acc[1][2] = fmaf(cu[2], swu * sx0, acc[1][2]);
                acc[1][3] = fmaf(cu[3], swu * sx1, acc[1][3]);
            }
            if (++s == S) {
                s = 0;
                ph ^= 1;
            }
        }
        if (!failed) store_rec<2>(acc, r, r.shared ? pts : pt);
    }
    if (tid == 0) trace_stamp(a.trace, 1, 3);
}

// ======================================================================= down
// One round of the down operand build of a row group. Four (task, K part) slots of
// partial sums: slot q holds part q % PP of task t0 + (q / PP) * kCons, where a task is
// the 128 values of one activation row's gate/up block and PP (1, 2 or 4) is the part
// count P rounded up, so a round covers 4 / PP tasks. Every load of the round is issued
// before any arithmetic (one memory round trip); then per task the parts are summed in
// part order (A + B of each), a = SiLU(g) * u is formed and quantised per 128 values
// (MXFP8: per 32) into the shared-memory operand.
template <bool kMX>
__device__ __forceinline__ void operand_round(const Partials& src, int P, int PP, int row_begin, int Nb, int ntask,
                                              int t0, uint8_t* s_hq, int hp, float* s_hs, int Nmax) {
    const int lane = threadIdx.x & 31;
    float4 ga[4], gb[4], ua[4], ub[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int task = t0 + (q / PP) * kCons, p = q % PP;
        if (task < ntask && p < P) {
            const int col = task / Nb, kbq = task % Nb;
            const size_t o = ((size_t)p * src.rows + row_begin + col) * src.N + kbq * kTile + 4 * lane;
            ga[q] = __ldcg(reinterpret_cast<const float4*>(src.A[0] + o));
            gb[q] = __ldcg(reinterpret_cast<const float4*>(src.B[0] + o));
            ua[q] = __ldcg(reinterpret_cast<const float4*>(src.A[1] + o));
            ub[q] = __ldcg(reinterpret_cast<const float4*>(src.B[1] + o));
        }
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int task = t0 + b * kCons;
        if (b * PP >= 4 || task >= ntask) break;  // warp-uniform
        const int col = task / Nb, kbq = task % Nb;
        float4 gv = make_float4(0.f, 0.f, 0.f, 0.f), uv = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 4; ++q)  // this task's slots in part order
            if (q / PP == b && q % PP < P) {
                gv.x += ga[q].x + gb[q].x;
                gv.y += ga[q].y + gb[q].y;
                gv.z += ga[q].z + gb[q].z;
                gv.w += ga[q].w + gb[q].w;
                uv.x += ua[q].x + ub[q].x;
                uv.y += ua[q].y + ub[q].y;
                uv.z += ua[q].z + ub[q].z;
                uv.w += ua[q].w + ub[q].w;
            }
        const float h0 = silu_mul(gv.x, uv.x), h1 = silu_mul(gv.y, uv.y);
        const float h2 = silu_mul(gv.z, uv.z), h3 = silu_mul(gv.w, uv.w);
        if constexpr (kMX) {  // per 32 values: E8M0 bytes [8][Nmax/32] in place of s_hs
            uint32_t s8;
            const uint32_t code = warp_quant_mx32(h0, h1, h2, h3, &s8);
            reinterpret_cast<uint32_t*>(s_hq + col * hp + kbq * kBlk)[lane] = code;
            if ((lane & 7) == 0)
                reinterpret_cast<uint8_t*>(s_hs)[col * (Nmax / 32) + kbq * 4 + (lane >> 3)] = (uint8_t)s8;
        } else {
            float sc;
            const uint32_t code = warp_quant_block128(h0, h1, h2, h3, &sc);
            reinterpret_cast<uint32_t*>(s_hq + col * hp + kbq * kBlk)[lane] = code;
            if (lane == 0) s_hs[col * (Nmax / kBlk) + kbq] = sc;
        }
    }
}

// Positions of token tok's routed rows j0 .. j0 + RB - 1 in the permuted order (-1 beyond
// top_k, or outside [0, T*k)), read through L2.
template <int RB>
__device__ __forceinline__ void combine_pos(const StreamArgs& a, int tok, int j0, int (&r)[RB]) {
    const int Tk = a.T * a.k;
#pragma unroll
    for (int jj = 0; jj < RB; ++jj) {
        r[jj] = j0 + jj < a.k ? __ldcg(a.inv_pos + tok * a.k + j0 + jj) : -1;
        if ((unsigned)r[jj] >= (unsigned)Tk) r[jj] = -1;
    }
}

// Combine of one token's four channels h..h+3: the k routed rows' down outputs in slot
// order (each row's K parts summed in order, A + B), then the shared row, then the
// residual, in fp32. r0: the positions of the first RB slots (combine_pos). RB rows at a
// time: all their loads (with the shared row's, in the first batch), then the sums in
// slot order; the result does not depend on RB.
template <int RB>
__device__ __forceinline__ float4 combine4(const StreamArgs& a, const Partials& pt, const Partials& pts, int P,
                                           int tok, int h, const int (&r0)[RB]) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f), ys = make_float4(0.f, 0.f, 0.f, 0.f);
    const bool shared = a.n_shared_groups > 0;
    for (int j0 = 0; j0 < a.k; j0 += RB) {
        int r[RB];
        if (j0 == 0) {
#pragma unroll
            for (int jj = 0; jj < RB; ++jj) r[jj] = r0[jj];
        } else {
            combine_pos<RB>(a, tok, j0, r);
        }
        float4 y[RB];
#pragma unroll
        for (int jj = 0; jj < RB; ++jj) y[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = 0; p < P; ++p) {
            float4 ya[RB], yb[RB], sa, sb;
#pragma unroll
            for (int jj = 0; jj < RB; ++jj)
                if (r[jj] >= 0) {
                    const size_t o = ((size_t)p * pt.rows + r[jj]) * pt.N + h;
                    ya[jj] = __ldcg(reinterpret_cast<const float4*>(pt.A[0] + o));
                    yb[jj] = __ldcg(reinterpret_cast<const float4*>(pt.B[0] + o));
                }
            if (j0 == 0 && shared) {
                const size_t o = ((size_t)p * pts.rows + tok) * pts.N + h;
                sa = __ldcg(reinterpret_cast<const float4*>(pts.A[0] + o));
                sb = __ldcg(reinterpret_cast<const float4*>(pts.B[0] + o));
            }
#pragma unroll
            for (int jj = 0; jj < RB; ++jj)
                if (r[jj] >= 0) {
                    y[jj].x += ya[jj].x + yb[jj].x;
                    y[jj].y += ya[jj].y + yb[jj].y;
                    y[jj].z += ya[jj].z + yb[jj].z;
                    y[jj].w += ya[jj].w + yb[jj].w;
                }
            if (j0 == 0 && shared) {
                ys.x += sa.x + sb.x;
                ys.y += sa.y + sb.y;
                ys.z += sa.z + sb.z;
                ys.w += sa.w + sb.w;
            }
        }
#pragma unroll
        for (int jj = 0; jj < RB; ++jj)
            if (r[jj] >= 0) {
                v.x += y[jj].x;
                v.y += y[jj].y;
                v.z += y[jj].z;
                v.w += y[jj].w;
            }
    }
    if (shared) {
        v.x += ys.x;
        v.y += ys.y;
        v.z += ys.z;
        v.w += ys.w;
    }
    if (a.residual) {
        const uint2 rr = *reinterpret_cast<const uint2*>(a.residual + (size_t)tok * a.H + h);
        v.x += __uint_as_float(rr.x << 16);
        v.y += __uint_as_float(rr.x & 0xFFFF0000u);
        v.z += __uint_as_float(rr.y << 16);
        v.w += __uint_as_float(rr.y & 0xFFFF0000u);
    }
    return v;
}

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* dst, float4 v) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&lo);
    o.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = o;
}

template <bool kMX, typename Ix, bool kLocal>
__global__ void __launch_bounds__(kThreads, 1)
    down_stream_kernel(const StreamArgs a, const __grid_constant__ TmaMap tm_d, const __grid_constant__ TmaMap tm_sd) {
    extern __shared__ uint8_t smem_raw[];
    const int S = a.stages_d;
    constexpr int SB = kBox;
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * SB);
    uint64_t* empty = full + S;
    const int Nmax = max(a.I, a.Is);
    const int hp = Nmax + 16;  // operand row pitch: the rows of a B fragment in distinct banks
    uint8_t* s_hq = reinterpret_cast<uint8_t*>(empty + S);               // [8][hp] FP8 operand
    float* s_hs = reinterpret_cast<float*>(s_hq + kGroupRows * hp);      // [8][Nmax/128] its scales
    __shared__ float s_w[kGroupRows];
    __shared__ RouteSmem s_route;
    __shared__ TileRec s_tab[kMaxTab];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int H = a.H, Ib = a.I / kBlk, Isb = a.Is / kBlk;
    const int slices = H / kTile;
    if (tid == 0) trace_stamp(a.trace, 2, 0);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCons);
        }
        fence_mbar_init();
    }

    // The routing data come from the router kernels, which completed before the gate/up
    // kernel (this kernel's predecessor) got past its own wait; down weights depend on
    // nothing else, so the tile table is built and the producer streams weights before
    // the gate/up results exist (load_route reads through L2 and ends with
    // __syncthreads). With routing inside the streaming kernels (up to 8 tokens) gate/up
    // CTA 0 published it: it is read after the wait (deriving it again here from the
    // logits took ~4 us per CTA, and these CTAs start only as gate/up CTAs retire).
    if constexpr (kLocal) pdl_wait();
    const RouteView rv = load_route(&s_route, a.ctrl, a.groups, a.max_groups, a.perm_src, a.topk_w, a.T * a.k, a.E,
                                    a.status, tid, kThreads);
    const Plan pl = down_plan<Ix>(a, rv.n_groups);
    const Plan pl_gu = gateup_plan<Ix>(a, rv.n_groups);  // the K parts of the gate/up partials
    const TileSpace<Ix> ts = down_space<Ix>(a, rv.n_groups, pl.P);
    const Range<Ix> rg = make_range(ts, pl.nb, blockIdx.x);
    const bool active = blockIdx.x < pl.nb && rg.u1 > rg.u0;
    const int ntiles = active ? build_table(s_tab, ts, rg, slices, slices, rv, a.T, a.k, tid, kThreads) : 0;
    __syncthreads();
    auto rec = [&](int i) {
        return i < kMaxTab ? s_tab[i] : make_rec_far(ts, rg, rg.first_tile + (Ix)i, slices, slices, rv, a.T, a.k);
    };

    if (warp == kCons) {
        if (lane == 0 && active) {
            prefetch_tmap(&tm_d);
            if (a.Is > 0) prefetch_tmap(&tm_sd);
            const uint64_t wpol = l2_policy_evict_first();  // the routed experts' weights, or all up to 8 tokens
            int s = 0, ph = 0;
            long q = 0;  // units issued
            bool stop = false;
            for (int i = 0; i < ntiles && !stop; ++i) {
                const TileRec r = rec(i);
                const int y = r.shared ? r.slice * kTile : r.expert * H + r.slice * kTile;
                const void* md = r.shared ? (const void*)&tm_sd : (const void*)&tm_d;
                for (int j = 0; j < r.n; ++j, ++q) {
                    if (q >= S && !mbar_wait_bounded(&empty[s], ph ^ 1)) {
                        set_status(a.status, kStatusTimeout);
                        stop = true;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], kBox);
                    if (a.stream_once || !r.shared)
                        tma_load_2d_hint(smem + s * SB, md, (r.kb0 + j) * kBlk, y, &full[s], wpol);
                    else
                        tma_load_2d(smem + s * SB, md, (r.kb0 + j) * kBlk, y, &full[s]);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
        }
        pdl_wait();
        pdl_launch_dependents();
        return;
    }

    pdl_wait();  // the gate/up tiles are complete
    pdl_launch_dependents();
    if (tid == 0) trace_stamp(a.trace, 2, 1);
    if (!active) return;

    const Partials gu_r{{a.g_r, a.u_r}, {a.gb_r, a.ub_r}, (long)a.T * a.k, a.I};
    const Partials gu_s{{a.g_s, a.u_s}, {a.gb_s, a.ub_s}, (long)a.T, a.Is};
    const Partials pt{{a.y_r, nullptr}, {a.yb_r, nullptr}, (long)a.T * a.k, H};
    const Partials pts{{a.y_s, nullptr}, {a.yb_s, nullptr}, (long)a.T, H};
    bool failed = false;

    // FP8 operand of one row group: a = SiLU(g) * u from the gate/up tiles, quantised
    // per 128 values (one gate/up slice = one down K block); as many tasks per warp and
    // round as 16 float4 registers of partial sums hold
    auto build_operand = [&](const TileRec& q) {
        const int N = q.shared ? a.Is : a.I;
        const int Nb = N / kBlk;
        const Partials& src = q.shared ? gu_s : gu_r;
        const int ntask = q.nrows * Nb, P = pl_gu.P;
        const int PP = P <= 1 ? 1 : (P <= 2 ? 2 : 4);
        for (int t0 = warp; t0 < ntask; t0 += kCons * (4 / PP))
            operand_round<kMX>(src, P, PP, q.row_begin, Nb, ntask, t0, s_hq, hp, s_hs, Nmax);
        if (tid < kGroupRows) s_w[tid] = q.w[tid];
        named_bar(1, kConsThreads);
    };

    // routed group index, or -1 - shared group index; INT_MIN: no operand built yet
    int cur_group = INT_MIN;
    int s = 0, ph = 0;
    const int nsb = Nmax / kBlk;
    for (int i = 0; i < ntiles; ++i) {
        const TileRec r = rec(i);
        const int grp = r.shared ? -1 - r.row_begin / kGroupRows : r.group;
        if (grp != cur_group) {
            named_bar(1, kConsThreads);  // every warp is done with the previous operand
            build_operand(r);
            if (tid == 0 && i == 0) trace_stamp(a.trace, 2, 2);
            cur_group = grp;
        }
        const float* swr = nullptr;
        const uint8_t* wd8 = nullptr;  // MXFP8: E8M0 row of this lane's weight row warp*16 + g
        const int Ns = (r.shared ? a.Is : a.I) / 32;
        if constexpr (kMX) {
            wd8 = (r.shared ? a.ss_down8 : a.s_down8 + (size_t)r.expert * H * Ns) +
                  ((size_t)r.slice * kTile + warp * 16 + g) * Ns;
        } else {
            swr = r.shared ? a.ss_down + (size_t)r.slice * Isb : a.s_down + ((size_t)r.expert * slices + r.slice) * Ib;
        }
        const bool v0 = 2 * t4 < r.nrows, v1 = 2 * t4 + 1 < r.nrows;
        float acc[1][4] = {};
        for (int j = 0; j < r.n; ++j) {
            const int kb = r.kb0 + j;
            if constexpr (kMX) {
                const uint32_t w0 = ldg32(wd8 + kb * 4), w1 = ldg32(wd8 + 8 * Ns + kb * 4);
                const uint8_t* hs8 = reinterpret_cast<const uint8_t*>(s_hs);
                const uint32_t x0 = v0 ? *reinterpret_cast<const uint32_t*>(hs8 + (2 * t4) * (Nmax / 32) + kb * 4) : 0u;
                const uint32_t x1 =
                    v1 ? *reinterpret_cast<const uint32_t*>(hs8 + (2 * t4 + 1) * (Nmax / 32) + kb * 4) : 0u;
                if (!failed && !mbar_wait_bounded(&full[s], ph)) {
                    set_status(a.status, kStatusTimeout);
                    failed = true;  // keep walking the units so every named barrier is still reached
                }
                float c[4][4] = {};
                if (!failed) {
                    box_dot_mx(c, smem + s * SB, s_hq + g * hp + kb * kBlk, g < r.nrows, warp, g, t4);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float a0 = v0 ? e8m0_to_float((x0 >> (8 * q)) & 0xFF) : 0.f;
                    const float a1 = v1 ? e8m0_to_float((x1 >> (8 * q)) & 0xFF) : 0.f;
                    const float ws0 = e8m0_to_float((w0 >> (8 * q)) & 0xFF), ws1 = e8m0_to_float((w1 >> (8 * q)) & 0xFF);
                    acc[0][0] = fmaf(c[q][0], ws0 * a0, acc[0][0]);
                    acc[0][1] = fmaf(c[q][1], ws0 * a1, acc[0][1]);
                    acc[0][2] = fmaf(c[q][2], ws1 * a0, acc[0][2]);
                    acc[0][3] = fmaf(c[q][3], ws1 * a1, acc[0][3]);
                }
            } else {
                const float sw = __ldg(swr + kb);
                const float sx0 = s_hs[(2 * t4) * nsb + kb];
                const float sx1 = s_hs[(2 * t4 + 1) * nsb + kb];
                if (!failed && !mbar_wait_bounded(&full[s], ph)) {
                    set_status(a.status, kStatusTimeout);
                    failed = true;  // keep walking the units so every named barrier is still reached
                }
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                if (!failed) {
                    box_dot(c, smem + s * SB, s_hq + g * hp + kb * kBlk, g < r.nrows, warp, g, t4);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                }
                acc[0][0] = fmaf(c[0], v0 ? sw * sx0 : 0.f, acc[0][0]);
                acc[0][1] = fmaf(c[1], v1 ? sw * sx1 : 0.f, acc[0][1]);
                acc[0][2] = fmaf(c[2], v0 ? sw * sx0 : 0.f, acc[0][2]);
                acc[0][3] = fmaf(c[3], v1 ? sw * sx1 : 0.f, acc[0][3]);
            }
            if (++s == S) {
                s = 0;
                ph ^= 1;
            }
        }
        if (!failed) {
            float vals[1][4];
#pragma unroll
            for (int q = 0; q < 4; ++q) vals[0][q] = acc[0][q] * s_w[2 * t4 + (q & 1)];
            store_rec<1>(vals, r, r.shared ? pts : pt);
        }
    }
    if (tid == 0) trace_stamp(a.trace, 2, 3);
}

// ==================================================================== combine
// out[t] = sum_j y(row inv_pos[t*k+j]) + y_shared(t) (+ residual[t]), fp32, one bf16
// rounding; or, for the stage API, the bf16 expert rows y_perm / y_shared themselves.
// Each thread owns 4 consecutive hidden channels of one token (or one row).
__global__ void __launch_bounds__(256) stream_combine_kernel(const StreamArgs a) {
    if (threadIdx.x == 0) trace_stamp(a.trace, 3, 0);
    // Before the dependency wait, what was written two or more kernels back, through L2:
    // the row-group count (for the down stage's K-part count) and this thread's first
    // token's row positions.
    const int down_P = down_plan<long long>(a, __ldcg(&a.ctrl->n_routed_groups)).P;
    const int H = a.H;
    const int H4 = H / 4;
    const int Tk = a.T * a.k;
    const long i0 = (long)blockIdx.x * blockDim.x + threadIdx.x, stride = (long)gridDim.x * blockDim.x;
    int r0[8];
    if (a.fuse_combine && i0 < (long)a.T * H4) combine_pos<8>(a, (int)(i0 / H4), 0, r0);
    pdl_wait();  // the down tiles are complete
    pdl_launch_dependents();
    if (threadIdx.x == 0) trace_stamp(a.trace, 3, 1);
    const Partials pt{{a.y_r, nullptr}, {a.yb_r, nullptr}, (long)Tk, H};
    const Partials pts{{a.y_s, nullptr}, {a.yb_s, nullptr}, (long)a.T, H};
    if (a.fuse_combine) {
        const long n = (long)a.T * H4;
        for (long i = i0; i < n; i += stride) {
            const int tok = (int)(i / H4), h = (int)(i % H4) * 4;
            if (i != i0) combine_pos<8>(a, tok, 0, r0);
            store_bf16x4(a.out + (size_t)tok * H + h, combine4<8>(a, pt, pts, down_P, tok, h, r0));
        }
        if (threadIdx.x == 0) trace_stamp(a.trace, 3, 3);
    } else {
        const long nr = (long)Tk * H4, ns = a.n_shared_groups > 0 ? (long)a.T * H4 : 0;
        for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < nr + ns; i += (long)gridDim.x * blockDim.x) {
            if (i < nr) {
                const int r = (int)(i / H4), h = (int)(i % H4) * 4;
                store_bf16x4(a.y_perm + (size_t)r * H + h, read4(pt, down_P, 0, r, h));
            } else {
                const long j = i - nr;
                const int tok = (int)(j / H4), h = (int)(j % H4) * 4;
                store_bf16x4(a.y_shared + (size_t)tok * H + h, read4(pts, down_P, 0, tok, h));
            }
        }
    }
}

size_t smem_gateup() { return (size_t)kStagesGU * (2 * kBox + kBRows) + 2 * kStagesGU * 8 + 1024; }
// Static shared memory of the down kernel beside its dynamic ring and operand: the tile
// table, the routing copies and small scalars.
constexpr long kDownStaticSmem = (long)kTabBytes + (long)sizeof(RouteSmem) + 256;
// Down-kernel ring depth: as many 16 KB stages (up to 10) as fit beside the FP8 operand.
int stages_down(int Nmax) {
    const long operand = (long)kGroupRows * (Nmax + 16) + (long)kGroupRows * (Nmax / kBlk) * 4;
    const long room = 227L * 1024 - 1024 - operand - kDownStaticSmem - 64;
    return (int)std::max<long>(2, std::min<long>(kMaxStagesD, room / (kBox + 16)));
}
size_t smem_down(int Nmax) {
    const int S = stages_down(Nmax);
    return (size_t)S * kBox + 2 * S * 8 + (size_t)kGroupRows * (Nmax + 16) + (size_t)kGroupRows * (Nmax / kBlk) * 4 +
           1024;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t set_smem(const void* fn, size_t bytes, size_t* done) {
    if (*done >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) *done = bytes;
    return e;
}

}  // namespace

int stream_grid() { return std::min(num_sms(), kMaxStreamCtas); }

int down_stages(int I, int Is) { return stages_down(std::max(I, Is)); }

int stream_max_parts(const moe_config_t& c, int64_t T) {
    // fewest units either streaming stage can have for T tokens, spread over the most
    // CTAs the kernels may use: the longest part must still fit in a range
    const int64_t Hb = c.hidden / kBlk, Ib = c.moe_inter / kBlk, Isb = (int64_t)c.n_shared * Ib;
    const int64_t groups = (T * c.top_k + kGroupRows - 1) / kGroupRows;
    const int64_t sgroups = c.n_shared > 0 ? (T + kGroupRows - 1) / kGroupRows : 0;
    const int64_t U = groups * Ib * Hb + sgroups * Isb * Hb;  // same count for gate/up and down
    const int64_t L = std::max<int64_t>(1, U / kMaxStreamCtas);
    const int64_t kcmax = std::max<int64_t>(Hb, std::max(Ib, Isb));
    return (int)std::max<int64_t>(1, std::min<int64_t>(kMaxParts, (kcmax + L - 1) / L));
}

cudaError_t launch_gateup_stream(const StreamArgs& a, const uint8_t* w_gate, const uint8_t* w_up, int E,
                                 cudaStream_t st) {
    static size_t smem_set[6] = {0, 0, 0, 0, 0, 0};
    using K = void (*)(const StreamArgs, const TmaMap, const TmaMap, const TmaMap, const TmaMap);
    const K kerns[6] = {gateup_stream_kernel<false, int, false>,       gateup_stream_kernel<true, int, false>,
                        gateup_stream_kernel<false, long long, false>, gateup_stream_kernel<true, long long, false>,
                        gateup_stream_kernel<false, int, true>,        gateup_stream_kernel<true, int, true>};
    const int v = a.local_route ? 4 + (a.mx ? 1 : 0) : (a.mx ? 1 : 0) + (a.wide ? 2 : 0);
    cudaError_t e = set_smem((const void*)kerns[v], smem_gateup(), &smem_set[v]);
    if (e != cudaSuccess) return e;
    TmaMap tg{}, tu{}, tsg{}, tsu{};
    if (!tmap_u8_2d(&tg, w_gate, (uint64_t)E * a.I, a.H, kBlk, kTile) ||
        !tmap_u8_2d(&tu, w_up, (uint64_t)E * a.I, a.H, kBlk, kTile))
        return cudaErrorInvalidValue;
    if (a.Is > 0 && (!tmap_u8_2d(&tsg, a.ws_gate, a.Is, a.H, kBlk, kTile) ||
                     !tmap_u8_2d(&tsu, a.ws_up, a.Is, a.H, kBlk, kTile)))
        return cudaErrorInvalidValue;
    return launch_pdl(kerns[v], a.grid_gu, kThreads, smem_gateup(), st, a, tg, tu, tsg, tsu);
}

cudaError_t launch_down_stream(const StreamArgs& a, const uint8_t* w_down, const uint8_t* ws_down, int E,
                               cudaStream_t st) {
    static size_t smem_set[6] = {0, 0, 0, 0, 0, 0};
    const size_t smem = smem_down(std::max(a.I, a.Is));
    using K = void (*)(const StreamArgs, const TmaMap, const TmaMap);
    const K kerns[6] = {down_stream_kernel<false, int, false>,       down_stream_kernel<true, int, false>,
                        down_stream_kernel<false, long long, false>, down_stream_kernel<true, long long, false>,
                        down_stream_kernel<false, int, true>,        down_stream_kernel<true, int, true>};
    const int v = a.local_route ? 4 + (a.mx ? 1 : 0) : (a.mx ? 1 : 0) + (a.wide ? 2 : 0);
    cudaError_t e = set_smem((const void*)kerns[v], smem, &smem_set[v]);
    if (e != cudaSuccess) return e;
    TmaMap td{}, tsd{};
    if (!tmap_u8_2d(&td, w_down, (uint64_t)E * a.H, a.I, kBlk, kTile)) return cudaErrorInvalidValue;
    if (a.Is > 0 && !tmap_u8_2d(&tsd, ws_down, a.H, a.Is, kBlk, kTile)) return cudaErrorInvalidValue;
    return launch_pdl(kerns[v], a.grid_d, kThreads, smem, st, a, td, tsd);
}

cudaError_t launch_stream_combine(const StreamArgs& a, cudaStream_t st) {
    const long n = a.fuse_combine ? (long)a.T * (a.H / 4)
                                  : (long)a.T * a.k * (a.H / 4) + (a.n_shared_groups > 0 ? (long)a.T * (a.H / 4) : 0);
    if (n == 0) return cudaSuccess;
    const int grid = (int)std::min<long>((n + 255) / 256, (long)num_sms() * 8);
    return launch_pdl(stream_combine_kernel, grid, 256, 0, st, a);
}

}  // namespace moe
