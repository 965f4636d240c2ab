// Device building blocks of expert selection shared by the router kernels
// (route.cu) and the fused small-T layer kernel (moe_fused.cu): group-limited
// top-k of one token by one warp, and the in-CTA counting-sort permutation.
#pragma once

#include <climits>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {
namespace routing {

constexpr int kMaxE = 256;

// Softmax over E logits and group-limited greedy top-k for one token, computed by
// one warp. lg[i] is the logit of expert lane + 32*i (-inf beyond E). scratch holds
// kMaxE words of shared memory private to this warp.
//
// A group is kept when fewer than topk_group groups beat it (higher score, or equal
// score and lower index). The experts are then taken in top_k rounds of a warp-wide
// arg-max over the candidates of kept groups (highest probability, ties to the lower
// index), so slot j holds the j-th best: the greedy order, with no serial scan.
__device__ inline void topk_warp(const float (&lg)[kMaxE / 32], int E, int G, int Gk, int k, float scale,
                                 float* scratch, int32_t* ids_out, float* w_out, int32_t* ids_smem) {
    const int lane = threadIdx.x & 31;
    float* sp = scratch;  // [E] probabilities
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) mx = fmaxf(mx, lg[i]);
    mx = warp_max(mx);
    float p[kMaxE / 32];
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        p[i] = (e < E) ? expf(lg[i] - mx) : 0.f;
        z += p[i];
    }
    z = warp_sum(z);
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        p[i] = p[i] / z;
        const int e = lane + 32 * i;
        if (e < E) sp[e] = p[i];
    }
    __syncwarp();
    // group score = max member score; groups are contiguous blocks of E/G experts
    const int per = E / G;
    float gs = -INFINITY;
    if (lane < G) {
        gs = sp[lane * per];
        for (int i = 1; i < per; ++i) gs = fmaxf(gs, sp[lane * per + i]);
    }
    int beaten = 0;
    for (int h = 0; h < G; ++h) {
        const float o = __shfl_sync(0xffffffffu, gs, h);
        beaten += (o > gs) || (o == gs && h < lane);
    }
    const unsigned kept = __ballot_sync(0xffffffffu, lane < G && beaten < Gk);
    // candidates: experts of kept groups (probabilities are >= 0; -1 marks "none")
    float cv[kMaxE / 32];
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        cv[i] = (e < E && ((kept >> (e / per)) & 1u)) ? p[i] : -1.f;
    }
    for (int j = 0; j < k; ++j) {
        // this lane's best (lowest index on ties: e grows with i), then the warp's
        float bv = -2.f;
        int be = INT_MAX;
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i)
            if (cv[i] > bv) {
                bv = cv[i];
                be = lane + 32 * i;
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) {  // the owner removes the winner from its candidates
#pragma unroll
            for (int i = 0; i < kMaxE / 32; ++i)
                if (lane + 32 * i == be) cv[i] = -1.f;
        }
        if (lane == 0) {
            ids_out[j] = be;
            w_out[j] = bv * scale;
            if (ids_smem) ids_smem[j] = be;
        }
    }
    __syncwarp();
}

// Exclusive scan of n (<= 256) ints in shared memory by one warp; returns the total.
__device__ inline int warp_exclusive_scan256(int* v, int n) {
    const int lane = threadIdx.x & 31;
    int loc[8];
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = lane * 8 + i;
        loc[i] = idx < n ? v[idx] : 0;
        s += loc[i];
    }
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int run = incl - s;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = lane * 8 + i;
        if (idx < n) v[idx] = run;
        run += loc[i];
    }
    __syncwarp();
    return total;
}

// Stable counting sort of n = T*k ids held in shared memory (n small) by one CTA,
// plus row groups of at most kGroupRows rows per expert.
__device__ inline void small_permute(const int32_t* s_ids, int n, int E, int* s_cnt, int* s_off, int* s_gcnt,
                              int* s_goff, int32_t* offsets, int32_t* perm_src, int32_t* inv_pos,
                              RowGroup* groups, int32_t* group_of_row, Ctrl* ctrl) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
        for (int f = 0; f < n; ++f) c += (s_ids[f] == e);
        s_cnt[e] = c;
        s_off[e] = c;
        s_gcnt[e] = (c + kGroupRows - 1) / kGroupRows;
        s_goff[e] = s_gcnt[e];
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int tot = warp_exclusive_scan256(s_off, E);
        const int gtot = warp_exclusive_scan256(s_goff, E);
        if (threadIdx.x == 0) {
            s_off[E] = tot;
            ctrl->n_routed_groups = gtot;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = s_off[e];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int pos = s_off[e];
        for (int f = 0; f < n; ++f) {
            if (s_ids[f] == e) {
                perm_src[pos] = f;
                inv_pos[f] = pos;
                ++pos;
            }
        }
        const int c = s_cnt[e];
        for (int g = 0; g < s_gcnt[e]; ++g) {
            RowGroup rg;
            rg.expert = e;
            rg.row_begin = s_off[e] + g * kGroupRows;
            rg.nrows = min(kGroupRows, c - g * kGroupRows);
            rg.pad = 0;
            groups[s_goff[e] + g] = rg;
            for (int r = 0; r < rg.nrows; ++r) group_of_row[rg.row_begin + r] = s_goff[e] + g;
        }
    }
}

}  // namespace routing
}  // namespace moe
