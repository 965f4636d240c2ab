// Device building blocks of expert selection shared by the router kernels
// (route.cu) and the fused small-T layer kernel (moe_fused.cu): group-limited
// top-k of one token by one warp, and the in-CTA counting-sort permutation.
#pragma once

#include "common.cuh"
#include "moe_internal.h"

namespace moe {
namespace routing {

constexpr int kMaxE = 256;

// Softmax over E logits and group-limited greedy top-k for one token, computed by
// one warp. lg[i] is the logit of expert lane + 32*i (-inf beyond E). scratch holds
// 2*kMaxE + 32 words of shared memory private to this warp.
//
// Selection by ranks instead of repeated arg-max rounds: a group is kept when fewer
// than topk_group groups beat it (higher score, or equal score and lower index); the
// candidates of kept groups are compacted with a ballot, and a candidate is selected
// when fewer than top_k candidates beat it, its rank being its output slot. Same
// result as the greedy rounds (ties to the lower index), with no serial dependency.
__device__ inline void topk_warp(const float (&lg)[kMaxE / 32], int E, int G, int Gk, int k, float scale,
                          float* scratch, int32_t* ids_out, float* w_out, int32_t* ids_smem) {
    const int lane = threadIdx.x & 31;
    float* sp = scratch;                                          // [E] probabilities
    int* cand = reinterpret_cast<int*>(scratch + kMaxE);          // [<= E] candidate ids
    float* gsc = scratch + 2 * kMaxE;                             // [G] group scores
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
    if (lane < G) {
        float m = sp[lane * per];
        for (int i = 1; i < per; ++i) m = fmaxf(m, sp[lane * per + i]);
        gsc[lane] = m;
    }
    __syncwarp();
    bool keep_g = false;
    if (lane < G) {
        const float mine = gsc[lane];
        int beaten = 0;
        for (int h = 0; h < G; ++h) {
            const float o = gsc[h];
            beaten += (o > mine) || (o == mine && h < lane);
        }
        keep_g = beaten < Gk;
    }
    const unsigned kept = __ballot_sync(0xffffffffu, keep_g);
    // compact the candidates (experts of kept groups), in expert order
    int n = 0;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        const bool c = e < E && ((kept >> (e / per)) & 1u);
        const unsigned m = __ballot_sync(0xffffffffu, c);
        if (c) cand[n + __popc(m & ((1u << lane) - 1u))] = e;
        n += __popc(m);
    }
    __syncwarp();
    for (int j = lane; j < n; j += 32) {
        const int e = cand[j];
        const float pe = sp[e];
        int beaten = 0;
        for (int q = 0; q < n; ++q) {
            const int o = cand[q];
            const float po = sp[o];
            beaten += (po > pe) || (po == pe && o < e);
        }
        if (beaten < k) {
            ids_out[beaten] = e;
            w_out[beaten] = pe * scale;
            if (ids_smem) ids_smem[beaten] = e;
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
