// Device building blocks of expert selection shared by the router kernels (route.cu):
// group-limited top-k of one token by one warp, and the in-CTA counting-sort
// permutation.
#pragma once

#include <climits>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {
namespace routing {

constexpr int kMaxE = 256;

// Total order of floats as unsigned keys (larger float -> larger key).
__device__ __forceinline__ unsigned float_key(float f) {
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Softmax over E logits and group-limited greedy top-k for one token, computed by
// one warp. lg[i] is the logit of expert lane + 32*i (-inf beyond E). scratch is
// unused (kept for the callers' shared-memory layout).
//
// The softmax is monotonic, so groups and experts are ranked on the logits themselves
// and probabilities are formed only for the chosen experts: p = exp(l - max) / sum.
// A group's score is its best member; a group is kept when fewer than topk_group
// groups beat it (higher score, or equal score and lower index). The experts are then
// taken in top_k rounds of a warp-wide arg-max over the members of kept groups (ties
// to the lower index), so slot j holds the j-th best: the greedy order.
//
// topk_warp_n runs NT tokens through the same steps side by side in one warp (token q's
// logits in lg[q]; its outputs through ids_out[q], w_out[q], ids_smem[q], each skipped when
// null): every token's arithmetic is exactly topk_warp's, and the NT independent chains of
// warp-wide reductions overlap their latencies.
template <int NT>
__device__ inline void topk_warp_n(const float (&lg)[NT][kMaxE / 32], int E, int G, int Gk, int k, float scale,
                                   int32_t* const (&ids_out)[NT], float* const (&w_out)[NT],
                                   int32_t* const (&ids_smem)[NT]) {
    const int lane = threadIdx.x & 31;
    const int per = E / G;
    float mx[NT];
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        mx[q] = -INFINITY;
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i) mx[q] = fmaxf(mx[q], lg[q][i]);
    }
#pragma unroll
    for (int q = 0; q < NT; ++q) mx[q] = warp_max(mx[q]);
    // group scores: lane g keeps the best key of group g
    int gid[kMaxE / 32];
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        gid[i] = e < E ? e / per : -1;
    }
    unsigned gkey[NT];
#pragma unroll
    for (int q = 0; q < NT; ++q) gkey[q] = 0u;
    for (int gi = 0; gi < G; ++gi) {
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            unsigned m = 0u;
#pragma unroll
            for (int i = 0; i < kMaxE / 32; ++i)
                if (gid[i] == gi) m = max(m, float_key(lg[q][i]));
            m = __reduce_max_sync(0xffffffffu, m);
            if (lane == gi) gkey[q] = m;
        }
    }
    int beaten[NT];
#pragma unroll
    for (int q = 0; q < NT; ++q) beaten[q] = 0;
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            const unsigned o = __shfl_sync(0xffffffffu, gkey[q], h);
            beaten[q] += (o > gkey[q]) || (o == gkey[q] && h < lane);
        }
    }
    // candidates: experts of kept groups, as keys (0: none; a real key is never 0)
    unsigned ck[NT][kMaxE / 32];
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        const unsigned kept = __ballot_sync(0xffffffffu, lane < G && beaten[q] < Gk);
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i)
            ck[q][i] = (gid[i] >= 0 && ((kept >> gid[i]) & 1u)) ? float_key(lg[q][i]) : 0u;
    }
    float lsel[NT];  // lane j < k: logit of the j-th choice
#pragma unroll
    for (int q = 0; q < NT; ++q) lsel[q] = 0.f;
    for (int j = 0; j < k; ++j) {
        unsigned top[NT], be[NT];
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            unsigned bk = 0u;
#pragma unroll
            for (int i = 0; i < kMaxE / 32; ++i) bk = max(bk, ck[q][i]);
            top[q] = __reduce_max_sync(0xffffffffu, bk);
        }
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            be[q] = 0xffffffffu;  // this lane's lowest expert holding the top key
#pragma unroll
            for (int i = kMaxE / 32 - 1; i >= 0; --i)
                if (ck[q][i] == top[q]) be[q] = (unsigned)(lane + 32 * i);
            be[q] = __reduce_min_sync(0xffffffffu, be[q]);
        }
#pragma unroll
        for (int q = 0; q < NT; ++q) {
#pragma unroll
            for (int i = 0; i < kMaxE / 32; ++i)
                if ((unsigned)(lane + 32 * i) == be[q]) ck[q][i] = 0u;  // the owner removes the winner
            const int owner = (int)(be[q] & 31u), slot = (int)(be[q] >> 5);
            float lw = 0.f;
#pragma unroll
            for (int i = 0; i < kMaxE / 32; ++i)
                if (i == slot) lw = lg[q][i];
            lw = __shfl_sync(0xffffffffu, lw, owner);
            if (lane == j) lsel[q] = lw;
            if (lane == 0) {
                if (ids_out[q]) ids_out[q][j] = (int)be[q];
                if (ids_smem[q]) ids_smem[q][j] = (int)be[q];
            }
        }
    }
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i) z += (lane + 32 * i < E) ? expf(lg[q][i] - mx[q]) : 0.f;
        z = warp_sum(z);
        if (lane < k && w_out[q]) w_out[q][lane] = expf(lsel[q] - mx[q]) / z * scale;
    }
    __syncwarp();
}

__device__ inline void topk_warp(const float (&lg)[kMaxE / 32], int E, int G, int Gk, int k, float scale,
                                 float* scratch, int32_t* ids_out, float* w_out, int32_t* ids_smem) {
    (void)scratch;
    const float(&l1)[1][kMaxE / 32] = *reinterpret_cast<const float(*)[1][kMaxE / 32]>(&lg);
    int32_t* const io[1] = {ids_out};
    float* const wo[1] = {w_out};
    int32_t* const so[1] = {ids_smem};
    topk_warp_n<1>(l1, E, G, Gk, k, scale, io, wo, so);
}

// Inverse of float_key.
__device__ __forceinline__ float key_float(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The same selection and weights as topk_warp for a single token, computed by a whole
// CTA of at least E threads (thread e holds expert e): group scores by shared-memory
// atomicMax, the kept groups by counting the groups that beat each one, and every
// candidate's rank by one pass over the candidates' keys (ties to the lower index), so
// slot j holds the j-th best; no rounds of warp-wide arg-max. The softmax sum runs per
// warp, then over the warps (another order than topk_warp's, so w may differ in the
// last bit). Scratch: key[kMaxE] (16-byte aligned), gkey[32], part[32].
__device__ inline void cta_topk1(const float* lg, int E, int G, int Gk, int k, float scale, unsigned* key_s,
                                 unsigned* gkey, float* part, int32_t* ids_out, float* w_out, int32_t* ids_smem) {
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5, nw = blockDim.x >> 5;
    const int per = E / G;
    const float l = e < E ? __ldcg(lg + e) : -INFINITY;
    const unsigned key = e < E ? float_key(l) : 0u;
    if (e < 32) gkey[e] = 0u;
    __syncthreads();
    if (e < E) atomicMax(&gkey[e / per], key);
    __syncthreads();
    unsigned mkey = 0u;  // the best logit's key
    for (int h = 0; h < G; ++h) mkey = max(mkey, gkey[h]);
    bool cand = false;
    if (e < E) {
        const int g = e / per;
        const unsigned gk = gkey[g];
        int beaten = 0;
        for (int h = 0; h < G; ++h) {
            const unsigned o = gkey[h];
            beaten += (o > gk) || (o == gk && h < g);
        }
        cand = beaten < Gk;
    }
    if (e < kMaxE) key_s[e] = cand ? key : 0u;  // a real key is never 0
    const float mx = key_float(mkey);
    float z = e < E ? expf(l - mx) : 0.f;
    z = warp_sum(z);
    if (lane == 0) part[warp] = z;
    __syncthreads();
    if (cand) {
        int rank = 0;
        const uint4* kv = reinterpret_cast<const uint4*>(key_s);
        for (int j4 = 0; j4 < (E + 3) / 4; ++j4) {
            const uint4 o = kv[j4];
            const int j = 4 * j4;
            rank += (o.x > key) || (o.x == key && j < e);
            rank += (o.y > key) || (o.y == key && j + 1 < e);
            rank += (o.z > key) || (o.z == key && j + 2 < e);
            rank += (o.w > key) || (o.w == key && j + 3 < e);
        }
        if (rank < k) {
            float Z = 0.f;
            for (int w = 0; w < nw; ++w) Z += part[w];
            ids_out[rank] = e;
            if (ids_smem) ids_smem[rank] = e;
            w_out[rank] = expf(l - mx) / Z * scale;
        }
    }
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

// Stable counting sort of n = T*k (<= 1024) ids held in shared memory by one CTA,
// plus row groups of at most kGroupRows rows per expert. The rank of each id among the
// earlier equal ids comes from one warp walking 32-id chunks in order (__match_any_sync
// inside a chunk, a running count per expert across chunks); the scatter is parallel.
// s_rank holds n ints of scratch.
__device__ inline void small_permute(const int32_t* s_ids, int n, int E, int* s_cnt, int* s_off, int* s_gcnt,
                                     int* s_goff, int* s_rank, int32_t* offsets, int32_t* perm_src, int32_t* inv_pos,
                                     RowGroup* groups, int32_t* group_of_row, int* n_groups) {
    const int lane = threadIdx.x & 31;
    if (n <= 32) {
        // One warp, no CTA barrier: a slot's row is the number of slots with a smaller id
        // plus its rank among the equal ids before it (the order of the general path
        // below), and a row group starts at every kGroupRows-th row of an expert, so its
        // index counts the group starts of smaller ids. The offsets come from counts.
        if (threadIdx.x < 32) {
            const int e = lane < n ? s_ids[lane] : INT_MAX;
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            const int rin = __popc(peers & ((1u << lane) - 1u));
            const int start = lane < n && e >= 0 && rin % kGroupRows == 0;
            int below = 0, gbelow = 0;
            for (int j = 0; j < n; ++j) {
                const int ej = __shfl_sync(0xffffffffu, e, j);
                const int sj = __shfl_sync(0xffffffffu, start, j);
                below += ej >= 0 && ej < e;
                gbelow += (ej >= 0 && ej < e) & sj;
            }
            const int pos = below + rin, gi = gbelow + rin / kGroupRows;
            if (lane < n && e >= 0) {
                perm_src[pos] = lane;
                inv_pos[lane] = pos;
                group_of_row[pos] = gi;
            }
            if (start) {
                RowGroup rg;
                rg.expert = e;
                rg.row_begin = pos;
                rg.nrows = min(kGroupRows, __popc(peers) - rin);
                rg.pad = 0;
                groups[gi] = rg;
            }
            const int ng = __popc(__ballot_sync(0xffffffffu, start));
            if (lane == 0) *n_groups = ng;
        }
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            int c = 0;
            for (int f = 0; f < n; ++f) c += s_ids[f] >= 0 && s_ids[f] < e;
            offsets[e] = c;
        }
        return;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    if (threadIdx.x < 32) {
        const unsigned lt = (1u << lane) - 1u;
        for (int c0 = 0; c0 < n; c0 += 32) {
            const int f = c0 + lane;
            const int e = f < n ? s_ids[f] : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            if (e >= 0) s_rank[f] = s_cnt[e] + __popc(peers & lt);
            __syncwarp();
            if (e >= 0 && (peers & lt) == 0u) s_cnt[e] += __popc(peers);  // one leader per expert
            __syncwarp();
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int c = s_cnt[e];
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
            *n_groups = gtot;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = s_off[e];
    for (int f = threadIdx.x; f < n; f += blockDim.x) {
        const int e = s_ids[f];
        if (e < 0) continue;
        const int r = s_rank[f];
        const int pos = s_off[e] + r;
        perm_src[pos] = f;
        inv_pos[f] = pos;
        group_of_row[pos] = s_goff[e] + r / kGroupRows;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int c = s_cnt[e];
        for (int g = 0; g < s_gcnt[e]; ++g) {
            RowGroup rg;
            rg.expert = e;
            rg.row_begin = s_off[e] + g * kGroupRows;
            rg.nrows = min(kGroupRows, c - g * kGroupRows);
            rg.pad = 0;
            groups[s_goff[e] + g] = rg;
        }
    }
}

}  // namespace routing
}  // namespace moe
