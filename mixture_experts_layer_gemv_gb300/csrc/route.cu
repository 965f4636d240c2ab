// Stage N (router) and stage O (softmax + group-limited greedy top-k) of the
// DeepSeek-V2 MoE layer ("DSV2-236B-MegaKernel", README stage flowchart, MoE
// subgraph), plus the FP8 activation quantisation the expert GEMMs consume.
//
// Two routes:
//  * small T (<= kSmallT): one launch. CTA e computes logits[:, e] (a GEMV over the
//    fp32 router row, K split across warps), every CTA quantises a share of x, and
//    the last CTA to arrive (an atomic arrival counter, no waiting) runs the
//    per-token softmax/top-k and, for the fused forward, the expert permutation and
//    the row-group work list. The README's stage O does the selection with
//    "ballot + popc + ctz"; here groups and experts are ranked (count of better
//    candidates, ties to the lower index) with a ballot-compacted candidate list.
//  * large T: a tiled fp32 SIMT GEMM for the logits (split-K partials, summed in a
//    fixed order), then one warp per token for softmax/top-k.
#include <algorithm>

#include "route_common.cuh"

namespace moe {

namespace {

constexpr int kRouteWarps = 8;

using namespace routing;

struct RouteSmallParams {
    int H, E, G, Gk, k, T;
    float scale;
    const uint16_t* x;
    const float* wr;
    const float* bias;
    float* logits;
    int32_t* ids;
    float* w;
    uint8_t* xq;
    float* xs;
    int32_t* offsets;
    int32_t* perm_src;
    int32_t* inv_pos;
    RowGroup* groups;
    int32_t* group_of_row;
    Ctrl* ctrl;
};

__global__ void __launch_bounds__(kRouteWarps * 32) route_small_kernel(RouteSmallParams p) {
    __shared__ float s_part[kRouteWarps][kSmallT];
    __shared__ float s_gs[kRouteWarps][kMaxE];
    __shared__ int32_t s_ids[kSmallT * 16];
    __shared__ int s_rank[kSmallT * 16];
    __shared__ int s_cnt[kMaxE], s_off[kMaxE + 1], s_gcnt[kMaxE], s_goff[kMaxE];
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x;
    const int H = p.H, T = p.T, Hb = H / kBlk;
    pdl_wait();  // x and the workspace are free (the previous kernel in the stream is done)
    pdl_launch_dependents();

    // ---- N: logits[:, e], K split over the CTA's warps (H/8 is a multiple of 16).
    // A warp's router slice sits in registers (up to 8 float4 per lane per chunk) and
    // four tokens' activations are loaded before any FMA, so a warp waits for one
    // memory round trip per chunk and four tokens, not one per load.
    const int slice = H / kRouteWarps;
    const int n4 = slice / 4;  // float4 per warp slice
    const float4* wrow = reinterpret_cast<const float4*>(p.wr + (size_t)e * H + warp * slice);
    for (int t = lane; t < T; t += 32) s_part[warp][t] = 0.f;
    __syncwarp();
    for (int c0 = 0; c0 < n4; c0 += 32 * 8) {
        float4 wv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = c0 + lane + 32 * j;
            wv[j] = i < n4 ? __ldg(wrow + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int t = 0; t < T; t += 4) {
            uint2 xv[4][8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint2* xr =
                    reinterpret_cast<const uint2*>(p.x + (size_t)min(t + q, T - 1) * H + warp * slice);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int i = c0 + lane + 32 * j;
                    xv[q][j] = i < n4 ? __ldg(xr + i) : make_uint2(0, 0);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    acc = fmaf(bf16_bits_to_float((uint16_t)(xv[q][j].x & 0xFFFF)), wv[j].x, acc);
                    acc = fmaf(bf16_bits_to_float((uint16_t)(xv[q][j].x >> 16)), wv[j].y, acc);
                    acc = fmaf(bf16_bits_to_float((uint16_t)(xv[q][j].y & 0xFFFF)), wv[j].z, acc);
                    acc = fmaf(bf16_bits_to_float((uint16_t)(xv[q][j].y >> 16)), wv[j].w, acc);
                }
                acc = warp_sum(acc);
                if (lane == 0 && t + q < T) s_part[warp][t + q] += acc;
            }
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < kRouteWarps; ++w) l += s_part[w][t];
        if (p.bias) l += p.bias[e];
        p.logits[(size_t)t * p.E + e] = l;
    }

    // ---- activation quantisation: this CTA's share of the T*H/128 blocks
    for (int b = blockIdx.x * kRouteWarps + warp; b < T * Hb; b += gridDim.x * kRouteWarps) {
        const int t = b / Hb, kb = b % Hb;
        const uint2 xv = __ldg(reinterpret_cast<const uint2*>(p.x + (size_t)t * H + kb * kBlk) + lane);
        float s;
        const uint32_t q = warp_quant_block128(
            bf16_bits_to_float((uint16_t)(xv.x & 0xFFFF)), bf16_bits_to_float((uint16_t)(xv.x >> 16)),
            bf16_bits_to_float((uint16_t)(xv.y & 0xFFFF)), bf16_bits_to_float((uint16_t)(xv.y >> 16)), &s);
        reinterpret_cast<uint32_t*>(p.xq + (size_t)t * H + kb * kBlk)[lane] = q;
        if (lane == 0) p.xs[(size_t)t * Hb + kb] = s;
    }

    // ---- last CTA to arrive: O (softmax + top-k) and the permutation
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&p.ctrl->route_arrived, 1u);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    for (int t = warp; t < T; t += kRouteWarps) {
        float lg[kMaxE / 32];
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i) {
            const int ee = lane + 32 * i;
            lg[i] = ee < p.E ? __ldcg(p.logits + (size_t)t * p.E + ee) : -INFINITY;
        }
        topk_warp(lg, p.E, p.G, p.Gk, p.k, p.scale, s_gs[warp], p.ids + (size_t)t * p.k, p.w + (size_t)t * p.k,
                  s_ids + t * p.k);
    }
    __syncthreads();
    if (p.offsets)
        small_permute(s_ids, T * p.k, p.E, s_cnt, s_off, s_gcnt, s_goff, s_rank, p.offsets, p.perm_src, p.inv_pos,
                      p.groups, p.group_of_row, p.ctrl);
    if (threadIdx.x == 0) p.ctrl->route_arrived = 0u;
}

// ---------------------------------------------------------------- large T
constexpr int kBM = 64, kBN = 64, kBK = 32;

struct RouterGemmParams {
    int H, E, T, kchunk;
    const uint16_t* x;
    const float* wr;
    float* part;  // [splits, T, E]
};

// part[s][t][e] = sum over this split's K range of x[t][h] * wr[e][h]; 256 threads,
// each owns a 4x4 register tile (rows ty+16i, cols tx+16j).
__global__ void __launch_bounds__(256) router_gemm_kernel(RouterGemmParams p) {
    __shared__ float As[kBK][kBM + 4];
    __shared__ float Bs[kBK][kBN + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN;
    const int k_begin = blockIdx.z * p.kchunk;
    const int k_end = min(p.H, k_begin + p.kchunk);
    float acc[4][4] = {};
    for (int k0 = k_begin; k0 < k_end; k0 += kBK) {
        {   // A: 64 rows x 32 bf16, 8 per thread
            const int r = tid >> 2, c = (tid & 3) * 8;
            const int t = m0 + r;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (t < p.T) v = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t * p.H + k0 + c));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                As[c + 2 * i][r] = bf16_bits_to_float((uint16_t)(w4[i] & 0xFFFF));
                As[c + 2 * i + 1][r] = bf16_bits_to_float((uint16_t)(w4[i] >> 16));
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // B: 64 rows x 32 fp32, 2 float4 per thread
            const int idx = tid + h * 256;
            const int r = idx >> 3, c = (idx & 7) * 4;
            const int e = n0 + r;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < p.E) v = __ldg(reinterpret_cast<const float4*>(p.wr + (size_t)e * p.H + k0 + c));
            Bs[c + 0][r] = v.x;
            Bs[c + 1][r] = v.y;
            Bs[c + 2][r] = v.z;
            Bs[c + 3][r] = v.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kBK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    float* out = p.part + (size_t)blockIdx.z * p.T * p.E;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = m0 + ty + 16 * i;
        if (t >= p.T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = n0 + tx + 16 * j;
            if (e < p.E) out[(size_t)t * p.E + e] = acc[i][j];
        }
    }
}

struct TopkParams {
    int E, G, Gk, k, T, splits;
    float scale;
    const float* part;
    const float* bias;
    int32_t* ids;
    float* w;
};

__global__ void __launch_bounds__(256) topk_kernel(TopkParams p) {
    __shared__ float s_gs[8][kMaxE];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= p.T) return;
    float lg[kMaxE / 32];
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        if (e < p.E) {
            float l = 0.f;
            for (int s = 0; s < p.splits; ++s) l += p.part[((size_t)s * p.T + t) * p.E + e];
            if (p.bias) l += p.bias[e];
            lg[i] = l;
        } else {
            lg[i] = -INFINITY;
        }
    }
    topk_warp(lg, p.E, p.G, p.Gk, p.k, p.scale, s_gs[warp], p.ids + (size_t)t * p.k, p.w + (size_t)t * p.k,
              nullptr);
}

// x [T, H] bf16 -> xq codes, xs scales; one warp per 128-block.
__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t* x, int T, int H, uint8_t* xq, float* xs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hb = H / kBlk;
    const long nb = (long)T * Hb;
    for (long b = (long)blockIdx.x * 8 + warp; b < nb; b += (long)gridDim.x * 8) {
        const long t = b / Hb;
        const int kb = (int)(b % Hb);
        const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + t * H + kb * kBlk) + lane);
        float s;
        const uint32_t q = warp_quant_block128(
            bf16_bits_to_float((uint16_t)(xv.x & 0xFFFF)), bf16_bits_to_float((uint16_t)(xv.x >> 16)),
            bf16_bits_to_float((uint16_t)(xv.y & 0xFFFF)), bf16_bits_to_float((uint16_t)(xv.y >> 16)), &s);
        reinterpret_cast<uint32_t*>(xq + t * H + kb * kBlk)[lane] = q;
        if (lane == 0) xs[t * Hb + kb] = s;
    }
}

}  // namespace

cudaError_t launch_quant_act(const void* x, int T, int H, uint8_t* xq, float* xs, cudaStream_t st) {
    const long nb = (long)T * (H / kBlk);
    const int grid = (int)std::min<long>((nb + 7) / 8, (long)num_sms() * 8);
    quant_act_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(x), T, H, xq, xs);
    return cudaGetLastError();
}

cudaError_t launch_route_small(const moe_config_t& c, const void* x, int T, const float* w_router,
                               const float* bias, int32_t* ids, float* w, float* logits, uint8_t* xq,
                               float* xs, int32_t* offsets, int32_t* perm_src, int32_t* inv_pos,
                               RowGroup* groups, int32_t* group_of_row, Ctrl* ctrl, cudaStream_t st) {
    RouteSmallParams p;
    p.H = c.hidden;
    p.E = c.n_routed;
    p.G = c.n_group;
    p.Gk = c.topk_group;
    p.k = c.top_k;
    p.T = T;
    p.scale = c.routed_scaling_factor;
    p.x = static_cast<const uint16_t*>(x);
    p.wr = w_router;
    p.bias = bias;
    p.logits = logits;
    p.ids = ids;
    p.w = w;
    p.xq = xq;
    p.xs = xs;
    p.offsets = offsets;
    p.perm_src = perm_src;
    p.inv_pos = inv_pos;
    p.groups = groups;
    p.group_of_row = group_of_row;
    p.ctrl = ctrl;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c.n_routed);
    cfg.blockDim = dim3(kRouteWarps * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_small_kernel, p);
}

cudaError_t launch_route_large(const moe_config_t& c, const void* x, int T, const float* w_router,
                               const float* bias, int32_t* ids, float* w, float* logits, int splits,
                               cudaStream_t st) {
    RouterGemmParams g;
    g.H = c.hidden;
    g.E = c.n_routed;
    g.T = T;
    const int Hb = c.hidden / kBlk;
    g.kchunk = ((Hb + splits - 1) / splits) * kBlk;
    g.x = static_cast<const uint16_t*>(x);
    g.wr = w_router;
    g.part = logits;
    dim3 grid((T + kBM - 1) / kBM, (c.n_routed + kBN - 1) / kBN, splits);
    router_gemm_kernel<<<grid, 256, 0, st>>>(g);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    TopkParams t;
    t.E = c.n_routed;
    t.G = c.n_group;
    t.Gk = c.topk_group;
    t.k = c.top_k;
    t.T = T;
    t.splits = splits;
    t.scale = c.routed_scaling_factor;
    t.part = logits;
    t.bias = bias;
    t.ids = ids;
    t.w = w;
    topk_kernel<<<(T + 7) / 8, 256, 0, st>>>(t);
    return cudaGetLastError();
}

}  // namespace moe
