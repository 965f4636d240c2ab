// Stage N (router) and stage O (softmax + group-limited greedy top-k) of the
// DeepSeek-V2 MoE layer ("DSV2-236B-MegaKernel", README stage flowchart, MoE
// subgraph), plus the FP8 activation quantisation the expert GEMMs consume.
//
// Two routes:
//  * small T (<= kSmallT): one launch. CTA e computes logits[:, e] (a GEMV over the
//    fp32 router row, K split across warps), every CTA quantises a share of x, and
//    the last CTA to arrive (an atomic arrival counter, no waiting) runs the
//    per-token softmax/top-k and, for the fused forward, the expert permutation and
//    the row-group work list. The README's stage O selects with warp ballots and
//    bit counts; here groups and experts are ranked (count of better candidates, ties
//    to the lower index) with a ballot-compacted candidate list.
//  * large T: a tiled fp32 SIMT GEMM for the logits (split-K partials, summed in a
//    fixed order), then one warp per token for softmax/top-k.
#include <algorithm>
#include <type_traits>

#include "route_common.cuh"

namespace moe {

namespace {

constexpr int kRouteWarps = 8;
constexpr int kTailNT = 4;  // tokens per warp in the last CTA's top-k (T > 1)

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
    const uint16_t* gamma;  // stage M in front of the router when not null
    float eps;
    uint8_t* xs8;           // MXFP8: E8M0 scales [T, H/32] (xs unused)
    uint64_t* trace;        // per-CTA timer stamps or null
    int tail;               // 1: the last CTA runs top-k and the permutation; 0: logits and x codes only
};

// kNorm: stage M in front of the router (p.gamma != nullptr); kMX: x quantised per 32
// values with E8M0 scales (p.xs8) instead of per 128 with fp32 scales (p.xs)
// (Two CTAs per SM without stage M: the 160 CTAs of a 160-expert layer in one wave.)
template <bool kNorm, bool kMX>
__global__ void __launch_bounds__(kRouteWarps * 32, kNorm ? 1 : 2) route_small_kernel(RouteSmallParams p) {
    __shared__ float s_part[kRouteWarps][kSmallT];
    __shared__ alignas(16) float s_gs[kRouteWarps][kMaxE];
    __shared__ int32_t s_ids[kSmallT * 16];
    __shared__ int s_rank[kSmallT * 16];
    __shared__ int s_cnt[kMaxE], s_off[kMaxE + 1], s_gcnt[kMaxE], s_goff[kMaxE];
    __shared__ int s_last;
    __shared__ float s_rstd[kSmallT];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x;
    const int H = p.H, T = p.T, Hb = H / kBlk;
    constexpr bool norm = kNorm;

    // A warp's slice of the router row (and of gamma) sits in registers, up to 8 float4
    // per lane per chunk of 256 float4. Nothing is read before the wait: this is the
    // layer's first kernel, and the one before it in the stream (the caller's) may have
    // written any of the inputs, the weights included; its writes are visible only
    // after the wait.
    const int slice = H / kRouteWarps;
    const int n4 = slice / 4;  // float4 per warp slice
    const float4* wrow = reinterpret_cast<const float4*>(p.wr + (size_t)e * H + warp * slice);
    const uint2* grow = norm ? reinterpret_cast<const uint2*>(p.gamma + warp * slice) : nullptr;
    float4 wv[8];
    uint2 gv[8];
    auto load_w = [&](int c0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = c0 + lane + 32 * j;
            wv[j] = i < n4 ? __ldg(wrow + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            gv[j] = norm && i < n4 ? __ldg(grow + i) : make_uint2(0, 0);
        }
    };
    trace_stamp(p.trace, 0, 0);
    pdl_wait();  // the previous kernel in the stream is done: inputs written, workspace free
    pdl_launch_dependents();
    trace_stamp(p.trace, 0, 1);
    load_w(0);
    const float bias_e = p.bias ? __ldg(p.bias + e) : 0.f;

    // ---- M (optional): every CTA derives the same 1/rms of each token itself
    if (norm) {
        for (int t = warp; t < T; t += kRouteWarps) {
            const float r = rms_rstd(warp_row_sumsq(p.x + (size_t)t * H, H), H, p.eps);
            if (lane == 0) s_rstd[t] = r;
        }
        __syncthreads();
    }

    // ---- N: logits[:, e], K split over the CTA's warps (H/8 is a multiple of 16).
    // Four tokens' activations are loaded before any FMA, so a warp waits for one
    // memory round trip per chunk and four tokens, not one per load.
    for (int t = lane; t < T; t += 32) s_part[warp][t] = 0.f;
    __syncwarp();
    for (int c0 = 0; c0 < n4; c0 += 32 * 8) {
        if (c0 > 0) load_w(c0);
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
            if (norm) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float r = s_rstd[min(t + q, T - 1)];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        xv[q][j] = make_uint2(rms_apply2(xv[q][j].x, r, gv[j].x), rms_apply2(xv[q][j].y, r, gv[j].y));
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
        if (p.bias) l += bias_e;
        p.logits[(size_t)t * p.E + e] = l;
    }
    trace_stamp(p.trace, 0, 2);

    // ---- activation quantisation: this CTA's share of the T*H/128 blocks
    for (int b = blockIdx.x * kRouteWarps + warp; b < T * Hb; b += gridDim.x * kRouteWarps) {
        const int t = b / Hb, kb = b % Hb;
        uint2 xv = __ldg(reinterpret_cast<const uint2*>(p.x + (size_t)t * H + kb * kBlk) + lane);
        if (norm) {
            const uint2 g = __ldg(reinterpret_cast<const uint2*>(p.gamma + kb * kBlk) + lane);
            xv = make_uint2(rms_apply2(xv.x, s_rstd[t], g.x), rms_apply2(xv.y, s_rstd[t], g.y));
        }
        const float v0 = bf16_bits_to_float((uint16_t)(xv.x & 0xFFFF)), v1 = bf16_bits_to_float((uint16_t)(xv.x >> 16));
        const float v2 = bf16_bits_to_float((uint16_t)(xv.y & 0xFFFF)), v3 = bf16_bits_to_float((uint16_t)(xv.y >> 16));
        if constexpr (kMX) {
            uint32_t s8;
            const uint32_t q = warp_quant_mx32(v0, v1, v2, v3, &s8);
            reinterpret_cast<uint32_t*>(p.xq + (size_t)t * H + kb * kBlk)[lane] = q;
            if ((lane & 7) == 0) p.xs8[(size_t)t * (H / 32) + kb * 4 + (lane >> 3)] = (uint8_t)s8;
        } else {
            float s;
            const uint32_t q = warp_quant_block128(v0, v1, v2, v3, &s);
            reinterpret_cast<uint32_t*>(p.xq + (size_t)t * H + kb * kBlk)[lane] = q;
            if (lane == 0) p.xs[(size_t)t * Hb + kb] = s;
        }
    }

    // ---- last CTA to arrive: O (softmax + top-k) and the permutation; with p.tail = 0
    // the kernels that follow derive the selection from the logits themselves
    if (!p.tail) {
        trace_stamp(p.trace, 0, 3);
        return;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&p.ctrl->route_arrived, 1u);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) {
        trace_stamp(p.trace, 0, 3);
        return;
    }
    __threadfence();

    if (T == 1 && p.E <= (int)blockDim.x) {
        // one token: the whole CTA ranks the experts (s_gs as scratch)
        unsigned* scratch = reinterpret_cast<unsigned*>(&s_gs[0][0]);
        cta_topk1(p.logits, p.E, p.G, p.Gk, p.k, p.scale, scratch, scratch + kMaxE,
                  reinterpret_cast<float*>(scratch + kMaxE + 32), p.ids, p.w, s_ids);
    } else {
        // kTailNT tokens per warp side by side (tokens t0 + q * kRouteWarps), all their
        // logits loaded at once
        for (int t0 = warp; t0 < T; t0 += kRouteWarps * kTailNT) {
            float lg[kTailNT][kMaxE / 32];
            int32_t* io[kTailNT];
            float* wo[kTailNT];
            int32_t* so[kTailNT];
#pragma unroll
            for (int q = 0; q < kTailNT; ++q) {
                const int t = t0 + q * kRouteWarps;
                const bool valid = t < T;
#pragma unroll
                for (int i = 0; i < kMaxE / 32; ++i) {
                    const int ee = lane + 32 * i;
                    lg[q][i] = valid && ee < p.E ? __ldcg(p.logits + (size_t)t * p.E + ee) : -INFINITY;
                }
                io[q] = valid ? p.ids + (size_t)t * p.k : nullptr;
                wo[q] = valid ? p.w + (size_t)t * p.k : nullptr;
                so[q] = valid ? s_ids + t * p.k : nullptr;
            }
            topk_warp_n<kTailNT>(lg, p.E, p.G, p.Gk, p.k, p.scale, io, wo, so);
        }
    }
    __syncthreads();
    if (p.offsets)
        small_permute(s_ids, T * p.k, p.E, s_cnt, s_off, s_gcnt, s_goff, s_rank, p.offsets, p.perm_src, p.inv_pos,
                      p.groups, p.group_of_row, &p.ctrl->n_routed_groups);
    if (threadIdx.x == 0) p.ctrl->route_arrived = 0u;
    trace_stamp(p.trace, 0, 3);
}

// ---------------------------------------------------------------- large T
// w -> (hi, mid, lo), each the bf16 rounding of what the previous parts leave:
// |w - hi - mid - lo| <= 2^-27 |w|, the precision of the fp32 weight itself, so that with
// x exact in bf16 the three bf16 products reproduce the fp32 router GEMM.
__device__ __forceinline__ void split3(float w, uint16_t& hi, uint16_t& mid, uint16_t& lo) {
    const __nv_bfloat16 h = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(h);
    const __nv_bfloat16 m = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(m);
    hi = __bfloat16_as_ushort(h);
    mid = __bfloat16_as_ushort(m);
    lo = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
}

// ---- large T: router GEMM on the tcgen05 tensor cores (kind::f16, fp32 in tensor memory).
// The fp32 router weights are split once per call into three bf16 parts (router_split_
// kernel: hi + mid + lo, as split3), stacked as [3][Ep][H] with zero rows from E to Ep;
// x is exact in bf16. A CTA takes 128 tokens x all experts over a range of K (split-K
// partials, summed in fixed order by topk_kernel), in 64-wide K steps: per step the three
// parts' products (12 MMAs of M=128, N=Ep, K=16, the small parts first) accumulate in a
// fresh TMEM accumulator (the tensor core truncates small products against a large
// accumulator), which the epilogue adds into fp32 registers while the tensor core fills
// the other accumulator with the next step. Warp 9: TMA producer (an x box of 128 rows
// and the three parts' boxes of Ep rows per step); warp 8: MMA issuer; warps 0-7:
// epilogue (warp w reads lanes 32*(w%4).. and the 16-column chunks c = w/4, w/4+2, ...).
constexpr int kRTM = 128;            // tokens per CTA (MMA M)
constexpr int kRTK = 64;             // bf16 per K step (128 bytes)
constexpr int kRTEpi = 8;
constexpr int kRTMma = kRTEpi;
constexpr int kRTProd = kRTEpi + 1;
constexpr int kRTThreads = (kRTEpi + 2) * 32;
constexpr int kRTSA = kRTM * kRTK * 2;   // 16 KB x box

// TMEM columns per accumulator buffer: the power of two >= Ep (two buffers per CTA)
__host__ __device__ constexpr uint32_t rt_buf_cols(int Ep) {
    uint32_t c = 16;
    while (c < (uint32_t)Ep) c <<= 1;
    return c;
}

struct RouterTcParams {
    int T, E, Ep, H, k_per_split, n_mt, stages;
    float* part;  // [splits, T, E]
    int* status;
};

__global__ void __launch_bounds__(256) router_split_kernel(const float* wr, int E, int Ep, int H, uint16_t* out) {
    const size_t plane = (size_t)Ep * H, n4 = plane / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const size_t o = 4 * i;
        const int e = (int)(o / H);
        const float4 v = e < E ? __ldg(reinterpret_cast<const float4*>(wr) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float w4[4] = {v.x, v.y, v.z, v.w};
        uint16_t h[4], m[4], l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) split3(w4[u], h[u], m[u], l[u]);
        *reinterpret_cast<uint2*>(out + o) = make_uint2(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16));
        *reinterpret_cast<uint2*>(out + plane + o) =
            make_uint2(m[0] | ((uint32_t)m[1] << 16), m[2] | ((uint32_t)m[3] << 16));
        *reinterpret_cast<uint2*>(out + 2 * plane + o) =
            make_uint2(l[0] | ((uint32_t)l[1] << 16), l[2] | ((uint32_t)l[3] << 16));
    }
}

template <int NCH>  // 16-column chunks of the accumulator: Ep = 16 * NCH
__global__ void __launch_bounds__(kRTThreads, 1)
    router_tc_kernel(const RouterTcParams p, const __grid_constant__ TmaMap tm_x, const __grid_constant__ TmaMap tm_w) {
    constexpr int Ep = 16 * NCH;
    constexpr int kSB = 3 * Ep * kRTK * 2;  // the three parts' boxes
    constexpr int kStage = kRTSA + kSB;     // a multiple of 1024 (Ep is a multiple of 16)
    constexpr int kMyCh = (NCH + 1) / 2;    // chunks per epilogue thread (at most)
    static_assert(kRTM * (Ep + 4) * 4 <= 2 * kStage, "the output block is staged in the (at least two) stages");
    constexpr uint32_t kIdesc = idesc_bf16_f32(kRTM, Ep);
    constexpr uint32_t kBuf = rt_buf_cols(Ep);
    constexpr uint32_t kAlloc = 2 * kBuf < 32 ? 32 : 2 * kBuf;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kStage);
    uint64_t* empty = full + S;
    uint64_t* acc_full = empty + S;   // [2]
    uint64_t* acc_empty = acc_full + 2;  // [2]
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(acc_empty + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x % p.n_mt, split = blockIdx.x / p.n_mt;
    const int k0 = split * p.k_per_split, k1 = min(p.H, k0 + p.k_per_split);
    const int nsteps = k1 > k0 ? (k1 - k0) / kRTK : 0;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kRTEpi);
        }
        fence_mbar_init();
    }
    if (warp == kRTMma) {
        tmem_alloc(s_tmem, kAlloc);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();
    pdl_launch_dependents();

    if (warp == kRTProd) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && nsteps > 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_w);
            int n = 0;
            for (; n < nsteps; ++n) {
                const int s = n % S;
                if (n >= S && !mbar_wait_bounded(&empty[s], ((n / S) - 1) & 1)) {
                    set_status(p.status, kStatusTimeout);
                    break;
                }
                uint8_t* st = smem + s * kStage;
                const int x = k0 + n * kRTK;
                mbar_arrive_expect_tx(&full[s], kStage);
                tma_load_2d(st, &tm_x, x, mt * kRTM, &full[s]);
#pragma unroll
                for (int part = 0; part < 3; ++part)
                    tma_load_2d(st + kRTSA + part * Ep * kRTK * 2, &tm_w, x, part * Ep, &full[s]);
            }
            // copies still in flight land before this CTA may exit
            for (int q = n > S ? n - S : 0; q < n; ++q) mbar_wait_bounded(&full[q % S], (q / S) & 1);
        }
    } else if (warp == kRTMma) {
        // -------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int n = 0;
            for (; n < nsteps; ++n) {
                const int s = n % S, b = n & 1;
                if ((n >= 2 && !mbar_wait_bounded(&acc_empty[b], ((n >> 1) - 1) & 1)) ||
                    !mbar_wait_bounded(&full[s], (n / S) & 1)) {
                    set_status(p.status, kStatusTimeout);
                    break;
                }
                tc_fence_after();
                const uint8_t* st = smem + s * kStage;
                const uint64_t da = smem_desc_sw128(st);
#pragma unroll
                for (int k = 0; k < 4; ++k)  // 4 x K=16 (32 bytes) inside the 128-byte swizzled rows
#pragma unroll
                    for (int part = 2; part >= 0; --part) {  // small parts first
                        const uint64_t db = smem_desc_sw128(st + kRTSA + part * Ep * kRTK * 2);
                        tc_mma_bf16(tmem + b * kBuf, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), kIdesc,
                                    (k | (2 - part)) != 0);
                    }
                tc_commit(&empty[s]);
                tc_commit(&acc_full[b]);
            }
            // every MMA issued has completed before the CTA frees tensor memory
            if (n > 0) mbar_wait_bounded(&acc_full[(n - 1) & 1], ((n - 1) >> 1) & 1);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q4 = warp & 3, half = warp >> 2;
        const int row = 32 * q4 + lane;
        const uint32_t t_row = tmem + ((uint32_t)(32 * q4) << 16);
        float acc[kMyCh][16];
#pragma unroll
        for (int c = 0; c < kMyCh; ++c)
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[c][j] = 0.f;
        bool ok = true;
        for (int n = 0; n < nsteps; ++n) {
            const int b = n & 1;
            if (ok && !mbar_wait_bounded(&acc_full[b], (n >> 1) & 1)) ok = false;
            ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
            tc_fence_after();
            if (ok) {
#pragma unroll
                for (int c = 0; c < kMyCh; ++c) {
                    const int ch = half + 2 * c;
                    if (ch < NCH) {
                        float v[16];
                        tmem_ld16(t_row + b * kBuf + 16 * ch, v);
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[c][j] += v[j];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
        if (!ok) set_status(p.status, kStatusTimeout);
        // The CTA's partial logits are one contiguous [rows, E] block of part: stage them
        // in shared memory (the stages are free: every copy was consumed by an MMA that
        // has completed) with a row pitch of Ep + 4 floats, so that a warp's 16-byte
        // stores of 32 rows fall in distinct banks, then store the block coalesced.
        constexpr int kPitch = Ep + 4;
        float* stg = reinterpret_cast<float*>(smem);
#pragma unroll
        for (int c = 0; c < kMyCh; ++c) {
            const int ch = half + 2 * c;
            if (ch < NCH)
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4*>(stg + row * kPitch + 16 * ch + j) =
                        make_float4(acc[c][j], acc[c][j + 1], acc[c][j + 2], acc[c][j + 3]);
        }
        named_bar(1, kRTEpi * 32);
        const int rows = min(kRTM, p.T - mt * kRTM), E = p.E;
        float* out = p.part + ((size_t)split * p.T + (size_t)mt * kRTM) * E;
        if ((E & 3) == 0) {
            const int q = E >> 2, n = rows * q;
            for (int i = tid; i < n; i += kRTEpi * 32) {
                const int r = i / q, c4 = i - r * q;
                reinterpret_cast<float4*>(out)[i] = *reinterpret_cast<const float4*>(stg + r * kPitch + 4 * c4);
            }
        } else {
            const int n = rows * E;
            for (int i = tid; i < n; i += kRTEpi * 32) {
                const int r = i / E;
                out[i] = stg[r * kPitch + (i - r * E)];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kRTMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kAlloc);
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
    pdl_wait();  // the logits (launched with programmatic serialization after the small-T router)
    pdl_launch_dependents();
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

// The permutation and row-group work list of up to kSmallT tokens from topk_kernel's ids,
// by one CTA (the small-T router's tail, split off when its last CTA would rank more
// than one token per warp).
__global__ void __launch_bounds__(256) route_permute_kernel(const int32_t* ids, int n, int E, int32_t* offsets,
                                                            int32_t* perm_src, int32_t* inv_pos, RowGroup* groups,
                                                            int32_t* group_of_row, int* n_groups) {
    __shared__ int32_t s_ids[kSmallT * 16];
    __shared__ int s_rank[kSmallT * 16];
    __shared__ int s_cnt[kMaxE], s_off[kMaxE + 1], s_gcnt[kMaxE], s_goff[kMaxE];
    pdl_wait();  // topk_kernel's ids
    pdl_launch_dependents();
    for (int f = threadIdx.x; f < n; f += blockDim.x) s_ids[f] = ids[f];
    __syncthreads();
    small_permute(s_ids, n, E, s_cnt, s_off, s_gcnt, s_goff, s_rank, offsets, perm_src, inv_pos, groups, group_of_row,
                  n_groups);
}

// x [T, H] bf16 -> xq codes + scales. Each thread takes 32 consecutive values. Per-128
// blocks (kMX false): four threads share a block (two shuffles for its maximum), one fp32
// scale per block in xs. MXFP8 (kMX true): a thread's 32 values are one block, its E8M0
// scale byte goes to xs8 [T, H/32].
template <bool kMX>
__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t* x, int T, int H, uint8_t* xq, float* xs,
                                                        uint8_t* xs8, const uint16_t* gamma, const float* rstd) {
    const int Hb = H / kBlk;
    const long nq = (long)T * Hb * 4;  // quarters of a 128-value block
    // the loop condition is the same for every lane of a warp (the shuffles need all 32)
    for (long base = (long)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < nq;
         base += (long)gridDim.x * blockDim.x) {
        const long i = base + (threadIdx.x & 31);
        const bool ok = i < nq;
        const long b = (ok ? i : nq - 1) >> 2;
        const int q = (int)(i & 3);
        const long t = b / Hb;
        const int kb = (int)(b % Hb);
        const uint4* src = reinterpret_cast<const uint4*>(x + t * H + kb * kBlk + q * 32);
        uint4 u[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) u[c] = __ldg(src + c);
        if (gamma) {  // stage M applied on the fly
            const uint4* gs = reinterpret_cast<const uint4*>(gamma + kb * kBlk + q * 32);
            const float r = rstd[t];
#pragma unroll
            for (int c = 0; c < 4; ++c) u[c] = rms_apply8(u[c], r, __ldg(gs + c));
        }
        float v[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[8 * c + 2 * h] = bf16_bits_to_float((uint16_t)(w[h] & 0xFFFF));
                v[8 * c + 2 * h + 1] = bf16_bits_to_float((uint16_t)(w[h] >> 16));
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
        float inv, sc = 0.f;
        uint32_t s8 = 0;
        if (kMX) {
            s8 = act_scale_e8m0(amax, &inv);
        } else {
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            sc = act_scale_pow2(amax, &inv);
        }
        if (ok) {
            uint32_t code[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                code[j] = pack_e4m3x4(v[4 * j] * inv, v[4 * j + 1] * inv, v[4 * j + 2] * inv, v[4 * j + 3] * inv);
            uint4* dst = reinterpret_cast<uint4*>(xq + t * H + kb * kBlk + q * 32);
            dst[0] = make_uint4(code[0], code[1], code[2], code[3]);
            dst[1] = make_uint4(code[4], code[5], code[6], code[7]);
            if (kMX)
                xs8[t * (H / 32) + kb * 4 + q] = (uint8_t)s8;
            else if (q == 0)
                xs[t * Hb + kb] = sc;
        }
    }
}

// ---- stage M as a kernel of its own (large T, and the stand-alone moe_rmsnorm):
// one warp per token row writes 1/rms (rstd != nullptr) and/or the normalised row.
__global__ void __launch_bounds__(256) rms_kernel(const uint16_t* x, int T, int H, const uint16_t* gamma, float eps,
                                                  float* rstd, uint16_t* x_out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    const uint16_t* row = x + (size_t)t * H;
    const float r = rms_rstd(warp_row_sumsq(row, H), H, eps);
    if (rstd && lane == 0) rstd[t] = r;
    if (x_out) {
        const uint4* src = reinterpret_cast<const uint4*>(row);
        const uint4* g = reinterpret_cast<const uint4*>(gamma);
        uint4* dst = reinterpret_cast<uint4*>(x_out + (size_t)t * H);
        for (int c = lane; c < H / 8; c += 32) dst[c] = rms_apply8(__ldg(src + c), r, __ldg(g + c));
    }
}

}  // namespace

cudaError_t launch_quant_act(const void* x, int T, int H, uint8_t* xq, float* xs, const NormArgs& nm,
                             cudaStream_t st) {
    const long nq = (long)T * (H / kBlk) * 4;
    const int grid = (int)std::min<long>((nq + 255) / 256, (long)num_sms() * 8);
    quant_act_kernel<false><<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(x), T, H, xq, xs, nullptr, nm.gamma,
                                                   nm.rstd);
    return cudaGetLastError();
}

cudaError_t launch_quant_act_mx(const void* x, int T, int H, uint8_t* xq, uint8_t* xs8, const NormArgs& nm,
                                cudaStream_t st) {
    const long nq = (long)T * (H / kBlk) * 4;
    const int grid = (int)std::min<long>((nq + 255) / 256, (long)num_sms() * 8);
    quant_act_kernel<true><<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(x), T, H, xq, nullptr, xs8, nm.gamma,
                                                 nm.rstd);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const void* x, int T, int H, const NormArgs& nm, void* x_out, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    rms_kernel<<<(T + 7) / 8, 256, 0, st>>>(static_cast<const uint16_t*>(x), T, H, nm.gamma, nm.eps, nm.rstd,
                                            static_cast<uint16_t*>(x_out));
    return cudaGetLastError();
}

cudaError_t launch_route_small(const moe_config_t& c, const void* x, int T, const float* w_router,
                               const float* bias, int32_t* ids, float* w, float* logits, uint8_t* xq,
                               float* xs, int32_t* offsets, int32_t* perm_src, int32_t* inv_pos,
                               RowGroup* groups, int32_t* group_of_row, Ctrl* ctrl, const NormArgs& nm,
                               cudaStream_t st, uint8_t* xs8, uint64_t* trace, bool tail) {
    // Above kRouteWarps tokens the last CTA would rank several tokens per warp on one SM
    // (~3 us each): the router then leaves the logits, and top-k (one warp per token
    // over T/8 CTAs) and the permutation run as two chained kernels.
    const bool split = tail && offsets != nullptr && T > kRouteWarps;
    RouteSmallParams p;
    p.tail = tail && !split ? 1 : 0;
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
    p.gamma = nm.gamma;
    p.eps = nm.eps;
    p.xs8 = nullptr;
    p.trace = trace;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c.n_routed);
    cfg.blockDim = dim3(kRouteWarps * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (xs8) {
        p.xs8 = xs8;
        e = nm.gamma ? cudaLaunchKernelEx(&cfg, route_small_kernel<true, true>, p)
                     : cudaLaunchKernelEx(&cfg, route_small_kernel<false, true>, p);
    } else {
        e = nm.gamma ? cudaLaunchKernelEx(&cfg, route_small_kernel<true, false>, p)
                     : cudaLaunchKernelEx(&cfg, route_small_kernel<false, false>, p);
    }
    if (e != cudaSuccess || !split) return e;
    TopkParams t;
    t.E = c.n_routed;
    t.G = c.n_group;
    t.Gk = c.topk_group;
    t.k = c.top_k;
    t.T = T;
    t.splits = 1;
    t.scale = c.routed_scaling_factor;
    t.part = logits;
    t.bias = nullptr;  // the router's logits include it
    t.ids = ids;
    t.w = w;
    cfg.gridDim = dim3((T + 7) / 8);
    cfg.blockDim = dim3(256);
    e = cudaLaunchKernelEx(&cfg, topk_kernel, t);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(1);
    return cudaLaunchKernelEx(&cfg, route_permute_kernel, static_cast<const int32_t*>(ids), T * c.top_k,
                              (int)c.n_routed, offsets, perm_src, inv_pos, groups, group_of_row,
                              &ctrl->n_routed_groups);
}

cudaError_t launch_route_large(const moe_config_t& c, const void* x, int T, const float* w_router,
                               const float* bias, int32_t* ids, float* w, float* logits, int splits,
                               uint16_t* w3, int* status, cudaStream_t st) {
    const int H = c.hidden, E = c.n_routed, Ep = (E + 15) & ~15;
    const int Hb = H / kBlk;
    const int k_per_split = ((Hb + splits - 1) / splits) * kBlk;
    cudaError_t e2 = cudaErrorInvalidValue;
    // split the router weights, then the GEMM
    if (!w3) return cudaErrorInvalidValue;
    {
        const size_t n4 = (size_t)Ep * H / 4;
        const unsigned blocks = (unsigned)std::min<size_t>(1024, (n4 + 255) / 256);
        router_split_kernel<<<blocks, 256, 0, st>>>(w_router, E, Ep, H, w3);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    TmaMap tx, tw;
    if (!tmap_bf16_2d(&tx, x, (uint64_t)T, (uint64_t)H, kRTK, kRTM) ||
        !tmap_bf16_2d(&tw, w3, (uint64_t)3 * Ep, (uint64_t)H, kRTK, (uint32_t)Ep))
        return cudaErrorInvalidValue;
    RouterTcParams p;
    p.T = T;
    p.E = E;
    p.Ep = Ep;
    p.H = H;
    p.k_per_split = k_per_split;
    p.n_mt = (T + kRTM - 1) / kRTM;
    p.part = logits;
    p.status = status;
    const size_t stage = (size_t)kRTSA + 3 * (size_t)Ep * kRTK * 2;
    const size_t room = 227 * 1024 - 1024 - 256;
    p.stages = (int)std::min<size_t>(4, room / stage);
    if (p.stages < 2) return cudaErrorInvalidValue;
    const size_t smem = 1024 + (size_t)p.stages * stage + 256;
    auto run = [&](auto kern) -> cudaError_t {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<p.n_mt * splits, kRTThreads, smem, st>>>(p, tx, tw);
        return cudaGetLastError();
    };
    auto pick = [&](auto nch) -> cudaError_t { return run(router_tc_kernel<decltype(nch)::value>); };
    switch (Ep / 16) {  // n_routed <= 256
        case 1: e2 = pick(std::integral_constant<int, 1>{}); break;
        case 2: e2 = pick(std::integral_constant<int, 2>{}); break;
        case 3: e2 = pick(std::integral_constant<int, 3>{}); break;
        case 4: e2 = pick(std::integral_constant<int, 4>{}); break;
        case 5: e2 = pick(std::integral_constant<int, 5>{}); break;
        case 6: e2 = pick(std::integral_constant<int, 6>{}); break;
        case 7: e2 = pick(std::integral_constant<int, 7>{}); break;
        case 8: e2 = pick(std::integral_constant<int, 8>{}); break;
        case 9: e2 = pick(std::integral_constant<int, 9>{}); break;
        case 10: e2 = pick(std::integral_constant<int, 10>{}); break;
        case 11: e2 = pick(std::integral_constant<int, 11>{}); break;
        case 12: e2 = pick(std::integral_constant<int, 12>{}); break;
        case 13: e2 = pick(std::integral_constant<int, 13>{}); break;
        case 14: e2 = pick(std::integral_constant<int, 14>{}); break;
        case 15: e2 = pick(std::integral_constant<int, 15>{}); break;
        case 16: e2 = pick(std::integral_constant<int, 16>{}); break;
    }
    if (e2 != cudaSuccess) return e2;
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
