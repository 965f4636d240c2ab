// Stages P1/P2 and Q1/Q2 of the DeepSeek-V2 MoE layer ("DSV2-236B-MegaKernel",
// README stage flowchart, MoE subgraph) for the weight-streaming regime: every
// expert sees a handful of tokens, so each FP8 weight byte is used by at most 8
// activation rows and the kernels are bound by HBM bandwidth (the lecture's
// "decode is a GEMV", DeepSeek-V4.1 Flash, "Skill 5").
//
// Both kernels are persistent loops over work items (row group x output tile)
// whose count comes from the device-side permutation, so no count ever travels to
// the host. The inner product runs on mma.m16n8k32 (E4M3 x E4M3 -> fp32): the MMA
// is used as a dequantising dot-product engine, with 16 weight rows as A and up to
// 8 activation rows as B. Each lane streams 16 contiguous weight bytes per row and
// K-step; because a dot product may visit K in any order as long as A and B agree,
// the lane's 16 bytes are split over the two k32 MMAs of a 64-wide K step and the
// activation fragment is loaded at the very same offsets. Per-128 block scales are
// applied after each 128-wide K block: acc += partial * s_w[block] * s_x[token, block].
#include <algorithm>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kGUWarps = 4;  // gate/up: warps of a CTA split K (strided 128-blocks)
constexpr int kGUNB = 2;     // 128-blocks in flight per warp per iteration
constexpr int kDWarps = 4;   // down: warps of a CTA own 16 output rows each
constexpr int kDNB = 4;

__device__ __forceinline__ void mma_step64(float (&c)[4], const uint4& ar, const uint4& ar8, const uint4& b) {
    mma_e4m3_16832(c, ar.x, ar8.x, ar.y, ar8.y, b.x, b.y);
    mma_e4m3_16832(c, ar.z, ar8.z, ar.w, ar8.w, b.z, b.w);
}

// One work item of gate/up: 16 rows of the gate and up matrices (output rows
// r0..r0+15 of the intermediate), K = H split over the CTA's warps, for <= 8 rows
// of activations. Writes a = SiLU(g) * u in fp32.
__global__ void __launch_bounds__(kGUWarps * 32) gateup_gemv_kernel(ExpertArgs a) {
    __shared__ float red[kGUWarps][2][32][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int H = a.H, Hb = H / kBlk;
    const int tilesR = a.I / 16, tilesS = a.Is / 16;
    const int nR = a.ctrl->n_routed_groups * tilesR;
    const int nS = a.n_shared_groups * tilesS;
    const int total = nR + nS;

    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        const bool shared = item >= nR;
        int tile, row_begin, nrows, N;
        const uint8_t *Wg, *Wu;
        const float *Sg, *Su;
        float* out;
        if (!shared) {
            const RowGroup rg = a.groups[item / tilesR];
            tile = item % tilesR;
            row_begin = rg.row_begin;
            nrows = rg.nrows;
            N = a.I;
            const size_t e = (size_t)rg.expert;
            Wg = a.w_gate + e * a.I * H;
            Wu = a.w_up + e * a.I * H;
            Sg = a.s_gate + e * (a.I / kBlk) * Hb;
            Su = a.s_up + e * (a.I / kBlk) * Hb;
            out = a.a_routed;
        } else {
            const int it = item - nR;
            tile = it % tilesS;
            row_begin = (it / tilesS) * kGroupRows;
            nrows = min(kGroupRows, a.T - row_begin);
            N = a.Is;
            Wg = a.ws_gate;
            Wu = a.ws_up;
            Sg = a.ss_gate;
            Su = a.ss_up;
            out = a.a_shared;
        }
        // Token of activation column col (-1: padding). A permuted row whose source
        // index lies outside [0, T*k) is treated as padding rather than read.
        auto token_of = [&](int col) -> int {
            if (col >= nrows) return -1;
            if (shared) return row_begin + col;
            const int f = a.perm_src[row_begin + col];
            return ((unsigned)f < (unsigned)(a.T * a.k)) ? f / a.k : -1;
        };
        const int tok_b = token_of(g);
        const int tok_c0 = token_of(2 * t4), tok_c1 = token_of(2 * t4 + 1);
        const int r0 = tile * 16;
        const uint8_t* ag = Wg + (size_t)(r0 + g) * H + 16 * t4;
        const uint8_t* ag8 = ag + 8 * (size_t)H;
        const uint8_t* au = Wu + (size_t)(r0 + g) * H + 16 * t4;
        const uint8_t* au8 = au + 8 * (size_t)H;
        const uint8_t* xb = tok_b >= 0 ? a.xq + (size_t)tok_b * H + 16 * t4 : nullptr;
        const float* sgr = Sg + (size_t)(r0 / kBlk) * Hb;
        const float* sur = Su + (size_t)(r0 / kBlk) * Hb;
        const float* xs0 = tok_c0 >= 0 ? a.xs + (size_t)tok_c0 * Hb : nullptr;
        const float* xs1 = tok_c1 >= 0 ? a.xs + (size_t)tok_c1 * Hb : nullptr;

        float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int kb = warp; kb < Hb; kb += kGUNB * kGUWarps) {
            uint4 A[kGUNB][2][4];
            uint4 B[kGUNB][2];
#pragma unroll
            for (int j = 0; j < kGUNB; ++j) {
                const int kbj = kb + j * kGUWarps;
                if (kbj < Hb) {
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        const int off = kbj * kBlk + s * 64;
                        A[j][s][0] = ld_stream_v4(ag + off);
                        A[j][s][1] = ld_stream_v4(ag8 + off);
                        A[j][s][2] = ld_stream_v4(au + off);
                        A[j][s][3] = ld_stream_v4(au8 + off);
                        B[j][s] = xb ? ld_v4(xb + off) : make_uint4(0, 0, 0, 0);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kGUNB; ++j) {
                const int kbj = kb + j * kGUWarps;
                if (kbj < Hb) {
                    float cg[4] = {0.f, 0.f, 0.f, 0.f}, cu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        mma_step64(cg, A[j][s][0], A[j][s][1], B[j][s]);
                        mma_step64(cu, A[j][s][2], A[j][s][3], B[j][s]);
                    }
                    const float swg = __ldg(sgr + kbj), swu = __ldg(sur + kbj);
                    const float sx0 = xs0 ? __ldg(xs0 + kbj) : 0.f;
                    const float sx1 = xs1 ? __ldg(xs1 + kbj) : 0.f;
                    accg[0] = fmaf(cg[0], swg * sx0, accg[0]);
                    accg[1] = fmaf(cg[1], swg * sx1, accg[1]);
                    accg[2] = fmaf(cg[2], swg * sx0, accg[2]);
                    accg[3] = fmaf(cg[3], swg * sx1, accg[3]);
                    accu[0] = fmaf(cu[0], swu * sx0, accu[0]);
                    accu[1] = fmaf(cu[1], swu * sx1, accu[1]);
                    accu[2] = fmaf(cu[2], swu * sx0, accu[2]);
                    accu[3] = fmaf(cu[3], swu * sx1, accu[3]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            red[warp][0][lane][i] = accg[i];
            red[warp][1][lane][i] = accu[i];
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float gs = 0.f, us = 0.f;
#pragma unroll
                for (int w = 0; w < kGUWarps; ++w) {
                    gs += red[w][0][lane][i];
                    us += red[w][1][lane][i];
                }
                const int col = 2 * t4 + (i & 1);
                const int row = r0 + g + (i >= 2 ? 8 : 0);
                if (col < nrows) out[(size_t)(row_begin + col) * N + row] = silu_mul(gs, us);
            }
        }
        __syncthreads();
    }
}

// One work item of down: 64 output rows (16 per warp) of Wd for <= 8 activation
// rows, K = I (or Is) in full. The CTA first quantises its activation rows to FP8
// (power-of-two scale per 128 values) into shared memory; every CTA of a group
// computes the same codes, so the result does not depend on which CTA ran first.
__global__ void __launch_bounds__(kDWarps * 32) down_gemv_kernel(ExpertArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int H = a.H;
    const int Nmax = max(a.I, a.Is);
    uint8_t* s_q = smem;                                             // [8][Nmax]
    float* s_s = reinterpret_cast<float*>(smem + kGroupRows * Nmax);  // [8][Nmax/128]
    float* s_w = s_s + kGroupRows * (Nmax / kBlk);                    // [8]
    const int tiles = H / (16 * kDWarps);
    const int nR = a.ctrl->n_routed_groups * tiles;
    const int nS = a.n_shared_groups * tiles;
    const int total = nR + nS;

    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        const bool shared = item >= nR;
        int tile, row_begin, nrows, N;
        const uint8_t* Wd;
        const float *Sd, *src;
        __nv_bfloat16* dst;
        if (!shared) {
            const RowGroup rg = a.groups[item / tiles];
            tile = item % tiles;
            row_begin = rg.row_begin;
            nrows = rg.nrows;
            N = a.I;
            const size_t e = (size_t)rg.expert;
            Wd = a.w_down + e * H * a.I;
            Sd = a.s_down + e * (H / kBlk) * (a.I / kBlk);
            src = a.a_routed;
            dst = a.y_perm;
        } else {
            const int it = item - nR;
            tile = it % tiles;
            row_begin = (it / tiles) * kGroupRows;
            nrows = min(kGroupRows, a.T - row_begin);
            N = a.Is;
            Wd = a.ws_down;
            Sd = a.ss_down;
            src = a.a_shared;
            dst = a.y_shared;
        }
        const int Nb = N / kBlk;
        __syncthreads();  // the previous item is done with shared memory
        for (int b = warp; b < nrows * Nb; b += kDWarps) {
            const int r = b / Nb, kb = b % Nb;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(src + (size_t)(row_begin + r) * N + kb * kBlk) + lane);
            float s;
            const uint32_t q = warp_quant_block128(v.x, v.y, v.z, v.w, &s);
            reinterpret_cast<uint32_t*>(s_q + r * Nmax + kb * kBlk)[lane] = q;
            if (lane == 0) s_s[r * (Nmax / kBlk) + kb] = s;
        }
        if (threadIdx.x < kGroupRows) {
            const int c = threadIdx.x;
            float wc = 0.f;
            if (c < nrows) {
                if (shared) {
                    wc = 1.f;
                } else {
                    const int f = a.perm_src[row_begin + c];
                    wc = ((unsigned)f < (unsigned)(a.T * a.k)) ? a.topk_w[f] : 0.f;
                }
            }
            s_w[c] = wc;
        }
        __syncthreads();

        const int o0 = tile * (16 * kDWarps) + warp * 16;
        const uint8_t* ar = Wd + (size_t)(o0 + g) * N + 16 * t4;
        const uint8_t* ar8 = ar + 8 * (size_t)N;
        const float* swr = Sd + (size_t)(o0 / kBlk) * Nb;
        const bool bvalid = g < nrows;
        const uint8_t* xb = s_q + g * Nmax + 16 * t4;
        const int c0 = 2 * t4, c1 = 2 * t4 + 1;
        const float* sx0 = s_s + c0 * (Nmax / kBlk);
        const float* sx1 = s_s + c1 * (Nmax / kBlk);
        const bool v0 = c0 < nrows, v1 = c1 < nrows;

        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int kb = 0; kb < Nb; kb += kDNB) {
            uint4 A[kDNB][2][2];
#pragma unroll
            for (int j = 0; j < kDNB; ++j) {
                if (kb + j < Nb) {
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        const int off = (kb + j) * kBlk + s * 64;
                        A[j][s][0] = ld_stream_v4(ar + off);
                        A[j][s][1] = ld_stream_v4(ar8 + off);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kDNB; ++j) {
                if (kb + j < Nb) {
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        const int off = (kb + j) * kBlk + s * 64;
                        const uint4 b = bvalid ? *reinterpret_cast<const uint4*>(xb + off) : make_uint4(0, 0, 0, 0);
                        mma_step64(c, A[j][s][0], A[j][s][1], b);
                    }
                    const float sw = __ldg(swr + kb + j);
                    const float f0 = v0 ? sw * sx0[kb + j] : 0.f;
                    const float f1 = v1 ? sw * sx1[kb + j] : 0.f;
                    acc[0] = fmaf(c[0], f0, acc[0]);
                    acc[1] = fmaf(c[1], f1, acc[1]);
                    acc[2] = fmaf(c[2], f0, acc[2]);
                    acc[3] = fmaf(c[3], f1, acc[3]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int col = (i & 1) ? c1 : c0;
            const int row = o0 + g + (i >= 2 ? 8 : 0);
            if (col < nrows)
                dst[(size_t)(row_begin + col) * H + row] = __float2bfloat16_rn(acc[i] * s_w[col]);
        }
    }
}

int occupancy_blocks(const void* fn, int threads, size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 1) n = 1;
    return n;
}

}  // namespace

cudaError_t launch_gateup_gemv(const ExpertArgs& a, cudaStream_t st) {
    static int occ = occupancy_blocks((const void*)gateup_gemv_kernel, kGUWarps * 32, 0);
    const long items = (long)a.max_groups * (a.I / 16) + (long)a.n_shared_groups * (a.Is / 16);
    if (items <= 0) return cudaSuccess;
    const int grid = (int)std::min<long>(items, (long)num_sms() * occ);
    gateup_gemv_kernel<<<grid, kGUWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_down_gemv(const ExpertArgs& a, cudaStream_t st) {
    const int Nmax = std::max(a.I, a.Is);
    const size_t smem = (size_t)kGroupRows * Nmax + (size_t)kGroupRows * (Nmax / kBlk) * 4 + kGroupRows * 4;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute((const void*)down_gemv_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const int occ = occupancy_blocks((const void*)down_gemv_kernel, kDWarps * 32, smem);
    const int tiles = a.H / (16 * kDWarps);
    const long items = (long)(a.max_groups + a.n_shared_groups) * tiles;
    if (items <= 0) return cudaSuccess;
    const int grid = (int)std::min<long>(items, (long)num_sms() * occ);
    down_gemv_kernel<<<grid, kDWarps * 32, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
