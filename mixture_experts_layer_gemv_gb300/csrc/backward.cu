// The layer's backward: gradients of sum(dout * out) with the forward's expert choice
// held fixed (the Mixture-of-Kittens page's training workload: Table 1's backward
// columns, and the abstract's training of the expert MLPs). The FP8 quantisers are straight-through and the
// weights enter at their dequantised FP8 values. Per routed row r = (t, j), expert e,
// routing weight w = s * p_e, with g, u, ahat the forward's values:
//   dau = Wd_e^T dout_t                       (unweighted)        dgrad of the down GEMM
//   dw  = <dau, ahat> = <dout_t, Wd_e ahat>
//   da  = w dau; dg = da u sig(g)(1 + g(1 - sig(g))); du = da g sig(g)
//   dx_r = Wg_e^T dg + Wu_e^T du                                  dgrad of gate/up
//   dWd_e = sum_r (w dout_t) (x) ahat;  dWg_e = sum_r dg (x) xhat_t;  dWu_e likewise
// the shared experts the same with w = 1; the router (softmax over all E, logits from
// the unquantised x): dp_e = s dw for the kept experts, dlogit = p (dp - <p, dp>),
// dx_t += Wr^T dlogit, dWr = sum_t dlogit (x) x_t, dbias = sum_t dlogit.
//
// The forward's g and u are recomputed by the grouped tcgen05 FP8 GEMM (mode 2, same
// tiles and arithmetic as the forward, so ahat is bit-identical to what the forward's
// down GEMM consumed). The contractions of the backward run in bf16 with fp32
// accumulation on the tcgen05 tensor cores (bwd_tc.cu), on operands prepared here: the
// FP8 weights decoded to bf16 and transposed so that K is contiguous (one bf16 rounding
// of weight x block scale), the activations decoded exactly, rows gathered into expert
// order, and the transposed operands of the weight gradients.
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// 16 E4M3 codes times a scale, as 16 bf16 in two uint4.
__device__ __forceinline__ void e4m3x16_to_bf16(uint4 q, float s, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h01 = __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFF), __NV_E4M3));
        const __half2 h23 = __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3));
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        o[2 * i] = pack_bf16x2(f01.x * s, f01.y * s);
        o[2 * i + 1] = pack_bf16x2(f23.x * s, f23.y * s);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// ---------------------------------------------------------------- operand preparation
// Transposed dequantisation for the tcgen05 dgrad operands: for each of nmat matrices
// q [R, Cc] of E4M3 codes (fp32 scales per 128 x 128 block), out[c, col0 + r] =
// bf16(dec(q[r, c]) * scale) in an output matrix [Cc, out_ld]. 64 x 64 tiles through
// shared memory: reads of 64-byte row pieces, writes of 128-byte row pieces.
__global__ void __launch_bounds__(256) dequant_t_kernel(const uint8_t* q, const float* s, int R, int Cc, int out_ld,
                                                        int col0, __nv_bfloat16* out) {
    __shared__ __nv_bfloat16 tile[64][64 + 8];
    const int mat = blockIdx.z, r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
    const uint8_t* qm = q + (size_t)mat * R * Cc;
    const float* sm = s + (size_t)mat * (R / kBlk) * (Cc / kBlk);
    {  // read: thread -> row r0 + tid/4, 16 columns from c0 + (tid%4)*16
        const int r = threadIdx.x >> 2, c = (threadIdx.x & 3) * 16;
        const uint4 v = *reinterpret_cast<const uint4*>(qm + (size_t)(r0 + r) * Cc + c0 + c);
        const float sc = sm[(size_t)((r0 + r) / kBlk) * (Cc / kBlk) + (c0 + c) / kBlk];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f01 = __half22float2(
                __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFF), __NV_E4M3)));
            const float2 f23 = __half22float2(
                __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3)));
            tile[c + 4 * i][r] = __float2bfloat16_rn(f01.x * sc);
            tile[c + 4 * i + 1][r] = __float2bfloat16_rn(f01.y * sc);
            tile[c + 4 * i + 2][r] = __float2bfloat16_rn(f23.x * sc);
            tile[c + 4 * i + 3][r] = __float2bfloat16_rn(f23.y * sc);
        }
    }
    __syncthreads();
    {  // write: thread -> output row c0 + tid/4, 16 values from r0 + (tid%4)*16
        const int c = threadIdx.x >> 2, r = (threadIdx.x & 3) * 16;
        const uint4* src = reinterpret_cast<const uint4*>(&tile[c][r]);
        uint4* dst = reinterpret_cast<uint4*>(out + (size_t)mat * Cc * out_ld + (size_t)(c0 + c) * out_ld + col0 + r0 + r);
        dst[0] = src[0];
        dst[1] = src[1];
    }
}

// The weight gradients' column layout: expert e's permuted rows occupy columns
// [poff[e], poff[e] + cnt_e) of the transposed operands, poff[e] = sum over e' < e of
// cnt_e' rounded up to 64, and the columns up to poff[e + 1] are padding (map -1).
// One block per expert; block E - 1 also writes poff[E].
__global__ void __launch_bounds__(256) pad_map_kernel(int E, const int32_t* offsets, int32_t* poff, int32_t* pmap) {
    const int e = blockIdx.x;
    int base = 0;
    for (int i = 0; i < e; ++i) base += (offsets[i + 1] - offsets[i] + 63) & ~63;
    const int o = offsets[e], cnt = offsets[e + 1] - o, padded = (cnt + 63) & ~63;
    for (int j = threadIdx.x; j < padded; j += blockDim.x) pmap[base + j] = j < cnt ? o + j : -1;
    if (threadIdx.x == 0) {
        poff[e] = base;
        if (e == E - 1) poff[E] = base + padded;
    }
}

// dst[c, j] = src[row(j), c] for the columns j < ncols (ncols_dev when given, else
// ncols), with row(j) = map[j] (or j when map is null and j < nsrc), and 0 where row(j)
// < 0 or j >= nsrc: bf16, src [*, C] rows, dst [C, ldd]. 64 x 64 tiles through shared
// memory; C and the column tiles multiples of 16 and 64.
__global__ void __launch_bounds__(256) transpose_kernel(const __nv_bfloat16* src, int C, const int32_t* map, int nsrc,
                                                        int ncols, const int32_t* ncols_dev, __nv_bfloat16* dst,
                                                        long ldd) {
    __shared__ __nv_bfloat16 tile[64][64 + 8];
    const int j0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
    const int nc = ncols_dev ? *ncols_dev : ncols;
    if (j0 >= nc) return;
    {  // read: column j0 + tid/4 (a source row), 16 channels from c0 + (tid%4)*16
        const int jj = threadIdx.x >> 2, cc = (threadIdx.x & 3) * 16;
        const int j = j0 + jj;
        int row = -1;
        if (j < nc) row = map ? map[j] : (j < nsrc ? j : -1);
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        if (row >= 0 && c0 + cc < C) {
            const uint4* sp = reinterpret_cast<const uint4*>(src + (size_t)row * C + c0 + cc);
            a = sp[0];
            b = sp[1];
        }
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            tile[cc + 2 * i][jj] = __ushort_as_bfloat16((unsigned short)(w[i] & 0xFFFF));
            tile[cc + 2 * i + 1][jj] = __ushort_as_bfloat16((unsigned short)(w[i] >> 16));
        }
    }
    __syncthreads();
    {  // write: row c0 + tid/4 of dst, 16 columns from j0 + (tid%4)*16
        const int c = threadIdx.x >> 2, jc = (threadIdx.x & 3) * 16;
        if (c0 + c < C) {
            const uint4* tp = reinterpret_cast<const uint4*>(&tile[c][jc]);
            uint4* dp = reinterpret_cast<uint4*>(dst + (size_t)(c0 + c) * ldd + j0 + jc);
            dp[0] = tp[0];
            dp[1] = tp[1];
        }
    }
}

// xhat[t, :] = dec(xq[t, :]) * xs[t, block] in bf16 (exact: a 3-bit significand times 2^k).
__global__ void __launch_bounds__(256) xhat_kernel(const uint8_t* xq, const float* xs, long T, int H,
                                                   __nv_bfloat16* out) {
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < T * H / 16; i += (long)gridDim.x * blockDim.x) {
        const long off = i * 16;
        const long t = off / H;
        const int h = (int)(off % H);
        uint4 lo, hi;
        e4m3x16_to_bf16(*reinterpret_cast<const uint4*>(xq + off), xs[t * (H / kBlk) + h / kBlk], lo, hi);
        reinterpret_cast<uint4*>(out + off)[0] = lo;
        reinterpret_cast<uint4*>(out + off)[1] = hi;
    }
}

// dst[r, :] = src[perm_src[r] / k, :] for the n_rows permuted rows (bf16 rows of H), a warp per row.
__global__ void __launch_bounds__(256) gather_bf16_kernel(const __nv_bfloat16* src, int H, const int32_t* perm_src,
                                                          int k, int n_rows, __nv_bfloat16* dst) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= n_rows) return;
    const int f = perm_src[r];
    const bool good = (unsigned)f < (unsigned)n_rows;  // else a row no valid id reached: zeros
    const uint4* s4 = reinterpret_cast<const uint4*>(src + (size_t)(good ? f / k : 0) * H);
    uint4* d4 = reinterpret_cast<uint4*>(dst + (size_t)r * H);
    for (int c = lane; c < H / 8; c += 32) d4[c] = good ? __ldg(s4 + c) : make_uint4(0, 0, 0, 0);
}

// dst [C, R] bf16 = src [R, C] fp32 transposed (the router weights as the K-contiguous
// operand of dx's router term: K = E), 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) f32_to_bf16_t_kernel(const float* src, int R, int C, __nv_bfloat16* dst) {
    __shared__ float tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int i = ty; i < 32; i += 8)
        if (r0 + i < R && c0 + tx < C) tile[i][tx] = src[(size_t)(r0 + i) * C + c0 + tx];
    __syncthreads();
    for (int i = ty; i < 32; i += 8)
        if (c0 + i < C && r0 + tx < R) dst[(size_t)(c0 + i) * R + r0 + tx] = __float2bfloat16_rn(tile[tx][i]);
}

// SwiGLU backward and the quantised intermediate, one warp per row (routed rows or
// tokens): ahat = the forward's FP8 intermediate (same arithmetic as its epilogue),
// dw = <dau, ahat> (routed rows: written at the row's (token, slot) index),
// dgu = [dg | du] with da = w dau, and wahat = w ahat in bf16 (the operand of the down
// weight gradient, which then reads dout rows as they are).
struct SwigluBwd {
    int rows, Iw, routed;
    const float *g, *u, *dau;
    const int32_t* perm_src;
    const float* topk_w;
    __nv_bfloat16* wahat;  // [rows, Iw]
    __nv_bfloat16* dgu;    // [rows, 2 Iw]
    float* dw;            // [T k]
};

__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const SwigluBwd p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + warp;
    if (r >= p.rows) return;
    const int f = p.routed ? p.perm_src[r] : 0;
    const bool good = !p.routed || (unsigned)f < (unsigned)p.rows;  // rows no valid id reached: weight 0
    const float w = p.routed ? (good ? p.topk_w[f] : 0.f) : 1.f;
    const size_t base = (size_t)r * p.Iw;
    float dw = 0.f;
    for (int b = 0; b < p.Iw; b += kBlk) {
        const int i = b + 4 * lane;
        const float4 g4 = *reinterpret_cast<const float4*>(p.g + base + i);
        const float4 u4 = *reinterpret_cast<const float4*>(p.u + base + i);
        const float4 d4 = *reinterpret_cast<const float4*>(p.dau + base + i);
        const float g[4] = {g4.x, g4.y, g4.z, g4.w}, u[4] = {u4.x, u4.y, u4.z, u4.w};
        const float d[4] = {d4.x, d4.y, d4.z, d4.w};
        float a[4], amax = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            a[q] = silu_mul(g[q], u[q]);
            amax = fmaxf(amax, fabsf(a[q]));
        }
        amax = warp_max(amax);
        float inv;
        const float scale = act_scale_pow2(amax, &inv);
        const uint32_t code = pack_e4m3x4(a[0] * inv, a[1] * inv, a[2] * inv, a[3] * inv);
        const float2 c01 = __half22float2(
            __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(code & 0xFFFF), __NV_E4M3)));
        const float2 c23 = __half22float2(
            __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(code >> 16), __NV_E4M3)));
        const float ah[4] = {c01.x * scale, c01.y * scale, c23.x * scale, c23.y * scale};
        float dg[4], du[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            dw = fmaf(d[q], ah[q], dw);
            const float da = w * d[q];
            const float sg = 1.f / (1.f + expf(-g[q]));
            dg[q] = da * u[q] * sg * (1.f + g[q] * (1.f - sg));
            du[q] = da * g[q] * sg;
        }
        *reinterpret_cast<uint2*>(p.wahat + base + i) =
            make_uint2(pack_bf16x2(w * ah[0], w * ah[1]), pack_bf16x2(w * ah[2], w * ah[3]));
        __nv_bfloat16* drow = p.dgu + (size_t)r * 2 * p.Iw;
        *reinterpret_cast<uint2*>(drow + i) = make_uint2(pack_bf16x2(dg[0], dg[1]), pack_bf16x2(dg[2], dg[3]));
        *reinterpret_cast<uint2*>(drow + p.Iw + i) =
            make_uint2(pack_bf16x2(du[0], du[1]), pack_bf16x2(du[2], du[3]));
    }
    dw = warp_sum(dw);
    if (p.routed && good && lane == 0) p.dw[f] = dw;
}

// Router backward, one warp per token: the forward's logits (split-K partials summed in
// the same fixed order as its top-k, plus the bias), softmax over all E, dp from the
// kept experts' dw, dlogit = p (dp - <p, dp>).
struct RouterBwd {
    int T, E, k, splits;
    float scale;
    const float* part;  // [splits, T, E]
    const float* bias;
    const int32_t* ids;
    const float* dw;    // [T k]
    float* dlogit;      // [T, E]
    __nv_bfloat16* dlogit_bf;  // [T, E], the GEMMs' operand
};

__global__ void __launch_bounds__(256) router_bwd_kernel(const RouterBwd p) {
    constexpr int kPer = 8;  // E <= 256
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= p.T) return;
    float l[kPer], dp[kPer];
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int e = lane + 32 * q;
        l[q] = -INFINITY;
        dp[q] = 0.f;
        if (e < p.E) {
            float v = 0.f;
            for (int s = 0; s < p.splits; ++s) v += p.part[((size_t)s * p.T + t) * p.E + e];
            if (p.bias) v += p.bias[e];
            l[q] = v;
            mx = fmaxf(mx, v);
        }
    }
    mx = warp_max(mx);
    float z = 0.f;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        l[q] = (lane + 32 * q < p.E) ? expf(l[q] - mx) : 0.f;
        z += l[q];
    }
    z = warp_sum(z);
    for (int j = 0; j < p.k; ++j) {
        const int e = p.ids[(size_t)t * p.k + j];
        const float v = p.scale * p.dw[(size_t)t * p.k + j];
#pragma unroll
        for (int q = 0; q < kPer; ++q)
            if (lane + 32 * q == e) dp[q] += v;
    }
    float pdp = 0.f;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        l[q] /= z;  // p
        pdp += l[q] * dp[q];
    }
    pdp = warp_sum(pdp);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int e = lane + 32 * q;
        if (e < p.E) {
            const float v = l[q] * (dp[q] - pdp);
            p.dlogit[(size_t)t * p.E + e] = v;
            p.dlogit_bf[(size_t)t * p.E + e] = __float2bfloat16_rn(v);
        }
    }
}

// dbias[e] = sum over tokens of dlogit[t, e]: 32 experts per block, 32 token slices
// (t = slice, slice + 32, ...) summed in slice order, so the result is deterministic.
__global__ void __launch_bounds__(1024) dbias_kernel(int T, int E, const float* dlogit, float* dbias) {
    __shared__ float part[32][33];
    const int le = threadIdx.x & 31, ts = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + le;
    float s = 0.f;
    if (e < E)
        for (int t = ts; t < T; t += 32) s += dlogit[(size_t)t * E + e];
    part[ts][le] = s;
    __syncthreads();
    if (ts == 0 && e < E) {
        float tot = 0.f;
        for (int i = 0; i < 32; ++i) tot += part[i][le];
        dbias[e] = tot;
    }
}

// dx[t, :] += sum_j dx_perm[inv_pos[t k + j], :] + dx_s[t, :], four channels per thread.
__global__ void __launch_bounds__(256) dx_combine_kernel(int T, int H, int k, const int32_t* inv_pos,
                                                         const float* dx_perm, const float* dx_s, float* dx) {
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    const long n4 = (long)T * (H / 4);
    if (i >= n4) return;
    const int t = (int)(i / (H / 4)), h = (int)(i % (H / 4)) * 4;
    float4 acc = *reinterpret_cast<const float4*>(dx + (size_t)t * H + h);
    for (int j = 0; j < k; ++j) {
        const int pos = inv_pos[(size_t)t * k + j];
        if ((unsigned)pos >= (unsigned)(T * k)) continue;  // an invalid id: no row (status reported)
        const float4 v = *reinterpret_cast<const float4*>(dx_perm + (size_t)pos * H + h);
        acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
    }
    if (dx_s) {
        const float4 v = *reinterpret_cast<const float4*>(dx_s + (size_t)t * H + h);
        acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
    }
    *reinterpret_cast<float4*>(dx + (size_t)t * H + h) = acc;
}

unsigned cdiv(long a, long b) { return (unsigned)((a + b - 1) / b); }
unsigned grid_for(long n, int per_thread) { return (unsigned)std::min<long>(4096, std::max<long>(1, cdiv(n / per_thread, 256))); }

}  // namespace

BwdLayout bwd_layout(const moe_config_t& c, int64_t T) {
    BwdLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    };
    const size_t H = c.hidden, I = c.moe_inter, E = c.n_routed, k = c.top_k, t = (size_t)T;
    const size_t Is = (size_t)c.n_shared * c.moe_inter, R = t * k;
    L.splits = router_splits_for(c, T);
    L.max_mtiles = (int)((R + 127) / 128 + std::min(E, R));
    L.ctrl = take(kCtrlRegionBytes);
    L.logits = take((size_t)L.splits * t * E * 4);
    L.router_w3 = take(router_w3_bytes(c));
    L.ids = take(R * 4);
    L.w = take(R * 4);
    L.xq = take(t * H);
    L.xs = take(t * (H / 128) * 4);
    L.offsets = take((E + 1) * 4);
    L.perm_src = take(R * 4);
    L.inv_pos = take(R * 4);
    L.perm_hist = take((size_t)permute_segments((int64_t)R) * E * 4);
    L.mtiles = take((size_t)L.max_mtiles * sizeof(MTile));
    L.xq_perm = take(R * H);
    L.g_r = take(R * I * 4);
    L.u_r = take(R * I * 4);
    L.dau_r = take(R * I * 4);
    L.wahat_r = take(R * I * 2);
    L.dgu_r = take(R * 2 * I * 2);
    L.dx_perm = take(R * H * 4);
    L.g_s = take(t * Is * 4);
    L.u_s = take(t * Is * 4);
    L.dau_s = take(t * Is * 4);
    L.wahat_s = take(t * Is * 2);
    L.dgu_s = take(t * 2 * Is * 2);
    L.dx_s = take(t * H * 4);
    L.dw = take(R * 4);
    L.dlogit = take(t * E * 4);
    L.dlogit_bf = take(t * E * 2);
    L.wdT = take(E * I * H * 2);
    L.wguT = take(E * H * 2 * I * 2);
    L.wsdT = take(Is * H * 2);
    L.wsguT = take(H * 2 * Is * 2);
    L.wr_bf = take(E * H * 2);
    L.xhat = take(t * H * 2);
    L.xhat_perm = take(R * H * 2);
    L.dout_perm = take(R * H * 2);
    // the weight gradients' transposed operands: routed rows in padded expert segments
    // (Rp columns), tokens padded to Tp
    L.Rp = (int)(((R + 63) & ~size_t(63)) + 64 * E);
    L.Tp = (int)((t + 63) & ~size_t(63));
    const size_t Rp = (size_t)L.Rp, Tp = (size_t)L.Tp;
    L.poff = take((E + 1) * 4);
    L.pmap = take(Rp * 4);
    L.dout_permT = take(H * Rp * 2);
    L.wahatT = take(I * Rp * 2);
    L.dguT = take(2 * I * Rp * 2);
    L.xhat_permT = take(H * Rp * 2);
    L.doutT = take(H * Tp * 2);
    L.wahat_sT = take(Is * Tp * 2);
    L.dgu_sT = take(2 * Is * Tp * 2);
    L.xhatT = take(H * Tp * 2);
    L.dlogitT = take(E * Tp * 2);
    L.xT = take(H * Tp * 2);
    L.total = off;
    return L;
}

// The backward's launches (one stream, in order); shapes and pointers checked by the caller.
cudaError_t launch_backward(const moe_config_t& c, const BwdArgs& a, void* ws, cudaStream_t st) {
    const int T = a.T, H = c.hidden, I = c.moe_inter, E = c.n_routed, k = c.top_k;
    const int Is = c.n_shared * c.moe_inter;
    const bool sh = Is > 0;
    const int R = T * k;
    const BwdLayout L = bwd_layout(c, T);
    auto at = [&](size_t o) { return static_cast<uint8_t*>(ws) + o; };
    auto bf = [&](size_t o) { return reinterpret_cast<__nv_bfloat16*>(at(o)); };
    auto f32 = [&](size_t o) { return reinterpret_cast<float*>(at(o)); };
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(at(L.ctrl));
    int32_t* perm_src = reinterpret_cast<int32_t*>(at(L.perm_src));
    int32_t* inv_pos = reinterpret_cast<int32_t*>(at(L.inv_pos));
    MTile* mtiles = reinterpret_cast<MTile*>(at(L.mtiles));
    uint8_t* xq = at(L.xq);
    float* xs = f32(L.xs);
    const __nv_bfloat16* dout = static_cast<const __nv_bfloat16*>(a.dout);
    cudaError_t e;
#define BWD_TRY(x)                             \
    do {                                       \
        if ((e = (x)) != cudaSuccess) return e; \
    } while (0)
    // optional events around the parts (slots of moe_stage_events_t, see moe.h)
    auto mark = [&](int slot, bool begin) -> cudaError_t {
        void* ev = a.ev ? (begin ? a.ev->start[slot] : a.ev->stop[slot]) : nullptr;
        return ev ? cudaEventRecord((cudaEvent_t)ev, st) : cudaSuccess;
    };
    BWD_TRY(mark(MOE_STAGE_ROUTE, true));

    // ---- forward quantities: activation codes, the router's logits, the permutation, g and u
    BWD_TRY(launch_quant_act(a.x, T, H, xq, xs, NormArgs{}, st));
    BWD_TRY(launch_route_large(c, a.x, T, a.W->w_router, a.W->router_bias, reinterpret_cast<int32_t*>(at(L.ids)),
                               f32(L.w), f32(L.logits), L.splits, reinterpret_cast<uint16_t*>(at(L.router_w3)),
                               &ctrl->status, st));
    BWD_TRY(launch_permute(c, a.topk_ids, T, reinterpret_cast<int32_t*>(at(L.offsets)), perm_src, inv_pos, nullptr,
                           nullptr, mtiles, reinterpret_cast<int32_t*>(at(L.perm_hist)), ctrl, st));
    BWD_TRY(launch_gather_rows(T, H, k, perm_src, xq, at(L.xq_perm), &ctrl->status, st));
    {
        GemmArgs g = {};
        g.mode = 2;
        g.H = H;
        g.I = I;
        g.Is = Is;
        g.T = T;
        g.k = k;
        g.K_r = g.K_s = H;
        g.nt_r = I / 128;
        g.nt_s = Is / 128;
        g.n_mt_s = sh ? (T + 127) / 128 : 0;
        g.ctrl = ctrl;
        g.mtiles = mtiles;
        g.perm_src = perm_src;
        g.topk_w = a.topk_w;
        g.xs = xs;
        g.s_gate = a.W->s_gate;
        g.s_up = a.W->s_up;
        g.ss_gate = a.W->ss_gate;
        g.ss_up = a.W->ss_up;
        g.g_out_r = f32(L.g_r);
        g.u_out_r = f32(L.u_r);
        g.g_out_s = f32(L.g_s);
        g.u_out_s = f32(L.u_s);
        g.status = &ctrl->status;
        TmaMaps m = {};
        if (!tmap_u8_2d(&m.a_r, at(L.xq_perm), (uint64_t)R, H, 128, 128) ||
            !tmap_u8_2d(&m.b0_r, a.W->w_gate, (uint64_t)E * I, H, 128, 128) ||
            !tmap_u8_2d(&m.b1_r, a.W->w_up, (uint64_t)E * I, H, 128, 128))
            return cudaErrorInvalidValue;
        if (sh && (!tmap_u8_2d(&m.a_s, xq, T, H, 128, 128) || !tmap_u8_2d(&m.b0_s, a.W->ws_gate, Is, H, 128, 128) ||
                   !tmap_u8_2d(&m.b1_s, a.W->ws_up, Is, H, 128, 128)))
            return cudaErrorInvalidValue;
        BWD_TRY(launch_expert_gemm(g, m, st));
    }
    // ---- bf16 operands of the contractions: weights dequantised, xhat, gathered rows
    // weights, dequantised and transposed for the tcgen05 dgrad (K contiguous):
    //   WdT [E][I][H] (dau = dout Wd), WguT [E][H][2I] ([Wg; Wu] stacked along K for dx)
    dequant_t_kernel<<<dim3(I / 64, H / 64, E), 256, 0, st>>>(a.W->w_down, a.W->s_down, H, I, H, 0, bf(L.wdT));
    dequant_t_kernel<<<dim3(H / 64, I / 64, E), 256, 0, st>>>(a.W->w_gate, a.W->s_gate, I, H, 2 * I, 0, bf(L.wguT));
    dequant_t_kernel<<<dim3(H / 64, I / 64, E), 256, 0, st>>>(a.W->w_up, a.W->s_up, I, H, 2 * I, I, bf(L.wguT));
    if (sh) {
        dequant_t_kernel<<<dim3(Is / 64, H / 64, 1), 256, 0, st>>>(a.W->ws_down, a.W->ss_down, H, Is, H, 0,
                                                                 bf(L.wsdT));
        dequant_t_kernel<<<dim3(H / 64, Is / 64, 1), 256, 0, st>>>(a.W->ws_gate, a.W->ss_gate, Is, H, 2 * Is, 0,
                                                                 bf(L.wsguT));
        dequant_t_kernel<<<dim3(H / 64, Is / 64, 1), 256, 0, st>>>(a.W->ws_up, a.W->ss_up, Is, H, 2 * Is, Is,
                                                                 bf(L.wsguT));
    }
    f32_to_bf16_t_kernel<<<dim3(cdiv(H, 32), cdiv(E, 32)), 256, 0, st>>>(a.W->w_router, E, H, bf(L.wr_bf));
    xhat_kernel<<<grid_for((long)T * H, 16), 256, 0, st>>>(xq, xs, T, H, bf(L.xhat));
    gather_bf16_kernel<<<cdiv(R, 8), 256, 0, st>>>(bf(L.xhat), H, perm_src, k, R, bf(L.xhat_perm));
    gather_bf16_kernel<<<cdiv(R, 8), 256, 0, st>>>(dout, H, perm_src, k, R, bf(L.dout_perm));
    BWD_TRY(cudaGetLastError());
    BWD_TRY(mark(MOE_STAGE_ROUTE, false));
    BWD_TRY(mark(MOE_STAGE_PERMUTE, true));

    // ---- dau = Wd^T dout: routed rows (tiles of the permutation), then the shared experts
    BWD_TRY(launch_bwd_tc(bf(L.dout_perm), (uint64_t)R, bf(L.wdT), (uint64_t)E, H, I, 1, 0, mtiles, ctrl,
                          f32(L.dau_r), &ctrl->status, st));
    if (sh)
        BWD_TRY(launch_bwd_tc(dout, (uint64_t)T, bf(L.wsdT), 1, H, Is, 0, T, mtiles, ctrl, f32(L.dau_s),
                              &ctrl->status, st));
    // ---- SwiGLU backward: w ahat, dgu, dw
    {
        SwigluBwd s;
        s.rows = R;
        s.Iw = I;
        s.routed = 1;
        s.g = f32(L.g_r);
        s.u = f32(L.u_r);
        s.dau = f32(L.dau_r);
        s.perm_src = perm_src;
        s.topk_w = a.topk_w;
        s.wahat = bf(L.wahat_r);
        s.dgu = bf(L.dgu_r);
        s.dw = f32(L.dw);
        swiglu_bwd_kernel<<<cdiv(s.rows, 8), 256, 0, st>>>(s);
        BWD_TRY(cudaGetLastError());
        if (sh) {
            s.rows = T;
            s.Iw = Is;
            s.routed = 0;
            s.g = f32(L.g_s);
            s.u = f32(L.u_s);
            s.dau = f32(L.dau_s);
            s.wahat = bf(L.wahat_s);
            s.dgu = bf(L.dgu_s);
            swiglu_bwd_kernel<<<cdiv(s.rows, 8), 256, 0, st>>>(s);
            BWD_TRY(cudaGetLastError());
        }
    }
    // ---- router: dlogit, dbias
    {
        RouterBwd r;
        r.T = T;
        r.E = E;
        r.k = k;
        r.splits = L.splits;
        r.scale = c.routed_scaling_factor;
        r.part = f32(L.logits);
        r.bias = a.W->router_bias;
        r.ids = a.topk_ids;
        r.dw = f32(L.dw);
        r.dlogit = f32(L.dlogit);
        r.dlogit_bf = bf(L.dlogit_bf);
        router_bwd_kernel<<<cdiv(T, 8), 256, 0, st>>>(r);
        BWD_TRY(cudaGetLastError());
        if (a.dbias) {
            dbias_kernel<<<cdiv(E, 32), 1024, 0, st>>>(T, E, f32(L.dlogit), a.dbias);
            BWD_TRY(cudaGetLastError());
        }
    }
    BWD_TRY(mark(MOE_STAGE_PERMUTE, false));
    // ---- dx: router term, then the routed rows and the shared experts, then their sum
    {
        BWD_TRY(mark(MOE_STAGE_COMBINE, true));
        // dx = dlogit [T, E] . Wr: K = E in 64-wide steps (columns past E read as zeros)
        BWD_TRY(launch_bwd_tc_wgrad(bf(L.dlogit_bf), T, bf(L.wr_bf), H, (uint64_t)E, nullptr, 1, (E + 63) / 64 * 64,
                                    a.dx, nullptr, 0, 0, &ctrl->status, st));
        BWD_TRY(launch_bwd_tc(bf(L.dgu_r), (uint64_t)R, bf(L.wguT), (uint64_t)E, 2 * I, H, 1, 0, mtiles, ctrl,
                              f32(L.dx_perm), &ctrl->status, st));
        if (sh)
            BWD_TRY(launch_bwd_tc(bf(L.dgu_s), (uint64_t)T, bf(L.wsguT), 1, 2 * Is, H, 0, T, mtiles, ctrl,
                                  f32(L.dx_s), &ctrl->status, st));
        const long n4 = (long)T * (H / 4);
        dx_combine_kernel<<<cdiv(n4, 256), 256, 0, st>>>(T, H, k, inv_pos, f32(L.dx_perm), sh ? f32(L.dx_s) : nullptr,
                                                        a.dx);
        BWD_TRY(cudaGetLastError());
        BWD_TRY(mark(MOE_STAGE_COMBINE, false));
    }
    // ---- weight gradients on the tcgen05 tensor cores: dWd_e = dout_perm^T (w ahat),
    // [dWg_e; dWu_e] = [dg | du]^T xhat_perm (routed, per expert over its padded columns),
    // the same over tokens for the shared experts, and dWr = dlogit^T x
    BWD_TRY(mark(MOE_STAGE_DOWN, true));
    {
        int32_t* poff = reinterpret_cast<int32_t*>(at(L.poff));
        int32_t* pmap = reinterpret_cast<int32_t*>(at(L.pmap));
        pad_map_kernel<<<E, 256, 0, st>>>(E, reinterpret_cast<int32_t*>(at(L.offsets)), poff, pmap);
        const long Rp = L.Rp, Tp = L.Tp;
        auto tr = [&](const __nv_bfloat16* src, int C, const int32_t* map, int nsrc, int ncols, const int32_t* ncd,
                      size_t dst, long ldd) {
            transpose_kernel<<<dim3(cdiv(ldd, 64), cdiv(C, 64)), 256, 0, st>>>(src, C, map, nsrc, ncols, ncd, bf(dst),
                                                                                ldd);
        };
        const int32_t* nc_r = poff + E;  // the routed columns in use
        tr(bf(L.dout_perm), H, pmap, R, 0, nc_r, L.dout_permT, Rp);
        tr(bf(L.wahat_r), I, pmap, R, 0, nc_r, L.wahatT, Rp);
        tr(bf(L.dgu_r), 2 * I, pmap, R, 0, nc_r, L.dguT, Rp);
        tr(bf(L.xhat_perm), H, pmap, R, 0, nc_r, L.xhat_permT, Rp);
        BWD_TRY(cudaGetLastError());
        BWD_TRY(launch_bwd_tc_wgrad(bf(L.dout_permT), H, bf(L.wahatT), I, (uint64_t)Rp, poff, E, 0, a.dw_down,
                                    nullptr, 0, (size_t)H * I, &ctrl->status, st));
        BWD_TRY(mark(MOE_STAGE_GATE_UP, true));
        BWD_TRY(launch_bwd_tc_wgrad(bf(L.dguT), 2 * I, bf(L.xhat_permT), H, (uint64_t)Rp, poff, E, 0, a.dw_gate,
                                    a.dw_up, I, (size_t)I * H, &ctrl->status, st));
        BWD_TRY(mark(MOE_STAGE_GATE_UP, false));
        if (sh) {
            tr(dout, H, nullptr, T, (int)Tp, nullptr, L.doutT, Tp);
            tr(bf(L.wahat_s), Is, nullptr, T, (int)Tp, nullptr, L.wahat_sT, Tp);
            tr(bf(L.dgu_s), 2 * Is, nullptr, T, (int)Tp, nullptr, L.dgu_sT, Tp);
            tr(bf(L.xhat), H, nullptr, T, (int)Tp, nullptr, L.xhatT, Tp);
            BWD_TRY(cudaGetLastError());
            BWD_TRY(launch_bwd_tc_wgrad(bf(L.doutT), H, bf(L.wahat_sT), Is, (uint64_t)Tp, nullptr, 1, (int)Tp,
                                        a.dws_down, nullptr, 0, 0, &ctrl->status, st));
            BWD_TRY(launch_bwd_tc_wgrad(bf(L.dgu_sT), 2 * Is, bf(L.xhatT), H, (uint64_t)Tp, nullptr, 1, (int)Tp,
                                        a.dws_gate, a.dws_up, Is, 0, &ctrl->status, st));
        }
        tr(bf(L.dlogit_bf), E, nullptr, T, (int)Tp, nullptr, L.dlogitT, Tp);
        tr(static_cast<const __nv_bfloat16*>(a.x), H, nullptr, T, (int)Tp, nullptr, L.xT, Tp);
        BWD_TRY(cudaGetLastError());
        BWD_TRY(launch_bwd_tc_wgrad(bf(L.dlogitT), E, bf(L.xT), H, (uint64_t)Tp, nullptr, 1, (int)Tp, a.dw_router,
                                    nullptr, 0, 0, &ctrl->status, st));
    }
    BWD_TRY(mark(MOE_STAGE_DOWN, false));
#undef BWD_TRY
    return cudaSuccess;
}

}  // namespace moe
