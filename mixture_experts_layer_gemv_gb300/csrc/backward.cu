// The layer's backward: gradients of sum(dout * out) with the forward's expert choice
// held fixed (the Mixture-of-Kittens page's training workload, Table 1 "Backward";
// "expert FFNs" forward and backward). The FP8 quantisers are straight-through and the
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
// accumulation on the mma.sync tensor path: one grouped GEMM kernel, specialised per
// operand access pattern, with the FP8 weights and activations decoded to bf16 (exact
// for activations, one bf16 rounding for weight x block scale) while they are staged
// in shared memory.
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kBM = 128, kBN = 128, kBK = 32;
constexpr int kAPitch = kBK + 8;  // bf16 per A row in shared memory (k contiguous)
constexpr int kATPitch = kBM + 8; // bf16 per A row of the transposed layout (m contiguous, one row per k)
constexpr int kBPitch = kBN + 8;  // bf16 per B row in shared memory (n contiguous)
constexpr int kGThr = 256;        // 8 warps: 2 along M (64 rows) x 4 along N (32 columns)

// The contractions (F_*) and how each reads its operands; C is fp32 [M, N] per group.
enum : int {
    F_DDOWN = 0,  // dau[r, i]   = sum_h dout[tok r, h] Wd_e[h, i]          rows r of a tile, K = H
    F_DGU = 1,    // dx_r[r, h]  = sum_i dgu[r, i] [Wg_e; Wu_e][i, h]       rows r of a tile, K = 2 Iw
    F_DXR = 2,    // dx[t, h]    = sum_e dlogit[t, e] Wr[e, h]              K = E
    F_WDOWN = 3,  // dWd_e[h, i] = sum_r w_r dout[tok r, h] ahat[r, i]      K = rows of e
    F_WGU = 4,    // [dWg_e; dWu_e][i, h] = sum_r dgu[r, i] xhat[tok r, h]  K = rows of e
    F_WR = 5,     // dWr[e, h]   = sum_t dlogit[t, e] x[t, h]               K = T
};

struct BwdGemm {
    int M, N, K;       // output extent; K of single-group problems
    int T, k, E;
    int Iw;            // intermediate width of the experts involved (I routed, Is shared)
    int H;
    int routed;        // rows are permuted rows (token via perm_src) or tokens
    const int32_t* perm_src;
    const MTile* mtiles;
    const Ctrl* ctrl;
    const int32_t* offsets;  // per-expert row ranges (wgrad of routed experts)
    int grouping;            // 0: one group; 1: the permutation's 128-row tiles; 2: per expert
    const __nv_bfloat16* dout;  // [T, H]
    const __nv_bfloat16* dgu;   // [rows, 2 Iw]
    const __nv_bfloat16* ahat;  // [rows, Iw]
    const float* topk_w;        // [T k] routing weights
    const float* dlogit;        // [T, E]
    const __nv_bfloat16* x;     // [T, H]
    const uint8_t* xq;          // [T, H] e4m3
    const float* xs;            // [T, H / 128]
    const uint8_t *w0, *w1;     // FP8 weights: w1 stacked under w0 along K (F_DGU)
    const float *s0, *s1;       // their block scales
    size_t w_estride, s_estride;  // per-expert strides (elements) of w0/w1 and s0/s1
    const float* wr;              // [E, H]
    float *c0, *c1;             // outputs; F_WGU rows >= Iw go to c1
    size_t c_estride;           // per-expert stride of c0/c1 (elements)
};

__device__ __forceinline__ int tok_of(const BwdGemm& p, int r) { return p.routed ? p.perm_src[r] / p.k : r; }

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

__device__ __forceinline__ void f32x16_to_bf16(const float* v, float mul, uint4& lo, uint4& hi) {
    lo = make_uint4(pack_bf16x2(v[0] * mul, v[1] * mul), pack_bf16x2(v[2] * mul, v[3] * mul),
                    pack_bf16x2(v[4] * mul, v[5] * mul), pack_bf16x2(v[6] * mul, v[7] * mul));
    hi = make_uint4(pack_bf16x2(v[8] * mul, v[9] * mul), pack_bf16x2(v[10] * mul, v[11] * mul),
                    pack_bf16x2(v[12] * mul, v[13] * mul), pack_bf16x2(v[14] * mul, v[15] * mul));
}

__device__ __forceinline__ void bf16x16_scaled(uint4 a, uint4 b, float mul, uint4& lo, uint4& hi) {
    if (mul == 1.f) {
        lo = a;
        hi = b;
        return;
    }
    float v[16];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    f32x16_to_bf16(v, mul, lo, hi);
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One 128 x 128 output tile of one group. A tile element (m, kk) and B tile element
// (kk, n) are read as 16 contiguous values per thread and staged as bf16: B as [k][n],
// A as [m][k] when its rows run along k (dgrad) and as [k][m] when they run along m
// (wgrad), two buffers each; fragments come from ldmatrix (.trans for the [k][*] ones).
template <int F>
__global__ void __launch_bounds__(kGThr) bwd_gemm_kernel(const BwdGemm p) {
    static_assert(kBM * kAPitch >= kBK * kATPitch, "one A buffer holds either layout");
    __shared__ __align__(16) __nv_bfloat16 A_s[2][kBM * kAPitch];
    __shared__ __align__(16) __nv_bfloat16 B_s[2][kBK * kBPitch];
    constexpr bool a_cols = F >= F_WDOWN;  // A(m, kk) contiguous along m (its rows are the K index)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- the group: output rows [m0, m0 + mv), columns [n0, N), K range [k0, k0 + kv)
    int e = 0, m0, mv, n0 = blockIdx.y * kBN, k0 = 0, kv = p.K, row0 = 0;
    if (p.grouping == 1) {  // a 128-row tile of the permutation (rows r = row0 + m)
        if ((int)blockIdx.x >= p.ctrl->n_mtiles) return;
        const MTile t = p.mtiles[blockIdx.x];
        e = t.expert;
        row0 = t.row0;
        m0 = 0;
        mv = t.nrows;
    } else {
        m0 = blockIdx.x * kBM;
        mv = min(kBM, p.M - m0);
        if (a_cols) {  // wgrad: M, N tiles on x, y, the group on z
            m0 = blockIdx.y * kBM;
            mv = min(kBM, p.M - m0);
            n0 = blockIdx.x * kBN;
        }
        if (p.grouping == 2) {
            e = blockIdx.z;
            k0 = p.offsets[e];
            kv = p.offsets[e + 1] - k0;
        }
    }
    if (mv <= 0 || n0 >= p.N) return;

    // ---- loader coordinates: 16 contiguous values per thread
    // A rows mode: m = tid / 2, k chunk (tid % 2) * 16; A cols mode: kk = tid / 8, m chunk (tid % 8) * 16
    // B: kk = tid / 8, n chunk (tid % 8) * 16
    const int am = a_cols ? (tid & 7) * 16 : tid >> 1;
    const int ak = a_cols ? tid >> 3 : (tid & 1) * 16;
    const int bk = tid >> 3, bn = (tid & 7) * 16;

    // A rows mode: the source row of this thread's m (fixed over the K loop)
    const __nv_bfloat16* arow_b = nullptr;
    const float* arow_f = nullptr;
    if (!a_cols && am < mv) {
        if (F == F_DDOWN) arow_b = p.dout + (size_t)tok_of(p, row0 + m0 + am) * p.H;
        if (F == F_DGU) arow_b = p.dgu + (size_t)(row0 + m0 + am) * (2 * p.Iw);
        if (F == F_DXR) arow_f = p.dlogit + (size_t)(m0 + am) * p.E;
    }
    const uint8_t* wq0 = p.w0 ? p.w0 + (size_t)e * p.w_estride : nullptr;
    const uint8_t* wq1 = p.w1 ? p.w1 + (size_t)e * p.w_estride : nullptr;
    const float* ws0 = p.s0 ? p.s0 + (size_t)e * p.s_estride : nullptr;
    const float* ws1 = p.s1 ? p.s1 + (size_t)e * p.s_estride : nullptr;

    uint4 ra0, ra1, rb0, rb1;  // staged bf16 (16 values each for A and B)
    auto load = [&](int kt) {
        const int kb = kt * kBK;
        // ---------------- A
        ra0 = ra1 = make_uint4(0, 0, 0, 0);
        if (!a_cols) {
            const int kk = kb + ak;
            if (am < mv && kk < kv) {
                if (F == F_DXR) {
                    float v[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 f = __ldg(reinterpret_cast<const float4*>(arow_f + kk) + q);
                        v[4 * q] = f.x, v[4 * q + 1] = f.y, v[4 * q + 2] = f.z, v[4 * q + 3] = f.w;
                    }
                    f32x16_to_bf16(v, 1.f, ra0, ra1);
                } else {
                    ra0 = __ldg(reinterpret_cast<const uint4*>(arow_b + kk));
                    ra1 = __ldg(reinterpret_cast<const uint4*>(arow_b + kk) + 1);
                }
            }
        } else {
            const int kk = kb + ak;  // a row of the group
            const int m = m0 + am;
            if (kk < kv && m < p.M) {
                const int r = k0 + kk;
                if (F == F_WDOWN) {
                    const float wmul = p.routed ? p.topk_w[p.perm_src[r]] : 1.f;
                    const uint4* src = reinterpret_cast<const uint4*>(p.dout + (size_t)tok_of(p, r) * p.H + m);
                    bf16x16_scaled(__ldg(src), __ldg(src + 1), wmul, ra0, ra1);
                } else if (F == F_WGU) {
                    const uint4* src = reinterpret_cast<const uint4*>(p.dgu + (size_t)r * (2 * p.Iw) + m);
                    ra0 = __ldg(src);
                    ra1 = __ldg(src + 1);
                } else {  // F_WR
                    float v[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 f = __ldg(reinterpret_cast<const float4*>(p.dlogit + (size_t)r * p.E + m) + q);
                        v[4 * q] = f.x, v[4 * q + 1] = f.y, v[4 * q + 2] = f.z, v[4 * q + 3] = f.w;
                    }
                    f32x16_to_bf16(v, 1.f, ra0, ra1);
                }
            }
        }
        // ---------------- B: row kk of the K range, columns n0 + bn .. + 15
        rb0 = rb1 = make_uint4(0, 0, 0, 0);
        const int kk = kb + bk, n = n0 + bn;
        if (kk < kv && n < p.N) {
            if (F == F_DDOWN) {  // Wd_e [H, Iw]: row kk = h
                const uint4 q = __ldg(reinterpret_cast<const uint4*>(wq0 + (size_t)kk * p.N + n));
                const float s = __ldg(ws0 + (size_t)(kk / kBlk) * (p.N / kBlk) + n / kBlk);
                e4m3x16_to_bf16(q, s, rb0, rb1);
            } else if (F == F_DGU) {  // [Wg_e; Wu_e], each [Iw, H]
                const bool up = kk >= p.Iw;
                const int kr = up ? kk - p.Iw : kk;
                const uint4 q = __ldg(reinterpret_cast<const uint4*>((up ? wq1 : wq0) + (size_t)kr * p.N + n));
                const float s = __ldg((up ? ws1 : ws0) + (size_t)(kr / kBlk) * (p.N / kBlk) + n / kBlk);
                e4m3x16_to_bf16(q, s, rb0, rb1);
            } else if (F == F_DXR) {  // Wr [E, H]
                float v[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 f = __ldg(reinterpret_cast<const float4*>(p.wr + (size_t)kk * p.N + n) + q);
                    v[4 * q] = f.x, v[4 * q + 1] = f.y, v[4 * q + 2] = f.z, v[4 * q + 3] = f.w;
                }
                f32x16_to_bf16(v, 1.f, rb0, rb1);
            } else if (F == F_WDOWN) {  // ahat [rows, Iw]
                const uint4* src = reinterpret_cast<const uint4*>(p.ahat + (size_t)(k0 + kk) * p.N + n);
                rb0 = __ldg(src);
                rb1 = __ldg(src + 1);
            } else if (F == F_WGU) {  // xhat of the row's token: codes x per-128 scale (exact in bf16)
                const int t = tok_of(p, k0 + kk);
                const uint4 q = __ldg(reinterpret_cast<const uint4*>(p.xq + (size_t)t * p.N + n));
                e4m3x16_to_bf16(q, __ldg(p.xs + (size_t)t * (p.N / kBlk) + n / kBlk), rb0, rb1);
            } else {  // F_WR: x [T, H]
                const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)(k0 + kk) * p.N + n);
                rb0 = __ldg(src);
                rb1 = __ldg(src + 1);
            }
        }
    };
    auto store = [&](int buf) {
        if (!a_cols) {
            uint4* d = reinterpret_cast<uint4*>(&A_s[buf][am * kAPitch + ak]);
            d[0] = ra0;
            d[1] = ra1;
        } else {  // row kk of the [k][m] layout: 16 consecutive m
            uint4* d = reinterpret_cast<uint4*>(&A_s[buf][ak * kATPitch + am]);
            d[0] = ra0;
            d[1] = ra1;
        }
        uint4* d = reinterpret_cast<uint4*>(&B_s[buf][bk * kBPitch + bn]);
        d[0] = rb0;
        d[1] = rb1;
    };

    float acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
    const int wm = warp & 1, wn = warp >> 1;
    const int nk = (kv + kBK - 1) / kBK;
    if (nk > 0) {
        load(0);
        store(0);
    }
    __syncthreads();
    for (int kt = 0; kt < nk; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < nk) load(kt + 1);  // global loads in flight during the MMAs
#pragma unroll
        for (int ks = 0; ks < kBK; ks += 16) {
            uint32_t af[4][4], bf[2][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (a_cols)  // matrices (m 0-7 | 8-15) x (k 0-7 | 8-15) from rows k of [k][m]
                    ldsm_x4_t(af[i], &A_s[buf][(ks + (lane & 7) + ((lane >> 4) & 1) * 8) * kATPitch + wm * 64 +
                                              i * 16 + ((lane >> 3) & 1) * 8]);
                else
                    ldsm_x4(af[i], &A_s[buf][(wm * 64 + i * 16 + (lane & 15)) * kAPitch + ks + (lane >> 4) * 8]);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
                ldsm_x4_t(bf[j], &B_s[buf][(ks + (lane & 15)) * kBPitch + wn * 32 + j * 16 + (lane >> 4) * 8]);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_bf16(acc[i][j], af[i], bf[j >> 1][2 * (j & 1)], bf[j >> 1][2 * (j & 1) + 1]);
        }
        if (kt + 1 < nk) store(buf ^ 1);
        __syncthreads();
    }

    // ---- epilogue: fp32 rows of C
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int m = wm * 64 + i * 16 + (lane >> 2) + 8 * h;
            if (m >= mv) continue;
            float* crow;
            if (F == F_DDOWN || F == F_DGU) {
                crow = p.c0 + (size_t)(row0 + m0 + m) * p.N;
            } else if (F == F_WGU) {
                const int mm = m0 + m;
                crow = mm < p.Iw ? p.c0 + (size_t)e * p.c_estride + (size_t)mm * p.N
                                 : p.c1 + (size_t)e * p.c_estride + (size_t)(mm - p.Iw) * p.N;
            } else {
                crow = p.c0 + (size_t)e * p.c_estride + (size_t)(m0 + m) * p.N;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + wn * 32 + j * 8 + (lane & 3) * 2;
                if (n < p.N) *reinterpret_cast<float2*>(crow + n) = make_float2(acc[i][j][2 * h], acc[i][j][2 * h + 1]);
            }
        }
}

// SwiGLU backward and the quantised intermediate, one warp per row (routed rows or
// tokens): ahat = the forward's FP8 intermediate (same arithmetic as its epilogue),
// dw = <dau, ahat> (routed rows: written at the row's (token, slot) index), and
// dgu = [dg | du] with da = w dau.
struct SwigluBwd {
    int rows, Iw, routed;
    const float *g, *u, *dau;
    const int32_t* perm_src;
    const float* topk_w;
    __nv_bfloat16* ahat;  // [rows, Iw]
    __nv_bfloat16* dgu;   // [rows, 2 Iw]
    float* dw;            // [T k]
};

__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const SwigluBwd p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + warp;
    if (r >= p.rows) return;
    const float w = p.routed ? p.topk_w[p.perm_src[r]] : 1.f;
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
        *reinterpret_cast<uint2*>(p.ahat + base + i) = make_uint2(pack_bf16x2(ah[0], ah[1]), pack_bf16x2(ah[2], ah[3]));
        __nv_bfloat16* drow = p.dgu + (size_t)r * 2 * p.Iw;
        *reinterpret_cast<uint2*>(drow + i) = make_uint2(pack_bf16x2(dg[0], dg[1]), pack_bf16x2(dg[2], dg[3]));
        *reinterpret_cast<uint2*>(drow + p.Iw + i) =
            make_uint2(pack_bf16x2(du[0], du[1]), pack_bf16x2(du[2], du[3]));
    }
    dw = warp_sum(dw);
    if (p.routed && lane == 0) p.dw[p.perm_src[r]] = dw;
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
        if (e < p.E) p.dlogit[(size_t)t * p.E + e] = l[q] * (dp[q] - pdp);
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
        const float4 v = *reinterpret_cast<const float4*>(dx_perm + (size_t)inv_pos[(size_t)t * k + j] * H + h);
        acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
    }
    if (dx_s) {
        const float4 v = *reinterpret_cast<const float4*>(dx_s + (size_t)t * H + h);
        acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
    }
    *reinterpret_cast<float4*>(dx + (size_t)t * H + h) = acc;
}

template <int F>
cudaError_t run_gemm(const BwdGemm& p, dim3 grid, cudaStream_t st) {
    if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
    bwd_gemm_kernel<F><<<grid, kGThr, 0, st>>>(p);
    return cudaGetLastError();
}

unsigned cdiv(long a, long b) { return (unsigned)((a + b - 1) / b); }

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
    L.ahat_r = take(R * I * 2);
    L.dgu_r = take(R * 2 * I * 2);
    L.dx_perm = take(R * H * 4);
    L.g_s = take(t * Is * 4);
    L.u_s = take(t * Is * 4);
    L.dau_s = take(t * Is * 4);
    L.ahat_s = take(t * Is * 2);
    L.dgu_s = take(t * 2 * Is * 2);
    L.dx_s = take(t * H * 4);
    L.dw = take(R * 4);
    L.dlogit = take(t * E * 4);
    L.total = off;
    return L;
}

// The backward's launches (one stream, in order); shapes and pointers checked by the caller.
cudaError_t launch_backward(const moe_config_t& c, const BwdArgs& a, void* ws, cudaStream_t st) {
    const int T = a.T, H = c.hidden, I = c.moe_inter, E = c.n_routed, k = c.top_k;
    const int Is = c.n_shared * c.moe_inter;
    const bool sh = Is > 0;
    const BwdLayout L = bwd_layout(c, T);
    auto at = [&](size_t o) { return static_cast<uint8_t*>(ws) + o; };
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(at(L.ctrl));
    int32_t* perm_src = reinterpret_cast<int32_t*>(at(L.perm_src));
    int32_t* inv_pos = reinterpret_cast<int32_t*>(at(L.inv_pos));
    MTile* mtiles = reinterpret_cast<MTile*>(at(L.mtiles));
    uint8_t* xq = at(L.xq);
    float* xs = reinterpret_cast<float*>(at(L.xs));
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

    // forward quantities: activation codes, the router's logits, the permutation, g and u
    BWD_TRY(launch_quant_act(a.x, T, H, xq, xs, NormArgs{}, st));
    BWD_TRY(launch_route_large(c, a.x, T, a.W->w_router, a.W->router_bias, reinterpret_cast<int32_t*>(at(L.ids)),
                               reinterpret_cast<float*>(at(L.w)), reinterpret_cast<float*>(at(L.logits)), L.splits,
                               NormArgs{}, st));
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
        g.g_out_r = reinterpret_cast<float*>(at(L.g_r));
        g.u_out_r = reinterpret_cast<float*>(at(L.u_r));
        g.g_out_s = reinterpret_cast<float*>(at(L.g_s));
        g.u_out_s = reinterpret_cast<float*>(at(L.u_s));
        g.status = &ctrl->status;
        TmaMaps m = {};
        if (!tmap_u8_2d(&m.a_r, at(L.xq_perm), (uint64_t)T * k, H, 128, 128) ||
            !tmap_u8_2d(&m.b0_r, a.W->w_gate, (uint64_t)E * I, H, 128, 128) ||
            !tmap_u8_2d(&m.b1_r, a.W->w_up, (uint64_t)E * I, H, 128, 128))
            return cudaErrorInvalidValue;
        if (sh && (!tmap_u8_2d(&m.a_s, xq, T, H, 128, 128) || !tmap_u8_2d(&m.b0_s, a.W->ws_gate, Is, H, 128, 128) ||
                   !tmap_u8_2d(&m.b1_s, a.W->ws_up, Is, H, 128, 128)))
            return cudaErrorInvalidValue;
        BWD_TRY(launch_expert_gemm(g, m, st));
    }
    BWD_TRY(mark(MOE_STAGE_ROUTE, false));
    BWD_TRY(mark(MOE_STAGE_PERMUTE, true));

    BwdGemm b = {};
    b.T = T;
    b.k = k;
    b.E = E;
    b.H = H;
    b.perm_src = perm_src;
    b.mtiles = mtiles;
    b.ctrl = ctrl;
    b.offsets = reinterpret_cast<int32_t*>(at(L.offsets));
    b.dout = static_cast<const __nv_bfloat16*>(a.dout);
    b.topk_w = a.topk_w;
    b.x = static_cast<const __nv_bfloat16*>(a.x);
    b.xq = xq;
    b.xs = xs;
    b.wr = a.W->w_router;
    b.dlogit = reinterpret_cast<float*>(at(L.dlogit));
    const unsigned mt_grid = (unsigned)L.max_mtiles;

    // dau = Wd^T dout (routed rows, then the shared experts' tokens)
    BwdGemm d = b;
    d.routed = 1;
    d.grouping = 1;
    d.Iw = I;
    d.N = I;
    d.K = H;
    d.w0 = a.W->w_down;
    d.s0 = a.W->s_down;
    d.w_estride = (size_t)H * I;
    d.s_estride = (size_t)(H / 128) * (I / 128);
    d.c0 = reinterpret_cast<float*>(at(L.dau_r));
    BWD_TRY(run_gemm<F_DDOWN>(d, dim3(mt_grid, cdiv(I, kBN)), st));
    if (sh) {
        BwdGemm ds = b;
        ds.routed = 0;
        ds.grouping = 0;
        ds.Iw = Is;
        ds.M = T;
        ds.N = Is;
        ds.K = H;
        ds.w0 = a.W->ws_down;
        ds.s0 = a.W->ss_down;
        ds.c0 = reinterpret_cast<float*>(at(L.dau_s));
        // a single group: the tile's rows are tokens m0 + m (row0 stays 0, m0 from blockIdx.x)
        BWD_TRY(run_gemm<F_DDOWN>(ds, dim3(cdiv(T, kBM), cdiv(Is, kBN)), st));
    }
    // SwiGLU backward: ahat, dgu, dw
    {
        SwigluBwd s;
        s.rows = T * k;
        s.Iw = I;
        s.routed = 1;
        s.g = reinterpret_cast<float*>(at(L.g_r));
        s.u = reinterpret_cast<float*>(at(L.u_r));
        s.dau = reinterpret_cast<float*>(at(L.dau_r));
        s.perm_src = perm_src;
        s.topk_w = a.topk_w;
        s.ahat = reinterpret_cast<__nv_bfloat16*>(at(L.ahat_r));
        s.dgu = reinterpret_cast<__nv_bfloat16*>(at(L.dgu_r));
        s.dw = reinterpret_cast<float*>(at(L.dw));
        swiglu_bwd_kernel<<<cdiv(s.rows, 8), 256, 0, st>>>(s);
        BWD_TRY(cudaGetLastError());
        if (sh) {
            s.rows = T;
            s.Iw = Is;
            s.routed = 0;
            s.g = reinterpret_cast<float*>(at(L.g_s));
            s.u = reinterpret_cast<float*>(at(L.u_s));
            s.dau = reinterpret_cast<float*>(at(L.dau_s));
            s.ahat = reinterpret_cast<__nv_bfloat16*>(at(L.ahat_s));
            s.dgu = reinterpret_cast<__nv_bfloat16*>(at(L.dgu_s));
            swiglu_bwd_kernel<<<cdiv(s.rows, 8), 256, 0, st>>>(s);
            BWD_TRY(cudaGetLastError());
        }
    }
    // router: dlogit, dbias
    {
        RouterBwd r;
        r.T = T;
        r.E = E;
        r.k = k;
        r.splits = L.splits;
        r.scale = c.routed_scaling_factor;
        r.part = reinterpret_cast<float*>(at(L.logits));
        r.bias = a.W->router_bias;
        r.ids = a.topk_ids;
        r.dw = reinterpret_cast<float*>(at(L.dw));
        r.dlogit = reinterpret_cast<float*>(at(L.dlogit));
        router_bwd_kernel<<<cdiv(T, 8), 256, 0, st>>>(r);
        BWD_TRY(cudaGetLastError());
        if (a.dbias) {
            dbias_kernel<<<cdiv(E, 32), 1024, 0, st>>>(T, E, b.dlogit, a.dbias);
            BWD_TRY(cudaGetLastError());
        }
    }
    BWD_TRY(mark(MOE_STAGE_PERMUTE, false));
    // dx: router term, then the routed rows and the shared experts
    {
        BWD_TRY(mark(MOE_STAGE_COMBINE, true));
        BwdGemm x = b;
        x.grouping = 0;
        x.M = T;
        x.N = H;
        x.K = E;
        x.c0 = a.dx;
        BWD_TRY(run_gemm<F_DXR>(x, dim3(cdiv(T, kBM), cdiv(H, kBN)), st));
        BwdGemm g = b;
        g.routed = 1;
        g.grouping = 1;
        g.Iw = I;
        g.N = H;
        g.K = 2 * I;
        g.dgu = reinterpret_cast<__nv_bfloat16*>(at(L.dgu_r));
        g.w0 = a.W->w_gate;
        g.w1 = a.W->w_up;
        g.s0 = a.W->s_gate;
        g.s1 = a.W->s_up;
        g.w_estride = (size_t)I * H;
        g.s_estride = (size_t)(I / 128) * (H / 128);
        g.c0 = reinterpret_cast<float*>(at(L.dx_perm));
        BWD_TRY(mark(MOE_STAGE_GATE_UP, true));
        BWD_TRY(run_gemm<F_DGU>(g, dim3(mt_grid, cdiv(H, kBN)), st));
        BWD_TRY(mark(MOE_STAGE_GATE_UP, false));
        if (sh) {
            BwdGemm gs = b;
            gs.routed = 0;
            gs.grouping = 0;
            gs.Iw = Is;
            gs.M = T;
            gs.N = H;
            gs.K = 2 * Is;
            gs.dgu = reinterpret_cast<__nv_bfloat16*>(at(L.dgu_s));
            gs.w0 = a.W->ws_gate;
            gs.w1 = a.W->ws_up;
            gs.s0 = a.W->ss_gate;
            gs.s1 = a.W->ss_up;
            gs.c0 = reinterpret_cast<float*>(at(L.dx_s));
            BWD_TRY(run_gemm<F_DGU>(gs, dim3(cdiv(T, kBM), cdiv(H, kBN)), st));
        }
        const long n4 = (long)T * (H / 4);
        dx_combine_kernel<<<cdiv(n4, 256), 256, 0, st>>>(T, H, k, inv_pos, reinterpret_cast<float*>(at(L.dx_perm)),
                                                        sh ? reinterpret_cast<float*>(at(L.dx_s)) : nullptr, a.dx);
        BWD_TRY(cudaGetLastError());
        BWD_TRY(mark(MOE_STAGE_COMBINE, false));
    }
    BWD_TRY(mark(MOE_STAGE_DOWN, true));
    // weight gradients: down, gate/up (routed per expert, shared over all tokens), router
    {
        BwdGemm w = b;
        w.routed = 1;
        w.grouping = 2;
        w.Iw = I;
        w.M = H;
        w.N = I;
        w.ahat = reinterpret_cast<__nv_bfloat16*>(at(L.ahat_r));
        w.c0 = a.dw_down;
        w.c_estride = (size_t)H * I;
        BWD_TRY(run_gemm<F_WDOWN>(w, dim3(cdiv(I, kBN), cdiv(H, kBM), E), st));
        BwdGemm u = b;
        u.routed = 1;
        u.grouping = 2;
        u.Iw = I;
        u.M = 2 * I;
        u.N = H;
        u.dgu = reinterpret_cast<__nv_bfloat16*>(at(L.dgu_r));
        u.c0 = a.dw_gate;
        u.c1 = a.dw_up;
        u.c_estride = (size_t)I * H;
        BWD_TRY(run_gemm<F_WGU>(u, dim3(cdiv(H, kBN), cdiv(2 * I, kBM), E), st));
        if (sh) {
            BwdGemm ws_ = b;
            ws_.routed = 0;
            ws_.grouping = 0;
            ws_.Iw = Is;
            ws_.M = H;
            ws_.N = Is;
            ws_.K = T;
            ws_.ahat = reinterpret_cast<__nv_bfloat16*>(at(L.ahat_s));
            ws_.c0 = a.dws_down;
            BWD_TRY(run_gemm<F_WDOWN>(ws_, dim3(cdiv(Is, kBN), cdiv(H, kBM), 1), st));
            BwdGemm us = b;
            us.routed = 0;
            us.grouping = 0;
            us.Iw = Is;
            us.M = 2 * Is;
            us.N = H;
            us.K = T;
            us.dgu = reinterpret_cast<__nv_bfloat16*>(at(L.dgu_s));
            us.c0 = a.dws_gate;
            us.c1 = a.dws_up;
            BWD_TRY(run_gemm<F_WGU>(us, dim3(cdiv(H, kBN), cdiv(2 * Is, kBM), 1), st));
        }
        BwdGemm r = b;
        r.grouping = 0;
        r.M = E;
        r.N = H;
        r.K = T;
        r.c0 = a.dw_router;
        BWD_TRY(run_gemm<F_WR>(r, dim3(cdiv(H, kBN), cdiv(E, kBM), 1), st));
    }
    BWD_TRY(mark(MOE_STAGE_DOWN, false));
#undef BWD_TRY
    return cudaSuccess;
}

}  // namespace moe
