// The backward's dgrad contractions on the tcgen05 tensor cores (kind::f16: bf16 x bf16
// -> fp32 in tensor memory):
//   C[r, n] = sum_k A[r, k] * Bt_e[n, k]
// A: bf16 rows [rows, K] (K contiguous): the permuted rows of an expert (the
//    permutation's 128-row tiles) or the shared experts' tokens;
// Bt_e: the expert's weights transposed and dequantised to bf16, [N, K] (K contiguous),
//    stacked over experts as [E * N, K].
// Used for dau = Wd^T dout (K = H, N = I) and dx_r = [Wg; Wu]^T [dg | du] (K = 2I, N = H).
// The weight gradients use the same kernel with transposed operands: C_e[m, n] =
// sum_j At[m, j] Bt[n, j] over an expert's columns j (its rows, laid out with each
// expert's segment starting at a multiple of 64 and zero-padded to one, so every K block
// is whole and every TMA offset aligned): dWd_e = (dout_perm^T)(w ahat), [dWg_e; dWu_e]
// = (dgu^T)(xhat_perm), and over tokens for the shared experts and the router.
//
// Tiles of 128 rows x 256 columns; a tile's whole K accumulates in one TMEM accumulator,
// and two accumulators (512 columns) let one tile's epilogue overlap the next tile's
// MMAs. One persistent CTA of 10 warps per SM:
//   warp 9      TMA producer: per 64-wide K block (128 bytes) an A box of 128 rows and two
//               B boxes of 128 rows (128-byte swizzle), a 4-stage ring
//   warp 8      MMA issuer (one thread): per K block 4 tcgen05.mma M=128 N=256 K=16
//   warps 0-7   epilogue: warp w reads lanes 32*(w%4).. and column half w/4 of the
//               accumulator, releases it, and stores the rows in fp32 through a per-warp
//               shared-memory block, so that each store instruction writes 128-byte
//               pieces of 4 rows (the weight gradients' short K makes the stores the
//               bottleneck otherwise).
#include <algorithm>

#include "gemm_common.cuh"

namespace moe {

namespace {

constexpr int kTM = 128, kTN = 256, kTK = 64;   // tile rows, columns; bf16 per K block
constexpr int kTStages = 4;
constexpr int kTEpiWarps = 8;
constexpr int kTMmaWarp = kTEpiWarps;
constexpr int kTProdWarp = kTEpiWarps + 1;
constexpr int kTThreads = (kTEpiWarps + 2) * 32;
constexpr int kTSA = kTM * kTK * 2;             // 16 KB A box
constexpr int kTSB = kTN * kTK * 2;             // 32 KB: two B boxes of 128 rows
constexpr int kTStage = kTSA + kTSB;
constexpr uint32_t kTTmemCols = 512;            // two 128 x 256 fp32 accumulators
constexpr uint32_t kTIdesc = idesc_bf16_f32(kTM, kTN);

// mode 0: dgrad over the permutation's tiles; 1: dgrad over rows [0, rows); 2: wgrad per
// expert (K range [poff[e], poff[e+1]) of the transposed operands); 3: wgrad, one group
// with K = K (a multiple of 64).
struct TcParams {
    int mode;
    int K, N;         // dgrad: reduction length and output width (Bt_e has N rows)
    int M;            // wgrad: output rows (rows of At)
    int rows;         // dgrad mode 1: rows of A
    int groups;       // wgrad mode 2: experts
    const MTile* mtiles;
    const Ctrl* ctrl;
    const int32_t* poff;  // wgrad mode 2: [groups + 1] padded column offsets
    float *C, *C2;    // output rows >= msplit go to C2 (row - msplit); C2 == nullptr: none
    int msplit;
    long ldc;
    size_t c_estride; // per-group stride of C and C2 (wgrad)
    int* status;
};

struct TcItem {
    int row0, nrows, brow, ncol, k0, kb, e;
};

__device__ __forceinline__ TcItem tc_item(const TcParams& p, int n_mt, int nt_per, int item) {
    TcItem it;
    const int g = item / (n_mt * nt_per), rest = item % (n_mt * nt_per);
    const int mt = rest / nt_per, nt = rest % nt_per;
    it.ncol = nt * kTN;
    it.e = 0;
    it.k0 = 0;
    if (p.mode == 0) {
        const MTile m = p.mtiles[mt];
        it.row0 = m.row0;
        it.nrows = m.nrows;
        it.brow = m.expert * p.N + it.ncol;
        it.kb = p.K / kTK;
    } else if (p.mode == 1) {
        it.row0 = mt * kTM;
        it.nrows = min(kTM, p.rows - it.row0);
        it.brow = it.ncol;
        it.kb = p.K / kTK;
    } else {
        it.row0 = mt * kTM;
        it.nrows = min(kTM, p.M - it.row0);
        it.brow = it.ncol;
        if (p.mode == 2) {
            it.e = g;
            it.k0 = p.poff[g];
            it.kb = (p.poff[g + 1] - it.k0) / kTK;
        } else {
            it.kb = p.K / kTK;
        }
    }
    return it;
}

__global__ void __launch_bounds__(kTThreads, 1)
    bwd_tc_kernel(const TcParams p, const __grid_constant__ TmaMap tm_a, const __grid_constant__ TmaMap tm_b) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = gemm::align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTStages * kTStage);
    uint64_t* empty = full + kTStages;
    uint64_t* acc_full = empty + kTStages;  // [2]
    uint64_t* acc_empty = acc_full + 2;     // [2]
    uint64_t* fin = acc_empty + 2;          // the MMA warp's last commit
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(fin + 1);
    float* s_epi = reinterpret_cast<float*>(s_tmem + 4);  // [8 warps][32 rows][33]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kTStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kTEpiWarps);
        }
        mbar_init(fin, 1);
        fence_mbar_init();
    }
    if (warp == kTMmaWarp) {
        tmem_alloc(s_tmem, kTTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();
    pdl_launch_dependents();

    const int nt_per = (p.N + kTN - 1) / kTN;
    const int n_mt = p.mode == 0 ? p.ctrl->n_mtiles
                   : p.mode == 1 ? (p.rows + kTM - 1) / kTM
                                 : (p.M + kTM - 1) / kTM;
    const int n_items = n_mt * nt_per * (p.mode == 2 ? p.groups : 1);

    if (warp == kTProdWarp) {
        // ----------------------------------------------------------- TMA producer
        if (lane == 0 && (int)blockIdx.x < n_items) {
            prefetch_tmap(&tm_a);
            prefetch_tmap(&tm_b);
            int n = 0;
            bool stop = false;
            for (int item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
                const TcItem it = tc_item(p, n_mt, nt_per, item);
                for (int kb = 0; kb < it.kb; ++kb, ++n) {
                    const int s = n % kTStages;
                    if (n >= kTStages && !mbar_wait_bounded(&empty[s], ((n / kTStages) - 1) & 1)) {
                        set_status(p.status, kStatusTimeout);
                        stop = true;
                        break;
                    }
                    uint8_t* st = smem + s * kTStage;
                    const int x = it.k0 + kb * kTK;
                    mbar_arrive_expect_tx(&full[s], kTStage);
                    tma_load_2d(st, &tm_a, x, it.row0, &full[s]);
                    tma_load_2d(st + kTSA, &tm_b, x, it.brow, &full[s]);
                    tma_load_2d(st + kTSA + kTSB / 2, &tm_b, x, it.brow + kTN / 2, &full[s]);
                }
            }
            // copies still in flight land before this CTA may exit
            for (int q = n > kTStages ? n - kTStages : 0; q < n; ++q)
                mbar_wait_bounded(&full[q % kTStages], (q / kTStages) & 1);
        }
    } else if (warp == kTMmaWarp) {
        // -------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int n = 0, t = 0;
            for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++t) {
                const int kbs = tc_item(p, n_mt, nt_per, item).kb;
                const int b = t & 1;
                if (t >= 2 && !mbar_wait_bounded(&acc_empty[b], ((t >> 1) - 1) & 1)) {
                    set_status(p.status, kStatusTimeout);
                    break;
                }
                tc_fence_after();
                bool stop = false;
                for (int kb = 0; kb < kbs; ++kb, ++n) {
                    const int s = n % kTStages;
                    if (!mbar_wait_bounded(&full[s], (n / kTStages) & 1)) {
                        set_status(p.status, kStatusTimeout);
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* st = smem + s * kTStage;
                    const uint64_t da = smem_desc_sw128(st);
                    const uint64_t db = smem_desc_sw128(st + kTSA);
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // 4 x K=16 (32 bytes) inside the 128-byte swizzled rows
                        tc_mma_bf16(tmem + b * kTN, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), kTIdesc,
                                    (kb | k) != 0);
                    tc_commit(&empty[s]);
                }
                if (stop) break;
                tc_commit(&acc_full[b]);  // with no K blocks (an expert without rows) it arrives at once
            }
            // every MMA issued has completed before the CTA frees tensor memory
            if (t > 0) {
                tc_commit(fin);
                mbar_wait_bounded(fin, 0);
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q4 = warp & 3, wg = warp >> 2;
        const uint32_t t_row = tmem + ((uint32_t)(32 * q4) << 16);
        bool ok = true;
        int t = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++t) {
            const TcItem it = tc_item(p, n_mt, nt_per, item);
            const int b = t & 1;
            if (ok && !mbar_wait_bounded(&acc_full[b], (t >> 1) & 1)) ok = false;
            ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
            tc_fence_after();
            float v0[32], v1[32], v2[32], v3[32];
            if (ok) {
                const uint32_t c0 = t_row + (uint32_t)(b * kTN + 128 * wg);
                tmem_ld32(c0, v0);
                tmem_ld32(c0 + 32, v1);
                tmem_ld32(c0 + 64, v2);
                tmem_ld32(c0 + 96, v3);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);  // the tile after next may start
            if (!ok) continue;
            // rows 32*q4 + rr of the tile, columns ncol + 128*wg + 32*c + 4*(lane%8)..: each store
            // instruction covers 4 rows x 128 bytes
            const bool zero = it.kb == 0;  // no K blocks: the accumulator was never written
            float* sb = s_epi + warp * 32 * 33;
            const int rsub = lane >> 3, cc = (lane & 7) * 4;
            auto put = [&](const float (&v)[32], int c) {
#pragma unroll
                for (int j = 0; j < 32; ++j) sb[lane * 33 + j] = zero ? 0.f : v[j];
                __syncwarp();
                const int col = it.ncol + 128 * wg + 32 * c + cc;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int rr = 4 * q + rsub;
                    const int trow = 32 * q4 + rr;
                    if (trow < it.nrows && col < p.N) {
                        const int mrow = it.row0 + trow;
                        float* crow = (p.C2 && mrow >= p.msplit)
                                          ? p.C2 + (size_t)it.e * p.c_estride + (size_t)(mrow - p.msplit) * p.ldc
                                          : p.C + (size_t)it.e * p.c_estride + (size_t)mrow * p.ldc;
                        const float* r = sb + rr * 33 + cc;
                        *reinterpret_cast<float4*>(crow + col) = make_float4(r[0], r[1], r[2], r[3]);
                    }
                }
                __syncwarp();
            };
            put(v0, 0);
            put(v1, 1);
            put(v2, 2);
            put(v3, 3);
        }
        if (!ok) set_status(p.status, kStatusTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTTmemCols);
    }
}

size_t tc_smem() { return (size_t)kTStages * kTStage + 1024 + (2 * kTStages + 5) * 8 + 16 + kTEpiWarps * 32 * 33 * 4; }

// A: bf16 [a_rows, cols], B: bf16 [b_rows, cols], both K contiguous.
cudaError_t launch_tc(const TcParams& p, const void* A, uint64_t a_rows, uint64_t cols, const void* B, uint64_t b_rows,
                      cudaStream_t st) {
    TmaMap ta, tb;
    if (!tmap_bf16_2d(&ta, A, a_rows, cols, kTK, kTM) || !tmap_bf16_2d(&tb, B, b_rows, cols, kTK, kTN / 2))
        return cudaErrorInvalidValue;
    static bool smem_set = false;
    const size_t smem = tc_smem();
    if (!smem_set) {
        const cudaError_t e =
            cudaFuncSetAttribute((const void*)bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(num_sms(), kMaxStreamCtas));
    cfg.blockDim = dim3(kTThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bwd_tc_kernel, p, ta, tb);
}

}  // namespace

// dgrad: C[r, :] = A[r, :] . Bt_e^T for the rows of the permutation's tiles (routed) or rows
// [0, rows) (one group, Bt = its only matrix). A: bf16 [rows_a, K]; Bt: bf16 [n_mat * N, K];
// K a multiple of 64, N a multiple of 8; C: fp32 [rows, N].
cudaError_t launch_bwd_tc(const void* A, uint64_t rows_a, const void* Bt, uint64_t n_mat, int K, int N, int routed,
                          int rows, const MTile* mtiles, const Ctrl* ctrl, float* C, int* status, cudaStream_t st) {
    TcParams p = {};
    p.mode = routed ? 0 : 1;
    p.K = K;
    p.N = N;
    p.rows = rows;
    p.mtiles = mtiles;
    p.ctrl = ctrl;
    p.C = C;
    p.ldc = N;
    p.status = status;
    return launch_tc(p, A, rows_a, (uint64_t)K, Bt, n_mat * (uint64_t)N, st);
}

// wgrad: C_g[m, n] = sum_j At[m, j] Bt[n, j] over the columns j of group g: [poff[g],
// poff[g+1]) (poff != nullptr: groups of them, each a multiple of 64) or [0, K) (one
// group). At: bf16 [M, cols]; Bt: bf16 [N, cols]; C_g = C + g * c_estride, [M, N] rows of
// N (rows >= msplit to C2 when given).
cudaError_t launch_bwd_tc_wgrad(const void* At, int M, const void* Bt, int N, uint64_t cols, const int32_t* poff,
                                int groups, int K, float* C, float* C2, int msplit, size_t c_estride, int* status,
                                cudaStream_t st) {
    TcParams p = {};
    p.mode = poff ? 2 : 3;
    p.K = K;
    p.N = N;
    p.M = M;
    p.groups = groups;
    p.poff = poff;
    p.C = C;
    p.C2 = C2;
    p.msplit = msplit;
    p.ldc = N;
    p.c_estride = c_estride;
    p.status = status;
    return launch_tc(p, At, (uint64_t)M, cols, Bt, (uint64_t)N, st);
}

}  // namespace moe
