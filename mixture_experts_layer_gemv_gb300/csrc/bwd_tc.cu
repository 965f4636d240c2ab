// The backward's dgrad contractions on the tcgen05 tensor cores (kind::f16: bf16 x bf16
// -> fp32 in tensor memory):
//   C[r, n] = sum_k A[r, k] * Bt_e[n, k]
// A: bf16 rows [rows, K] (K contiguous): the permuted rows of an expert (the
//    permutation's 128-row tiles) or the shared experts' tokens;
// Bt_e: the expert's weights transposed and dequantised to bf16, [N, K] (K contiguous),
//    stacked over experts as [E * N, K].
// Used for dau = Wd^T dout (K = H, N = I) and dx_r = [Wg; Wu]^T [dg | du] (K = 2I, N = H).
//
// Tiles of 128 rows x 256 columns; a tile's whole K accumulates in one TMEM accumulator,
// and two accumulators (512 columns) let one tile's epilogue overlap the next tile's
// MMAs. One persistent CTA of 10 warps per SM:
//   warp 9      TMA producer: per 64-wide K block (128 bytes) an A box of 128 rows and two
//               B boxes of 128 rows (128-byte swizzle), a 4-stage ring
//   warp 8      MMA issuer (one thread): per K block 4 tcgen05.mma M=128 N=256 K=16
//   warps 0-7   epilogue: warp w reads lanes 32*(w%4).. and column half w/4 of the
//               accumulator, releases it, and stores the rows in fp32.
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

struct TcParams {
    int K, N;         // reduction length, output width (Bt_e has N rows)
    int routed;       // 1: tiles of the permutation (rows row0.., B of the tile's expert); 0: one group
    int rows;         // rows of A in the one-group case
    const MTile* mtiles;
    const Ctrl* ctrl;
    float* C;         // [rows, N] fp32
    int* status;
};

struct TcItem {
    int row0, nrows, brow, ncol;
};

__device__ __forceinline__ TcItem tc_item(const TcParams& p, int nt_per, int item) {
    TcItem it;
    const int mt = item / nt_per, nt = item % nt_per;
    it.ncol = nt * kTN;
    if (p.routed) {
        const MTile m = p.mtiles[mt];
        it.row0 = m.row0;
        it.nrows = m.nrows;
        it.brow = m.expert * p.N + it.ncol;
    } else {
        it.row0 = mt * kTM;
        it.nrows = min(kTM, p.rows - it.row0);
        it.brow = it.ncol;
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
    const int n_mt = p.routed ? p.ctrl->n_mtiles : (p.rows + kTM - 1) / kTM;
    const int n_items = n_mt * nt_per;
    const int Kb = p.K / kTK;
    const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int total = my_items * Kb;

    if (warp == kTProdWarp) {
        // ----------------------------------------------------------- TMA producer
        if (lane == 0 && total > 0) {
            prefetch_tmap(&tm_a);
            prefetch_tmap(&tm_b);
            int n = 0, item = blockIdx.x;
            TcItem it = tc_item(p, nt_per, item);
            int kb = 0;
            for (; n < total; ++n) {
                const int s = n % kTStages;
                if (n >= kTStages && !mbar_wait_bounded(&empty[s], ((n / kTStages) - 1) & 1)) {
                    set_status(p.status, kStatusTimeout);
                    break;
                }
                uint8_t* st = smem + s * kTStage;
                const int x = kb * kTK;
                mbar_arrive_expect_tx(&full[s], kTStage);
                tma_load_2d(st, &tm_a, x, it.row0, &full[s]);
                tma_load_2d(st + kTSA, &tm_b, x, it.brow, &full[s]);
                tma_load_2d(st + kTSA + kTSB / 2, &tm_b, x, it.brow + kTN / 2, &full[s]);
                if (++kb == Kb) {
                    kb = 0;
                    item += gridDim.x;
                    if (item < n_items) it = tc_item(p, nt_per, item);
                }
            }
            // copies still in flight land before this CTA may exit
            for (int q = n > kTStages ? n - kTStages : 0; q < n; ++q)
                mbar_wait_bounded(&full[q % kTStages], (q / kTStages) & 1);
        }
    } else if (warp == kTMmaWarp) {
        // -------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int n = 0;
            for (int t = 0; t < my_items; ++t) {
                const int b = t & 1;
                if (t >= 2 && !mbar_wait_bounded(&acc_empty[b], ((t >> 1) - 1) & 1)) {
                    set_status(p.status, kStatusTimeout);
                    break;
                }
                tc_fence_after();
                bool stop = false;
                for (int kb = 0; kb < Kb; ++kb, ++n) {
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
                tc_commit(&acc_full[b]);
            }
            // every MMA issued has completed before the CTA frees tensor memory
            if (n > 0) {
                tc_commit(fin);
                mbar_wait_bounded(fin, 0);
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q4 = warp & 3, wg = warp >> 2;
        const int row = 32 * q4 + lane;
        const uint32_t t_row = tmem + ((uint32_t)(32 * q4) << 16);
        bool ok = true;
        int t = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++t) {
            const TcItem it = tc_item(p, nt_per, item);
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
            if (!ok || row >= it.nrows) continue;
            float* dst = p.C + (size_t)(it.row0 + row) * p.N + it.ncol + 128 * wg;
            const int ncols = min(128, p.N - it.ncol - 128 * wg);
            const float* vs[4] = {v0, v1, v2, v3};
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                if (4 * c >= ncols) break;
                const float* v = vs[c >> 3];
                const int j = 4 * (c & 7);
                reinterpret_cast<float4*>(dst)[c] = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
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

size_t tc_smem() { return (size_t)kTStages * kTStage + 1024 + (2 * kTStages + 5) * 8 + 16; }

}  // namespace

// C[r, :] = A[r, :] . Bt_e^T for the rows of the permutation's tiles (routed) or rows
// [0, rows) (one group, Bt = its only matrix). A: bf16 [rows_a, K]; Bt: bf16 [n_mat * N, K];
// K a multiple of 64, N a multiple of 8; C: fp32 [rows, N].
cudaError_t launch_bwd_tc(const void* A, uint64_t rows_a, const void* Bt, uint64_t n_mat, int K, int N, int routed,
                          int rows, const MTile* mtiles, const Ctrl* ctrl, float* C, int* status, cudaStream_t st) {
    TmaMap ta, tb;
    if (!tmap_bf16_2d(&ta, A, rows_a, (uint64_t)K, kTK, kTM) ||
        !tmap_bf16_2d(&tb, Bt, n_mat * (uint64_t)N, (uint64_t)K, kTK, kTN / 2))
        return cudaErrorInvalidValue;
    static bool smem_set = false;
    const size_t smem = tc_smem();
    if (!smem_set) {
        const cudaError_t e =
            cudaFuncSetAttribute((const void*)bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = true;
    }
    TcParams p;
    p.K = K;
    p.N = N;
    p.routed = routed;
    p.rows = rows;
    p.mtiles = mtiles;
    p.ctrl = ctrl;
    p.C = C;
    p.status = status;
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

}  // namespace moe
