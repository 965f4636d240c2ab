// Stages P1/P2 and Q1/Q2 of the DeepSeek-V2 MoE layer ("DSV2-236B-MegaKernel", README
// stage flowchart, MoE subgraph) when experts see many tokens: a grouped FP8 GEMM on
// the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Tiles are 128 permuted token rows (one expert's segment, or the shared experts'
// tokens) x 256 weight rows. For gate/up the 256 rows are 128 gate rows and the same
// 128 up rows, so one thread's accumulator row holds g and u for the same intermediate
// channels; for down they are 256 rows of the hidden dimension.
//
// Block scales. The weights carry arbitrary fp32 scales per 128x128 block and the
// activations a power-of-two scale per (row, 128 channels), so the tensor core cannot
// apply them: every 128-wide K block is accumulated on its own (4 MMAs of K=32) into
// one of two TMEM accumulators, and the epilogue warps promote it,
//     acc[m][n] += D_kb[m][n] * s_x[m][kb] * s_w[n-block][kb],
// while the MMA warp fills the other accumulator with the next K block.
//
// Warp roles (one CTA per SM, persistent over tiles):
//   warp 9      TMA producer: A box (128 rows x 128 B), B boxes (2 x 128 rows x 128 B),
//               the tile rows' activation scales for this K block, into a 4-stage ring
//   warp 8      MMA issuer (one thread): 4 x tcgen05.mma kind::f8f6f4 per K block,
//               commits to the stage's "empty" barrier and the accumulator's "full"
//   warps 0-7   epilogue: warpgroup g covers columns [64g, 64g+64) of gate and of up
//               (or [128g, 128g+128) of down); TMEM lanes 32*(warp%4).. are its rows
// Epilogue at the end of a tile: gate/up -> a = SiLU(g) * u, quantised per 128 values
// to E4M3 with a power-of-two scale (the down GEMM's operand); down -> w * y in bf16.
#include <algorithm>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kGM = 128;                  // token rows per tile (MMA M)
constexpr int kGN = 256;                  // weight rows per tile (MMA N)
constexpr int kGStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kGThreads = (kEpiWarps + 2) * 32;
constexpr int kProducerWarp = kEpiWarps + 1;
constexpr int kMmaWarp = kEpiWarps;
constexpr int kSA = kGM * kBlk;           // 16 KB A tile
constexpr int kSB = kGN * kBlk;           // 32 KB B tile
constexpr int kSXF = 132;                 // activation scales loaded per stage (floats)
constexpr int kStageBytes = ((kSA + kSB + kSXF * 4) + 1023) & ~1023;
constexpr uint32_t kTmemCols = 512;       // two 128 x 256 fp32 accumulators
constexpr uint32_t kPolls = 1u << 22;
constexpr uint32_t kIdesc = idesc_f8_f32(kGM, kGN);

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

struct Item {
    int shared;  // shared experts' segment
    int expert;
    int row0;    // first row of the tile in the A tensor (permuted row, or token)
    int nrows;   // valid rows (<= 128)
    int ntile;   // 256-row weight tile index
};

__device__ __forceinline__ Item decode_item(const GemmArgs& a, int n_mt_r, int item) {
    Item it;
    const int n_r = n_mt_r * a.nt_r;
    if (item < n_r) {
        const MTile mt = a.mtiles[item / a.nt_r];
        it.shared = 0;
        it.expert = mt.expert;
        it.row0 = mt.row0;
        it.nrows = mt.nrows;
        it.ntile = (int)(item % a.nt_r);
    } else {
        const int v = item - n_r;
        const int m = (int)(v / a.nt_s);
        it.shared = 1;
        it.expert = -1;
        it.row0 = m * kGM;
        it.nrows = min(kGM, a.T - it.row0);
        it.ntile = (int)(v % a.nt_s);
    }
    return it;
}

template <int kMode>  // 0: gate/up, 1: down
__global__ void __launch_bounds__(kGThreads, 1)
    expert_gemm_kernel(const GemmArgs a, const __grid_constant__ TmaMap tm_a_r, const __grid_constant__ TmaMap tm_a_s,
                       const __grid_constant__ TmaMap tm_b0_r, const __grid_constant__ TmaMap tm_b1_r,
                       const __grid_constant__ TmaMap tm_b0_s, const __grid_constant__ TmaMap tm_b1_s,
                       const __grid_constant__ TmaMap tm_sx_r, const __grid_constant__ TmaMap tm_sx_s) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGStages * kStageBytes);
    uint64_t* empty = full + kGStages;
    uint64_t* acc_full = empty + kGStages;   // [2]
    uint64_t* acc_empty = acc_full + 2;      // [2]
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(acc_empty + 2);
    float* s_amax = reinterpret_cast<float*>(s_tmem + 4);  // [2][128]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + kEpiWarps);  // MMA commit + every epilogue warp (activation scales read)
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiWarps);
        }
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();
    pdl_launch_dependents();

    const int n_mt_r = a.ctrl->n_mtiles;
    const int n_items = n_mt_r * a.nt_r + a.n_mt_s * a.nt_s;
    constexpr bool gateup = kMode == 0;

    if (warp == kProducerWarp) {
        // ----------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_a_r);
            prefetch_tmap(&tm_b0_r);
            prefetch_tmap(&tm_sx_r);
            if (a.n_mt_s > 0) {
                prefetch_tmap(&tm_a_s);
                prefetch_tmap(&tm_b0_s);
                prefetch_tmap(&tm_sx_s);
            }
            int n = 0;  // K blocks issued
            bool ok = true;
            for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                const Item it = decode_item(a, n_mt_r, item);
                const int Kb = (it.shared ? a.K_s : a.K_r) / kBlk;
                const void* ma = it.shared ? (const void*)&tm_a_s : (const void*)&tm_a_r;
                const void* mb0 = it.shared ? (const void*)&tm_b0_s : (const void*)&tm_b0_r;
                const void* mb1 = it.shared ? (const void*)&tm_b1_s : (const void*)&tm_b1_r;
                const void* msx = it.shared ? (const void*)&tm_sx_s : (const void*)&tm_sx_r;
                // weight rows of this tile in the 2-D [E * rows_per_expert, K] view
                int yb0, yb1;
                if (gateup) {
                    const int base = it.shared ? 0 : it.expert * a.I;
                    yb0 = base + it.ntile * kBlk;  // gate rows
                    yb1 = yb0;                     // the same rows of up
                } else {
                    const int base = it.shared ? 0 : it.expert * a.H;
                    yb0 = base + it.ntile * kGN;
                    yb1 = yb0 + kBlk;
                }
                const int x0 = it.row0 & ~3;  // TMA inner coordinate must be 16-byte aligned
                for (int kb = 0; kb < Kb; ++kb, ++n) {
                    const int s = (int)(n % kGStages);
                    if (n >= kGStages && !mbar_wait_bounded(&empty[s], ((n / kGStages) - 1) & 1, kPolls)) {
                        set_status(a.status, kStatusTimeout);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * kStageBytes;
                    mbar_arrive_expect_tx(&full[s], kSA + kSB + kSXF * 4);
                    tma_load_2d(st, ma, kb * kBlk, it.row0, &full[s]);
                    tma_load_2d(st + kSA, mb0, kb * kBlk, yb0, &full[s]);
                    tma_load_2d(st + kSA + kSB / 2, mb1, kb * kBlk, yb1, &full[s]);
                    tma_load_2d(st + kSA + kSB, msx, x0, kb, &full[s]);
                }
            }
            // copies still in flight land before this CTA may exit
            const int done_from = n > kGStages ? n - kGStages : 0;
            for (int q = done_from; q < n; ++q)
                mbar_wait_bounded(&full[q % kGStages], (q / kGStages) & 1, kPolls);
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int n = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                const Item it = decode_item(a, n_mt_r, item);
                const int Kb = (it.shared ? a.K_s : a.K_r) / kBlk;
                for (int kb = 0; kb < Kb; ++kb, ++n) {
                    const int s = (int)(n % kGStages);
                    const int b = (int)(n & 1);
                    if (n >= 2 && !mbar_wait_bounded(&acc_empty[b], ((n >> 1) - 1) & 1, kPolls)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait_bounded(&full[s], (n / kGStages) & 1, kPolls)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* st = smem + s * kStageBytes;
                    const uint64_t da = smem_desc_sw128(st);
                    const uint64_t db = smem_desc_sw128(st + kSA);
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // 4 x K=32 bytes inside the 128-byte swizzled rows
                        tc_mma_f8(tmem + b * kGN, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), kIdesc, k > 0);
                    tc_commit(&empty[s]);
                    tc_commit(&acc_full[b]);
                }
            }
            if (!ok) set_status(a.status, kStatusTimeout);
            // every MMA issued has completed before the CTA frees tensor memory
            if (n > 0) mbar_wait_bounded(&acc_full[(n - 1) & 1], ((n - 1) >> 1) & 1, kPolls);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;          // TMEM lane quadrant: rows 32q .. 32q+31
        const int wg = warp >> 2;        // column half
        const int row = 32 * q + lane;   // tile row of this thread
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        int n = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            const Item it = decode_item(a, n_mt_r, item);
            const int Kb = (it.shared ? a.K_s : a.K_r) / kBlk;
            // weight block scales of this tile's rows, one per K block
            const float* sw0;
            const float* sw1;
            if (gateup) {
                const size_t r = it.shared ? (size_t)it.ntile : (size_t)it.expert * (a.I / kBlk) + it.ntile;
                sw0 = (it.shared ? a.ss_gate : a.s_gate) + r * Kb;
                sw1 = (it.shared ? a.ss_up : a.s_up) + r * Kb;
            } else {
                const size_t r = (it.shared ? 0 : (size_t)it.expert * (a.H / kBlk)) + (size_t)it.ntile * 2 + wg;
                sw0 = (it.shared ? a.ss_down : a.s_down) + r * Kb;
                sw1 = sw0;
            }
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0.f;
            const int sx_off = it.row0 - (it.row0 & ~3) + row;
            for (int kb = 0; kb < Kb; ++kb, ++n) {
                const int s = (int)(n % kGStages);
                const int b = (int)(n & 1);
                if (ok && !mbar_wait_bounded(&acc_full[b], (n >> 1) & 1, kPolls)) ok = false;
                if (ok && !mbar_wait_bounded(&full[s], (n / kGStages) & 1, kPolls)) ok = false;
                tc_fence_after();
                const float sx = ok ? reinterpret_cast<const float*>(smem + s * kStageBytes + kSA + kSB)[sx_off] : 0.f;
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                const float c0 = sx * __ldg(sw0 + kb);
                const float c1 = sx * __ldg(sw1 + kb);
                if (ok) {
                    const uint32_t tb = tmem + lane_off + (uint32_t)(b * kGN);
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        // gate/up: chunks 0-3 = gate cols 64wg.., chunks 4-7 = up cols 128+64wg..
                        // down: chunks 0-7 = cols 128wg..
                        const int col = gateup ? (h < 4 ? 64 * wg + 16 * h : 128 + 64 * wg + 16 * (h - 4))
                                               : 128 * wg + 16 * h;
                        float v[16];
                        tmem_ld16(tb + col, v);
                        const float c = (gateup && h >= 4) ? c1 : c0;
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[16 * h + j] = fmaf(v[j], c, acc[16 * h + j]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[b]);
            }
            if (!ok) set_status(a.status, kStatusTimeout);
            // after a timeout this warp still takes every named barrier below (its sibling
            // warpgroup waits there) but writes nothing
            const bool valid = ok && row < it.nrows;
            const int grow = it.row0 + row;  // row in the output tensors
            if (gateup) {
                // a = SiLU(g) * u for 64 intermediate channels; the 128-channel scale
                // block spans both warpgroups: combine their maxima through shared memory
                float amax = 0.f;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    acc[j] = silu_mul(acc[j], acc[64 + j]);
                    amax = fmaxf(amax, fabsf(acc[j]));
                }
                s_amax[wg * kGM + row] = amax;
                named_bar(1, kEpiWarps * 32);
                amax = fmaxf(s_amax[row], s_amax[kGM + row]);
                float inv;
                const float scale = act_scale_pow2(amax, &inv);
                if (valid) {
                    const int N = it.shared ? a.Is : a.I;
                    uint8_t* dst = (it.shared ? a.hq_s : a.hq_r) + (size_t)grow * N + it.ntile * kBlk + 64 * wg;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 w;
                        w.x = pack_e4m3x4(acc[16 * c + 0] * inv, acc[16 * c + 1] * inv, acc[16 * c + 2] * inv,
                                          acc[16 * c + 3] * inv);
                        w.y = pack_e4m3x4(acc[16 * c + 4] * inv, acc[16 * c + 5] * inv, acc[16 * c + 6] * inv,
                                          acc[16 * c + 7] * inv);
                        w.z = pack_e4m3x4(acc[16 * c + 8] * inv, acc[16 * c + 9] * inv, acc[16 * c + 10] * inv,
                                          acc[16 * c + 11] * inv);
                        w.w = pack_e4m3x4(acc[16 * c + 12] * inv, acc[16 * c + 13] * inv, acc[16 * c + 14] * inv,
                                          acc[16 * c + 15] * inv);
                        reinterpret_cast<uint4*>(dst)[c] = w;
                    }
                    if (wg == 0) {  // transposed scales: [I/128][rows] (the down GEMM's TMA layout)
                        float* hsT = it.shared ? a.hsT_s : a.hsT_r;
                        const long ld = it.shared ? a.ld_s : a.ld_r;
                        hsT[(size_t)it.ntile * ld + grow] = scale;
                    }
                }
                named_bar(1, kEpiWarps * 32);  // s_amax is reused by the next tile
            } else if (valid) {
                float wrow = 1.f;
                if (!it.shared) {
                    const int f = a.perm_src[grow];
                    wrow = ((unsigned)f < (unsigned)(a.T * a.k)) ? a.topk_w[f] : 0.f;
                }
                __nv_bfloat16* dst = (it.shared ? a.y_shared : a.y_perm) + (size_t)grow * a.H + it.ntile * kGN + 128 * wg;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    uint4 o;
                    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const __nv_bfloat162 h2 =
                            __floats2bfloat162_rn(acc[8 * c + 2 * p] * wrow, acc[8 * c + 2 * p + 1] * wrow);
                        ow[p] = *reinterpret_cast<const uint32_t*>(&h2);
                    }
                    reinterpret_cast<uint4*>(dst)[c] = o;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

size_t gemm_smem() { return (size_t)kGStages * kStageBytes + 1024 + 2 * kGStages * 8 + 4 * 8 + 16 + 2 * kGM * 4; }

}  // namespace

bool gemm_supported(const moe_config_t& c) {
    // 256-row down tiles, whole 128-row intermediate tiles, and the scale rows of a
    // K block must fit the epilogue's per-lane registers (K <= 256 blocks)
    const int Is = c.n_shared * c.moe_inter;
    return c.hidden % kGN == 0 && c.hidden / kBlk <= 256 && c.moe_inter / kBlk <= 256 && Is / kBlk <= 256;
}

cudaError_t launch_expert_gemm(const GemmArgs& g, const TmaMaps& m, cudaStream_t st) {
    static size_t smem_set[2] = {0, 0};
    const size_t smem = gemm_smem();
    const int mode = g.mode == 0 ? 0 : 1;
    auto kern = mode == 0 ? expert_gemm_kernel<0> : expert_gemm_kernel<1>;
    if (smem_set[mode] < smem) {
        const cudaError_t e =
            cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set[mode] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(num_sms(), kMaxStreamCtas));
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, g, m.a_r, m.a_s, m.b0_r, m.b1_r, m.b0_s, m.b1_s, m.sx_r, m.sx_s);
}

}  // namespace moe
