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
// one of two TMEM accumulators, and the epilogue promotes it into registers,
//     acc[m][n] += D_kb[m][n] * s_x[m][kb] * s_w[n-block][kb],
// while the tensor core fills the other accumulator with the next K block.
//
// One CTA of 12 warps per SM, persistent over tiles, warp-specialised:
//   warp 9      TMA producer: per K block an A box (128 rows x 128 B) and two B boxes
//               (128 rows x 128 B) into a 4-stage ring; a stage is refilled as soon as
//               the MMAs that read it have completed
//   warp 8      MMA issuer (one thread): 4 x tcgen05.mma kind::f8f6f4 per K block into
//               accumulator n%2 once the epilogue has drained it
//   warps 0-7   epilogue: warp w reads TMEM lanes 32*(w%4).. (its 32 rows) and, with
//               g = w/4, columns [64g, 64g+64) of gate and of up (or [128g, 128g+128) of
//               down), so each thread keeps a 128-float accumulator row in registers
//   warps 10-11 idle (they complete the third warpgroup)
// Registers: the CTA is launched with 168 per thread (three warps on each of the four
// 16K-register sub-partition files); the third warpgroup (MMA, producer, idle) then
// gives back all but 56 of its registers (setmaxnreg) and the two epilogue warpgroups
// grow to 224, room for the accumulator row plus a 64-column TMEM slice.
// Per K block an epilogue thread loads its two 64-column halves from TMEM in turn, each
// followed by its multiply-adds (packed FP32 pairs), and then releases the accumulator
// to the MMA warp. (Releasing it before the second half's multiply-adds measured
// slower: 1.05 against 1.03 ms for the T=4096 gate/up GEMM.)
// Activation scales come from global memory (row-major, one row per thread) and the
// weight scales of the tile's row blocks too; both are loaded one K block ahead.
// Epilogue at the end of a tile: gate/up -> a = SiLU(g) * u, quantised per 128 values
// to E4M3 with a power-of-two scale (the down GEMM's operand); down -> w * y in bf16.
#include <algorithm>

#include "gemm_common.cuh"

namespace moe {

namespace {

using namespace gemm;

constexpr int kGStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kMmaWarp = kEpiWarps;
constexpr int kProducerWarp = kEpiWarps + 1;
constexpr int kGThreads = (kEpiWarps + 4) * 32;  // + a warpgroup: MMA, producer, two idle warps
constexpr int kLaunchRegs = 168;                  // per thread at launch (__launch_bounds__ below)
constexpr int kEpiRegs = 224, kCtlRegs = 56;      // after the split
static_assert(kEpiWarps * 32 * kEpiRegs + 128 * kCtlRegs == kGThreads * kLaunchRegs,
              "the register split hands over exactly what the launch holds");
constexpr int kSA = kGM * kBlk;           // 16 KB A tile
constexpr int kSB = kGN * kBlk;           // 32 KB B tile
constexpr int kStageBytes = kSA + kSB;    // a multiple of 1024 (128-byte swizzle atoms)
constexpr uint32_t kTmemCols = 512;       // two 128 x 256 fp32 accumulators
constexpr uint32_t kIdesc = idesc_f8_f32(kGM, kGN);

struct Maps {
    const void *a_r, *a_s, *b0_r, *b1_r, *b0_s, *b1_s;
};

__device__ __forceinline__ void issue_loads(uint8_t* stage, uint64_t* bar, const LoadCursor& c, const Maps& m) {
    mbar_arrive_expect_tx(bar, kStageBytes);
    const int x = c.kb * kBlk;
    tma_load_2d(stage, c.shared ? m.a_s : m.a_r, x, c.row0, bar);
    tma_load_2d(stage + kSA, c.shared ? m.b0_s : m.b0_r, x, c.yb0, bar);
    tma_load_2d(stage + kSA + kSB / 2, c.shared ? m.b1_s : m.b1_r, x, c.yb1, bar);
}

template <int kMode>  // 0: gate/up, 1: down, 2: gate/up with g and u written as they are (fp32)
__global__ void __launch_bounds__(kGThreads, 1)
    expert_gemm_kernel(const GemmArgs a, const __grid_constant__ TmaMap tm_a_r, const __grid_constant__ TmaMap tm_a_s,
                       const __grid_constant__ TmaMap tm_b0_r, const __grid_constant__ TmaMap tm_b1_r,
                       const __grid_constant__ TmaMap tm_b0_s, const __grid_constant__ TmaMap tm_b1_s) {
    constexpr bool gateup = kMode != 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGStages * kStageBytes);
    uint64_t* empty = full + kGStages;
    uint64_t* acc_full = empty + kGStages;  // [2]
    uint64_t* acc_empty = acc_full + 2;     // [2]
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(acc_empty + 2);
    float* s_amax = reinterpret_cast<float*>(s_tmem + 4);  // [2][128]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);  // the MMA warp's commit
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
    const int n_r = n_mt_r * a.nt_r;
    const int n_items = n_r + a.n_mt_s * a.nt_s;
    // K blocks this CTA runs, over all its items
    const int total = items_in(0, n_r) * (a.K_r / kBlk) + items_in(n_r, n_items) * (a.K_s / kBlk);

    if (warp >= kEpiWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtlRegs));
    if (warp == kProducerWarp) {
        // ----------------------------------------------------------- TMA producer
        if (lane == 0 && total > 0) {
            const Maps maps{&tm_a_r, &tm_a_s, &tm_b0_r, &tm_b1_r, &tm_b0_s, &tm_b1_s};
            prefetch_tmap(&tm_a_r);
            prefetch_tmap(&tm_b0_r);
            prefetch_tmap(&tm_b1_r);
            if (a.n_mt_s > 0) {
                prefetch_tmap(&tm_a_s);
                prefetch_tmap(&tm_b0_s);
                prefetch_tmap(&tm_b1_s);
            }
            LoadCursor lc;
            lc.item = blockIdx.x;
            lc.kb = 0;
            lc.set(a, n_mt_r, n_items, gateup);
            int n = 0;
            for (; n < total; ++n) {
                const int s = n % kGStages;
                if (n >= kGStages && !mbar_wait_bounded(&empty[s], ((n / kGStages) - 1) & 1)) {
                    set_status(a.status, kStatusTimeout);
                    break;
                }
                issue_loads(smem + s * kStageBytes, &full[s], lc, maps);
                lc.next(a, n_mt_r, n_items, gateup);
            }
            // copies still in flight land before this CTA may exit
            for (int q = n > kGStages ? n - kGStages : 0; q < n; ++q)
                mbar_wait_bounded(&full[q % kGStages], (q / kGStages) & 1);
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int n = 0;
            for (; n < total; ++n) {
                const int s = n % kGStages, b = n & 1;
                if ((n >= 2 && !mbar_wait_bounded(&acc_empty[b], ((n >> 1) - 1) & 1)) ||
                    !mbar_wait_bounded(&full[s], (n / kGStages) & 1)) {
                    set_status(a.status, kStatusTimeout);
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
            // every MMA issued has completed before the CTA frees tensor memory
            if (n > 0) mbar_wait_bounded(&acc_full[(n - 1) & 1], ((n - 1) >> 1) & 1);
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
        // ---------------------------------------------------------------- epilogue
        const int q4 = warp & 3;          // TMEM lane quadrant: rows 32q .. 32q+31
        const int wg = warp >> 2;         // column half
        const int row = 32 * q4 + lane;   // tile row of this thread
        const uint32_t t_row = tmem + ((uint32_t)(32 * q4) << 16);
        int n = 0;  // K blocks consumed
        bool ok = true;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            int Kb, grow;
            bool valid_row;
            const float *sxp, *sw0, *sw1;
            {
                const Item it = decode_item(a, n_mt_r, item);
                Kb = (it.shared ? a.K_s : a.K_r) / kBlk;
                valid_row = row < it.nrows;
                grow = it.row0 + row;  // row in the A tensor and the output tensors
                // this row's activation scales (row-major, Kb per row) and the weight scales
                if (gateup) {
                    int tok = grow;
                    if (!it.shared) {
                        const int f = valid_row ? a.perm_src[grow] : 0;
                        tok = ((unsigned)f < (unsigned)(a.T * a.k)) ? f / a.k : 0;
                    }
                    sxp = a.xs + (size_t)(valid_row ? tok : 0) * Kb;
                    const size_t r = it.shared ? (size_t)it.ntile : (size_t)it.expert * (a.I / kBlk) + it.ntile;
                    sw0 = (it.shared ? a.ss_gate : a.s_gate) + r * Kb;
                    sw1 = (it.shared ? a.ss_up : a.s_up) + r * Kb;
                } else {
                    sxp = (it.shared ? a.hs_s : a.hs_r) + (size_t)(valid_row ? grow : 0) * Kb;
                    const size_t r = (it.shared ? 0 : (size_t)it.expert * (a.H / kBlk)) + (size_t)it.ntile * 2 + wg;
                    sw0 = (it.shared ? a.ss_down : a.s_down) + r * Kb;
                    sw1 = sw0;
                }
            }
            // raw scales of the next K block, loaded one block ahead of their use
            float nx = __ldg(sxp), nw0 = __ldg(sw0), nw1 = gateup ? __ldg(sw1) : 0.f;

            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0.f;

            for (int kb = 0; kb < Kb; ++kb, ++n) {
                const int b = n & 1;
                const float c0 = nx * nw0, c1 = gateup ? nx * nw1 : c0;
                if (kb + 1 < Kb) {
                    nx = __ldg(sxp + kb + 1);
                    nw0 = __ldg(sw0 + kb + 1);
                    if (gateup) nw1 = __ldg(sw1 + kb + 1);
                }
                if (ok && !mbar_wait_bounded(&acc_full[b], (n >> 1) & 1)) ok = false;
                // tcgen05.ld is warp-collective: the whole warp reads, or none of it
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                // half h: gate/up: 0 = gate cols 64wg.., 1 = up cols 128+64wg..; down: cols 128wg + 64h
                const uint32_t tb = t_row + (uint32_t)(b * kGN);
                if (ok) {
                    float v[64];
                    tmem_ld64(tb + (gateup ? 64 * wg : 128 * wg), v);
#pragma unroll
                    for (int j = 0; j < 64; j += 2) fma2(acc[j], acc[j + 1], v[j], v[j + 1], c0);
                    tmem_ld64(tb + (gateup ? 128 + 64 * wg : 128 * wg + 64), v);
#pragma unroll
                    for (int j = 0; j < 64; j += 2) fma2(acc[64 + j], acc[64 + j + 1], v[j], v[j + 1], c1);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[b]);
            }
            if (!ok) set_status(a.status, kStatusTimeout);
            // after a timeout every warp still takes the named barriers below, but writes nothing
            const bool valid = ok && valid_row;
            const Item it = decode_item(a, n_mt_r, item);
            if (kMode == 2) {
                // the backward's recompute: g and u of 64 intermediate channels each
                if (valid) {
                    const int N = it.shared ? a.Is : a.I;
                    const size_t o = (size_t)grow * N + it.ntile * kBlk + 64 * wg;
                    float4* dg = reinterpret_cast<float4*>((it.shared ? a.g_out_s : a.g_out_r) + o);
                    float4* du = reinterpret_cast<float4*>((it.shared ? a.u_out_s : a.u_out_r) + o);
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        dg[c] = make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
                        du[c] = make_float4(acc[64 + 4 * c], acc[64 + 4 * c + 1], acc[64 + 4 * c + 2],
                                            acc[64 + 4 * c + 3]);
                    }
                }
            } else if (gateup) {
                // a = SiLU(g) * u for 64 intermediate channels; the 128-channel scale block
                // spans both column halves: combine their maxima through shared memory
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
                    if (wg == 0)  // row-major [rows, N/128]: the down GEMM's activation scales
                        (it.shared ? a.hs_s : a.hs_r)[(size_t)grow * (N / kBlk) + it.ntile] = scale;
                }
                named_bar(1, kEpiWarps * 32);  // s_amax is reused by the next tile
            } else if (valid) {
                float wrow = 1.f;
                if (!it.shared) {
                    const int f = a.perm_src[grow];
                    wrow = ((unsigned)f < (unsigned)(a.T * a.k)) ? a.topk_w[f] : 0.f;
                }
                __nv_bfloat16* dst =
                    (it.shared ? a.y_shared : a.y_perm) + (size_t)grow * a.H + it.ntile * kGN + 128 * wg;
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
    // 256-row down tiles; intermediate tiles are whole 128-row blocks by the ABI's checks
    return c.hidden % kGN == 0;
}

cudaError_t launch_expert_gemm(const GemmArgs& g, const TmaMaps& m, cudaStream_t st) {
    static size_t smem_set[3] = {0, 0, 0};
    const size_t smem = gemm_smem();
    const int mode = g.mode == 0 ? 0 : g.mode == 1 ? 1 : 2;
    auto kern = mode == 0 ? expert_gemm_kernel<0> : mode == 1 ? expert_gemm_kernel<1> : expert_gemm_kernel<2>;
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
    return cudaLaunchKernelEx(&cfg, kern, g, m.a_r, m.a_s, m.b0_r, m.b1_r, m.b0_s, m.b1_s);
}

}  // namespace moe
