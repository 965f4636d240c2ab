// Stages P1/P2 and Q1/Q2 of the MoE layer in the MXFP8 variant: E4M3 codes with one
// UE8M0 (power-of-two) scale per row and 32 consecutive K, for weights and activations
// (Mixture-of-Kittens Table 2, its MXFP8 routed-expert rows; the DeepSeek-V4.1 Flash
// lecture, "Round 1->2": converting the weights' 128-block scales to the MX layout
// so that the GEMMs run on Blackwell's block-scaled MXFP8 MMA).
//
// Such scales go through the tensor core (tcgen05.mma kind::mxf8f6f4, scale factors in
// tensor memory), so a tile's whole K reduction accumulates in one TMEM accumulator and
// the epilogue runs once per tile instead of once per 128-wide K block.
//
// Tiles as in expert_gemm.cu: 128 permuted token rows x 256 weight rows (gate/up: 128
// gate rows and the same 128 up rows; down: 256 hidden rows), one M=128 N=256 MMA per
// 32-wide K step. One CTA of 11 warps per SM:
//   warp 9      TMA producer: per 128-wide K block an A box and two B boxes (4-stage
//               ring)
//   warp 10     scale producer: per group of 4 K blocks the scale bytes of the tile's
//               128 A rows and 256 B rows, read by its 32 lanes from the row-major scale
//               tensors (16 bytes = 4 K blocks x 4 steps per row) and stored rearranged
//               into the tensor core's scale layout (below), a 2-slot ring
//   warp 8      MMA issuer (one thread): per group twelve tcgen05.cp 32x128b.warpx4
//               (A, B half 0, B half 1; 4 K blocks each) into tensor memory, then per K
//               block 4 tcgen05.mma, the descriptor's scale-factor ids picking the step's
//               byte
//   warps 0-7   epilogue: drains the accumulator into registers (warp w: lanes
//               32*(w%4).., column half w/4), releases it, then gate/up -> a = SiLU(g)*u
//               quantised per 32 values to E4M3 + E8M0 (the down GEMM's operand), or
//               down -> w * y in bf16.
// Scale layout. For one K block, the scales of 128 rows (A, or one half of B) form a
// 512-byte atom: 16 bytes per i = 0..31 holding the 4-byte words (the 4 K steps) of
// rows i, i+32, i+64, i+96. tcgen05.cp 32x128b.warpx4 puts the atom into 4 columns of
// every lane quadrant, and the MMA reads row 32q + i from lane 32q + i of column q; the
// 256 rows of B take two such groups side by side (rows 128.. in the next 4 columns).
// Tensor memory: columns 0-255 the accumulator; scale slot j at 256 + 64j: A at +4kb
// (4 columns per K block of the group), B at +16 + 8kb (8 columns per K block).
#include <algorithm>

#include "gemm_common.cuh"

namespace moe {

namespace {

using namespace gemm;

constexpr int kXStages = 4;
constexpr int kXEpiWarps = 8;
constexpr int kXMmaWarp = kXEpiWarps;
constexpr int kXProducerWarp = kXEpiWarps + 1;
constexpr int kXScaleWarp = kXEpiWarps + 2;
constexpr int kXThreads = (kXEpiWarps + 3) * 32;
constexpr int kXSA = kGM * kBlk;           // 16 KB A tile
constexpr int kXSB = kGN * kBlk;           // 32 KB B tile
constexpr int kXStage = kXSA + kXSB;
constexpr int kSfGroup = 4;                // K blocks per scale group
constexpr int kSfRow = 16;                 // scale bytes per row and group
constexpr int kSfAtom = 512;               // one K block of 128 rows
constexpr int kSfA = kSfGroup * kSfAtom;   // 2 KB
constexpr int kSfB = 2 * kSfGroup * kSfAtom;  // 4 KB: two 128-row halves
constexpr int kSfStage = kSfA + kSfB;
constexpr int kSfSlots = 4;  // TMEM: 256 + 4 x 64 columns = 512
constexpr uint32_t kXTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kSfSlotCols = 64;

struct MapsMX {
    const void *a_r, *a_s, *b0_r, *b1_r, *b0_s, *b1_s;
};

__device__ __forceinline__ uint32_t word(const uint4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

template <int kMode>  // 0: gate/up, 1: down
__global__ void __launch_bounds__(kXThreads, 1)
    expert_gemm_mx_kernel(const GemmArgs a, const __grid_constant__ TmaMaps tm) {
    constexpr bool gateup = kMode == 0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* sf_smem = smem + kXStages * kXStage;
    uint64_t* full = reinterpret_cast<uint64_t*>(sf_smem + kSfSlots * kSfStage);
    uint64_t* empty = full + kXStages;
    uint64_t* sf_full = empty + kXStages;    // [kSfSlots]
    uint64_t* sf_empty = sf_full + kSfSlots; // [kSfSlots]
    uint64_t* acc_full = sf_empty + kSfSlots;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* fin = acc_empty + 1;           // the MMA warp's last commit
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(fin + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);  // the MMA warp's commit
        }
        for (int j = 0; j < kSfSlots; ++j) {
            mbar_init(&sf_full[j], 1);
            mbar_init(&sf_empty[j], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kXEpiWarps);
        mbar_init(fin, 1);
        fence_mbar_init();
    }
    if (warp == kXMmaWarp) {
        tmem_alloc(s_tmem, kXTmemCols);
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
    const int total = items_in(0, n_r) * (a.K_r / kBlk) + items_in(n_r, n_items) * (a.K_s / kBlk);

    if (warp == kXProducerWarp) {
        // ----------------------------------------------------------- TMA producer
        if (lane == 0 && total > 0) {
            const MapsMX m{&tm.a_r, &tm.a_s, &tm.b0_r, &tm.b1_r, &tm.b0_s, &tm.b1_s};
            prefetch_tmap(m.a_r);
            prefetch_tmap(m.b0_r);
            prefetch_tmap(m.b1_r);
            LoadCursor lc;
            lc.item = blockIdx.x;
            lc.kb = 0;
            lc.set(a, n_mt_r, n_items, gateup);
            int n = 0;
            for (; n < total; ++n) {
                const int s = n % kXStages;
                if (n >= kXStages && !mbar_wait_bounded(&empty[s], ((n / kXStages) - 1) & 1)) {
                    set_status(a.status, kStatusTimeout);
                    break;
                }
                uint8_t* st = smem + s * kXStage;
                const int x = lc.kb * kBlk;
                mbar_arrive_expect_tx(&full[s], kXStage);
                tma_load_2d(st, lc.shared ? m.a_s : m.a_r, x, lc.row0, &full[s]);
                tma_load_2d(st + kXSA, lc.shared ? m.b0_s : m.b0_r, x, lc.yb0, &full[s]);
                tma_load_2d(st + kXSA + kXSB / 2, lc.shared ? m.b1_s : m.b1_r, x, lc.yb1, &full[s]);
                lc.next(a, n_mt_r, n_items, gateup);
            }
            // copies still in flight land before this CTA may exit
            for (int q = n > kXStages ? n - kXStages : 0; q < n; ++q)
                mbar_wait_bounded(&full[q % kXStages], (q / kXStages) & 1);
        }
    } else if (warp == kXScaleWarp) {
        // ------------------------------------------------------- scale producer
        // all 32 lanes; every tile's K blocks come in whole groups of 4 (K % 512 == 0)
        if (total > 0) {
            const int rows_r = a.T * a.k;
            LoadCursor gc;
            gc.item = blockIdx.x;
            gc.kb = 0;
            gc.set(a, n_mt_r, n_items, gateup);
            // scale rows of a group: A rows row0 + lane + 32*m1, B half h rows yb_h + lane + 32*m1
            // (16 bytes each). Two register sets: the loads of groups g+1 and g+2 are in flight
            // while group g waits for its slot, so a group's load latency spans two groups' MMAs.
            auto fetch = [&](uint4 (&pa)[4], uint4 (&pb)[8]) {
                if (gc.item >= n_items) return;
                const int Kg = (gc.shared ? a.K_s : a.K_r) / 32;  // scale bytes per row
                const size_t off = (size_t)(gc.kb / kSfGroup) * kSfRow;
                const uint8_t* sa = gc.shared ? a.sfa_s : a.sfa_r;
                const int ra = gc.shared ? a.T : rows_r;
#pragma unroll
                for (int m1 = 0; m1 < 4; ++m1) {
                    const int r = gc.row0 + lane + 32 * m1;
                    pa[m1] = r < ra ? __ldg(reinterpret_cast<const uint4*>(sa + (size_t)r * Kg + off))
                                    : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint8_t* sb = h == 0 ? (gc.shared ? a.sfb0_s : a.sfb0_r) : (gc.shared ? a.sfb1_s : a.sfb1_r);
                    const int y = h == 0 ? gc.yb0 : gc.yb1;
#pragma unroll
                    for (int m1 = 0; m1 < 4; ++m1)
                        pb[4 * h + m1] =
                            __ldg(reinterpret_cast<const uint4*>(sb + (size_t)(y + lane + 32 * m1) * Kg + off));
                }
                // advance to the next group: 4 K blocks on, or the next tile
                gc.kb += kSfGroup;
                if (gc.kb >= gc.Kb) {
                    gc.kb = 0;
                    gc.item += gridDim.x;
                    gc.set(a, n_mt_r, n_items, gateup);
                }
            };
            // waits for slot g % kSfSlots, stores the group as 512-byte atoms, hands it over
            auto publish = [&](int g, const uint4 (&pa)[4], const uint4 (&pb)[8]) -> bool {
                const int j = g % kSfSlots;
                bool ok = true;
                if (g >= kSfSlots && lane == 0) ok = mbar_wait_bounded(&sf_empty[j], ((g / kSfSlots) - 1) & 1);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    if (lane == 0) set_status(a.status, kStatusTimeout);
                    return false;
                }
                uint8_t* sf = sf_smem + j * kSfStage;
#pragma unroll
                for (int jj = 0; jj < kSfGroup; ++jj) {
                    reinterpret_cast<uint4*>(sf + jj * kSfAtom)[lane] =
                        make_uint4(word(pa[0], jj), word(pa[1], jj), word(pa[2], jj), word(pa[3], jj));
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        reinterpret_cast<uint4*>(sf + kSfA + (h * kSfGroup + jj) * kSfAtom)[lane] =
                            make_uint4(word(pb[4 * h], jj), word(pb[4 * h + 1], jj), word(pb[4 * h + 2], jj),
                                       word(pb[4 * h + 3], jj));
                }
                fence_proxy_async_smem();  // the tensor core reads these through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_full[j]);
                return true;
            };
            uint4 pa0[4], pb0[8], pa1[4], pb1[8];
            fetch(pa0, pb0);
            fetch(pa1, pb1);
            const int groups = total / kSfGroup;
            for (int g = 0; g < groups; g += 2) {
                if (!publish(g, pa0, pb0)) break;
                fetch(pa0, pb0);
                if (g + 1 < groups) {
                    if (!publish(g + 1, pa1, pb1)) break;
                    fetch(pa1, pb1);
                }
            }
        }
    } else if (warp == kXMmaWarp) {
        // -------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int n = 0, g = 0, tile = 0;
            bool stop = false;
            for (int item = blockIdx.x; item < n_items && !stop; item += gridDim.x, ++tile) {
                const Item it = decode_item(a, n_mt_r, item);
                const int Kb = (it.shared ? a.K_s : a.K_r) / kBlk;
                if (tile > 0 && !mbar_wait_bounded(acc_empty, (tile - 1) & 1)) {
                    set_status(a.status, kStatusTimeout);
                    break;
                }
                tc_fence_after();
                uint32_t sfc = 0;
                for (int kb = 0; kb < Kb; ++kb, ++n) {
                    if (kb % kSfGroup == 0) {
                        const int j = g % kSfSlots;
                        if (!mbar_wait_bounded(&sf_full[j], (g / kSfSlots) & 1)) {
                            set_status(a.status, kStatusTimeout);
                            stop = true;
                            break;
                        }
                        tc_fence_after();
                        const uint8_t* sf = sf_smem + j * kSfStage;
                        sfc = tmem + kAccCols + j * kSfSlotCols;
#pragma unroll
                        for (int jj = 0; jj < kSfGroup; ++jj) {
                            tc_cp_32x128b_x4(sfc + 4 * jj, smem_desc_rows16(sf + jj * kSfAtom));
                            tc_cp_32x128b_x4(sfc + 16 + 8 * jj, smem_desc_rows16(sf + kSfA + jj * kSfAtom));
                            tc_cp_32x128b_x4(sfc + 16 + 8 * jj + 4,
                                             smem_desc_rows16(sf + kSfA + (kSfGroup + jj) * kSfAtom));
                        }
                        ++g;
                    }
                    const int s = n % kXStages;
                    if (!mbar_wait_bounded(&full[s], (n / kXStages) & 1)) {
                        set_status(a.status, kStatusTimeout);
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* st = smem + s * kXStage;
                    const uint64_t da = smem_desc_sw128(st);
                    const uint64_t db = smem_desc_sw128(st + kXSA);
                    const uint32_t col = 4u * (uint32_t)(kb % kSfGroup);  // this K block's scale columns
#pragma unroll
                    for (int k = 0; k < 4; ++k)      // one N=256 MMA per K step
                        tc_mma_mx(tmem, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc_mx_f32(kGM, 256, k),
                                  sfc + col, sfc + 16 + 2 * col, (kb | k) != 0);
                    tc_commit(&empty[s]);
                    if (kb % kSfGroup == kSfGroup - 1 || kb == Kb - 1) tc_commit(&sf_empty[(g - 1) % kSfSlots]);
                }
                if (stop) break;
                tc_commit(acc_full);
            }
            // every tcgen05 operation issued (MMAs and scale copies) has completed before the
            // CTA frees tensor memory; a barrier of its own, so no other wait sees the arrival
            if (n > 0 || g > 0) {
                tc_commit(fin);
                mbar_wait_bounded(fin, 0);
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q4 = warp & 3;          // TMEM lane quadrant: rows 32q .. 32q+31
        const int wg = warp >> 2;         // column half
        const int row = 32 * q4 + lane;   // tile row of this thread
        const uint32_t t_row = tmem + ((uint32_t)(32 * q4) << 16);
        bool ok = true;
        int tile = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++tile) {
            const Item it = decode_item(a, n_mt_r, item);
            const bool valid_row = row < it.nrows;
            const int grow = it.row0 + row;  // row in the A tensor and the output tensors
            float wrow = 1.f;                // routing weight of this row (down)
            if (!gateup && !it.shared && valid_row) {
                const int f = a.perm_src[grow];
                wrow = ((unsigned)f < (unsigned)(a.T * a.k)) ? a.topk_w[f] : 0.f;
            }
            if (ok && !mbar_wait_bounded(acc_full, tile & 1)) ok = false;
            ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
            tc_fence_after();
            float v0[32], v1[32], v2[32], v3[32];
            if (ok) {
                // gate/up: gate cols 64wg.. (v0, v1) and up cols 128+64wg.. (v2, v3);
                // down: cols 128wg.. (v0..v3)
                const uint32_t c0 = gateup ? 64 * wg : 128 * wg;
                const uint32_t c2 = gateup ? 128 + 64 * wg : 128 * wg + 64;
                tmem_ld32(t_row + c0, v0);
                tmem_ld32(t_row + c0 + 32, v1);
                tmem_ld32(t_row + c2, v2);
                tmem_ld32(t_row + c2 + 32, v3);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);  // the next tile's MMAs may start
            if (!ok || !valid_row) continue;
            if (gateup) {
                // a = SiLU(g) * u for 64 channels, two MX blocks of 32 per thread
                const int N = it.shared ? a.Is : a.I;
                uint8_t* dst = (it.shared ? a.hq_s : a.hq_r) + (size_t)grow * N + it.ntile * kBlk + 64 * wg;
                uint32_t sb[2];
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    float* h = blk == 0 ? v0 : v1;  // a overwrites g in place
                    const float* u = blk == 0 ? v2 : v3;
                    float amax = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        h[j] = silu_mul(h[j], u[j]);
                        amax = fmaxf(amax, fabsf(h[j]));
                    }
                    float inv;
                    sb[blk] = act_scale_e8m0(amax, &inv);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint4 w;
                        w.x = pack_e4m3x4(h[16 * c + 0] * inv, h[16 * c + 1] * inv, h[16 * c + 2] * inv,
                                          h[16 * c + 3] * inv);
                        w.y = pack_e4m3x4(h[16 * c + 4] * inv, h[16 * c + 5] * inv, h[16 * c + 6] * inv,
                                          h[16 * c + 7] * inv);
                        w.z = pack_e4m3x4(h[16 * c + 8] * inv, h[16 * c + 9] * inv, h[16 * c + 10] * inv,
                                          h[16 * c + 11] * inv);
                        w.w = pack_e4m3x4(h[16 * c + 12] * inv, h[16 * c + 13] * inv, h[16 * c + 14] * inv,
                                          h[16 * c + 15] * inv);
                        reinterpret_cast<uint4*>(dst + 32 * blk)[c] = w;
                    }
                }
                // row-major [rows, N/32] E8M0: the down GEMM's A scale bytes
                uint8_t* sdst = (it.shared ? a.hs8_s : a.hs8_r) + (size_t)grow * (N / 32) + it.ntile * 4 + 2 * wg;
                *reinterpret_cast<uint16_t*>(sdst) = (uint16_t)(sb[0] | (sb[1] << 8));
            } else {
                __nv_bfloat16* dst =
                    (it.shared ? a.y_shared : a.y_perm) + (size_t)grow * a.H + it.ntile * kGN + 128 * wg;
                const float* vs[4] = {v0, v1, v2, v3};
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    uint4 o;
                    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const int j = 8 * c + 2 * p;
                        const __nv_bfloat162 h2 =
                            __floats2bfloat162_rn(vs[j >> 5][j & 31] * wrow, vs[(j + 1) >> 5][(j + 1) & 31] * wrow);
                        ow[p] = *reinterpret_cast<const uint32_t*>(&h2);
                    }
                    reinterpret_cast<uint4*>(dst)[c] = o;
                }
            }
        }
        if (!ok) set_status(a.status, kStatusTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kXMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kXTmemCols);
    }
}

size_t gemm_mx_smem() {
    return (size_t)kXStages * kXStage + (size_t)kSfSlots * kSfStage + 1024 + (2 * kXStages + 2 * kSfSlots + 3) * 8 + 16;
}

}  // namespace

bool gemm_mx_supported(const moe_config_t& c) {
    // 256-row down tiles; scale rows of whole 16-byte groups (4 K blocks of 128)
    return c.hidden % kGN == 0 && c.hidden % 512 == 0 && c.moe_inter % 512 == 0;
}

cudaError_t launch_expert_gemm_mx(const GemmArgs& g, const TmaMaps& m, cudaStream_t st) {
    static size_t smem_set[2] = {0, 0};
    const size_t smem = gemm_mx_smem();
    const int mode = g.mode == 0 ? 0 : 1;
    auto kern = mode == 0 ? expert_gemm_mx_kernel<0> : expert_gemm_mx_kernel<1>;
    if (smem_set[mode] < smem) {
        const cudaError_t e =
            cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set[mode] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(num_sms(), kMaxStreamCtas));
    cfg.blockDim = dim3(kXThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, g, m);
}

}  // namespace moe
