// Internal interfaces between the C ABI (moe_api.cu) and the kernel files.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"  // include/ (on the include path)

namespace moe {

// Rows of activations one weight-streaming work item carries (the N=8 of the
// m16n8k32 MMA).
constexpr int kGroupRows = 8;
// Up to this many tokens the router + top-k + permutation run as one fused kernel.
constexpr int kSmallT = 64;
// Up to this many tokens the fused forward's streaming kernels derive the routing from the
// router's logits themselves (every CTA the same selection), so the router has no serial
// tail on the layer's critical path.
constexpr int kLocalT = 8;

// Control words at the start of the workspace (256 bytes, zeroed by
// moe_workspace_init and returned to zero by every call that changes them).
struct Ctrl {
    int status;              // device error bits (kStatusTimeout ...)
    unsigned route_arrived;  // last-block-done counter of the fused router
    int n_routed_groups;     // work descriptors written by the permutation
    int n_mtiles;            // 128-row token tiles of the routed experts (grouped GEMM)
    unsigned inject;         // fault injection for failure-detection tests (moe_debug_set), normally 0
    int pad[59];
};
static_assert(sizeof(Ctrl) == 256, "control block is 256 bytes");

// One activation row group of the expert GEMVs: up to kGroupRows rows of one expert
// (expert >= 0: permuted rows [row_begin, row_begin + nrows)) or of the shared experts
// (expert == -1: tokens [row_begin, row_begin + nrows)).
struct alignas(16) RowGroup {
    int expert;
    int row_begin;
    int nrows;
    int pad;
};

// One 128-row tile of an expert's permuted token rows (grouped GEMM work list).
struct MTile {
    int expert;
    int row0;
    int nrows;
    int pad;
};

// The grouped FP8 GEMM (tcgen05) of the large-T path; mode 0: gate/up -> SiLU(g)*u
// quantised to FP8, mode 1: down -> routing-weighted bf16 rows, mode 2: gate/up -> g and
// u in fp32 (the backward's recompute of the forward's pre-activations).

// Byte offsets of every workspace region for a given (config, T).
struct WsLayout {
    size_t ctrl;
    size_t logits;     // fp32 [splits, T, E] router partial logits
    size_t ids;        // int32 [T, k]
    size_t w;          // fp32 [T, k]
    size_t xq;         // u8 [T, H]
    size_t xs;         // fp32 [T, H/128]
    size_t rstd;       // fp32 [T] 1/rms of each token (stage M, large T)
    size_t offsets;    // int32 [E+1]
    size_t perm_src;   // int32 [T*k]
    size_t inv_pos;    // int32 [T*k]
    size_t groups;     // RowGroup [max_groups]
    size_t group_of_row;  // int32 [T*k]
    size_t perm_hist;  // int32 [ceil(T*k/1024), E] per-segment expert counts of the permutation
    size_t g_r, u_r, gb_r, ub_r;  // fp32 [P][T*k, I] each
    size_t g_s, u_s, gb_s, ub_s;  // fp32 [P][T, Is] each
    size_t y_r, yb_r;             // fp32 [P][T*k, H] each
    size_t y_s, yb_s;             // fp32 [P][T, H] each
    size_t xq_perm;    // u8 [T*k, H]                 (grouped GEMM path)
    size_t hq_r, hq_s;   // u8 [T*k, I], [T, Is]
    size_t hs_r, hs_s;   // fp32 [T*k, I/128], [T, Is/128]
    size_t mtiles;       // MTile [max_mtiles]
    int max_mtiles;
    size_t xs8, xs8_perm;  // MXFP8 variant: E8M0 activation scales [T, H/32], [T*k, H/32]
    size_t hs8_r, hs8_s;   //                and of the intermediate [T*k, I/32], [T, Is/32]
    size_t y_perm;     // bf16 [T*k, H]
    size_t y_shared;   // bf16 [T, H]
    size_t router_w3;  // bf16 [3][Ep][H]: the router weights' three-way split (large T)
    size_t total;
    int router_splits;
    int max_groups;
};

// mx: the MXFP8 variant's layout (E8M0 activation and intermediate scales added)
WsLayout ws_layout(const moe_config_t& c, int64_t T, bool mx = false);
int router_splits_for(const moe_config_t& c, int64_t T);
int max_routed_groups(const moe_config_t& c, int64_t T);

// Optional stage M in front of a kernel: gamma == nullptr means the input is used
// as it is. rstd: per-token 1/rms computed by rms_kernel (large T) or in-kernel.
struct NormArgs {
    const uint16_t* gamma = nullptr;  // bf16 [H]
    float eps = 0.f;
    float* rstd = nullptr;            // fp32 [T] workspace
};

// ------------------------------------------------------------ launchers
// All launchers enqueue on `st` and return cudaGetLastError().
// nm.gamma != nullptr: x is first normalised (stage M) with the 1/rms values in nm.rstd.
cudaError_t launch_quant_act(const void* x, int T, int H, uint8_t* xq, float* xs, const NormArgs& nm,
                             cudaStream_t st);

// Stage M alone: nm.rstd[t] = 1/rms of row t (if nm.rstd) and x_out = the normalised
// rows in bf16 (if x_out).
cudaError_t launch_rmsnorm(const void* x, int T, int H, const NormArgs& nm, void* x_out, cudaStream_t st);

// Fused small-T route: (stage M when nm.gamma, computed in-kernel), logits, x
// quantisation (MXFP8, per 32 values into xs8, when xs8 != nullptr), softmax + top-k, and (when offsets != nullptr) the permutation and
// row-group descriptors.
cudaError_t launch_route_small(const moe_config_t& c, const void* x, int T, const float* w_router,
                               const float* bias, int32_t* ids, float* w, float* logits,
                               uint8_t* xq, float* xs, int32_t* offsets, int32_t* perm_src,
                               int32_t* inv_pos, RowGroup* groups, int32_t* group_of_row, Ctrl* ctrl,
                               const NormArgs& nm, cudaStream_t st, uint8_t* xs8 = nullptr,
                               uint64_t* trace = nullptr, bool tail = true);

// Large-T route: router GEMM on tcgen05 (split-K partials) + softmax/top-k per token;
// w3 (router_w3_bytes) receives the weights' three-way bf16 split. With stage M the
// caller passes the normalised rows (launch_rmsnorm's x_out). logits: [splits, T, E] fp32.
cudaError_t launch_route_large(const moe_config_t& c, const void* x, int T, const float* w_router,
                               const float* bias, int32_t* ids, float* w, float* logits, int splits,
                               uint16_t* w3, int* status, cudaStream_t st);
// bytes of the three-way split router weights: bf16 [3][E rounded up to 16][H]
inline size_t router_w3_bytes(const moe_config_t& c) {
    return (size_t)3 * ((c.n_routed + 15) & ~15) * c.hidden * 2;
}

// Stable counting sort of the T*k pairs by expert; writes row groups when groups != nullptr.
// seg_hist: int32 [permute_segments(T*k), E] scratch.
int permute_segments(int64_t n);
cudaError_t launch_permute(const moe_config_t& c, const int32_t* ids, int T, int32_t* offsets,
                           int32_t* perm_src, int32_t* inv_pos, RowGroup* groups, int32_t* group_of_row,
                           MTile* mtiles, int32_t* seg_hist, Ctrl* ctrl, cudaStream_t st);

// Row groups from existing expert offsets (stage API path).
cudaError_t launch_build_groups(const moe_config_t& c, const int32_t* offsets, int n_rows, RowGroup* groups,
                                int32_t* group_of_row, MTile* mtiles, Ctrl* ctrl, cudaStream_t st);

// Opaque 128-byte TMA descriptor (a CUtensorMap), passed to kernels by value.
struct alignas(64) TmaMap {
    unsigned char bytes[128];
};

// 2-D tensor map of an 8-bit row-major [rows, cols] tensor with a box of
// box_rows x box_cols bytes and 128-byte swizzle (cached per address/shape/box).
bool tmap_bf16_2d(TmaMap* out, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                  uint32_t box_rows);
bool tmap_u8_2d(TmaMap* out, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows);

// Upper bound on the CTAs of the weight-streaming kernels (sizes the hand-off slots).
constexpr int kMaxStreamCtas = 512;

constexpr size_t kCtrlRegionBytes = sizeof(Ctrl);

struct StreamArgs {
    int H, I, Is, T, k, E, n_shared_groups;
    int grid_gu, grid_d, stages_d;  // launch shapes (the readers of partial tiles need them)
    int max_parts;                  // K parts the A buffers have room for
    int max_groups;                 // row-group capacity of the workspace
    int wide;                       // 1: unit indices may exceed 2^31 (64-bit tile arithmetic)
    int stream_once;                // 1: every weight byte is read by one row group (T <= 8): evict-first loads
                                    // of the shared experts too (the routed experts' always)
    const Ctrl* ctrl;
    const RowGroup* groups;
    const int32_t* group_of_row;  // [T*k] row group of each permuted row
    const int32_t* perm_src;
    const float* topk_w;
    const int32_t* inv_pos;
    // gate/up
    const float *s_gate, *s_up, *ss_gate, *ss_up;
    const uint8_t *ws_gate, *ws_up;  // raw pointers of the shared weights (L2 prefetch)
    const uint8_t* xq;
    const float* xs;
    float *g_r, *u_r;    // fp32 gate/up partial sums of routed rows [P][T*k, I]: A buffers
    float *gb_r, *ub_r;  // and B buffers (rest of a cut tile, or zeros)
    float *g_s, *u_s;    // shared rows [P][T, Is]
    float *gb_s, *ub_s;
    // down
    const float *s_down, *ss_down;
    float *y_r, *yb_r;  // fp32 weighted expert rows [P][T*k, H]: A and B buffers
    float *y_s, *yb_s;  // shared rows [P][T, H]
    // MXFP8 variant (mx = 1): E8M0 scales, one byte per row and 32 K, replace the fp32
    // block scales above; the activation scales xs8 [T, H/32] replace xs
    int mx;
    const uint8_t *s_gate8, *s_up8, *ss_gate8, *ss_up8, *s_down8, *ss_down8;
    const uint8_t* xs8;
    // combine
    int fuse_combine;  // 1: out (bf16) = sum of rows + shared (+ residual); 0: y_perm / y_shared (bf16)
    // Routing derived inside every streaming CTA (local_route = 1, up to kLocalT tokens):
    // the router leaves logits [T, E] only; each gate/up and down CTA runs top-k and the
    // permutation itself, and gate/up CTA 0 publishes them (ids, weights, perm_src, inv_pos,
    // offsets, row groups and their count) for the combine and the caller.
    int local_route;
    int G, Gk;
    float scale;
    const float* logits;
    int32_t* pub_ids;
    float* pub_w;
    int32_t* pub_perm;
    int32_t* pub_inv;
    int32_t* pub_offsets;
    RowGroup* pub_groups;
    int32_t* pub_group_of_row;
    int* pub_n_groups;
    __nv_bfloat16* y_perm;
    __nv_bfloat16* y_shared;
    const __nv_bfloat16* residual;
    __nv_bfloat16* out;
    int* status;
    uint64_t* trace;  // per-CTA timer stamps (moe_forward_trace) or null
};

struct GemmArgs {
    int mode;
    int H, I, Is, T, k;
    int K_r, K_s;      // reduction length of routed / shared tiles
    int nt_r, nt_s;    // weight tiles per token tile (routed / shared)
    int n_mt_s;        // shared token tiles
    const Ctrl* ctrl;
    const MTile* mtiles;
    const int32_t* perm_src;
    const float* topk_w;
    const float* xs;   // activation scales [T, H/128] (token order)
    const float *s_gate, *s_up, *s_down, *ss_gate, *ss_up, *ss_down;
    uint8_t *hq_r, *hq_s;   // FP8 intermediate (gate/up output, down input)
    float *hs_r, *hs_s;     // its scales, row-major [rows, width/128]
    uint8_t *hs8_r, *hs8_s; // MXFP8 variant: its E8M0 scales, row-major [rows, width/32]
    // MXFP8 variant: E8M0 scale rows [rows, K/32] of the A operand (routed, shared) and
    // of the two 128-row halves of the B tile (routed, shared)
    const uint8_t *sfa_r, *sfa_s, *sfb0_r, *sfb1_r, *sfb0_s, *sfb1_s;
    __nv_bfloat16* y_perm;
    __nv_bfloat16* y_shared;
    float *g_out_r, *u_out_r, *g_out_s, *u_out_s;  // mode 2: g and u [rows, width] fp32
    int* status;
};
struct TmaMaps {
    TmaMap a_r, a_s, b0_r, b1_r, b0_s, b1_s;
};
bool gemm_supported(const moe_config_t& c);
cudaError_t launch_expert_gemm(const GemmArgs& g, const TmaMaps& m, cudaStream_t st);

// MXFP8 variant: the same tiles and operand maps, E8M0 scales (GemmArgs::sfa_*, sfb*_*)
// through the tensor core.
bool gemm_mx_supported(const moe_config_t& c);
cudaError_t launch_expert_gemm_mx(const GemmArgs& g, const TmaMaps& m, cudaStream_t st);
// MXFP8 activation quantisation: per (token, 32 values) one E8M0 scale byte.
cudaError_t launch_quant_act_mx(const void* x, int T, int H, uint8_t* xq, uint8_t* xs8, const NormArgs& nm,
                                cudaStream_t st);

// xq_perm[r] = xq[token of r] (the routed rows in expert order); with xs8 != nullptr also
// xs8_perm[r] = xs8[token of r] (E8M0 rows of H/32 bytes). A row whose perm_src entry is
// outside [0, T*k) is written as zeros and sets kStatusBadId.
cudaError_t launch_gather_rows(int T, int H, int k, const int32_t* perm_src, const uint8_t* xq, uint8_t* xq_perm,
                               int* status, cudaStream_t st, const uint8_t* xs8 = nullptr,
                               uint8_t* xs8_perm = nullptr);

// ------------------------------------------------------------------ backward
// Workspace regions of the layer backward (byte offsets), for T tokens.
struct BwdLayout {
    size_t ctrl, logits, ids, w, xq, xs, offsets, perm_src, inv_pos, perm_hist, mtiles, xq_perm;
    size_t router_w3;                                 // bf16 [3][Ep][H]: split router weights
    size_t g_r, u_r, dau_r, wahat_r, dgu_r, dx_perm;  // routed rows: fp32 [R, I] x3, bf16 [R, I], [R, 2I], fp32 [R, H]
    size_t g_s, u_s, dau_s, wahat_s, dgu_s, dx_s;     // shared experts' tokens, the same with Is
    size_t dw, dlogit, dlogit_bf;                     // fp32 [T k], fp32 and bf16 [T, E]
    size_t wdT, wguT, wsdT, wsguT, wr_bf;  // bf16 weights: dequantised and transposed (K contiguous); router
    size_t xhat, xhat_perm, dout_perm;                // bf16 [T, H], [R, H], [R, H]
    size_t poff, pmap;                                // int32 [E + 1], [Rp]: padded expert columns
    size_t dout_permT, wahatT, dguT, xhat_permT;      // bf16 [H | I | 2I | H, Rp]
    size_t doutT, wahat_sT, dgu_sT, xhatT, dlogitT, xT;  // bf16 [H | Is | 2Is | H | E | H, Tp]
    int Rp, Tp;                                       // padded column counts (multiples of 64)
    size_t total;
    int splits, max_mtiles;
};
BwdLayout bwd_layout(const moe_config_t& c, int64_t T);
struct BwdArgs {
    int T;
    const void* x;                 // bf16 [T, H]
    const moe_weights_t* W;
    const int32_t* topk_ids;       // [T, k] the forward's expert choice
    const float* topk_w;           // [T, k] the forward's routing weights
    const void* dout;              // bf16 [T, H]
    float *dx, *dw_gate, *dw_up, *dw_down, *dws_gate, *dws_up, *dws_down, *dw_router, *dbias;
    const moe_stage_events_t* ev = nullptr;  // optional: events around the parts (moe_backward_profiled)
};
cudaError_t launch_backward(const moe_config_t& c, const BwdArgs& a, void* ws, cudaStream_t st);
// The backward's contractions on the tcgen05 tensor cores (bwd_tc.cu): dgrad C[r, :] =
// A[r, :] Bt_e^T; wgrad C_g = At Bt^T over the columns of group g.
cudaError_t launch_bwd_tc_wgrad(const void* At, int M, const void* Bt, int N, uint64_t cols, const int32_t* poff,
                                int groups, int K, float* C, float* C2, int msplit, size_t c_estride, int* status,
                                cudaStream_t st);
cudaError_t launch_bwd_tc(const void* A, uint64_t rows_a, const void* Bt, uint64_t n_mat, int K, int N, int routed,
                          int rows, const MTile* mtiles, const Ctrl* ctrl, float* C, int* status, cudaStream_t st);

int stream_grid();
int down_stages(int I, int Is);
int stream_max_parts(const moe_config_t& c, int64_t T);  // K parts the workspace provides for
cudaError_t launch_gateup_stream(const StreamArgs& a, const uint8_t* w_gate, const uint8_t* w_up, int E,
                                 cudaStream_t st);
cudaError_t launch_down_stream(const StreamArgs& a, const uint8_t* w_down, const uint8_t* ws_down, int E,
                               cudaStream_t st);
cudaError_t launch_stream_combine(const StreamArgs& a, cudaStream_t st);
cudaError_t launch_combine(int T, int H, int k, const __nv_bfloat16* y_perm, const int32_t* inv_pos,
                           const __nv_bfloat16* y_shared, const __nv_bfloat16* residual,
                           __nv_bfloat16* out, cudaStream_t st);

int num_sms();

}  // namespace moe
