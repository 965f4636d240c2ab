// Internal interfaces between the C ABI (moe_api.cu) and the kernel files.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Rows of activations one weight-streaming work item carries (the N=8 of the
// m16n8k32 MMA).
constexpr int kGroupRows = 8;
// Up to this many tokens the router + top-k + permutation run as one fused kernel.
constexpr int kSmallT = 64;

// Control words at the start of the workspace (256 bytes, zeroed by
// moe_workspace_init and returned to zero by every call that changes them).
struct Ctrl {
    int status;              // device error bits (kStatusTimeout ...)
    unsigned route_arrived;  // last-block-done counter of the fused router
    int n_routed_groups;     // work descriptors written by the permutation
    int pad[61];
};
static_assert(sizeof(Ctrl) == 256, "control block is 256 bytes");

// One activation row group of the expert GEMVs: up to kGroupRows rows of one expert
// (expert >= 0: permuted rows [row_begin, row_begin + nrows)) or of the shared experts
// (expert == -1: tokens [row_begin, row_begin + nrows)).
struct RowGroup {
    int expert;
    int row_begin;
    int nrows;
    int pad;
};

// Byte offsets of every workspace region for a given (config, T).
struct WsLayout {
    size_t ctrl;
    size_t logits;     // fp32 [splits, T, E] router partial logits
    size_t ids;        // int32 [T, k]
    size_t w;          // fp32 [T, k]
    size_t xq;         // u8 [T, H]
    size_t xs;         // fp32 [T, H/128]
    size_t offsets;    // int32 [E+1]
    size_t perm_src;   // int32 [T*k]
    size_t inv_pos;    // int32 [T*k]
    size_t groups;     // RowGroup [max_groups]
    size_t a_routed;   // fp32 [T*k, I]
    size_t a_shared;   // fp32 [T, Is]
    size_t y_perm;     // bf16 [T*k, H]
    size_t y_shared;   // bf16 [T, H]
    size_t total;
    int router_splits;
    int max_groups;
};

WsLayout ws_layout(const moe_config_t& c, int64_t T);
int router_splits_for(const moe_config_t& c, int64_t T);
int max_routed_groups(const moe_config_t& c, int64_t T);

// ------------------------------------------------------------ launchers
// All launchers enqueue on `st` and return cudaGetLastError().
cudaError_t launch_quant_act(const void* x, int T, int H, uint8_t* xq, float* xs, cudaStream_t st);

// Fused small-T route: logits, x quantisation, softmax + top-k, and (when
// offsets != nullptr) the permutation and row-group descriptors.
cudaError_t launch_route_small(const moe_config_t& c, const void* x, int T, const float* w_router,
                               const float* bias, int32_t* ids, float* w, float* logits,
                               uint8_t* xq, float* xs, int32_t* offsets, int32_t* perm_src,
                               int32_t* inv_pos, RowGroup* groups, Ctrl* ctrl, cudaStream_t st);

// Large-T route: tiled fp32 router (split-K partials) + softmax/top-k per token.
cudaError_t launch_route_large(const moe_config_t& c, const void* x, int T, const float* w_router,
                               const float* bias, int32_t* ids, float* w, float* logits, int splits,
                               cudaStream_t st);

// Stable counting sort of the T*k pairs by expert; writes row groups when groups != nullptr.
cudaError_t launch_permute(const moe_config_t& c, const int32_t* ids, int T, int32_t* offsets,
                           int32_t* perm_src, int32_t* inv_pos, RowGroup* groups, Ctrl* ctrl,
                           cudaStream_t st);

// Row groups from existing expert offsets (stage API path).
cudaError_t launch_build_groups(const moe_config_t& c, const int32_t* offsets, int n_rows, RowGroup* groups,
                                Ctrl* ctrl, cudaStream_t st);

struct ExpertArgs {
    int H, I, Is, T, k, n_shared_groups;
    const uint8_t *w_gate, *w_up, *w_down;
    const float *s_gate, *s_up, *s_down;
    const uint8_t *ws_gate, *ws_up, *ws_down;
    const float *ss_gate, *ss_up, *ss_down;
    const uint8_t* xq;
    const float* xs;
    const int32_t* perm_src;
    const float* topk_w;
    const RowGroup* groups;
    const Ctrl* ctrl;
    float* a_routed;
    float* a_shared;
    __nv_bfloat16* y_perm;
    __nv_bfloat16* y_shared;
    int max_groups;
};

cudaError_t launch_gateup_gemv(const ExpertArgs& a, cudaStream_t st);
cudaError_t launch_down_gemv(const ExpertArgs& a, cudaStream_t st);

cudaError_t launch_combine(int T, int H, int k, const __nv_bfloat16* y_perm, const int32_t* inv_pos,
                           const __nv_bfloat16* y_shared, const __nv_bfloat16* residual,
                           __nv_bfloat16* out, cudaStream_t st);

int num_sms();

}  // namespace moe
