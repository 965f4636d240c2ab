// The C ABI of include/moe.h: host-side argument checks, workspace carving and
// the launch sequence of each entry point. No entry point allocates memory or
// synchronises the host, except moe_read_device_status (documented).
#include <algorithm>
#include <cstddef>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

int num_sms() {
    static const int n = [] {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return 152;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 152;
        return v;
    }();
    return n;
}

static_assert(kTraceCtas == MOE_TRACE_CTAS, "trace layout of moe.h");

static size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

int router_splits_for(const moe_config_t& c, int64_t T) {
    if (T <= kSmallT) return 1;  // the fused small-T route kernel
    const int64_t tiles = (T + 127) / 128;  // router CTAs: 128 tokens x all experts each
    int64_t s = 152 / tiles;                // at most one CTA per SM of a 152-SM part
    const int64_t hb = c.hidden / 128;
    if (s > 8) s = 8;
    if (s > hb) s = hb;
    return (int)(s < 1 ? 1 : s);
}

int max_routed_groups(const moe_config_t& c, int64_t T) {
    const int64_t n = T * c.top_k;
    const int64_t touched = n < c.n_routed ? n : c.n_routed;
    return (int)(n / kGroupRows + touched + 1);
}

// Many tokens per expert: the grouped tensor-core GEMM instead of the streaming GEMVs.
bool use_gemm(const moe_config_t& c, int64_t T) { return T > kSmallT && gemm_supported(c); }

WsLayout ws_layout(const moe_config_t& c, int64_t T, bool mx) {
    WsLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    };
    const size_t H = c.hidden, I = c.moe_inter, E = c.n_routed, k = c.top_k;
    const size_t Is = (size_t)c.n_shared * c.moe_inter;
    const size_t t = (size_t)T;
    L.router_splits = router_splits_for(c, T);
    L.max_groups = max_routed_groups(c, T);
    L.ctrl = take(kCtrlRegionBytes);
    L.logits = take((size_t)L.router_splits * t * E * 4);  // router split-K partials
    L.ids = take(t * k * 4);
    L.w = take(t * k * 4);
    L.xq = take(t * H);
    L.xs = take(t * (H / 128) * 4);
    L.rstd = take(t * 4);
    L.offsets = take((E + 1) * 4);
    L.perm_src = take(t * k * 4);
    L.inv_pos = take(t * k * 4);
    L.groups = take((size_t)L.max_groups * sizeof(RowGroup));
    L.group_of_row = take(t * k * 4);
    L.perm_hist = take((size_t)permute_segments((int64_t)(t * k)) * E * 4);
    // the streaming GEMVs' partial sums; on the GEMM path they stay sized for kSmallT
    // tokens so that the workspace size never shrinks as T grows
    // the MXFP8 variant streams at T <= 64 too, and its GEMM needs no 256-multiple hidden
    const bool gemm = mx ? T > kSmallT : use_gemm(c, T);
    const size_t ts = gemm ? (size_t)kSmallT : t;
    const size_t P = (size_t)stream_max_parts(c, (int64_t)ts);
    {
        const size_t t = ts;
    L.g_r = take(P * t * k * I * 4);
    L.u_r = take(P * t * k * I * 4);
    L.gb_r = take(P * t * k * I * 4);
    L.ub_r = take(P * t * k * I * 4);
    L.g_s = take(P * t * Is * 4);
    L.u_s = take(P * t * Is * 4);
    L.gb_s = take(P * t * Is * 4);
    L.ub_s = take(P * t * Is * 4);
    L.y_r = take(P * t * k * H * 4);
    L.yb_r = take(P * t * k * H * 4);
    L.y_s = take(P * t * H * 4);
    L.yb_s = take(P * t * H * 4);
    }
    L.max_mtiles = 0;
    L.xq_perm = L.hq_r = L.hq_s = L.hs_r = L.hs_s = L.mtiles = 0;
    if (gemm) {
        L.max_mtiles = (int)((t * k + 127) / 128 + std::min(E, t * k));
        L.xq_perm = take(t * k * H);
        L.hq_r = take(t * k * I);
        L.hq_s = take(t * Is);
        L.hs_r = take(t * k * (I / 128) * 4);
        L.hs_s = take(t * (Is / 128) * 4);
        L.mtiles = take((size_t)L.max_mtiles * sizeof(MTile));
    }
    L.xs8 = L.xs8_perm = L.hs8_r = L.hs8_s = 0;
    if (mx) {
        L.xs8 = take(t * (H / 32));
        L.xs8_perm = take(t * k * (H / 32));
        L.hs8_r = take(t * k * (I / 32));
        L.hs8_s = take(t * (Is / 32));
    }
    L.y_perm = take(t * k * H * 2);
    L.y_shared = take(t * H * 2);
    L.router_w3 = T > kSmallT ? take(router_w3_bytes(c)) : 0;
    L.total = off;
    return L;
}

}  // namespace moe

using namespace moe;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

moe_status_t check_cfg(const moe_config_t* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->hidden <= 0 || c->hidden % 128 || c->hidden > 32768) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->moe_inter <= 0 || c->moe_inter % 128 || c->moe_inter > 16384) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->n_routed < 1 || c->n_routed > 256) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->n_group < 1 || c->n_group > 32 || c->n_routed % c->n_group) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->topk_group < 1 || c->topk_group > c->n_group) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->top_k < 1 || c->top_k > 16 || c->top_k > c->topk_group * (c->n_routed / c->n_group))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->n_shared < 0 || (int64_t)c->n_shared * c->moe_inter > 16384) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!std::isfinite(c->routed_scaling_factor)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

moe_status_t check_T(const moe_config_t* c, int32_t T) {
    if (T < 0) return MOE_ERR_INVALID_ARG;
    // flat (token, slot) indices and row offsets are int32
    if ((int64_t)T * c->top_k > (int64_t)INT32_MAX / 2) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

moe_status_t check_ws(const moe_config_t* c, int32_t T, const void* ws, size_t ws_bytes) {
    if (!ws || !aligned16(ws)) return MOE_ERR_WORKSPACE;
    if (ws_bytes < ws_layout(*c, T).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status_t check_weights(const moe_config_t* c, const moe_weights_t* w, bool need_router) {
    if (!w) return MOE_ERR_INVALID_ARG;
    const void* req[] = {w->w_gate, w->w_up, w->w_down, w->s_gate, w->s_up, w->s_down};
    for (const void* p : req)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (c->n_shared > 0) {
        const void* sh[] = {w->ws_gate, w->ws_up, w->ws_down, w->ss_gate, w->ss_up, w->ss_down};
        for (const void* p : sh)
            if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    }
    if (need_router) {
        if (!w->w_router || !aligned16(w->w_router)) return MOE_ERR_INVALID_ARG;
        if (w->router_bias && !aligned4(w->router_bias)) return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

#define MOE_TRY(expr)                         \
    do {                                      \
        const moe_status_t _s = (expr);       \
        if (_s != MOE_OK) return _s;          \
    } while (0)

#define MOE_CUDA(expr)                                   \
    do {                                                 \
        if ((expr) != cudaSuccess) return MOE_ERR_CUDA;  \
    } while (0)

template <class T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// The streaming kernels need 64-bit unit indices: the most units a stage can have (every
// row group and shared group times the 128-row slices of its matrix times its K blocks,
// the same count for gate/up and down), times the CTAs, may pass 2^31.
bool stream_wide(const moe_config_t* c, int32_t T, const WsLayout& L) {
    const int64_t sgroups = c->n_shared > 0 ? (T + kGroupRows - 1) / kGroupRows : 0;
    const int64_t units = ((int64_t)L.max_groups * (c->moe_inter / kBlk) +
                           sgroups * ((int64_t)c->n_shared * c->moe_inter / kBlk)) * (c->hidden / kBlk);
    return units > (int64_t)INT32_MAX / (2 * kMaxStreamCtas);
}

StreamArgs stream_args(const moe_config_t* c, int32_t T, const moe_weights_t* W, const WsLayout& L, void* ws,
                       const int32_t* perm_src, const float* topk_w) {
    StreamArgs a = {};
    a.H = c->hidden;
    a.I = c->moe_inter;
    a.Is = c->n_shared * c->moe_inter;
    a.T = T;
    a.k = c->top_k;
    a.E = c->n_routed;
    a.n_shared_groups = c->n_shared > 0 ? (T + kGroupRows - 1) / kGroupRows : 0;
    a.grid_gu = stream_grid();
    a.grid_d = stream_grid();
    a.stages_d = down_stages(a.I, a.Is);
    a.max_parts = stream_max_parts(*c, T);
    a.max_groups = L.max_groups;
    a.wide = stream_wide(c, T, L) ? 1 : 0;
    // up to 8 tokens every routed expert's rows form one row group and the shared experts'
    // tokens another, so each weight byte is streamed exactly once
    a.stream_once = T <= kGroupRows ? 1 : 0;
    a.ctrl = at<Ctrl>(ws, L.ctrl);
    a.groups = at<RowGroup>(ws, L.groups);
    a.group_of_row = at<int32_t>(ws, L.group_of_row);
    a.perm_src = perm_src;
    a.topk_w = topk_w;
    a.inv_pos = at<int32_t>(ws, L.inv_pos);
    a.s_gate = W->s_gate;
    a.s_up = W->s_up;
    a.ss_gate = W->ss_gate;
    a.ss_up = W->ss_up;
    a.ws_gate = W->ws_gate;
    a.ws_up = W->ws_up;
    a.xq = at<uint8_t>(ws, L.xq);
    a.xs = at<float>(ws, L.xs);
    a.g_r = at<float>(ws, L.g_r);
    a.u_r = at<float>(ws, L.u_r);
    a.gb_r = at<float>(ws, L.gb_r);
    a.ub_r = at<float>(ws, L.ub_r);
    a.g_s = at<float>(ws, L.g_s);
    a.u_s = at<float>(ws, L.u_s);
    a.gb_s = at<float>(ws, L.gb_s);
    a.ub_s = at<float>(ws, L.ub_s);
    a.s_down = W->s_down;
    a.ss_down = W->ss_down;
    a.y_r = at<float>(ws, L.y_r);
    a.yb_r = at<float>(ws, L.yb_r);
    a.y_s = at<float>(ws, L.y_s);
    a.yb_s = at<float>(ws, L.yb_s);
    a.status = &at<Ctrl>(ws, L.ctrl)->status;
    return a;
}

// Routing inside the streaming kernels (T <= kLocalT): the router leaves logits only; the
// gate/up kernel's CTA 0 publishes the selection and the permutation into the workspace.
void set_local_route(StreamArgs* a, const moe_config_t* c, const WsLayout& L, void* ws) {
    a->local_route = 1;
    a->G = c->n_group;
    a->Gk = c->topk_group;
    a->scale = c->routed_scaling_factor;
    a->logits = at<float>(ws, L.logits);
    a->pub_ids = at<int32_t>(ws, L.ids);
    a->pub_w = at<float>(ws, L.w);
    a->pub_perm = at<int32_t>(ws, L.perm_src);
    a->pub_inv = at<int32_t>(ws, L.inv_pos);
    a->pub_offsets = at<int32_t>(ws, L.offsets);
    a->pub_groups = at<RowGroup>(ws, L.groups);
    a->pub_group_of_row = at<int32_t>(ws, L.group_of_row);
    a->pub_n_groups = &at<Ctrl>(ws, L.ctrl)->n_routed_groups;
}

// The streaming kernels' arguments for MXFP8 weights (E8M0 scale rows).
StreamArgs stream_args_mx(const moe_config_t* c, int32_t T, const moe_weights_mx_t* W, const WsLayout& L, void* ws,
                          const int32_t* perm_src, const float* topk_w) {
    moe_weights_t Wb = {};  // codes and router only; the fp32 scale pointers stay null
    Wb.w_gate = W->w_gate;
    Wb.w_up = W->w_up;
    Wb.w_down = W->w_down;
    Wb.ws_gate = W->ws_gate;
    Wb.ws_up = W->ws_up;
    Wb.ws_down = W->ws_down;
    StreamArgs a = stream_args(c, T, &Wb, L, ws, perm_src, topk_w);
    a.mx = 1;
    a.s_gate8 = W->s_gate;
    a.s_up8 = W->s_up;
    a.s_down8 = W->s_down;
    a.ss_gate8 = W->ss_gate;
    a.ss_up8 = W->ss_up;
    a.ss_down8 = W->ss_down;
    a.xs8 = at<uint8_t>(ws, L.xs8);
    return a;
}

struct StageMark {
    const moe_stage_events_t* ev;
    cudaStream_t st;
    moe_status_t begin(moe_stage_t s) const {
        if (ev && ev->start[s] && cudaEventRecord((cudaEvent_t)ev->start[s], st) != cudaSuccess) return MOE_ERR_CUDA;
        return MOE_OK;
    }
    moe_status_t end(moe_stage_t s) const {
        if (ev && ev->stop[s] && cudaEventRecord((cudaEvent_t)ev->stop[s], st) != cudaSuccess) return MOE_ERR_CUDA;
        return MOE_OK;
    }
};

// Both grouped-GEMM launches of the large-T path: gate/up (x -> FP8 SiLU(g)*u) and
// down (-> routing-weighted bf16 rows in y_perm, shared experts' rows in y_shared).
cudaError_t run_expert_gemms(const moe_config_t* c, int32_t T, const moe_weights_t* W, const WsLayout& L, void* ws,
                             const int32_t* perm_src, const float* topk_w, __nv_bfloat16* y_perm,
                             __nv_bfloat16* y_shared, const StageMark* mark) {
    const int H = c->hidden, I = c->moe_inter, E = c->n_routed, k = c->top_k;
    const int Is = c->n_shared * c->moe_inter;
    const bool sh = Is > 0;
    const uint64_t n = (uint64_t)T * k;
    cudaStream_t st = mark->st;
    GemmArgs g = {};
    g.H = H;
    g.I = I;
    g.Is = Is;
    g.T = T;
    g.k = k;
    g.n_mt_s = sh ? (T + 127) / 128 : 0;
    g.ctrl = at<Ctrl>(ws, L.ctrl);
    g.mtiles = at<MTile>(ws, L.mtiles);
    g.perm_src = perm_src;
    g.topk_w = topk_w;
    g.xs = at<float>(ws, L.xs);
    g.s_gate = W->s_gate;
    g.s_up = W->s_up;
    g.s_down = W->s_down;
    g.ss_gate = W->ss_gate;
    g.ss_up = W->ss_up;
    g.ss_down = W->ss_down;
    g.hq_r = at<uint8_t>(ws, L.hq_r);
    g.hq_s = at<uint8_t>(ws, L.hq_s);
    g.hs_r = at<float>(ws, L.hs_r);
    g.hs_s = at<float>(ws, L.hs_s);
    g.y_perm = y_perm;
    g.y_shared = y_shared;
    g.status = &at<Ctrl>(ws, L.ctrl)->status;

    TmaMaps m = {};
    // gate/up: A = permuted activation codes (routed) / token-order codes (shared)
    g.mode = 0;
    g.K_r = g.K_s = H;
    g.nt_r = I / 128;
    g.nt_s = Is / 128;
    if (!tmap_u8_2d(&m.a_r, at<uint8_t>(ws, L.xq_perm), n, H, 128, 128) ||
        !tmap_u8_2d(&m.b0_r, W->w_gate, (uint64_t)E * I, H, 128, 128) ||
        !tmap_u8_2d(&m.b1_r, W->w_up, (uint64_t)E * I, H, 128, 128))
        return cudaErrorInvalidValue;
    if (sh && (!tmap_u8_2d(&m.a_s, at<uint8_t>(ws, L.xq), T, H, 128, 128) ||
               !tmap_u8_2d(&m.b0_s, W->ws_gate, Is, H, 128, 128) ||
               !tmap_u8_2d(&m.b1_s, W->ws_up, Is, H, 128, 128)))
        return cudaErrorInvalidValue;
    if (mark->begin(MOE_STAGE_GATE_UP) != MOE_OK) return cudaErrorUnknown;
    cudaError_t e = launch_expert_gemm(g, m, st);
    if (e != cudaSuccess) return e;
    if (mark->end(MOE_STAGE_GATE_UP) != MOE_OK) return cudaErrorUnknown;

    // down: A = the FP8 intermediate, B = 256 hidden rows per tile
    g.mode = 1;
    g.K_r = I;
    g.K_s = Is;
    g.nt_r = g.nt_s = H / 256;
    m = TmaMaps{};
    if (!tmap_u8_2d(&m.a_r, g.hq_r, n, I, 128, 128) ||
        !tmap_u8_2d(&m.b0_r, W->w_down, (uint64_t)E * H, I, 128, 128))
        return cudaErrorInvalidValue;
    m.b1_r = m.b0_r;
    if (sh && (!tmap_u8_2d(&m.a_s, g.hq_s, T, Is, 128, 128) || !tmap_u8_2d(&m.b0_s, W->ws_down, H, Is, 128, 128)))
        return cudaErrorInvalidValue;
    m.b1_s = m.b0_s;
    if (mark->begin(MOE_STAGE_DOWN) != MOE_OK) return cudaErrorUnknown;
    e = launch_expert_gemm(g, m, st);
    if (e != cudaSuccess) return e;
    if (mark->end(MOE_STAGE_DOWN) != MOE_OK) return cudaErrorUnknown;
    return cudaSuccess;
}

// The MXFP8 variant's two grouped-GEMM launches (scales through the tensor core).
cudaError_t run_expert_gemms_mx(const moe_config_t* c, int32_t T, const moe_weights_mx_t* W, const WsLayout& L,
                                void* ws, const int32_t* perm_src, const float* topk_w, __nv_bfloat16* y_perm,
                                __nv_bfloat16* y_shared, const StageMark* mark) {
    const int H = c->hidden, I = c->moe_inter, E = c->n_routed, k = c->top_k;
    const int Is = c->n_shared * c->moe_inter;
    const bool sh = Is > 0;
    const uint64_t n = (uint64_t)T * k;
    cudaStream_t st = mark->st;
    GemmArgs g = {};
    g.H = H;
    g.I = I;
    g.Is = Is;
    g.T = T;
    g.k = k;
    g.n_mt_s = sh ? (T + 127) / 128 : 0;
    g.ctrl = at<Ctrl>(ws, L.ctrl);
    g.mtiles = at<MTile>(ws, L.mtiles);
    g.perm_src = perm_src;
    g.topk_w = topk_w;
    g.hq_r = at<uint8_t>(ws, L.hq_r);
    g.hq_s = at<uint8_t>(ws, L.hq_s);
    g.hs8_r = at<uint8_t>(ws, L.hs8_r);
    g.hs8_s = at<uint8_t>(ws, L.hs8_s);
    g.y_perm = y_perm;
    g.y_shared = y_shared;
    g.status = &at<Ctrl>(ws, L.ctrl)->status;

    TmaMaps m = {};
    // gate/up: A = permuted activation codes (routed) / token-order codes (shared)
    g.mode = 0;
    g.K_r = g.K_s = H;
    g.nt_r = I / 128;
    g.nt_s = Is / 128;
    g.sfa_r = at<uint8_t>(ws, L.xs8_perm);
    g.sfa_s = at<uint8_t>(ws, L.xs8);
    g.sfb0_r = W->s_gate;
    g.sfb1_r = W->s_up;
    g.sfb0_s = W->ss_gate;
    g.sfb1_s = W->ss_up;
    if (!tmap_u8_2d(&m.a_r, at<uint8_t>(ws, L.xq_perm), n, H, 128, 128) ||
        !tmap_u8_2d(&m.b0_r, W->w_gate, (uint64_t)E * I, H, 128, 128) ||
        !tmap_u8_2d(&m.b1_r, W->w_up, (uint64_t)E * I, H, 128, 128))
        return cudaErrorInvalidValue;
    if (sh && (!tmap_u8_2d(&m.a_s, at<uint8_t>(ws, L.xq), T, H, 128, 128) ||
               !tmap_u8_2d(&m.b0_s, W->ws_gate, Is, H, 128, 128) || !tmap_u8_2d(&m.b1_s, W->ws_up, Is, H, 128, 128)))
        return cudaErrorInvalidValue;
    if (mark->begin(MOE_STAGE_GATE_UP) != MOE_OK) return cudaErrorUnknown;
    cudaError_t e = launch_expert_gemm_mx(g, m, st);
    if (e != cudaSuccess) return e;
    if (mark->end(MOE_STAGE_GATE_UP) != MOE_OK) return cudaErrorUnknown;

    // down: A = the FP8 intermediate, B = 256 hidden rows per tile (two 128-row halves)
    g.mode = 1;
    g.K_r = I;
    g.K_s = Is;
    g.nt_r = g.nt_s = H / 256;
    m = TmaMaps{};
    g.sfa_r = g.hs8_r;
    g.sfa_s = g.hs8_s;
    g.sfb0_r = g.sfb1_r = W->s_down;  // the B halves are rows yb0 and yb0 + 128 of one tensor
    g.sfb0_s = g.sfb1_s = W->ss_down;
    if (!tmap_u8_2d(&m.a_r, g.hq_r, n, I, 128, 128) || !tmap_u8_2d(&m.b0_r, W->w_down, (uint64_t)E * H, I, 128, 128))
        return cudaErrorInvalidValue;
    m.b1_r = m.b0_r;
    if (sh && (!tmap_u8_2d(&m.a_s, g.hq_s, T, Is, 128, 128) || !tmap_u8_2d(&m.b0_s, W->ws_down, H, Is, 128, 128)))
        return cudaErrorInvalidValue;
    m.b1_s = m.b0_s;
    if (mark->begin(MOE_STAGE_DOWN) != MOE_OK) return cudaErrorUnknown;
    e = launch_expert_gemm_mx(g, m, st);
    if (e != cudaSuccess) return e;
    if (mark->end(MOE_STAGE_DOWN) != MOE_OK) return cudaErrorUnknown;
    return cudaSuccess;
}

moe_status_t check_weights_mx(const moe_config_t* c, const moe_weights_mx_t* w) {
    if (!w) return MOE_ERR_INVALID_ARG;
    const void* req[] = {w->w_gate, w->w_up, w->w_down, w->s_gate, w->s_up, w->s_down, w->w_router};
    for (const void* p : req)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (c->n_shared > 0) {
        const void* sh[] = {w->ws_gate, w->ws_up, w->ws_down, w->ss_gate, w->ss_up, w->ss_down};
        for (const void* p : sh)
            if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    }
    if (w->router_bias && !aligned4(w->router_bias)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

size_t moe_workspace_size(const moe_config_t* cfg, int32_t max_tokens) {
    if (check_cfg(cfg) != MOE_OK || max_tokens < 0 || check_T(cfg, max_tokens) != MOE_OK) return 0;
    return ws_layout(*cfg, max_tokens).total;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || ws_bytes < sizeof(Ctrl)) return MOE_ERR_WORKSPACE;
    MOE_CUDA(cudaMemsetAsync(ws, 0, ws_bytes < kCtrlRegionBytes ? ws_bytes : kCtrlRegionBytes,
                             (cudaStream_t)stream));
    return MOE_OK;
}

moe_status_t moe_debug_set(void* ws, size_t ws_bytes, uint32_t inject, void* stream) {
    static_assert(kInjectSkipGateupLoads == MOE_INJECT_SKIP_GATEUP_LOADS, "inject bit of moe.h");
    if (!ws || ws_bytes < sizeof(Ctrl)) return MOE_ERR_WORKSPACE;
    if (inject & ~kInjectSkipGateupLoads) return MOE_ERR_INVALID_ARG;
    const uint32_t word = inject;  // staged by the copy before it returns
    MOE_CUDA(cudaMemcpyAsync(static_cast<uint8_t*>(ws) + offsetof(Ctrl, inject), &word, sizeof(word),
                             cudaMemcpyHostToDevice, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status_t moe_read_device_status(void* ws, void* stream) {
    if (!ws) return MOE_ERR_WORKSPACE;
    int h = 0;
    cudaStream_t st = (cudaStream_t)stream;
    MOE_CUDA(cudaMemcpyAsync(&h, ws, sizeof(int), cudaMemcpyDeviceToHost, st));
    MOE_CUDA(cudaStreamSynchronize(st));
    if (h == 0) return MOE_OK;
    MOE_CUDA(cudaMemsetAsync(ws, 0, sizeof(int), st));
    MOE_CUDA(cudaStreamSynchronize(st));
    if (h & kStatusTimeout) return MOE_ERR_DEVICE_TIMEOUT;
    return MOE_ERR_INVALID_ARG;
}

size_t moe_backward_workspace_size(const moe_config_t* cfg, int32_t max_tokens) {
    if (check_cfg(cfg) != MOE_OK || max_tokens < 0 || check_T(cfg, max_tokens) != MOE_OK || !gemm_supported(*cfg) ||
        cfg->n_routed % 16)
        return 0;
    return bwd_layout(*cfg, max_tokens).total;
}

moe_status_t moe_backward_profiled(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                                   const moe_weights_t* weights, const int32_t* topk_ids, const float* topk_w,
                                   const void* dout_bf16, float* dx, float* dw_gate, float* dw_up, float* dw_down,
                                   float* dws_gate, float* dws_up, float* dws_down, float* dw_router, float* dbias,
                                   void* ws, size_t ws_bytes, void* stream, const moe_stage_events_t* events) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_T(cfg, T));
    if (!gemm_supported(*cfg) || cfg->n_routed % 16) return MOE_ERR_UNSUPPORTED_SHAPE;
    MOE_TRY(check_weights(cfg, weights, true));
    const void* req[] = {dw_gate, dw_up, dw_down, dw_router};  // the per-token arrays only when T > 0
    for (const void* p : req)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    const void* treq[] = {x_bf16, topk_ids, topk_w, dout_bf16, dx};
    for (const void* p : treq)
        if (T > 0 && (!p || !aligned16(p))) return MOE_ERR_INVALID_ARG;
    const bool sh = cfg->n_shared > 0;
    if (sh) {
        const void* sreq[] = {dws_gate, dws_up, dws_down};
        for (const void* p : sreq)
            if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    }
    if (dbias && !aligned4(dbias)) return MOE_ERR_INVALID_ARG;
    if (!ws || !aligned16(ws) || ws_bytes < bwd_layout(*cfg, T).total) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t H = cfg->hidden, I = cfg->moe_inter, E = cfg->n_routed, Is = (size_t)cfg->n_shared * I;
    if (T == 0) {  // sums over no tokens
        MOE_CUDA(cudaMemsetAsync(dw_gate, 0, E * I * H * 4, st));
        MOE_CUDA(cudaMemsetAsync(dw_up, 0, E * I * H * 4, st));
        MOE_CUDA(cudaMemsetAsync(dw_down, 0, E * H * I * 4, st));
        MOE_CUDA(cudaMemsetAsync(dw_router, 0, E * H * 4, st));
        if (dbias) MOE_CUDA(cudaMemsetAsync(dbias, 0, E * 4, st));
        if (sh) {
            MOE_CUDA(cudaMemsetAsync(dws_gate, 0, Is * H * 4, st));
            MOE_CUDA(cudaMemsetAsync(dws_up, 0, Is * H * 4, st));
            MOE_CUDA(cudaMemsetAsync(dws_down, 0, H * Is * 4, st));
        }
        return MOE_OK;
    }
    BwdArgs a;
    a.T = T;
    a.x = x_bf16;
    a.W = weights;
    a.topk_ids = topk_ids;
    a.topk_w = topk_w;
    a.dout = dout_bf16;
    a.dx = dx;
    a.dw_gate = dw_gate;
    a.dw_up = dw_up;
    a.dw_down = dw_down;
    a.dws_gate = sh ? dws_gate : nullptr;
    a.dws_up = sh ? dws_up : nullptr;
    a.dws_down = sh ? dws_down : nullptr;
    a.dw_router = dw_router;
    a.dbias = dbias;
    a.ev = events;
    MOE_CUDA(launch_backward(*cfg, a, ws, st));
    return MOE_OK;
}

moe_status_t moe_backward(const moe_config_t* cfg, const void* x_bf16, int32_t T, const moe_weights_t* weights,
                          const int32_t* topk_ids, const float* topk_w, const void* dout_bf16, float* dx,
                          float* dw_gate, float* dw_up, float* dw_down, float* dws_gate, float* dws_up,
                          float* dws_down, float* dw_router, float* dbias, void* ws, size_t ws_bytes, void* stream) {
    return moe_backward_profiled(cfg, x_bf16, T, weights, topk_ids, topk_w, dout_bf16, dx, dw_gate, dw_up, dw_down,
                                 dws_gate, dws_up, dws_down, dw_router, dbias, ws, ws_bytes, stream, nullptr);
}

moe_status_t moe_quant_act(const void* x_bf16, int32_t T, int32_t H, uint8_t* xq, float* xs, void* stream) {
    if (T < 0 || H <= 0 || H % 128) return T < 0 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !xq || !xs || !aligned16(x_bf16) || !aligned16(xq) || !aligned16(xs)) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_quant_act(x_bf16, T, H, xq, xs, NormArgs{}, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status_t moe_rmsnorm(const void* h_bf16, int32_t T, int32_t H, const void* gamma_bf16, float eps,
                         void* x_bf16, void* stream) {
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (H <= 0 || H % 8 || H > 65536) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!std::isfinite(eps) || eps < 0.f) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!h_bf16 || !gamma_bf16 || !x_bf16 || !aligned16(h_bf16) || !aligned16(gamma_bf16) || !aligned16(x_bf16))
        return MOE_ERR_INVALID_ARG;
    NormArgs nm;
    nm.gamma = static_cast<const uint16_t*>(gamma_bf16);
    nm.eps = eps;
    MOE_CUDA(launch_rmsnorm(h_bf16, T, H, nm, x_bf16, (cudaStream_t)stream));
    return MOE_OK;
}

static moe_status_t route_impl(const moe_config_t* cfg, const void* x_bf16, int32_t T, const float* w_router,
                               const float* router_bias, int32_t* topk_ids, float* topk_w, void* ws,
                               size_t ws_bytes, void* stream, NormArgs nm) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_T(cfg, T));
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !w_router || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(w_router) || !aligned16(topk_ids) || !aligned16(topk_w))
        return MOE_ERR_INVALID_ARG;
    if (router_bias && !aligned4(router_bias)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
    const WsLayout L = ws_layout(*cfg, T);
    cudaStream_t st = (cudaStream_t)stream;
    if (T <= kSmallT) {
        MOE_CUDA(launch_route_small(*cfg, x_bf16, T, w_router, router_bias, topk_ids, topk_w, at<float>(ws, L.logits),
                                    at<uint8_t>(ws, L.xq), at<float>(ws, L.xs), nullptr, nullptr, nullptr, nullptr,
                                    nullptr, at<Ctrl>(ws, L.ctrl), nm, st));
    } else {
        const void* xr = x_bf16;
        if (nm.gamma) {  // the normalised rows, in the y_perm region (free until the expert GEMMs)
            nm.rstd = at<float>(ws, L.rstd);
            MOE_CUDA(launch_rmsnorm(x_bf16, T, cfg->hidden, nm, at<uint16_t>(ws, L.y_perm), st));
            xr = at<uint16_t>(ws, L.y_perm);
        }
        MOE_CUDA(launch_route_large(*cfg, xr, T, w_router, router_bias, topk_ids, topk_w, at<float>(ws, L.logits),
                                    L.router_splits, at<uint16_t>(ws, L.router_w3), &at<Ctrl>(ws, L.ctrl)->status,
                                    st));
    }
    return MOE_OK;
}

moe_status_t moe_route(const moe_config_t* cfg, const void* x_bf16, int32_t T, const float* w_router,
                       const float* router_bias, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
                       void* stream) {
    return route_impl(cfg, x_bf16, T, w_router, router_bias, topk_ids, topk_w, ws, ws_bytes, stream, NormArgs{});
}

moe_status_t moe_route_rmsnorm(const moe_config_t* cfg, const void* h_bf16, int32_t T, const void* gamma_bf16,
                               float eps, const float* w_router, const float* router_bias, int32_t* topk_ids,
                               float* topk_w, void* ws, size_t ws_bytes, void* stream) {
    if (!gamma_bf16 || !aligned16(gamma_bf16) || !std::isfinite(eps) || eps < 0.f) return MOE_ERR_INVALID_ARG;
    NormArgs nm;
    nm.gamma = static_cast<const uint16_t*>(gamma_bf16);
    nm.eps = eps;
    return route_impl(cfg, h_bf16, T, w_router, router_bias, topk_ids, topk_w, ws, ws_bytes, stream, nm);
}

moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_ids, int32_t T, int32_t* expert_offsets,
                         int32_t* perm_src, int32_t* inv_pos, void* ws, size_t ws_bytes, void* stream) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_T(cfg, T));
    if (T == 0) return MOE_OK;
    const void* req[] = {topk_ids, expert_offsets, perm_src, inv_pos};
    for (const void* p : req)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
    const WsLayout L = ws_layout(*cfg, T);
    MOE_CUDA(launch_permute(*cfg, topk_ids, T, expert_offsets, perm_src, inv_pos, nullptr, nullptr, nullptr,
                            at<int32_t>(ws, L.perm_hist), at<Ctrl>(ws, L.ctrl), (cudaStream_t)stream));
    return MOE_OK;
}

moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* x_bf16, int32_t T, const moe_weights_t* weights,
                            const int32_t* expert_offsets, const int32_t* perm_src, const float* topk_w,
                            void* y_perm_bf16, void* y_shared_bf16, void* ws, size_t ws_bytes, void* stream) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_T(cfg, T));
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights(cfg, weights, false));
    const void* req[] = {x_bf16, expert_offsets, perm_src, topk_w, y_perm_bf16};
    for (const void* p : req)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (cfg->n_shared > 0 && (!y_shared_bf16 || !aligned16(y_shared_bf16))) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
    const WsLayout L = ws_layout(*cfg, T);
    cudaStream_t st = (cudaStream_t)stream;
    MOE_CUDA(launch_quant_act(x_bf16, T, cfg->hidden, at<uint8_t>(ws, L.xq), at<float>(ws, L.xs), NormArgs{}, st));
    if (use_gemm(*cfg, T)) {
        MOE_CUDA(launch_build_groups(*cfg, expert_offsets, T * cfg->top_k, nullptr, nullptr, at<MTile>(ws, L.mtiles),
                                     at<Ctrl>(ws, L.ctrl), st));
        MOE_CUDA(launch_gather_rows(T, cfg->hidden, cfg->top_k, perm_src, at<uint8_t>(ws, L.xq),
                                    at<uint8_t>(ws, L.xq_perm), &at<Ctrl>(ws, L.ctrl)->status, st));
        const StageMark mark{nullptr, st};
        MOE_CUDA(run_expert_gemms(cfg, T, weights, L, ws, perm_src, topk_w, static_cast<__nv_bfloat16*>(y_perm_bf16),
                                  static_cast<__nv_bfloat16*>(y_shared_bf16), &mark));
        return MOE_OK;
    }
    MOE_CUDA(launch_build_groups(*cfg, expert_offsets, T * cfg->top_k, at<RowGroup>(ws, L.groups),
                                 at<int32_t>(ws, L.group_of_row), nullptr, at<Ctrl>(ws, L.ctrl), st));
    StreamArgs a = stream_args(cfg, T, weights, L, ws, perm_src, topk_w);
    a.fuse_combine = 0;
    a.y_perm = static_cast<__nv_bfloat16*>(y_perm_bf16);
    a.y_shared = static_cast<__nv_bfloat16*>(y_shared_bf16);
    MOE_CUDA(launch_gateup_stream(a, weights->w_gate, weights->w_up, cfg->n_routed, st));
    MOE_CUDA(launch_down_stream(a, weights->w_down, weights->ws_down, cfg->n_routed, st));
    MOE_CUDA(launch_stream_combine(a, st));
    return MOE_OK;
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* y_perm_bf16, const int32_t* inv_pos,
                         const void* y_shared_bf16, const void* residual_bf16, int32_t T, void* out_bf16,
                         void* stream) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_T(cfg, T));
    if (T == 0) return MOE_OK;
    const void* req[] = {y_perm_bf16, inv_pos, out_bf16};
    for (const void* p : req)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if ((y_shared_bf16 && !aligned16(y_shared_bf16)) || (residual_bf16 && !aligned16(residual_bf16)))
        return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_combine(T, cfg->hidden, cfg->top_k, static_cast<const __nv_bfloat16*>(y_perm_bf16), inv_pos,
                            static_cast<const __nv_bfloat16*>(y_shared_bf16),
                            static_cast<const __nv_bfloat16*>(residual_bf16), static_cast<__nv_bfloat16*>(out_bf16),
                            (cudaStream_t)stream));
    return MOE_OK;
}

static moe_status_t forward_impl(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                                 const moe_weights_t* weights, const void* residual_bf16, void* out_bf16,
                                 int32_t* topk_ids_out, void* ws, size_t ws_bytes, void* stream,
                                 const moe_stage_events_t* events, NormArgs nm, uint64_t* trace = nullptr) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_T(cfg, T));
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights(cfg, weights, true));
    if (!x_bf16 || !out_bf16 || !aligned16(x_bf16) || !aligned16(out_bf16)) return MOE_ERR_INVALID_ARG;
    if ((residual_bf16 && !aligned16(residual_bf16)) || (topk_ids_out && !aligned4(topk_ids_out)))
        return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
    const WsLayout L = ws_layout(*cfg, T);
    cudaStream_t st = (cudaStream_t)stream;
    const StageMark mark{events, st};
    int32_t* ids = at<int32_t>(ws, L.ids);
    float* w = at<float>(ws, L.w);
    int32_t* perm_src = at<int32_t>(ws, L.perm_src);
    int32_t* inv_pos = at<int32_t>(ws, L.inv_pos);
    Ctrl* ctrl = at<Ctrl>(ws, L.ctrl);
    RowGroup* groups = at<RowGroup>(ws, L.groups);

    // the streaming kernels route (see set_local_route)
    const bool local = T <= kLocalT && !stream_wide(cfg, T, L);
    MOE_TRY(mark.begin(MOE_STAGE_ROUTE));
    if (T <= kSmallT) {
        MOE_CUDA(launch_route_small(*cfg, x_bf16, T, weights->w_router, weights->router_bias, ids, w,
                                    at<float>(ws, L.logits), at<uint8_t>(ws, L.xq), at<float>(ws, L.xs),
                                    at<int32_t>(ws, L.offsets), perm_src, inv_pos, groups,
                                    at<int32_t>(ws, L.group_of_row), ctrl, nm, st, nullptr, trace, !local));
        MOE_TRY(mark.end(MOE_STAGE_ROUTE));
    } else {
        const void* xr = x_bf16;
        if (nm.gamma) {  // the normalised rows, in the y_perm region (free until the expert GEMMs)
            nm.rstd = at<float>(ws, L.rstd);
            MOE_CUDA(launch_rmsnorm(x_bf16, T, cfg->hidden, nm, at<uint16_t>(ws, L.y_perm), st));
            xr = at<uint16_t>(ws, L.y_perm);
        }
        MOE_CUDA(launch_route_large(*cfg, xr, T, weights->w_router, weights->router_bias, ids, w,
                                    at<float>(ws, L.logits), L.router_splits, at<uint16_t>(ws, L.router_w3),
                                    &ctrl->status, st));
        MOE_CUDA(launch_quant_act(x_bf16, T, cfg->hidden, at<uint8_t>(ws, L.xq), at<float>(ws, L.xs), nm, st));
        MOE_TRY(mark.end(MOE_STAGE_ROUTE));
        MOE_TRY(mark.begin(MOE_STAGE_PERMUTE));
        if (use_gemm(*cfg, T)) {
            MOE_CUDA(launch_permute(*cfg, ids, T, at<int32_t>(ws, L.offsets), perm_src, inv_pos, nullptr, nullptr,
                                    at<MTile>(ws, L.mtiles), at<int32_t>(ws, L.perm_hist), ctrl, st));
            MOE_CUDA(launch_gather_rows(T, cfg->hidden, cfg->top_k, perm_src, at<uint8_t>(ws, L.xq),
                                        at<uint8_t>(ws, L.xq_perm), &ctrl->status, st));
            MOE_TRY(mark.end(MOE_STAGE_PERMUTE));
            __nv_bfloat16* y_perm = at<__nv_bfloat16>(ws, L.y_perm);
            __nv_bfloat16* y_shared = cfg->n_shared > 0 ? at<__nv_bfloat16>(ws, L.y_shared) : nullptr;
            MOE_CUDA(run_expert_gemms(cfg, T, weights, L, ws, perm_src, w, y_perm, y_shared, &mark));
            MOE_TRY(mark.begin(MOE_STAGE_COMBINE));
            MOE_CUDA(launch_combine(T, cfg->hidden, cfg->top_k, y_perm, inv_pos, y_shared,
                                    static_cast<const __nv_bfloat16*>(residual_bf16),
                                    static_cast<__nv_bfloat16*>(out_bf16), st));
            MOE_TRY(mark.end(MOE_STAGE_COMBINE));
            if (topk_ids_out)
                MOE_CUDA(cudaMemcpyAsync(topk_ids_out, ids, (size_t)T * cfg->top_k * sizeof(int32_t),
                                         cudaMemcpyDeviceToDevice, st));
            return MOE_OK;
        }
        MOE_CUDA(launch_permute(*cfg, ids, T, at<int32_t>(ws, L.offsets), perm_src, inv_pos, groups,
                                at<int32_t>(ws, L.group_of_row), nullptr, at<int32_t>(ws, L.perm_hist), ctrl, st));
        MOE_TRY(mark.end(MOE_STAGE_PERMUTE));
    }
    StreamArgs a = stream_args(cfg, T, weights, L, ws, perm_src, w);
    a.fuse_combine = 1;
    if (local) set_local_route(&a, cfg, L, ws);
    a.residual = static_cast<const __nv_bfloat16*>(residual_bf16);
    a.out = static_cast<__nv_bfloat16*>(out_bf16);
    a.trace = trace;
    MOE_TRY(mark.begin(MOE_STAGE_GATE_UP));
    MOE_CUDA(launch_gateup_stream(a, weights->w_gate, weights->w_up, cfg->n_routed, st));
    MOE_TRY(mark.end(MOE_STAGE_GATE_UP));
    MOE_TRY(mark.begin(MOE_STAGE_DOWN));
    MOE_CUDA(launch_down_stream(a, weights->w_down, weights->ws_down, cfg->n_routed, st));
    MOE_TRY(mark.end(MOE_STAGE_DOWN));
    MOE_TRY(mark.begin(MOE_STAGE_COMBINE));
    MOE_CUDA(launch_stream_combine(a, st));
    MOE_TRY(mark.end(MOE_STAGE_COMBINE));
    if (topk_ids_out)
        MOE_CUDA(cudaMemcpyAsync(topk_ids_out, ids, (size_t)T * cfg->top_k * sizeof(int32_t),
                                 cudaMemcpyDeviceToDevice, st));
    return MOE_OK;
}

moe_status_t moe_forward_profiled(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                                  const moe_weights_t* weights, const void* residual_bf16, void* out_bf16,
                                  int32_t* topk_ids_out, void* ws, size_t ws_bytes, void* stream,
                                  const moe_stage_events_t* events) {
    return forward_impl(cfg, x_bf16, T, weights, residual_bf16, out_bf16, topk_ids_out, ws, ws_bytes, stream,
                        events, NormArgs{});
}

moe_status_t moe_forward(const moe_config_t* cfg, const void* x_bf16, int32_t T, const moe_weights_t* weights,
                         const void* residual_bf16, void* out_bf16, int32_t* topk_ids_out, void* ws,
                         size_t ws_bytes, void* stream) {
    return forward_impl(cfg, x_bf16, T, weights, residual_bf16, out_bf16, topk_ids_out, ws, ws_bytes, stream,
                        nullptr, NormArgs{});
}

moe_status_t moe_forward_trace(const moe_config_t* cfg, const void* x_bf16, int32_t T, const moe_weights_t* weights,
                               const void* residual_bf16, void* out_bf16, void* ws, size_t ws_bytes, void* stream,
                               uint64_t* trace) {
    if (!trace || !aligned16(trace)) return MOE_ERR_INVALID_ARG;
    return forward_impl(cfg, x_bf16, T, weights, residual_bf16, out_bf16, nullptr, ws, ws_bytes, stream, nullptr,
                        NormArgs{}, trace);
}

moe_status_t moe_forward_rmsnorm_profiled(const moe_config_t* cfg, const void* h_bf16, int32_t T,
                                          const void* gamma_bf16, float eps, const moe_weights_t* weights,
                                          void* out_bf16, int32_t* topk_ids_out, void* ws, size_t ws_bytes,
                                          void* stream, const moe_stage_events_t* events) {
    if (!gamma_bf16 || !aligned16(gamma_bf16) || !std::isfinite(eps) || eps < 0.f) return MOE_ERR_INVALID_ARG;
    if (out_bf16 == h_bf16) return MOE_ERR_INVALID_ARG;  // h is also the residual
    NormArgs nm;
    nm.gamma = static_cast<const uint16_t*>(gamma_bf16);
    nm.eps = eps;
    return forward_impl(cfg, h_bf16, T, weights, h_bf16, out_bf16, topk_ids_out, ws, ws_bytes, stream, events, nm);
}

moe_status_t moe_forward_rmsnorm(const moe_config_t* cfg, const void* h_bf16, int32_t T, const void* gamma_bf16,
                                 float eps, const moe_weights_t* weights, void* out_bf16, int32_t* topk_ids_out,
                                 void* ws, size_t ws_bytes, void* stream) {
    return moe_forward_rmsnorm_profiled(cfg, h_bf16, T, gamma_bf16, eps, weights, out_bf16, topk_ids_out, ws,
                                        ws_bytes, stream, nullptr);
}

size_t moe_workspace_size_mx(const moe_config_t* cfg, int32_t max_tokens) {
    if (check_cfg(cfg) != MOE_OK || max_tokens < 0 || check_T(cfg, max_tokens) != MOE_OK) return 0;
    if (!gemm_mx_supported(*cfg)) return 0;
    return ws_layout(*cfg, max_tokens, true).total;
}

moe_status_t moe_quant_act_mx(const void* x_bf16, int32_t T, int32_t H, uint8_t* xq, uint8_t* xs_e8m0,
                              void* stream) {
    if (T < 0 || H <= 0 || H % 128) return T < 0 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !xq || !xs_e8m0 || !aligned16(x_bf16) || !aligned16(xq)) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_quant_act_mx(x_bf16, T, H, xq, xs_e8m0, NormArgs{}, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status_t moe_forward_mx_profiled(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                                     const moe_weights_mx_t* weights, const void* residual_bf16, void* out_bf16,
                                     int32_t* topk_ids_out, void* ws, size_t ws_bytes, void* stream,
                                     const moe_stage_events_t* events) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_T(cfg, T));
    if (!gemm_mx_supported(*cfg)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights_mx(cfg, weights));
    if (!x_bf16 || !out_bf16 || !aligned16(x_bf16) || !aligned16(out_bf16)) return MOE_ERR_INVALID_ARG;
    if ((residual_bf16 && !aligned16(residual_bf16)) || (topk_ids_out && !aligned4(topk_ids_out)))
        return MOE_ERR_INVALID_ARG;
    if (!ws || !aligned16(ws)) return MOE_ERR_WORKSPACE;
    const WsLayout L = ws_layout(*cfg, T, true);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const StageMark mark{events, st};
    int32_t* ids = at<int32_t>(ws, L.ids);
    float* w = at<float>(ws, L.w);
    int32_t* perm_src = at<int32_t>(ws, L.perm_src);
    int32_t* inv_pos = at<int32_t>(ws, L.inv_pos);
    Ctrl* ctrl = at<Ctrl>(ws, L.ctrl);

    MOE_TRY(mark.begin(MOE_STAGE_ROUTE));
    if (T <= kSmallT) {
        // decode: the fused route (x quantised per 32), then the weight-streaming kernels
        const bool local = T <= kLocalT && !stream_wide(cfg, T, L);  // the streaming kernels route
        MOE_CUDA(launch_route_small(*cfg, x_bf16, T, weights->w_router, weights->router_bias, ids, w,
                                    at<float>(ws, L.logits), at<uint8_t>(ws, L.xq), at<float>(ws, L.xs),
                                    at<int32_t>(ws, L.offsets), perm_src, inv_pos, at<RowGroup>(ws, L.groups),
                                    at<int32_t>(ws, L.group_of_row), ctrl, NormArgs{}, st, at<uint8_t>(ws, L.xs8),
                                    nullptr, !local));
        MOE_TRY(mark.end(MOE_STAGE_ROUTE));
        StreamArgs a = stream_args_mx(cfg, T, weights, L, ws, perm_src, w);
        a.fuse_combine = 1;
        if (local) set_local_route(&a, cfg, L, ws);
        a.residual = static_cast<const __nv_bfloat16*>(residual_bf16);
        a.out = static_cast<__nv_bfloat16*>(out_bf16);
        MOE_TRY(mark.begin(MOE_STAGE_GATE_UP));
        MOE_CUDA(launch_gateup_stream(a, weights->w_gate, weights->w_up, cfg->n_routed, st));
        MOE_TRY(mark.end(MOE_STAGE_GATE_UP));
        MOE_TRY(mark.begin(MOE_STAGE_DOWN));
        MOE_CUDA(launch_down_stream(a, weights->w_down, weights->ws_down, cfg->n_routed, st));
        MOE_TRY(mark.end(MOE_STAGE_DOWN));
        MOE_TRY(mark.begin(MOE_STAGE_COMBINE));
        MOE_CUDA(launch_stream_combine(a, st));
        MOE_TRY(mark.end(MOE_STAGE_COMBINE));
        if (topk_ids_out)
            MOE_CUDA(cudaMemcpyAsync(topk_ids_out, ids, (size_t)T * cfg->top_k * sizeof(int32_t),
                                     cudaMemcpyDeviceToDevice, st));
        return MOE_OK;
    }
    MOE_CUDA(launch_route_large(*cfg, x_bf16, T, weights->w_router, weights->router_bias, ids, w,
                                at<float>(ws, L.logits), L.router_splits, at<uint16_t>(ws, L.router_w3),
                                &ctrl->status, st));
    MOE_CUDA(launch_quant_act_mx(x_bf16, T, cfg->hidden, at<uint8_t>(ws, L.xq), at<uint8_t>(ws, L.xs8), NormArgs{},
                                 st));
    MOE_TRY(mark.end(MOE_STAGE_ROUTE));
    MOE_TRY(mark.begin(MOE_STAGE_PERMUTE));
    MOE_CUDA(launch_permute(*cfg, ids, T, at<int32_t>(ws, L.offsets), perm_src, inv_pos, nullptr, nullptr,
                            at<MTile>(ws, L.mtiles), at<int32_t>(ws, L.perm_hist), ctrl, st));
    MOE_CUDA(launch_gather_rows(T, cfg->hidden, cfg->top_k, perm_src, at<uint8_t>(ws, L.xq), at<uint8_t>(ws, L.xq_perm),
                                &ctrl->status, st, at<uint8_t>(ws, L.xs8), at<uint8_t>(ws, L.xs8_perm)));
    MOE_TRY(mark.end(MOE_STAGE_PERMUTE));
    __nv_bfloat16* y_perm = at<__nv_bfloat16>(ws, L.y_perm);
    __nv_bfloat16* y_shared = cfg->n_shared > 0 ? at<__nv_bfloat16>(ws, L.y_shared) : nullptr;
    MOE_CUDA(run_expert_gemms_mx(cfg, T, weights, L, ws, perm_src, w, y_perm, y_shared, &mark));
    MOE_TRY(mark.begin(MOE_STAGE_COMBINE));
    MOE_CUDA(launch_combine(T, cfg->hidden, cfg->top_k, y_perm, inv_pos, y_shared,
                            static_cast<const __nv_bfloat16*>(residual_bf16), static_cast<__nv_bfloat16*>(out_bf16),
                            st));
    MOE_TRY(mark.end(MOE_STAGE_COMBINE));
    if (topk_ids_out)
        MOE_CUDA(cudaMemcpyAsync(topk_ids_out, ids, (size_t)T * cfg->top_k * sizeof(int32_t),
                                 cudaMemcpyDeviceToDevice, st));
    return MOE_OK;
}

moe_status_t moe_forward_mx(const moe_config_t* cfg, const void* x_bf16, int32_t T, const moe_weights_mx_t* weights,
                            const void* residual_bf16, void* out_bf16, int32_t* topk_ids_out, void* ws,
                            size_t ws_bytes, void* stream) {
    return moe_forward_mx_profiled(cfg, x_bf16, T, weights, residual_bf16, out_bf16, topk_ids_out, ws, ws_bytes,
                                   stream, nullptr);
}

}  // extern "C"
