/*
 * moe.h - C ABI of the GB300 (sm_103a) MoE-layer forward library (libmoe_gb300.so).
 *
 * The layer is the DeepSeek-style mixture-of-experts block described on
 * "DSV2-236B-MegaKernel" (README, stage flowchart, MoE subgraph, stages M..R):
 *   router GEMV -> softmax + group-limited greedy top-k, w = score * routed_scaling_factor
 *   -> routed experts: FP8 block-scaled gate/up, SiLU(g) * u, down, times w
 *   -> shared experts (same MLP, weight 1) -> h = shared_out + sum of routed (+ residual).
 *
 * Conventions for every entry point
 *   - Pointers named *_bf16, *_ids, *_w, weights and ws are DEVICE pointers, owned by
 *     the caller; the library allocates no memory. All of them must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream). A returned MOE_OK means the work was enqueued.
 *   - Arguments are validated on the host before anything is launched; a failed check
 *     returns an error code and launches nothing.
 *   - T = 0 is a valid no-op that returns MOE_OK.
 *   - Row-major layouts everywhere. E4M3 = OCP FP8 E4M3FN, one byte per value.
 *   - The library keeps no state between calls; concurrent calls need distinct workspaces.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The layer's arguments, named as in the DeepSeek-V2 configuration the README's
 * "Model geometry" paragraph quotes (hidden 5120, moe_intermediate_size 1536, 160 routed
 * experts in 8 groups, top-3 groups, top-6 experts, x16.0, 2 shared experts).
 * Constraints (checked, MOE_ERR_UNSUPPORTED_SHAPE otherwise):
 *   hidden % 128 == 0 and moe_inter % 128 == 0 (the 128-wide FP8 scale block,
 *   README "Results": a TP=8 shard of 1536 is 192, not a multiple of 128);
 *   1 <= n_routed <= 256; n_routed % n_group == 0; 1 <= n_group <= 32;
 *   1 <= topk_group <= n_group; 1 <= top_k <= min(16, topk_group * n_routed / n_group);
 *   0 <= n_shared; the shared experts are fused into one MLP of width n_shared*moe_inter. */
typedef struct moe_config {
    int32_t hidden;                /* H */
    int32_t moe_inter;             /* I */
    int32_t n_routed;              /* E */
    int32_t n_group;               /* G */
    int32_t topk_group;            /* Gk */
    int32_t top_k;                 /* k */
    int32_t n_shared;              /* S; shared width Is = S * I */
    float routed_scaling_factor;   /* s; w = softmax score * s, no renormalisation */
} moe_config_t;

/* One layer's weights (device pointers). Expert weights are E4M3 codes with one fp32
 * scale per 128x128 block: value[o][i] = e4m3(code[o][i]) * scale[o/128][i/128].
 *   w_gate, w_up   [E, I, H]  codes     s_gate, s_up  [E, I/128, H/128] fp32
 *   w_down         [E, H, I]  codes     s_down        [E, H/128, I/128] fp32
 *   ws_gate, ws_up [Is, H]    codes     ss_gate, ss_up [Is/128, H/128]  fp32
 *   ws_down        [H, Is]    codes     ss_down        [H/128, Is/128]  fp32
 *   w_router       [E, H]     fp32      router_bias    [E] fp32 or NULL
 * The shared pointers may be NULL when n_shared == 0. */
typedef struct moe_weights {
    const uint8_t *w_gate, *w_up, *w_down;
    const float *s_gate, *s_up, *s_down;
    const uint8_t *ws_gate, *ws_up, *ws_down;
    const float *ss_gate, *ss_up, *ss_down;
    const float *w_router, *router_bias;
} moe_weights_t;

/* One layer's weights in the MXFP8 variant (Mixture-of-Kittens Table 2, its MXFP8
 * routed-expert rows; the DeepSeek-V4.1 Flash lecture's conversion of block scales to
 * the MX layout): E4M3 codes as in
 * moe_weights_t, with one UE8M0 scale byte b (value 2^(b-127)) per row and 32
 * consecutive K instead of the fp32 128x128 block scales:
 *   s_gate, s_up   [E, I, H/32]   s_down [E, H, I/32]
 *   ss_gate, ss_up [Is, H/32]     ss_down [H, Is/32]        (u8, row-major) */
typedef struct moe_weights_mx {
    const uint8_t *w_gate, *w_up, *w_down;
    const uint8_t *s_gate, *s_up, *s_down;
    const uint8_t *ws_gate, *ws_up, *ws_down;
    const uint8_t *ss_gate, *ss_up, *ss_down;
    const float *w_router, *router_bias;
} moe_weights_mx_t;

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,       /* NULL / misaligned pointer, negative T */
    MOE_ERR_UNSUPPORTED_SHAPE = -2, /* config outside the constraints above */
    MOE_ERR_WORKSPACE = -3,         /* ws NULL or ws_bytes < moe_workspace_size(cfg, T) */
    MOE_ERR_CUDA = -4,              /* a CUDA launch or runtime call failed */
    MOE_ERR_DEVICE_TIMEOUT = -5     /* a bounded device-side wait ran out (see below) */
} moe_status_t;

/* Which kernel launch moe_forward_profiled brackets with CUDA events. */
typedef enum moe_stage {
    MOE_STAGE_ROUTE = 0,    /* router + top-k (+ permutation when fused) */
    MOE_STAGE_PERMUTE = 1,  /* permutation (large T) */
    MOE_STAGE_GATE_UP = 2,  /* routed + shared gate/up, SiLU(g) * u */
    MOE_STAGE_DOWN = 3,     /* routed + shared down, times w */
    MOE_STAGE_COMBINE = 4,  /* sum into the hidden vector */
    MOE_STAGE_COUNT = 5
} moe_stage_t;

/* cudaEvent_t handles (or NULL) recorded on the call's stream immediately before and
 * after the named stage's kernels. */
typedef struct moe_stage_events {
    void* start[MOE_STAGE_COUNT];
    void* stop[MOE_STAGE_COUNT];
} moe_stage_events_t;

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status_t status);

/* Bytes of device workspace every entry point below needs for up to max_tokens tokens
 * (0 if the config is invalid). Workspace contents need no initialisation except the
 * control region at its start (status word and hand-off counters), which
 * moe_workspace_init zeroes; the library returns the counters to zero by the end of
 * every call, so one init after allocation suffices. */
size_t moe_workspace_size(const moe_config_t* cfg, int32_t max_tokens);

/* Zero the control region at the start of ws (asynchronous memset on stream). */
moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Device-side error word of ws: copies it to the host (synchronising `stream`), clears
 * it, and returns MOE_OK or the recorded error:
 *   MOE_ERR_DEVICE_TIMEOUT  a bounded wait inside a kernel gave up (that kernel skips its
 *                           remaining work and returns instead of hanging; every bounded
 *                           wait has a time and an iteration limit, none traps);
 *   MOE_ERR_INVALID_ARG     a kernel met invalid device data and left it out: an expert id
 *                           outside [0, E) given to moe_permute, a perm_src entry outside
 *                           [0, T*k), expert offsets that do not cover the permuted rows, or
 *                           a row-group work record outside the routing's bounds (in a build
 *                           with -DMOE_DEBUG also: a weight-streaming or grouped-GEMM tile
 *                           outside its K range, slice, part or rows).
 * A timeout takes precedence when both were recorded. The outputs of a call that recorded
 * an error are unspecified. */
moe_status_t moe_read_device_status(void* ws, void* stream);

/* Failure-detection test hook (the pages have no counterpart; a test uses it to make a
 * device-side wait run out on purpose, in the permitted form: a flag that nothing sets).
 * Sets the workspace's fault-injection word for the calls that follow on it,
 * asynchronously on `stream`:
 *   MOE_INJECT_SKIP_GATEUP_LOADS  the decode gate/up kernel (T <= 64 tokens) issues no
 *       copies, so its consumers' bounded waits run out (after about one second) with
 *       nothing in flight; such a call records MOE_ERR_DEVICE_TIMEOUT
 *       (moe_read_device_status) and its outputs are unspecified;
 *   0  clears it.
 * Other words of the workspace are not touched. Errors: MOE_ERR_WORKSPACE (ws NULL or
 * ws_bytes below the control region), MOE_ERR_INVALID_ARG (an unknown bit). */
#define MOE_INJECT_SKIP_GATEUP_LOADS 1u
moe_status_t moe_debug_set(void* ws, size_t ws_bytes, uint32_t inject, void* stream);

/* Activation quantisation, the FP8 operand of the expert GEMMs: per token and block of
 * 128 channels, scale = the smallest power of two 2^k with amax <= 448 * 2^k
 * (amax = 0 -> scale 1), code = round-to-nearest-even E4M3 of x / scale.
 * This is the reading of the pages' FP8 block-scaled expert GEMMs ("Results") with
 * UE8M0 (power-of-two) scale factors (README "Layout", quant/fp8_block_quant.py).
 *   x_bf16 [T, H] -> xq [T, H] E4M3 codes, xs [T, H/128] fp32 scales. */
moe_status_t moe_quant_act(const void* x_bf16, int32_t T, int32_t H, uint8_t* xq, float* xs,
                           void* stream);

/* Stage M: RMSNorm in front of the router (DSV2-236B-MegaKernel stage flowchart, MoE
 * subgraph: the hidden state normalised and scaled by gamma). Per token row t:
 *   x[t][i] = bf16( h[t][i] * rstd[t] * gamma[i] ),  rstd[t] = 1 / sqrt(mean_i h[t][i]^2 + eps),
 * the mean and 1/rms in fp32, one round-to-nearest-even to bf16 per element.
 *   h_bf16 [T, H], gamma_bf16 [H] -> x_bf16 [T, H] (must not alias h).
 * H % 8 == 0 (MOE_ERR_UNSUPPORTED_SHAPE otherwise); eps >= 0 and finite. The fused
 * entry points below compute exactly these x values inside their own kernels. */
moe_status_t moe_rmsnorm(const void* h_bf16, int32_t T, int32_t H, const void* gamma_bf16, float eps,
                         void* x_bf16, void* stream);

/* Stage N + O: router GEMV/GEMM and group-limited greedy top-k.
 *   logits[t][e] = sum_h x[t][h] * w_router[e][h] (+ router_bias[e])   (fp32)
 *   p = softmax over all E; group j = experts [j*E/G, (j+1)*E/G) scores max p;
 *   the topk_group best groups are kept (ties: lower group index); the top_k best
 *   experts inside them are selected (ties: lower expert index).
 * Outputs: topk_ids int32 [T, k] (score-descending), topk_w fp32 [T, k] = p * s.
 * README, stage flowchart "N" and "O"; per-stage table rows "M+N" and "O". */
moe_status_t moe_route(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                       const float* w_router, const float* router_bias, int32_t* topk_ids,
                       float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* moe_route on RMSNorm(h) (stage M fused into the router's kernels: the normalised
 * activation never goes to memory). Same outputs as moe_rmsnorm followed by moe_route;
 * the workspace afterwards holds the FP8 codes of the normalised rows. */
moe_status_t moe_route_rmsnorm(const moe_config_t* cfg, const void* h_bf16, int32_t T, const void* gamma_bf16,
                               float eps, const float* w_router, const float* router_bias, int32_t* topk_ids,
                               float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* moe_route without a workspace, for callers that cannot allocate device memory:
 * a framework that owns the whole device memory pool and forbids cudaMalloc while it
 * serves (cudaMalloc can synchronise the device and stall other streams), or a plugin
 * inside one with no allocator hook. The pages have no counterpart of this call; it
 * computes exactly what moe_route computes, with the same arguments minus ws.
 * Its scratch is one fixed device array of 606,464 bytes inside the library, held by
 * every GPU that loads it until the process exits; it covers T <= 64, n_routed <= 256
 * and hidden <= 8192, and larger sizes return MOE_ERR_UNSUPPORTED_SHAPE.
 * The first call on a device looks up that array's device address (once per device,
 * with the device current); make that first call before any stream capture.
 * Every call shares the array: calls whose work overlaps on the GPU (other streams,
 * other host threads) race and may return wrong results; serialise them. */
moe_status_t moe_route_noalloc(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                               const float* w_router, const float* router_bias, int32_t* topk_ids,
                               float* topk_w, void* stream);

/* Token permutation by expert: a stable counting sort of the T*k (token, slot) pairs.
 * Pair (t, j) has flat index f = t*k + j.
 *   expert_offsets int32 [E+1]: pairs routed to experts < e (exclusive prefix sum)
 *   perm_src       int32 [T*k]: flat index of the pair at each permuted position
 *   inv_pos        int32 [T*k]: permuted position of each flat index
 * Within one expert the pairs keep ascending f. An id outside [0, E) is checked on the
 * device: its pair is left out of the permutation and the workspace status records it
 * (moe_read_device_status then returns MOE_ERR_INVALID_ARG); ids from moe_route are
 * always valid.
 * (The router produces the layout the expert GEMMs consume: DeepSeek-V4.1 Flash
 * lecture, "Rounds 12-15" table; MoK's GPU-side dispatch scheduling, abstract.) */
moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_ids, int32_t T,
                         int32_t* expert_offsets, int32_t* perm_src, int32_t* inv_pos,
                         void* ws, size_t ws_bytes, void* stream);

/* Stages P1/P2 and Q1/Q2: the expert MLPs on FP8 block-scaled weights.
 * For permuted row r of expert e (token t = perm_src[r] / k, weight w = topk_w[perm_src[r]]):
 *   g = Wg_e . xhat_t, u = Wu_e . xhat_t, a = SiLU(g) * u, ahat = FP8-quantised a
 *   (as in moe_quant_act), y_perm[r] = w * (Wd_e . ahat)            -> bf16 [T*k, H]
 * and for the shared experts (width Is, weight 1): y_shared[t]     -> bf16 [T, H]
 * xhat is the moe_quant_act quantisation of x. y_shared may be NULL only if
 * n_shared == 0. */
moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                            const moe_weights_t* weights, const int32_t* expert_offsets,
                            const int32_t* perm_src, const float* topk_w, void* y_perm_bf16,
                            void* y_shared_bf16, void* ws, size_t ws_bytes, void* stream);

/* Stage R's local part: out[t] = sum_j y_perm[inv_pos[t*k + j]] + y_shared[t] (+ residual[t]),
 * summed in fp32, rounded once to bf16 (README flowchart, stage R: the shared and routed
 * outputs added into h).
 * y_shared / residual may be NULL (treated as zero). out must not alias the inputs. */
moe_status_t moe_combine(const moe_config_t* cfg, const void* y_perm_bf16, const int32_t* inv_pos,
                         const void* y_shared_bf16, const void* residual_bf16, int32_t T,
                         void* out_bf16, void* stream);

/* The whole layer: route, permute, expert MLPs, shared experts, combine.
 *   x_bf16 [T, H] -> out_bf16 [T, H]; residual_bf16 [T, H] or NULL;
 *   topk_ids_out int32 [T, k] or NULL (a copy of the routing decision).
 * No host synchronisation: expert counts and offsets never leave the device.
 * (MoK abstract: "no CPU-GPU synchronisation".) */
moe_status_t moe_forward(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                         const moe_weights_t* weights, const void* residual_bf16, void* out_bf16,
                         int32_t* topk_ids_out, void* ws, size_t ws_bytes, void* stream);

/* moe_forward with CUDA events recorded around each stage (events may be NULL). */
moe_status_t moe_forward_profiled(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                                  const moe_weights_t* weights, const void* residual_bf16,
                                  void* out_bf16, int32_t* topk_ids_out, void* ws, size_t ws_bytes,
                                  void* stream, const moe_stage_events_t* events);

/* moe_forward with per-CTA timestamps, for attributing the layer's time to its kernels
 * the way the DSV2-236B-MegaKernel README's per-stage table does (that page stamps each
 * stage with in-kernel clocks). trace is a DEVICE array of MOE_TRACE_WORDS uint64 owned by
 * the caller (16-byte aligned; NULL returns MOE_ERR_INVALID_ARG). The call writes
 *   trace[(kernel * MOE_TRACE_CTAS + cta) * 4 + event] = GPU global timer (ns)
 * for kernel 0 router (+ top-k and permutation), 1 gate/up, 2 down, 3 combine; event 0
 * CTA start, 1 its wait for the previous kernel returned, 2 first data consumed (router:
 * logits stored; down: first operand built), 3 CTA done. Only the decode kernels (T <= 64)
 * stamp; entries no CTA writes keep their previous contents, so clear the array first.
 * The stamps cost a few stores per CTA; the results equal moe_forward's. */
#define MOE_TRACE_CTAS 512
#define MOE_TRACE_WORDS (4 * MOE_TRACE_CTAS * 4)
moe_status_t moe_forward_trace(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                               const moe_weights_t* weights, const void* residual_bf16, void* out_bf16,
                               void* ws, size_t ws_bytes, void* stream, uint64_t* trace);

/* Stages M..R of the MoE block in one call, the residual stream in and out:
 *   out = h + layer(RMSNorm(h))      (stage M as in moe_rmsnorm, the layer as in
 *                                     moe_forward with residual = h)
 * h_bf16 [T, H] is the hidden state before the norm; out_bf16 must not alias it.
 * The normalised activation is formed inside the router and quantisation kernels
 * (README flowchart: stage M, then N..R, and stage R adds the shared and routed outputs
 * into h). */
moe_status_t moe_forward_rmsnorm(const moe_config_t* cfg, const void* h_bf16, int32_t T, const void* gamma_bf16,
                                 float eps, const moe_weights_t* weights, void* out_bf16, int32_t* topk_ids_out,
                                 void* ws, size_t ws_bytes, void* stream);

/* moe_forward_rmsnorm with CUDA events around each stage (stage M counts as routing). */
moe_status_t moe_forward_rmsnorm_profiled(const moe_config_t* cfg, const void* h_bf16, int32_t T,
                                          const void* gamma_bf16, float eps, const moe_weights_t* weights,
                                          void* out_bf16, int32_t* topk_ids_out, void* ws, size_t ws_bytes,
                                          void* stream, const moe_stage_events_t* events);

/* ------------------------------------------------------------ MXFP8 variant
 * The layer with moe_weights_mx_t weights and MXFP8 activations: x and the
 * intermediate a = SiLU(g) * u are quantised per token and 32 consecutive values
 * (scale = the smallest 2^k, k >= -126, with amax <= 448 * 2^k; codes RNE E4M3), and
 * for T > 64 the expert GEMMs apply all scales inside the tensor core (tcgen05.mma
 * kind::mxf8f6f4); for T <= 64 the weight-streaming kernels apply each 32-wide block's
 * scales to its own MMA partial. Routing is that of moe_route. Shapes: hidden % 512 == 0
 * and moe_inter % 512 == 0 (MOE_ERR_UNSUPPORTED_SHAPE otherwise; moe_workspace_size_mx
 * returns 0). */
size_t moe_workspace_size_mx(const moe_config_t* cfg, int32_t max_tokens);

/* MXFP8 activation quantisation: x_bf16 [T, H] -> xq [T, H] E4M3 codes and
 * xs_e8m0 [T, H/32] scale bytes. */
moe_status_t moe_quant_act_mx(const void* x_bf16, int32_t T, int32_t H, uint8_t* xq, uint8_t* xs_e8m0,
                              void* stream);

/* moe_forward in the MXFP8 variant (workspace from moe_workspace_size_mx). */
moe_status_t moe_forward_mx(const moe_config_t* cfg, const void* x_bf16, int32_t T, const moe_weights_mx_t* weights,
                            const void* residual_bf16, void* out_bf16, int32_t* topk_ids_out, void* ws,
                            size_t ws_bytes, void* stream);

/* moe_forward_mx with CUDA events around each stage. */
moe_status_t moe_forward_mx_profiled(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                                     const moe_weights_mx_t* weights, const void* residual_bf16, void* out_bf16,
                                     int32_t* topk_ids_out, void* ws, size_t ws_bytes, void* stream,
                                     const moe_stage_events_t* events);

/* ---------------------------------------------------------------- backward
 * The layer's backward (the Mixture-of-Kittens page's training workload, Table 1
 * "Backward"): the gradients of L = sum(dout * out) for the layer of moe_forward
 * (no residual, no stage M) with its expert choice held fixed. topk_ids / topk_w [T, k]
 * are the forward's routing as moe_route returns it; dout_bf16 [T, H] is dL/d(out).
 * Reading: the FP8 activation quantisers are straight-through, the weights enter at
 * their dequantised FP8 values, and the router receives gradient through the kept
 * experts' weights w = routed_scaling_factor * softmax(W_router x + bias)_e.
 * Outputs: fp32 device arrays, overwritten:
 *   dx [T, H]; dw_gate, dw_up [E, I, H]; dw_down [E, H, I];
 *   dws_gate, dws_up [Is, H], dws_down [H, Is] (required when n_shared > 0, else ignored);
 *   dw_router [E, H]; dbias [E] (NULL: not computed).
 * Arithmetic: g and u are recomputed by the forward's FP8 grouped GEMM; the backward's
 * contractions run in bf16 x bf16 -> fp32 (weights decoded from E4M3 x block scale to
 * bf16). Needs hidden % 256 == 0 and n_routed % 16 == 0 (MOE_ERR_UNSUPPORTED_SHAPE
 * otherwise, and moe_backward_workspace_size returns 0). T = 0 zeroes the weight gradients.
 * Errors as for moe_forward; the workspace's status word is read by
 * moe_read_device_status. */
size_t moe_backward_workspace_size(const moe_config_t* cfg, int32_t max_tokens);
moe_status_t moe_backward(const moe_config_t* cfg, const void* x_bf16, int32_t T, const moe_weights_t* weights,
                          const int32_t* topk_ids, const float* topk_w, const void* dout_bf16, float* dx,
                          float* dw_gate, float* dw_up, float* dw_down, float* dws_gate, float* dws_up,
                          float* dws_down, float* dw_router, float* dbias, void* ws, size_t ws_bytes, void* stream);

/* moe_backward with CUDA events around its parts, in the slots of moe_stage_events_t:
 * ROUTE: the forward recompute (activation codes, router logits, permutation, row
 * gather, g and u) and the bf16 operands (weights dequantised and transposed, xhat,
 * gathered rows); PERMUTE: dgrad of down, SwiGLU and router backward; COMBINE: the dx
 * terms and their sum; DOWN: the weight gradients, which contain GATE_UP: the routed
 * experts' weight gradient of gate/up alone. */
moe_status_t moe_backward_profiled(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                                   const moe_weights_t* weights, const int32_t* topk_ids, const float* topk_w,
                                   const void* dout_bf16, float* dx, float* dw_gate, float* dw_up, float* dw_down,
                                   float* dws_gate, float* dws_up, float* dws_down, float* dw_router, float* dbias,
                                   void* ws, size_t ws_bytes, void* stream, const moe_stage_events_t* events);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
