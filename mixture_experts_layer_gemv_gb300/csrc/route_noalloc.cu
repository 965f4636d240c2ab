// moe_route_noalloc: the fused small-T router + top-k with its scratch memory in a
// file-scope device array, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all, or cannot hand the library a
// workspace: a host framework that owns the whole device memory pool and forbids
// allocation once it is serving (cudaMalloc may synchronise the device and stall
// every other stream), or a plugin loaded into such a framework with no allocator
// hook. This entry point needs nothing from them but the inputs and outputs.
//
// The scratch (control words for the last-CTA-done counter, router logits and the
// activation codes the fused kernel also writes) lives in g_route_scratch below,
// sized for T <= 64 tokens, E <= 256 experts and H <= 8192. Every GPU that loads
// this library holds the array (606,464 bytes) until the process exits.
#include <mutex>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kNoAllocMaxT = 64;
constexpr int kNoAllocMaxE = 256;
constexpr int kNoAllocMaxH = 8192;
constexpr size_t kCtrlBytes = sizeof(Ctrl);
constexpr size_t kLogitsBytes = (size_t)kNoAllocMaxT * kNoAllocMaxE * sizeof(float);
constexpr size_t kXqBytes = (size_t)kNoAllocMaxT * kNoAllocMaxH;
constexpr size_t kXsBytes = (size_t)kNoAllocMaxT * (kNoAllocMaxH / kBlk) * sizeof(float);
constexpr size_t kScratchBytes = kCtrlBytes + kLogitsBytes + kXqBytes + kXsBytes;
static_assert(kScratchBytes == 606464, "documented scratch size");

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

// In host code g_route_scratch names a host-side stand-in, not device memory: the
// device address comes from cudaGetSymbolAddress, taken once per device with that
// device current (on the first call made on it).
constexpr int kMaxDevices = 64;
struct DeviceScratch {
    std::once_flag once;
    void* ptr = nullptr;
    cudaError_t err = cudaSuccess;
};
DeviceScratch g_scratch[kMaxDevices];

void* scratch_address(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    DeviceScratch& d = g_scratch[dev];
    std::call_once(d.once, [&d] { d.err = cudaGetSymbolAddress(&d.ptr, g_route_scratch); });
    *err = d.err;
    return d.err == cudaSuccess ? d.ptr : nullptr;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_noalloc(const moe_config_t* cfg, const void* x_bf16, int32_t T,
                                          const float* w_router, const float* router_bias, int32_t* topk_ids,
                                          float* topk_w, void* stream) {
    using namespace moe;
    if (!cfg) return MOE_ERR_INVALID_ARG;
    if (moe_workspace_size(cfg, 0) == 0) return MOE_ERR_UNSUPPORTED_SHAPE;  // config checks of the ABI
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T > kNoAllocMaxT || cfg->n_routed > kNoAllocMaxE || cfg->hidden > kNoAllocMaxH)
        return MOE_ERR_UNSUPPORTED_SHAPE;  // beyond the fixed scratch array
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !w_router || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(w_router, 16) || !aligned(topk_ids, 16) || !aligned(topk_w, 16))
        return MOE_ERR_INVALID_ARG;
    if (router_bias && !aligned(router_bias, 4)) return MOE_ERR_INVALID_ARG;
    cudaError_t err;
    unsigned char* base = static_cast<unsigned char*>(scratch_address(&err));
    if (!base) return MOE_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    // the last-CTA-done counter must start at zero, whatever an earlier call left behind
    if (cudaMemsetAsync(base, 0, kCtrlBytes, st) != cudaSuccess) return MOE_ERR_CUDA;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(base);
    float* logits = reinterpret_cast<float*>(base + kCtrlBytes);
    uint8_t* xq = base + kCtrlBytes + kLogitsBytes;
    float* xs = reinterpret_cast<float*>(base + kCtrlBytes + kLogitsBytes + kXqBytes);
    if (launch_route_small(*cfg, x_bf16, T, w_router, router_bias, topk_ids, topk_w, logits, xq, xs, nullptr,
                           nullptr, nullptr, nullptr, nullptr, ctrl, NormArgs{}, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
