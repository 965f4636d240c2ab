// Stage R's local part of the DeepSeek-V2 MoE layer ("DSV2-236B-MegaKernel",
// README stage flowchart: the shared and routed outputs added into h): a sorted-segment
// gather.
// Token t sums its k weighted expert rows (found through inv_pos), the shared
// experts' row and the optional residual in fp32, in a fixed order, and rounds
// once to bf16. No atomics, so the result is deterministic.
#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(w[i] << 16);
        acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__global__ void __launch_bounds__(256) combine_kernel(int T, int H, int k, const __nv_bfloat16* y_perm,
                                                      const int32_t* inv_pos, const __nv_bfloat16* y_shared,
                                                      const __nv_bfloat16* residual, __nv_bfloat16* out) {
    const int H8 = H / 8;
    const long n = (long)T * H8;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const long t = i / H8;
        const int c = (int)(i % H8);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            const long r = inv_pos[t * k + j];
            if ((unsigned long)r < (unsigned long)T * k)  // rows outside y_perm are not read
                add_bf16x8(acc, __ldcs(reinterpret_cast<const uint4*>(y_perm + r * H) + c));
        }
        if (y_shared) add_bf16x8(acc, __ldcs(reinterpret_cast<const uint4*>(y_shared + t * H) + c));
        if (residual) add_bf16x8(acc, __ldg(reinterpret_cast<const uint4*>(residual + t * H) + c));
        uint4 o;
        uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
            ow[q] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        reinterpret_cast<uint4*>(out + t * H)[c] = o;
    }
}

}  // namespace

cudaError_t launch_combine(int T, int H, int k, const __nv_bfloat16* y_perm, const int32_t* inv_pos,
                           const __nv_bfloat16* y_shared, const __nv_bfloat16* residual, __nv_bfloat16* out,
                           cudaStream_t st) {
    const long n = (long)T * (H / 8);
    if (n == 0) return cudaSuccess;
    const long want = (n + 255) / 256;
    const int grid = (int)(want < (long)num_sms() * 8 ? want : (long)num_sms() * 8);
    combine_kernel<<<grid, 256, 0, st>>>(T, H, k, y_perm, inv_pos, y_shared, residual, out);
    return cudaGetLastError();
}

}  // namespace moe
