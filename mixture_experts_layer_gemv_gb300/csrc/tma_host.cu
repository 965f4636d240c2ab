// Host-side TMA tensor-map encoding for the weight tensors, through the driver's
// cuTensorMapEncodeTiled (looked up once via the runtime, so the library does not
// link libcuda directly). Encoded maps are cached by (address, shape, box): a map
// only describes an address range, so a cached entry stays valid for any tensor
// that later occupies the same range with the same shape.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <tuple>

#include "moe_internal.h"

namespace moe {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// (address, rows, cols, row pitch in bytes, box, element kind)
using Key = std::tuple<uintptr_t, uint64_t, uint64_t, uint64_t, uint32_t, uint32_t, int>;
std::mutex g_mu;
std::map<Key, CUtensorMap> g_cache;

// kind 0: u8 with 128-byte swizzle; 1: fp32, no swizzle; 2: bf16 with 128-byte swizzle
bool encode_2d(TmaMap* out, const void* base, uint64_t rows, uint64_t cols, uint64_t pitch_bytes, uint32_t box_cols,
               uint32_t box_rows, int kind) {
    static_assert(sizeof(TmaMap) == sizeof(CUtensorMap), "opaque map size");
    const bool f32 = kind == 1;
    const Key key{(uintptr_t)base, rows, cols, pitch_bytes, box_cols, box_rows, kind};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_cache.find(key);
        if (it != g_cache.end()) {
            *reinterpret_cast<CUtensorMap*>(out) = it->second;
            return true;
        }
    }
    auto fn = encode_fn();
    if (!fn) return false;
    CUtensorMap m;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r =
        fn(&m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : kind == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
           2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           kind == 1 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_cache.size() > 4096) g_cache.clear();
        g_cache[key] = m;
    }
    *reinterpret_cast<CUtensorMap*>(out) = m;
    return true;
}

}  // namespace

// bf16 [rows, cols], dense rows, 128-byte swizzle (box_cols must be 64: 128 bytes)
bool tmap_bf16_2d(TmaMap* out, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                  uint32_t box_rows) {
    return encode_2d(out, base, rows, cols, cols * 2, box_cols, box_rows, 2);
}

// u8 [rows, cols], dense rows, 128-byte swizzle (box_cols must be 128)
bool tmap_u8_2d(TmaMap* out, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                uint32_t box_rows) {
    return encode_2d(out, base, rows, cols, cols, box_cols, box_rows, 0);
}


}  // namespace moe
