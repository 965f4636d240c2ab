// Tile bookkeeping shared by the grouped tensor-core GEMMs (expert_gemm.cu: fp32 block
// scales promoted in software; expert_gemm_mx.cu: UE8M0 scales in the tensor core).
// Tiles are 128 permuted token rows (one expert's segment, or the shared experts'
// tokens) x 256 weight rows; CTA b takes items b, b + gridDim.x, ...
#pragma once

#include "common.cuh"
#include "moe_internal.h"

namespace moe {
namespace gemm {

constexpr int kGM = 128;  // token rows per tile (MMA M)
constexpr int kGN = 256;  // weight rows per tile

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
        it.ntile = item % a.nt_r;
    } else {
        const int v = item - n_r;
        it.shared = 1;
        it.expert = -1;
        it.row0 = (v / a.nt_s) * kGM;
        it.nrows = min(kGM, a.T - it.row0);
        it.ntile = v % a.nt_s;
    }
#ifdef MOE_DEBUG
    // debug builds: a tile must lie inside its A tensor (a tile that does not is reported
    // and computed as rows 0.. of expert 0, none of them stored)
    if (it.nrows < 0 || it.nrows > kGM || it.row0 < 0 || it.row0 + it.nrows > (it.shared ? a.T : a.T * a.k) ||
        (!it.shared && it.expert < 0)) {
        set_status(a.status, kStatusBadId);
        it.row0 = 0;
        it.nrows = 0;
        it.expert = it.shared ? -1 : 0;
    }
#endif
    return it;
}

// Number of this CTA's items (blockIdx.x, blockIdx.x + gridDim.x, ...) in [from, to).
__device__ __forceinline__ int items_in(int from, int to) {
    const int b = blockIdx.x, g = gridDim.x;
    const int first = from <= b ? b : b + ((from - b + g - 1) / g) * g;
    return first < to ? (to - 1 - first) / g + 1 : 0;
}

// Walks this CTA's K blocks in order (the TMA side of the pipeline).
struct LoadCursor {
    int item, kb, Kb, shared, row0, yb0, yb1;
    __device__ __forceinline__ void set(const GemmArgs& a, int n_mt_r, int n_items, bool gateup) {
        if (item >= n_items) return;
        const Item it = decode_item(a, n_mt_r, item);
        Kb = (it.shared ? a.K_s : a.K_r) / kBlk;
        shared = it.shared;
        row0 = it.row0;
        if (gateup) {  // 128 gate rows and the same 128 rows of up
            yb0 = (it.shared ? 0 : it.expert * a.I) + it.ntile * kBlk;
            yb1 = yb0;
        } else {       // 256 consecutive rows of down
            yb0 = (it.shared ? 0 : it.expert * a.H) + it.ntile * kGN;
            yb1 = yb0 + kBlk;
        }
    }
    __device__ __forceinline__ void next(const GemmArgs& a, int n_mt_r, int n_items, bool gateup) {
        if (++kb == Kb) {
            kb = 0;
            item += gridDim.x;
            set(a, n_mt_r, n_items, gateup);
        }
    }
};

}  // namespace gemm
}  // namespace moe
