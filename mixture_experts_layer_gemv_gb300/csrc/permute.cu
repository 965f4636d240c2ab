// Token permutation by expert: a deterministic, stable counting sort of the
// T*k (token, slot) pairs, done on the device so that expert counts and offsets
// never travel to the host (MoK abstract: no CPU-GPU synchronisation; the
// DeepSeek-V4.1 Flash lecture, "Rounds 12-15": the router produces the data layout
// the expert GEMMs consume).
//
// Two launches over segments of 1024 flat indices, one CTA of 8 warps each:
// permute_count_kernel writes every segment's expert histogram; permute_scatter_kernel
// turns the histograms into each segment's base per expert (totals scanned expert-major,
// earlier segments first), recounts its segment per warp, and each warp then walks its
// 128 indices in order, ranking equal experts inside each 32-wide chunk with
// __match_any_sync. The result equals a sequential stable sort. CTA 0 also writes the
// expert offsets and the work list of the expert kernels: row groups of <= 8 rows for
// the streaming GEMVs, or 128-row tiles for the grouped GEMM.
#include <climits>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kPermWarps = 8;
constexpr int kPermSeg = 1024;                     // flat indices per CTA
constexpr int kWarpSeg = kPermSeg / kPermWarps;    // 128 per warp: 4 chunks of 32
constexpr int kMaxE = 256;

__device__ int scan_exclusive_warp256(int* v, int n) {
    const int lane = threadIdx.x & 31;
    int loc[8];
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = lane * 8 + i;
        loc[i] = idx < n ? v[idx] : 0;
        s += loc[i];
    }
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int run = incl - s;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = lane * 8 + i;
        if (idx < n) v[idx] = run;
        run += loc[i];
    }
    __syncwarp();
    return total;
}

// Write the row groups (<= kGroupRows rows of one expert each) from per-expert
// counts in s_cnt and exclusive offsets in s_off. s_gcnt/s_goff are scratch.
__device__ void write_groups(const int* s_cnt, const int* s_off, int* s_goff, int E, RowGroup* groups,
                             int32_t* group_of_row, Ctrl* ctrl) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_goff[e] = (s_cnt[e] + kGroupRows - 1) / kGroupRows;
    __syncthreads();
    if (threadIdx.x < 32) {
        const int gtot = scan_exclusive_warp256(s_goff, E);
        if (threadIdx.x == 0) ctrl->n_routed_groups = gtot;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int c = s_cnt[e];
        const int ng = (c + kGroupRows - 1) / kGroupRows;
        for (int g = 0; g < ng; ++g) {
            RowGroup rg;
            rg.expert = e;
            rg.row_begin = s_off[e] + g * kGroupRows;
            rg.nrows = min(kGroupRows, c - g * kGroupRows);
            rg.pad = 0;
            groups[s_goff[e] + g] = rg;
            for (int r = 0; r < rg.nrows; ++r) group_of_row[rg.row_begin + r] = s_goff[e] + g;
        }
    }
}

// Write the 128-row token tiles of every expert segment (the grouped GEMM's work
// list) from per-expert counts and offsets; s_tmp is scratch.
__device__ void write_mtiles(const int* s_cnt, const int* s_off, int* s_tmp, int E, MTile* mtiles, Ctrl* ctrl) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_tmp[e] = (s_cnt[e] + 127) / 128;
    __syncthreads();
    if (threadIdx.x < 32) {
        const int tot = scan_exclusive_warp256(s_tmp, E);
        if (threadIdx.x == 0) ctrl->n_mtiles = tot;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int c = s_cnt[e];
        for (int j = 0; 128 * j < c; ++j) {
            MTile m;
            m.expert = e;
            m.row0 = s_off[e] + 128 * j;
            m.nrows = min(128, c - 128 * j);
            m.pad = 0;
            mtiles[s_tmp[e] + j] = m;
        }
    }
}

struct PermuteParams {
    int E, n;
    const int32_t* ids;
    int32_t* offsets;
    int32_t* perm_src;
    int32_t* inv_pos;
    int32_t* seg_hist;  // [segments, E] expert counts of each segment
    RowGroup* groups;
    int32_t* group_of_row;
    MTile* mtiles;
    Ctrl* ctrl;
};

// The 4 x 32 expert ids of this warp's slice of a segment (-1 past the end or out of range).
__device__ __forceinline__ void load_warp_ids(const PermuteParams& p, int f0, int (&ev)[kWarpSeg / 32], bool flag) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int u = 0; u < kWarpSeg / 32; ++u) {
        const int f = f0 + lane + 32 * u;
        int e = -1;
        if (f < p.n) {
            e = __ldg(p.ids + f);
            if (e < 0 || e >= p.E) {
                if (flag) set_status(&p.ctrl->status, kStatusBadId);
                e = -1;
            }
        }
        ev[u] = e;
    }
}

__global__ void __launch_bounds__(kPermWarps * 32) permute_count_kernel(PermuteParams p) {
    __shared__ int hist[kMaxE];
    const int warp = threadIdx.x >> 5;
    pdl_launch_dependents();  // the scatter kernel waits for this grid's completion itself
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    int ev[kWarpSeg / 32];
    load_warp_ids(p, blockIdx.x * kPermSeg + warp * kWarpSeg, ev, true);
#pragma unroll
    for (int u = 0; u < kWarpSeg / 32; ++u)
        if (ev[u] >= 0) atomicAdd(&hist[ev[u]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) p.seg_hist[(size_t)blockIdx.x * p.E + e] = hist[e];
}

__global__ void __launch_bounds__(kPermWarps * 32) permute_scatter_kernel(PermuteParams p) {
    __shared__ int hist[kPermWarps][kMaxE];
    __shared__ int s_cnt[kMaxE], s_off[kMaxE + 1], s_pre[kMaxE], s_goff[kMaxE];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E, seg = blockIdx.x, n_seg = gridDim.x;
    int ev[kWarpSeg / 32];
    load_warp_ids(p, seg * kPermSeg + warp * kWarpSeg, ev, false);  // ids come from before the count kernel
    for (int i = threadIdx.x; i < kPermWarps * kMaxE; i += blockDim.x) (&hist[0][0])[i] = 0;
    pdl_wait();  // the segment histograms
    // per expert: pairs in earlier segments (s_pre) and in all segments (s_cnt)
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int pre = 0, tot = 0;
        for (int c = 0; c < n_seg; ++c) {
            const int h = p.seg_hist[(size_t)c * E + e];
            pre += c < seg ? h : 0;
            tot += h;
        }
        s_pre[e] = pre;
        s_cnt[e] = tot;
        s_off[e] = tot;
    }
    __syncthreads();
    if (warp == 0) {
        const int tot = scan_exclusive_warp256(s_off, E);
        if (lane == 0) s_off[E] = tot;
    }
#pragma unroll
    for (int u = 0; u < kWarpSeg / 32; ++u)
        if (ev[u] >= 0) atomicAdd(&hist[warp][ev[u]], 1);
    __syncthreads();
    if (seg == 0)
        for (int e = threadIdx.x; e <= E; e += blockDim.x) p.offsets[e] = s_off[e];
    // hist[w][e] <- first row of expert e for warp w of this segment
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = s_off[e] + s_pre[e];
        for (int w = 0; w < kPermWarps; ++w) {
            const int c = hist[w][e];
            hist[w][e] = run;
            run += c;
        }
    }
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    const int f0 = seg * kPermSeg + warp * kWarpSeg;
#pragma unroll
    for (int u = 0; u < kWarpSeg / 32; ++u) {
        const int f = f0 + lane + 32 * u;
        const int e = ev[u];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt_mask);
        if (e >= 0) {
            const int pos = hist[warp][e] + rank;
            p.perm_src[pos] = f;
            p.inv_pos[f] = pos;
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) hist[warp][e] += __popc(peers);
        __syncwarp();
    }
    if (seg != 0) return;
    if (p.groups) {
        __syncthreads();
        write_groups(s_cnt, s_off, s_goff, E, p.groups, p.group_of_row, p.ctrl);
    }
    if (p.mtiles) {
        __syncthreads();
        write_mtiles(s_cnt, s_off, s_goff, E, p.mtiles, p.ctrl);
    }
}

struct BuildGroupsParams {
    int E, n_rows;
    const int32_t* offsets;
    RowGroup* groups;
    int32_t* group_of_row;
    MTile* mtiles;
    Ctrl* ctrl;
};

// Work lists from caller-supplied offsets. Offsets that are not a non-decreasing
// sequence inside [0, T*k] would make the work list point outside the buffers, so
// they are rejected on the device: the error bit is set and no work is listed.
__global__ void __launch_bounds__(256) build_groups_kernel(BuildGroupsParams p) {
    __shared__ int s_cnt[kMaxE], s_off[kMaxE], s_goff[kMaxE];
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        const int a = p.offsets[e], b = p.offsets[e + 1];
        if (a < 0 || b < a || b > p.n_rows) s_bad = 1;
        s_off[e] = a;
        s_cnt[e] = b - a;
    }
    __syncthreads();
    if (s_bad) {
        if (threadIdx.x == 0) {
            p.ctrl->n_routed_groups = 0;
            p.ctrl->n_mtiles = 0;
            set_status(&p.ctrl->status, kStatusBadId);
        }
        return;
    }
    if (p.groups) write_groups(s_cnt, s_off, s_goff, p.E, p.groups, p.group_of_row, p.ctrl);
    if (p.mtiles) {
        __syncthreads();
        write_mtiles(s_cnt, s_off, s_goff, p.E, p.mtiles, p.ctrl);
    }
}

// Activation-code rows of the grouped GEMM in permuted order: one warp per row.
constexpr int kGatherRows = 32;

__global__ void __launch_bounds__(256) gather_rows_kernel(int T, int H, int k, const int32_t* perm_src,
                                                          const uint8_t* xq, uint8_t* xq_perm, int* status,
                                                          const uint8_t* xs8, uint8_t* xs8_perm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long n = (long)T * k;
    const int H16 = H / 16;
    for (long r = (long)blockIdx.x * kGatherRows + warp; r < n && r < (long)(blockIdx.x + 1) * kGatherRows; r += 8) {
        const int f = perm_src[r];
        const bool good = (unsigned)f < (unsigned)n;
        if (!good && lane == 0) set_status(status, kStatusBadId);
        const uint4* src = reinterpret_cast<const uint4*>(xq + (size_t)(good ? f / k : 0) * H);
        uint4* dst = reinterpret_cast<uint4*>(xq_perm + (size_t)r * H);
        for (int c0 = 0; c0 < H16; c0 += 32 * 8) {  // 8 loads in flight per lane, then the stores
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = c0 + lane + 32 * u;
                v[u] = good && c < H16 ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < H16) dst[c] = v[u];
            }
        }
        if (xs8) {  // the row's E8M0 scales: H/32 bytes, a multiple of 16 (H % 512 == 0)
            const uint4* ss = reinterpret_cast<const uint4*>(xs8 + (size_t)(good ? f / k : 0) * (H / 32));
            uint4* sd = reinterpret_cast<uint4*>(xs8_perm + (size_t)r * (H / 32));
            for (int c = lane; c < H / 512; c += 32) sd[c] = good ? __ldg(ss + c) : make_uint4(0, 0, 0, 0);
        }
    }
}

}  // namespace

int permute_segments(int64_t n) { return n > 0 ? (int)((n + kPermSeg - 1) / kPermSeg) : 1; }

cudaError_t launch_permute(const moe_config_t& c, const int32_t* ids, int T, int32_t* offsets,
                           int32_t* perm_src, int32_t* inv_pos, RowGroup* groups, int32_t* group_of_row,
                           MTile* mtiles, int32_t* seg_hist, Ctrl* ctrl, cudaStream_t st) {
    PermuteParams p;
    p.E = c.n_routed;
    p.n = T * c.top_k;
    p.ids = ids;
    p.offsets = offsets;
    p.perm_src = perm_src;
    p.inv_pos = inv_pos;
    p.seg_hist = seg_hist;
    p.groups = groups;
    p.group_of_row = group_of_row;
    p.mtiles = mtiles;
    p.ctrl = ctrl;
    const int segs = permute_segments(p.n);
    permute_count_kernel<<<segs, kPermWarps * 32, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the scatter's id loads and shared-memory set-up overlap the count kernel's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(segs);
    cfg.blockDim = dim3(kPermWarps * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, permute_scatter_kernel, p);
}

cudaError_t launch_build_groups(const moe_config_t& c, const int32_t* offsets, int n_rows, RowGroup* groups,
                                int32_t* group_of_row, MTile* mtiles, Ctrl* ctrl, cudaStream_t st) {
    BuildGroupsParams p;
    p.E = c.n_routed;
    p.n_rows = n_rows;
    p.offsets = offsets;
    p.groups = groups;
    p.group_of_row = group_of_row;
    p.mtiles = mtiles;
    p.ctrl = ctrl;
    build_groups_kernel<<<1, 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(int T, int H, int k, const int32_t* perm_src, const uint8_t* xq, uint8_t* xq_perm,
                               int* status, cudaStream_t st, const uint8_t* xs8, uint8_t* xs8_perm) {
    const long n = (long)T * k;
    if (n == 0) return cudaSuccess;
    gather_rows_kernel<<<(unsigned)((n + kGatherRows - 1) / kGatherRows), 256, 0, st>>>(T, H, k, perm_src, xq,
                                                                                        xq_perm, status, xs8,
                                                                                        xs8_perm);
    return cudaGetLastError();
}

}  // namespace moe
