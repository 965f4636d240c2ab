// Device helpers shared by the MoE kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kBlk = 128;       // FP8 scale block (weights: 128x128, activations: 1x128)
constexpr float kE4M3Max = 448.f;

// ---------------------------------------------------------------- loads
// Streaming 16-byte load for weights that are read exactly once: bypass L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte load of data that other CTAs also read (activations): normal caching.
__device__ __forceinline__ uint4 ld_v4(const void* p) { return *reinterpret_cast<const uint4*>(p); }

// ------------------------------------------------------------ warp helpers
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// ------------------------------------------------ activation quantisation
// Power-of-two block scale: the smallest 2^k with amax <= 448 * 2^k. With
// amax = m * 2^e (m in [0.5, 1)) and 448 = 0.875 * 2^9 this is k = e - 9 when
// m <= 0.875 and k = e - 8 otherwise. amax = 0 gives scale 1. k is clamped at
// -126 so both the scale and its inverse stay normal fp32 numbers.
__device__ __forceinline__ float act_scale_pow2(float amax, float* inv_scale) {
    if (!(amax > 0.f)) {
        *inv_scale = 1.f;
        return 1.f;
    }
    int e;
    const float m = frexpf(amax, &e);
    int k = (m <= 0.875f) ? e - 9 : e - 8;
    k = k < -126 ? -126 : k;
    *inv_scale = ldexpf(1.f, -k);
    return ldexpf(1.f, k);
}

// The same scale as an E8M0 byte (k + 127) for the MXFP8 variant.
__device__ __forceinline__ uint32_t act_scale_e8m0(float amax, float* inv_scale) {
    if (!(amax > 0.f)) {
        *inv_scale = 1.f;
        return 127u;
    }
    int e;
    const float m = frexpf(amax, &e);
    int k = (m <= 0.875f) ? e - 9 : e - 8;
    k = k < -126 ? -126 : k;
    *inv_scale = ldexpf(1.f, -k);
    return (uint32_t)(k + 127);
}

// E8M0 byte -> its value 2^(b-127) (b = 0: 2^-127, a subnormal; 0xFF, NaN, is not
// expected here).
__device__ __forceinline__ float e8m0_to_float(uint32_t b) {
    return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// Four fp32 values -> four E4M3 codes (round to nearest even, saturating), packed
// little-endian in one 32-bit word (value 0 in the low byte).
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// One 128-value block held by a warp, four consecutive values per lane
// (lane l holds values 4l..4l+3): returns the packed codes of this lane and
// writes the block scale (identical in every lane).
__device__ __forceinline__ uint32_t warp_quant_block128(float v0, float v1, float v2, float v3,
                                                        float* scale_out) {
    float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
    amax = warp_max(amax);
    float inv;
    const float s = act_scale_pow2(amax, &inv);
    *scale_out = s;
    return pack_e4m3x4(v0 * inv, v1 * inv, v2 * inv, v3 * inv);
}

// MXFP8: the same 128 values, four per lane, as four blocks of 32 (8 lanes each):
// returns this lane's packed codes and writes the E8M0 byte of its block.
__device__ __forceinline__ uint32_t warp_quant_mx32(float v0, float v1, float v2, float v3, uint32_t* s8_out) {
    float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    float inv;
    *s8_out = act_scale_e8m0(amax, &inv);
    return pack_e4m3x4(v0 * inv, v1 * inv, v2 * inv, v3 * inv);
}

// ------------------------------------------------------------- FP8 MMA
// D(16x8, f32) += A(16x32, e4m3, row) * B(32x8, e4m3, col). Used as a dequantising
// dot-product engine for weight-streaming GEMVs with up to 8 activation columns.
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// (a0, a1) = (v0 * c + a0, v1 * c + a1) in one packed FP32 instruction (fma.rn.f32x2:
// each lane rounds once, as fmaf does); halves the issue slots of a scale promotion.
__device__ __forceinline__ void fma2(float& a0, float& a1, float v0, float v1, float c) {
    unsigned long long A, V, C, D;
    asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(V) : "f"(v0), "f"(v1));
    asm("mov.b64 %0, {%1, %1};" : "=l"(C) : "f"(c));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(D) : "l"(V), "l"(C), "l"(A));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(D));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float((uint32_t)b << 16);
}

// ------------------------------------------------- stage M: RMSNorm x gamma
// x = h * rstd * gamma with rstd = 1 / sqrt(mean(h^2) + eps), rounded once to bf16
// (stage M of the DSV2-236B-MegaKernel stage flowchart, MoE subgraph: the hidden state
// normalised and scaled by its gamma before the router).
// Every kernel that reads a normalised activation derives it from the raw row with
// these functions (rstd always from warp_row_sumsq), so all of them see the same
// bf16 values.

// Sum of squares of one bf16 row of H values (H a multiple of 8), by one warp in
// a fixed order: lane l accumulates the 8-value chunks l, l+32, ... in order, then
// a xor-shuffle tree. Returns the sum in every lane.
__device__ __forceinline__ float warp_row_sumsq(const uint16_t* row, int H) {
    const uint4* r = reinterpret_cast<const uint4*>(row);
    const int lane = threadIdx.x & 31, n8 = H / 8;
    float ss = 0.f;
    for (int c0 = 0; c0 < n8; c0 += 32 * 8) {  // up to 8 loads in flight per lane
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = c0 + lane + 32 * j;
            v[j] = c < n8 ? __ldg(r + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float a = bf16_bits_to_float((uint16_t)(w[q] & 0xFFFF));
                const float b = bf16_bits_to_float((uint16_t)(w[q] >> 16));
                ss = fmaf(a, a, ss);
                ss = fmaf(b, b, ss);
            }
        }
    }
    return warp_sum(ss);
}

__device__ __forceinline__ float rms_rstd(float sumsq, int H, float eps) {
    return 1.f / sqrtf(sumsq / (float)H + eps);
}

// Two packed bf16 values (low half first) normalised, repacked as bf16 bits.
__device__ __forceinline__ uint32_t rms_apply2(uint32_t h2, float rstd, uint32_t g2) {
    const __nv_bfloat16 lo = __float2bfloat16_rn(bf16_bits_to_float((uint16_t)(h2 & 0xFFFF)) * rstd *
                                                 bf16_bits_to_float((uint16_t)(g2 & 0xFFFF)));
    const __nv_bfloat16 hi = __float2bfloat16_rn(bf16_bits_to_float((uint16_t)(h2 >> 16)) * rstd *
                                                 bf16_bits_to_float((uint16_t)(g2 >> 16)));
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

__device__ __forceinline__ uint4 rms_apply8(uint4 h8, float rstd, uint4 g8) {
    return make_uint4(rms_apply2(h8.x, rstd, g8.x), rms_apply2(h8.y, rstd, g8.y), rms_apply2(h8.z, rstd, g8.z),
                      rms_apply2(h8.w, rstd, g8.w));
}



// ------------------------------------------------------ mbarrier / TMA (sm_90+)
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Trace stamps (moe_forward_trace): trace[(kernel * kTraceCtas + cta) * 4 + event] = the
// global timer in ns; kernel 0 route, 1 gate/up, 2 down, 3 combine; event 0 CTA entry,
// 1 dependency wait returned, 2 first data consumed, 3 CTA done. Null: nothing recorded.
constexpr int kTraceCtas = 512;
__device__ __forceinline__ void trace_stamp(uint64_t* tr, int kernel, int ev) {
    if (tr != nullptr && blockIdx.x < (unsigned)kTraceCtas)
        tr[((size_t)kernel * kTraceCtas + blockIdx.x) * 4 + ev] = globaltimer_ns();
}

// Upper bound on the wall time of one wait; no legitimate wait in this library comes
// near it (the longest are TMA copies from HBM, microseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Bounded wait on an mbarrier phase: gives up after about kWaitLimitNs of wall time
// (each try_wait may itself suspend the thread for a while, so the bound is on time,
// not on the number of polls) and returns false; the caller then records a timeout
// in the status word and leaves instead of hanging the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; i != 0; ++i) {  // wraps after 2^32 polls at the latest
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

// mbar_wait_bounded for a whole warp: lane 0 alone polls the barrier (32 lanes polling one
// mbarrier contend with the thread that fills the stages) and the warp then synchronises,
// which orders the other lanes' reads of the stage after lane 0's observation of the
// completed phase. Every lane gets the same result. Call with the whole warp.
__device__ __forceinline__ bool warp_wait_bounded(uint64_t* bar, uint32_t parity) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// 2-D tiled TMA load of box {x (inner, bytes of an 8-bit tensor), y (rows)} into
// shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(smem_dst)), "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// L2 cache policy for TMA loads of data read exactly once (the weights of a decode layer
// that no other row group reads): evict first, so that the stream does not push out lines
// written for the next kernel.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// tma_load_2d with an L2 cache policy (l2_policy_evict_first).
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const void* tmap, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Prefetch of a global range into L2 (no shared-memory destination).
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

// Prefetch of one 2-D TMA box into L2.
__device__ __forceinline__ void tma_prefetch_2d(const void* tmap, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start launching,
// and wait until the previous kernel has completed with its memory visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Named barrier over the first `threads` threads of the CTA (id 1..15).
__device__ __forceinline__ void named_bar(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}


// ------------------------------------------------------------ tcgen05 / TMEM
// Tensor-memory allocation by one warp: writes the TMEM base address to *smem_dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D(tmem, fp32) (+)= A(smem desc) * B(smem desc)^T, E4M3 inputs, one thread issues.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D(tmem, fp32) (+)= A(smem desc) * B(smem desc)^T, bf16 inputs, one thread issues.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on an mbarrier once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread).
// The load and its wait sit in one asm statement, so no use of v can be scheduled
// before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes, load and wait in one statement.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this warp's 32 TMEM lanes, load and wait in one statement.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* p) {
    const uint64_t addr = smem_u32(p);
    uint64_t d = 0;
    d |= (addr & 0x3FFFFull) >> 4;    // start address
    d |= (uint64_t)1 << 16;           // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32; // stride byte offset: 8-row group pitch
    d |= (uint64_t)1 << 46;           // descriptor version
    d |= (uint64_t)2 << 61;           // layout: 128-byte swizzle
    return d;
}

// Shared-memory descriptor of a plain row-major matrix of 16-byte rows (no swizzle):
// 8-row core matrices 128 bytes apart. The source of a 128x128b tcgen05.cp.
__device__ __forceinline__ uint64_t smem_desc_rows16(const void* p) {
    const uint64_t addr = smem_u32(p);
    uint64_t d = 0;
    d |= (addr & 0x3FFFFull) >> 4;    // start address
    d |= (uint64_t)1 << 16;           // leading byte offset (one core matrix along K: unused)
    d |= (uint64_t)(128 >> 4) << 32;  // stride byte offset: 8-row group pitch
    d |= (uint64_t)1 << 46;           // descriptor version
    return d;                         // layout field 0: no swizzle
}

// Copy 32 rows x 16 bytes of shared memory into tensor memory, the same data into each
// of the four 32-lane quadrants: row i -> lane 32q + i of 4 consecutive 32-bit columns
// from taddr (q = 0..3). Ordered with the issuing thread's later tcgen05.mma; its
// completion is tracked by tcgen05.commit like an MMA's.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t s_desc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(s_desc) : "memory");
}

// Make this thread's generic shared-memory writes visible to the async proxy
// (tcgen05.cp / tcgen05.mma operand reads) that a later barrier hand-off orders.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D(tmem, fp32) (+)= (A * 2^(sfA-127)) * (B * 2^(sfB-127))^T with E4M3 operands and one
// UE8M0 scale factor per row and 32-wide K step, read from tensor memory. A scale
// group of 128 rows occupies 4 columns from sfa_tmem (sfb_tmem, a multiple of 4): the
// rows of lane quadrant q are read from column q, lane 32q + i holding the four K-step
// bytes of row 32q + i; with N = 256, B's rows 128.. are the next group of 4 columns.
// The descriptor's scale-factor ids pick the byte.
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of kind::mxf8f6f4: E4M3 x E4M3 -> fp32, both K-major, M x N,
// UE8M0 scale factors, byte sf_id of the A and B scale words.
__host__ __device__ constexpr uint32_t idesc_mx_f32(int M, int N, int sf_id) {
    return ((uint32_t)sf_id << 4)           // B scale-factor byte
           | (0u << 7) | (0u << 10)         // A, B: E4M3
           | ((uint32_t)(N >> 3) << 17)     // N / 8
           | (1u << 23)                     // scale factors: UE8M0
           | ((uint32_t)(M >> 4) << 24)     // M / 16
           | ((uint32_t)sf_id << 29);       // A scale-factor byte
}

// Instruction descriptor of kind::f16: bf16 x bf16 -> fp32, both operands K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                        // D format fp32
           | (1u << 7) | (1u << 10)         // A, B: bf16 (the same type for both)
           | ((uint32_t)(N >> 3) << 17)     // N / 8
           | ((uint32_t)(M >> 4) << 24);    // M / 16
}

// Instruction descriptor: E4M3 x E4M3 -> fp32, both operands K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f8_f32(int M, int N) {
    return (1u << 4)                        // D format fp32
           | (0u << 7) | (0u << 10)         // A, B: E4M3
           | ((uint32_t)(N >> 3) << 17)     // N / 8
           | ((uint32_t)(M >> 4) << 24);    // M / 16
}

// Fault-injection bits of Ctrl::inject (failure-detection tests): the decode gate/up
// kernel's producer issues no copies, so its consumers' bounded waits run out.
enum : unsigned { kInjectSkipGateupLoads = 1u };

// ----------------------------------------------------------- status word
// kStatusTimeout: a bounded wait gave up; kStatusBadId: an expert id outside [0, E)
// reached the permutation (the offending item is skipped).
enum : int { kStatusTimeout = 1, kStatusBadId = 2 };

__device__ __forceinline__ void set_status(int* status, int bit) { atomicOr(status, bit); }

}  // namespace moe
