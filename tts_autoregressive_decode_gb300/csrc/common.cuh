// common.cuh -- device helpers shared by the decode kernels (sm_103a).
//
// Inline PTX for programmatic dependent launch, mbarriers, bulk (TMA) copies and the packed
// f32x2 FMA; warp reductions; bf16 widening.  Every wait on an mbarrier is bounded: when the
// bound is hit the kernel records a flag in the device check word and returns.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"

namespace dec {

__device__ __forceinline__ void flag_check(unsigned* status, unsigned bit) {
    if (status) atomicOr(status, bit);
}

// ---- programmatic dependent launch -------------------------------------------------------
// pdl_trigger: this CTA allows the next kernel in the stream to be scheduled.
// pdl_wait: block until every prerequisite grid has completed and its writes are visible.
// Both are no-ops when the kernel was not launched with the programmatic attribute.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- shared-memory addresses, mbarriers, bulk copies ---------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Barrier over the first `nthreads` threads that name barrier `id` (ids 1..15; 0 is
// __syncthreads).  nthreads is a multiple of 32.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// arrive at named barrier `id` without waiting (the waiters use named_bar_sync)
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on phase `parity`.  try_wait suspends the thread for a hardware-bounded time
// per call, so the loop bound turns into a wall-clock bound of well under a few seconds.
constexpr int kWaitIters = 1 << 22;
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < kWaitIters; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// 1-D bulk copy global -> shared, completion counted in bytes on the mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 1-D bulk copy global -> shared with an L2 policy (weights, cached K/V: evict_first)
__device__ __forceinline__ void bulk_g2s_pol(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// ---- L2 cache policy -----------------------------------------------------------------------
// evict_first: data streamed once (weights), so it does not push out data that is reused
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// evict_normal: data read twice in a row by the same CTA (the first of two passes over rows)
__device__ __forceinline__ uint64_t l2_evict_normal() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Order this thread's earlier generic-proxy accesses to shared memory before later async-proxy
// (bulk copy) accesses: needed before a bulk copy overwrites shared memory that threads have read
// or written since the previous copy.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- loads ---------------------------------------------------------------------------------
// Streaming 16-byte load of data that is read once (weights): bypass L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ... with an L2 policy (weights: evict_first)
__device__ __forceinline__ uint4 ld_stream16(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

// ---- arithmetic ----------------------------------------------------------------------------
// (a.x*b.x + c.x, a.y*b.y + c.y), each lane rounded once (fma.rn.f32x2)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

// a 32-bit word holding two bf16 values (low half first) -> the two exact f32 values
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// PER (2 or 4) consecutive floats from shared memory as one 8- or 16-byte access
template <int PER>
__device__ __forceinline__ void load_vec(float* dst, const float* src) {
    if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        dst[0] = v.x;
        dst[1] = v.y;
        dst[2] = v.z;
        dst[3] = v.w;
    } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        dst[0] = v.x;
        dst[1] = v.y;
    }
}

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

}  // namespace dec
