// sv_ptx.cuh -- thin inline-PTX wrappers used by the verification kernel
// (sm_90+ instructions; the library is built for sm_103a only).
//
//  * cluster rank, cluster barrier (arrive.release / wait.acquire) and
//    distributed-shared-memory stores (mapa + st.shared::cluster);
//  * mbarrier init / arrive.expect_tx / bounded try_wait;
//  * the non-tensor bulk copy global -> shared (cp.async.bulk, the 1-D TMA
//    path), completing on an mbarrier transaction count, with an L2
//    evict-first hint, and the bulk prefetch into L2;
//  * st.async: a store into another cluster CTA's shared memory that
//    completes on that CTA's mbarrier transaction count;
//  * ex2.approx, the NaN-propagating max (scalar, three-input and bf16x2) and
//    the packed two-lane fp32 arithmetic of sm_100+ (add/sub/mul/fma .f32x2,
//    each lane rounded to nearest like its scalar form).
#pragma once

#include <stdint.h>

namespace sv {

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA in the cluster must execute these (aligned form).
__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory variable in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_addr, uint32_t rank)
{
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(local_addr), "r"(rank));
    return out;
}

__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}

// Make mbarrier.init visible to the bulk-copy (async) proxy before any copy
// that completes on the barrier is issued.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t addr, uint32_t tx_bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(addr), "r"(tx_bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t addr)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok) : "r"(addr), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after `max_spins` polls
// (each poll may suspend the thread for a system-dependent time; no suspend
// hint is given: with a 1 us hint workload 3 ran 2% slower).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t addr, uint32_t parity, uint32_t max_spins)
{
    for (uint32_t s = 0; s < max_spins; ++s)
        if (mbar_try_wait(addr, parity))
            return true;
    return false;
}

// 1-D bulk copy global -> shared; src, dst 16-byte aligned, bytes % 16 == 0.
// An L2 cache policy that evicts first what it tags: rows that are read once.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// As bulk_copy_g2s, the source lines tagged with an L2 cache policy.
__device__ __forceinline__ void bulk_copy_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                                   uint32_t mbar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar), "l"(policy) : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t mbar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}

// Bring [src, src + bytes) into L2 ahead of its bulk copy (16-byte aligned
// address, size a multiple of 16); no completion is tracked.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before its
// later bulk-copy (async-proxy) writes into the same buffer.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max_nan(float a, float b)
{
    float y;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
    return y;
}

// max of three with NaN propagation (sm_100+ three-input form)
__device__ __forceinline__ float max3_nan(float a, float b, float c)
{
    float y;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

// lane-wise max of two packed bf16 pairs, NaN-propagating
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b)
{
    uint32_t y;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
}

// Two fp32 values in one 64-bit register pair: lo in bits 0..31.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t y;
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(lo), "f"(hi));
    return y;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t y;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(a), "l"(b));
    return y;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t y;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(a), "l"(b));
    return y;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t y;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(y) : "l"(a), "l"(b), "l"(c));
    return y;
}

__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b)
{
    uint64_t y;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(a), "l"(b));
    return y;
}

// 16-byte store into cluster shared memory completing `bytes` on the
// destination CTA's mbarrier (both addresses from mapa).
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t mbar)
{
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
        ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(mbar) : "memory");
}

__device__ __forceinline__ void st_async_v2(uint32_t addr, float2 v, uint32_t mbar)
{
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
        ::"r"(addr), "f"(v.x), "f"(v.y), "r"(mbar) : "memory");
}

}  // namespace sv
