// pa_device.cuh -- device helpers shared by the kernels of libpa (sm_103a).
//
// Inline PTX for the shared-memory mbarrier, the bulk asynchronous copy
// (global -> this CTA's shared memory, completion counted on an mbarrier) and
// bounded waits.  Every wait has a wall-clock limit: when it runs out the
// kernel records PA_DEVERR_TIMEOUT in the device error word, raises a
// per-CTA abort flag and returns false, so a logic error can never spin a GPU
// forever.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// A pipeline wait that has not completed after this long gives up.
constexpr unsigned long long kWaitTimeoutNs = 1000000000ull;   // 1 s
// Secondary bound in case the global timer does not advance.
constexpr uint32_t kWaitMaxPolls = 1u << 30;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async proxy and other threads;
// follow with __syncthreads().
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the phase of `bar` with the given parity has completed.
// Returns false (without waiting further) if *abort_flag is raised by another
// thread of the CTA, or after the time limit, in which case it records a
// timeout in *err and raises *abort_flag itself.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          volatile int *abort_flag, unsigned int *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long start = global_timer_ns();
    for (uint32_t polls = 1;; ++polls) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((polls & 31u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - start > kWaitTimeoutNs || polls >= kWaitMaxPolls) {
                atomicOr(err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Like mbar_wait but ignores the abort flag: used on the way out to let
// copies already in flight land before the CTA exits.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long start = global_timer_ns();
    for (uint32_t polls = 1; polls < kWaitMaxPolls; ++polls) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((polls & 31u) == 0 && global_timer_ns() - start > kWaitTimeoutNs) return false;
    }
    return false;
}

// Wait until a shared-memory word equals `want` (same limits as mbar_wait).
__device__ __forceinline__ bool wait_value(const volatile uint32_t *word, uint32_t want,
                                           volatile int *abort_flag, unsigned int *err) {
    if (*word == want) return true;
    const unsigned long long start = global_timer_ns();
    for (uint32_t polls = 1;; ++polls) {
        __nanosleep(32);
        if (*word == want) return true;
        if ((polls & 31u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - start > kWaitTimeoutNs || polls >= kWaitMaxPolls) {
                atomicOr(err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Bulk asynchronous copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global memory into this CTA's shared memory.  Completion
// decrements the transaction count of `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                              uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Same, with an L2 eviction-priority hint (a policy from make_l2_policy_*).
__device__ __forceinline__ void bulk_copy_g2s_hint(void *smem_dst, const void *gmem_src,
                                                   uint32_t bytes, uint64_t *bar,
                                                   uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t make_l2_policy_evict_first() {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

__device__ __forceinline__ uint64_t make_l2_policy_evict_last() {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while the previous kernel on the stream is still
// running; grid_dependency_wait() blocks until that kernel has completed and
// its memory is visible, and must precede every global-memory access that
// could depend on it.  allow_dependents_to_launch() lets the next such kernel
// become resident early (it still waits for this one to finish).  Both are
// no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents_to_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Global loads that bypass L1: used for partial results written by other CTAs
// of the same launch.
__device__ __forceinline__ float2 ld_cg_f2(const float2 *p) { return __ldcg(p); }
__device__ __forceinline__ float4 ld_cg_f4(const float4 *p) { return __ldcg(p); }
__device__ __forceinline__ float2 ld_cg_f2x(const float *p) {
    return __ldcg(reinterpret_cast<const float2 *>(p));
}

}  // namespace pa
