// Thin inline-PTX wrappers for sm_103a: shared-memory mbarriers, TMA tile
// loads, the global timer, and the bounded wait every kernel of this library
// uses instead of an unbounded spin.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace sg {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// One non-blocking probe: true once the phase with parity `parity` completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Hard cap on probes, in addition to the time limit, so that the loop ends
// even if the global timer were to stall.
constexpr uint32_t kMaxWaitProbes = 1u << 30;

// Bounded wait on an mbarrier phase.  Returns false if the phase did not
// complete within `timeout_ns` (or kMaxWaitProbes probes); never spins forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t probe = 1; probe < kMaxWaitProbes; ++probe) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((probe & 63u) == 0 && globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return false;
}

// Global-memory flag used between CTAs: release store / acquire load at GPU scope.
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait for a global flag to become nonzero (the CTAs involved are
// all resident: the persistent grid never exceeds one wave).
__device__ __forceinline__ bool flag_wait_bounded(const uint32_t *p, uint64_t timeout_ns) {
    if (ld_acquire_gpu(p) != 0) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t probe = 1; probe < kMaxWaitProbes; ++probe) {
        __nanosleep(64);
        if (ld_acquire_gpu(p) != 0) return true;
        if ((probe & 15u) == 0 && globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return false;
}

// Error word layout: bits 24..31 = which wait expired, bits 0..23 = CTA index.
enum WaitSite : uint32_t {
    kSiteConsumerFull = 1, kSiteProducerEmpty = 2, kSiteSelfTest = 3,
    kSiteStreamKFlag = 4, kSiteCtaSync = 5
};

__device__ __forceinline__ void record_error(uint32_t *err, uint32_t site) {
    if (err != nullptr)
        atomicCAS(err, 0u, (site << 24) | (blockIdx.x & 0xFFFFFFu));
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D TMA tile load into this CTA's shared memory; completion is signalled
// as transaction bytes on `bar`.  c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map,
                                            uint64_t *bar, int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)),
           "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

}  // namespace sg
