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

// One probe: true once the phase with parity `parity` completed.  The
// thread may be suspended inside the probe until the phase completes or a
// system-dependent time passes.  CLUSTER: acquire at cluster scope, for a
// barrier that threads or copies of another CTA of the cluster arrive on.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    if constexpr (CLUSTER)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return done != 0;
}

// The same probe, suspended at most about `hint_ns` nanoseconds (it still
// returns as soon as the phase completes), so that a waiting loop looks at
// the clock often enough for its limit to mean what it says.
constexpr uint32_t kProbeSuspendNs = 2000;
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t done;
    if constexpr (CLUSTER)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
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
// complete within `timeout_ns` (or kMaxWaitProbes probes); never spins
// forever.  The clock is read every 16 probes of at most kProbeSuspendNs,
// so the limit is overshot by some 32 us at most.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
    if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t probe = 1; probe < kMaxWaitProbes; ++probe) {
        if (mbar_try_wait_hint<CLUSTER>(bar, parity, kProbeSuspendNs)) return true;
        if ((probe & 15u) == 0 && globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return false;
}

// Limit of a wait whose signal depends on another wait of the same CTA
// (a consumer's wait for data the TMA issuer loads once it has a free
// stage): twice the upstream limit, so that when the upstream wait runs
// out first, its site -- the root cause -- is the one recorded.
__device__ __forceinline__ uint64_t downstream_limit(uint64_t timeout_ns) { return 2 * timeout_ns; }

// Global-memory flag used between CTAs: release store / acquire load at GPU scope.
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add_gpu(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Bounded wait until a global word equals `tag` (acquire).  The CTAs
// involved are all resident: the persistent grid never exceeds one wave.
__device__ __forceinline__ bool tag_wait_bounded(const uint32_t *p, uint32_t tag, uint64_t timeout_ns) {
    if (ld_acquire_gpu(p) == tag) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t probe = 1; probe < kMaxWaitProbes; ++probe) {
        __nanosleep(64);
        if (ld_acquire_gpu(p) == tag) return true;
        if ((probe & 15u) == 0 && globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return false;
}

// Stream-K launch tags.  The partial-tile flags of a launch carry a tag no
// earlier launch used, so a flag left from an earlier launch (or from one
// whose waits gave up) never reads as ready.  seq[0] holds the tag of the
// last launch that completed, seq[1] counts the CTAs of the running launch
// that finished; the last of them publishes the new tag.  Both live in
// device memory, so a replayed CUDA graph gets a fresh tag every time.
__device__ __forceinline__ uint32_t sk_launch_tag(const uint32_t *seq) {
    const uint32_t t = ld_relaxed_gpu(seq) + 1u;
    return t == 0u ? 1u : t;    // 0 is what a fresh flag holds
}
// Called once per CTA (one thread), after the CTA has read the tag.
__device__ __forceinline__ void sk_launch_done(uint32_t *seq, uint32_t tag) {
    if (atom_add_acq_rel_gpu(seq + 1, 1u) == gridDim.x - 1u) {
        st_relaxed_gpu(seq + 1, 0u);
        st_relaxed_gpu(seq, tag);
    }
}

// Bounded wait until a global counter reaches `target` (acquire).  The
// CTAs involved are all resident: the persistent grid never exceeds one
// wave.
__device__ __forceinline__ bool count_wait_bounded(const uint32_t *p, uint32_t target, uint64_t timeout_ns) {
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t probe = 1; probe < kMaxWaitProbes; ++probe) {
        __nanosleep(64);
        if (ld_acquire_gpu(p) >= target) return true;
        if ((probe & 15u) == 0 && globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return false;
}

// Error word layout: bits 24..31 = which wait expired, bits 0..23 = CTA index.
enum WaitSite : uint32_t {
    kSiteConsumerFull = 1, kSiteProducerEmpty = 2, kSiteSelfTest = 3, kSiteStreamKFlag = 4
};

// Test hook for failure detection: a signal the kernels leave out on purpose,
// so that the bounded wait for it runs out and the expiry path (record the
// site, let the CTA's own copies land, return) runs without any fault.
//   kWithholdStreamKFlag: CTAs holding a partial tile never publish it (the
//     finishing CTA's flag wait, site 4, expires);
//   kWithholdRefill: the TMA issuer stops after filling the ring once (the
//     consumers' data wait, site 1, expires);
//   kWithholdRelease: consumers never release a stage (the issuer's slot
//     wait, site 2, expires).
enum Withhold : int {
    kWithholdNone = 0, kWithholdStreamKFlag = 1, kWithholdRefill = 2, kWithholdRelease = 3
};

__device__ __forceinline__ void record_error(uint32_t *err, uint32_t site) {
    if (err != nullptr)
        atomicCAS(err, 0u, (site << 24) | (blockIdx.x & 0xFFFFFFu));
}

// Programmatic dependent launch.  A kernel launched with programmatic
// stream serialisation may start while the kernel before it in the stream is
// still running: it must wait for that kernel (its completion and memory
// flush) before it reads or writes any global memory.  Signalling early
// lets the next kernel's CTAs be placed on SMs as this one's finish.
// Without the launch attribute both are no-ops.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// Round an FP32 value to TF32 (10 explicit mantissa bits), to nearest with
// ties away from zero; the result is an FP32 value whose low 13 bits are 0.
__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// The TF32 value a kind::tf32 MMA takes from an FP32 operand: its low 13
// mantissa bits dropped (rounding toward zero).  Measured: with the FP32
// values themselves as the high parts and residuals x - tf32_trunc(x), the
// 3xTF32 products keep their accuracy (mean error 1.8e-8 of sum |a b| at
// 1024^3, against 1.5e-8 with rounded high parts); had the MMA rounded to
// nearest, they would be off by up to 2^-11 relative.
__device__ __forceinline__ float tf32_trunc(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// Prefetch a 3-D TMA tile into L2 (no destination, no completion).  A hint
// only: L2 is where every write of the device lands, so data read later (by
// a TMA load after griddepcontrol.wait) is current even if the tile was
// written after the prefetch.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int32_t c0, int32_t c1, int32_t c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2) : "memory");
}

// 3-D TMA tile load (c0 innermost, c2 the batch index).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)),
           "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Thread-block clusters.  This CTA's rank in its cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Shared-memory address (shared::cluster window) of the variable at the same
// offset as `p` in the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
    return out;
}
// Every thread of every CTA of the cluster: release what came before, then
// acquire what the others released.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive (release, cluster scope) on an mbarrier of a CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(cluster_bar) : "memory");
}
// 3-D TMA tile load into this CTA's shared memory whose completion bytes go
// to an mbarrier of either CTA of this CTA's pair (`cluster_bar`, a
// shared::cluster address): how both CTAs of an SM pair fill the stage that
// the pair's MMAs read.
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *map, uint32_t cluster_bar,
                                                 int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)),
           "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

}  // namespace sg

// ---------------------------------------------------------------------------
// Tensor memory and 5th-generation tensor-core MMA (tcgen05), cta_group::1.
namespace sg {

// Allocate nCols (power of two >= 32) TMEM columns; the base address is
// written to shared memory.  Executed by one full warp.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::tf32, issued by one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on an mbarrier when all tcgen05 operations this thread
// issued so far have completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

// The same operations for an SM pair (cta_group::2: the two CTAs of a
// cluster of 2, ranks 0 and 1).  A kernel uses one group size throughout.
// Allocation and release are collective: one warp of each CTA of the pair
// executes them, and both get the same columns.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}
// Issued by one thread of rank 0: M = 256 rows, 128 from each CTA's shared
// memory (A) into each CTA's TMEM lanes, B's N columns split between the
// two CTAs' shared memory (first half in rank 0); the descriptors name
// offsets that hold in both CTAs.
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at `bar`'s offset in each CTA of `cta_mask`
// when the pair MMAs this thread issued so far have completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        :: "r"(smem_u32(bar)), "h"(cta_mask) : "memory");
}
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory operand descriptor for a K-major tile stored with the
// 128-byte swizzle (8-row x 128-byte atoms, the layout TMA's 128-byte swizzle
// writes): start address, stride between 8-row groups (1024 B), descriptor
// version 1, swizzle mode "128B".  The leading offset is unused for this
// layout.  The tile must start on a 1024-byte boundary; advancing K inside
// the 128-byte row is done by adding bytes to the start address.
__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // bits  0-13 start address >> 4
    d |= (uint64_t)1u << 16;                           // bits 16-29 leading offset (unused)
    d |= (uint64_t)(1024u >> 4) << 32;                 // bits 32-45 stride offset >> 4
    d |= (uint64_t)1u << 46;                           // bits 46-47 descriptor version
    d |= (uint64_t)2u << 61;                           // bits 61-63 swizzle: 128B
    return d;
}

// Instruction descriptor, kind::tf32: D f32, A and B tf32, both K-major,
// no negation, dense, M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4)                       // D format: f32
         | (2u << 7)                       // A format: tf32
         | (2u << 10)                      // B format: tf32
         | ((uint32_t)(N >> 3) << 17)      // N / 8
         | ((uint32_t)(M >> 4) << 24);     // M / 16
}

}  // namespace sg
