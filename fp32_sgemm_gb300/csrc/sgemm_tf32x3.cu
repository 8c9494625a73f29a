// FP32 SGEMM on the 5th-generation tensor cores, error-compensated 3xTF32:
//
//   x = x_hi + x_lo,  x_hi = x truncated to TF32 (what the MMA reads of an
//                     FP32 operand), x_lo = x - x_hi rounded to nearest TF32
//   A.B ~= A_hi.B_hi + A_hi.B_lo + A_lo.B_hi                  (FP32 accumulation)
//
// The dropped term A_lo.B_lo and the rounding of x_lo leave a relative
// error per product near 2^-21, far inside the FP32 acceptance bound, while
// the products run at tensor-core rate.  TF32 is only mentioned on the pages
// as a different contest ("Matmul I", section 1; "The Final Kernel", "What
// Could Be Improved"); the splitting is the error-compensated TF32 method of
// Ootomo & Yokota (2022).  Integer-valued inputs up to 2^11 in magnitude are
// exact in TF32 (x_lo = 0), so those products stay bit exact.
//
// Two kinds of kernel:
//   * split (sgemm_aux.cu): A -> A_hi, A_lo (row major, K contiguous) and
//     B -> B_hi^T, B_lo^T (N x K, K contiguous), so both tensor-core operands
//     are K-major and can be staged with TMA's 128-byte swizzle, the layout
//     the MMA descriptors name; an operand already stored that way is read
//     in place as its own high part;
//   * main: persistent CTAs (or SM pairs) of 2 + EPI_WARPS warps.  Warp 0
//     lane 0 streams the four operand tiles of each 32-wide K slice into a
//     shared-memory ring (TMA); warp 1 lane 0 (of rank 0 in a pair) issues
//     tcgen05.mma (K=8, kind::tf32) into TMEM; the epilogue warps read TMEM
//     back (tcgen05.ld, each warp a 32-lane quarter and a column slab) and
//     write C = alpha*acc (+ beta*C).
//
// Chunked accumulation.  The tensor core's FP32 accumulation does not round
// to nearest: summing all of K into one TMEM accumulator, whose sign and
// magnitude persist, lets those rounding errors pile up in one direction
// (measured: error growing linearly with K, 3x over the FP32 bound at
// K = 8192).  So the MMAs restart a fresh accumulator every CHUNK_KB K
// slices (two TMEM buffers alternate; the chunk length trades speed for
// error, see the configurations below), and the epilogue warps add each chunk
// into an FP32 register sum with ordinary round-to-nearest additions while
// the next chunk is being multiplied.  Chunk sums change sign at random, so
// what is left of the tensor core's rounding averages out.
// Every wait is bounded; a CTA that gives up records the error, lets its own
// TMA copies and MMAs finish, and releases its TMEM before returning.
#include <algorithm>

#include "kernel_table.h"

namespace sg {

// PAIR: the tile is computed by an SM pair (a cluster of 2 CTAs,
// tcgen05 cta_group::2): 256 rows, each CTA loading its own 128 rows of A
// and half of B's BN columns, rank 0 issuing M = 256 MMAs that read both
// CTAs' shared memory and write each CTA's 128 rows into its own TMEM.  Each
// SM then stages and reads half of B per MMA, which is what bounds the
// single-SM kernel (its shared-memory port).
template <int BN_, int STAGES_, int CHUNK_KB_, int EPI_WARPS_, bool PAIR_ = false>
struct Tf32x3Config {
    static constexpr bool PAIR = PAIR_;
    static constexpr int BM = 128, BN = BN_, BK = 32, STAGES = STAGES_;
    static constexpr int TILE_M = PAIR ? 2 * BM : BM;  // rows of C per tile
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // columns of B this CTA loads
    static constexpr int CHUNK_KB = CHUNK_KB_;     // K slices per TMEM accumulator chunk
    // Epilogue warps: 4 lane quarters of TMEM x EPI_WARPS/4 column slabs.
    static constexpr int EPI_WARPS = EPI_WARPS_;
    static constexpr int SLAB = BN / (EPI_WARPS / 4);   // columns per epilogue thread
    static constexpr int A_BYTES = BM * BK * 4;     // one of A_hi / A_lo
    static constexpr int B_BYTES = B_ROWS * BK * 4; // one of B_hi / B_lo
    static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;   // per CTA
    // Two accumulators of BN columns; the allocation is a power of two.
    static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
    static constexpr int THREADS = (2 + EPI_WARPS) * 32;
    static constexpr int NUM_BARRIERS = 2 * STAGES + 5;
    // Per epilogue warp, a padded 32 x 33 float tile to turn its rows into
    // coalesced row segments of C (the staged epilogue).
    static constexpr int XPOSE_BYTES = EPI_WARPS * 32 * 33 * 4;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + NUM_BARRIERS * 8 + 16 + XPOSE_BYTES + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(BN % 16 == 0 && BN >= 64 && BN <= 256, "UMMA N for M = 128");
    static_assert(!PAIR || (BN % 32 == 0 && B_ROWS % 8 == 0), "UMMA N for M = 256 across a pair");
    static_assert(EPI_WARPS % 4 == 0 && SLAB % 32 == 0 && SLAB * (EPI_WARPS / 4) == BN, "epilogue slabs");
    static_assert(TMEM_COLS >= 32 && (TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS <= 512, "TMEM");
    static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "align");
};

// Work of one slot (a CTA, or an SM pair: the cluster) as segments, K
// slices [kb0, kb1) of tile t: whole tiles slot, slot + slots, ... below
// sk_tile0, then an equal contiguous share of the (tile, slice) units of the
// tiles from sk_tile0 on ("stream-K").  A tile cut between slots is
// finished by the slot holding its first slice, whose last segment that is;
// the others (each slot has at most one such segment, its first) store
// partial sums.  All three roles of the CTA (of both CTAs of a pair) walk
// the same sequence.
template <bool PAIR>
__device__ __forceinline__ int tc_slot() { return PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x; }
template <bool PAIR>
__device__ __forceinline__ int tc_slots() { return PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x; }
struct TcSegment {
    int t, kb0, kb1;
};

template <bool PAIR>
struct TcWork {
    int t, u, u_end;
    __device__ __forceinline__ void begin(const Tf32x3Args &p) {
        const int slot = tc_slot<PAIR>(), slots = tc_slots<PAIR>();
        t = slot;
        const int64_t base = (int64_t)p.sk_tile0 * p.k_blocks;
        const int64_t W = (int64_t)(p.num_tiles - p.sk_tile0) * p.k_blocks;
        u = (int)(base + (int64_t)slot * W / slots);
        u_end = (int)(base + (int64_t)(slot + 1) * W / slots);
    }
    __device__ __forceinline__ bool get(const Tf32x3Args &p, TcSegment &s) const {
        if (t < p.sk_tile0) {
            s.t = t;
            s.kb0 = 0;
            s.kb1 = p.k_blocks;
            return true;
        }
        if (u >= u_end) return false;
        s.t = u / p.k_blocks;
        s.kb0 = u - s.t * p.k_blocks;
        s.kb1 = min(p.k_blocks, s.kb0 + (u_end - u));
        return true;
    }
    __device__ __forceinline__ void advance(const Tf32x3Args &p, const TcSegment &s) {
        if (t < p.sk_tile0) t += tc_slots<PAIR>();
        else u += s.kb1 - s.kb0;
    }
};

// The slot whose stream-K unit range contains unit u.
template <bool PAIR>
__device__ __forceinline__ int tc_slot_of_unit(int u, const Tf32x3Args &p) {
    const int64_t base = (int64_t)p.sk_tile0 * p.k_blocks;
    const int64_t W = (int64_t)(p.num_tiles - p.sk_tile0) * p.k_blocks;
    return (int)((((int64_t)u - base + 1) * tc_slots<PAIR>() - 1) / W);
}

__device__ __forceinline__ void prefetch_l2(const float *p) {
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

template <class Cfg, bool BETA_ZERO, bool C_VEC>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
sgemm_tf32x3_kernel(const __grid_constant__ CUtensorMap tmAhi, const __grid_constant__ CUtensorMap tmAlo,
                    const __grid_constant__ CUtensorMap tmBhi, const __grid_constant__ CUtensorMap tmBlo,
                    const Tf32x3Args p)
{
    constexpr bool PAIR = Cfg::PAIR;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int TILE_M = Cfg::TILE_M, B_ROWS = Cfg::B_ROWS;
    constexpr uint32_t IDESC = idesc_tf32(TILE_M, BN);

    extern __shared__ unsigned char smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    unsigned char *smem = smem_raw + pad;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * Cfg::STAGE_BYTES);
    uint64_t *full = bars;                      // TMA -> MMA, per stage
    uint64_t *empty = bars + STAGES;            // MMA -> TMA, per stage
    uint64_t *tfull = bars + 2 * STAGES;        // MMA -> epilogue, per accumulator
    uint64_t *tempty = tfull + 2;               // epilogue -> MMA, per accumulator
    uint64_t *drain = tempty + 2;               // MMA completion before teardown
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);   // [1]: stream-K launch tag
    float *xpose = reinterpret_cast<float *>(tmem_slot + 4);     // 16 bytes after the barriers

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Pair: rank 0 issues the MMAs and owns the barriers both CTAs' copies
    // and epilogues report to (full, tempty); both CTAs' empty and tfull
    // barriers receive rank 0's MMA completions.
    const uint32_t rank = PAIR ? cluster_rank() : 0u;

    if (warp == 0) {
        if constexpr (PAIR) tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        else tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], (PAIR ? 2 : 1) * Cfg::EPI_WARPS);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
        prefetch_tensormap(&tmAhi);
        prefetch_tensormap(&tmAlo);
        prefetch_tensormap(&tmBhi);
        prefetch_tensormap(&tmBlo);
    }
    // Shared memory, tensor memory and parameters only so far: wait for the
    // kernel before this one (the operand split) before touching global
    // memory.
    griddep_launch_dependents();
    griddep_wait();
    const bool stream_k = p.sk_tile0 < p.num_tiles;
    if (threadIdx.x == 32 && stream_k) tmem_slot[1] = sk_launch_tag(p.sk_seq);
    tc_fence_before();
    // A pair's CTAs signal each other's barriers from here on: both must
    // have initialised theirs.
    if constexpr (PAIR) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    const uint32_t sk_tag = stream_k ? reinterpret_cast<volatile uint32_t *>(tmem_slot)[1] : 0u;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        TcWork<PAIR> w;
        w.begin(p);
        TcSegment seg;
        while (ok && w.get(p, seg)) {
            int bt, tm, tn;
            tile_coords(seg.t, p.tiles_m, p.tiles_n, p.group_m, bt, tm, tn);
            const int ya = tm * TILE_M + (int)rank * BM;      // this CTA's rows of A
            const int yb = tn * BN + (int)rank * B_ROWS;      // this CTA's columns of B
            for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
                if (p.withhold == kWithholdRefill && issued >= STAGES) {
                    ok = false;     // test hook: stop after one ring fill (drain below)
                    break;
                }
                if (!mbar_wait_bounded<PAIR>(&empty[stage], phase ^ 1u, p.timeout_ns)) {
                    record_error(p.err, kSiteProducerEmpty);
                    ok = false;
                    break;
                }
                unsigned char *st = smem + stage * Cfg::STAGE_BYTES;
                if constexpr (PAIR) {
                    // Both CTAs' copies complete on rank 0's barrier, which
                    // rank 0 arms with the pair's bytes.
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * Cfg::STAGE_BYTES);
                    const uint32_t fb = cluster_addr(&full[stage], 0);
                    tma_load_3d_pair(st, &tmAhi, fb, kb * BK, ya, bt);
                    tma_load_3d_pair(st + Cfg::A_BYTES, &tmAlo, fb, kb * BK, ya, bt);
                    tma_load_3d_pair(st + 2 * Cfg::A_BYTES, &tmBhi, fb, kb * BK, yb, bt);
                    tma_load_3d_pair(st + 2 * Cfg::A_BYTES + Cfg::B_BYTES, &tmBlo, fb, kb * BK, yb, bt);
                } else {
                    mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
                    tma_load_3d(st, &tmAhi, &full[stage], kb * BK, ya, bt);
                    tma_load_3d(st + Cfg::A_BYTES, &tmAlo, &full[stage], kb * BK, ya, bt);
                    tma_load_3d(st + 2 * Cfg::A_BYTES, &tmBhi, &full[stage], kb * BK, yb, bt);
                    tma_load_3d(st + 2 * Cfg::A_BYTES + Cfg::B_BYTES, &tmBlo, &full[stage], kb * BK, yb, bt);
                }
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            w.advance(p, seg);
        }
        if (!ok) {
            // Let this CTA's own copies land before it can exit.  Rank 1 of
            // a pair cannot see its copies complete (they count on rank 0's
            // barrier): it waits for its stages to be released instead,
            // which happens only after they landed, or for the limit, far
            // longer than any copy takes.
            const int pending = issued < STAGES ? issued : STAGES;
            for (int back = 1; back <= pending; ++back) {
                int s = stage - back;
                uint32_t ph = phase;
                if (s < 0) { s += STAGES; ph ^= 1u; }
                mbar_wait_bounded<PAIR>(rank == 0 ? &full[s] : &empty[s], ph, p.timeout_ns);
            }
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---------------- MMA issuer (rank 0 of a pair) ----------------
        int stage = 0;
        uint32_t phase = 0;
        int gc = 0;             // chunk counter across segments: TMEM buffer gc & 1
        bool ok = true;
        // One accumulator chunk: K slices [kb0, kb1) into TMEM buffer gc & 1.
        auto chunk = [&](int kb0, int kb1) {
            const int ab = gc & 1;
            const uint32_t use = (uint32_t)(gc >> 1);
            ++gc;
            if (!mbar_wait_bounded<PAIR>(&tempty[ab], (use & 1u) ^ 1u, p.timeout_ns)) {
                record_error(p.err, kSiteConsumerFull);
                ok = false;
                return;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(ab * BN);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_bounded<PAIR>(&full[stage], phase, downstream_limit(p.timeout_ns))) {
                    record_error(p.err, kSiteConsumerFull);
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint32_t s_ahi = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                const uint32_t s_alo = s_ahi + Cfg::A_BYTES;
                const uint32_t s_bhi = s_ahi + 2 * Cfg::A_BYTES;
                const uint32_t s_blo = s_bhi + Cfg::B_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 8; ++kk) {
                    // K = 8 tf32 values = 32 bytes per MMA along the swizzled row.
                    const uint32_t off = (uint32_t)kk * 32u;
                    const uint64_t a_hi = smem_desc_k_sw128(s_ahi + off);
                    const uint64_t a_lo = smem_desc_k_sw128(s_alo + off);
                    const uint64_t b_hi = smem_desc_k_sw128(s_bhi + off);
                    const uint64_t b_lo = smem_desc_k_sw128(s_blo + off);
                    const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
                    // Small terms first, then the dominant product.
                    if constexpr (PAIR) {
                        mma_tf32_pair(d_tmem, a_lo, b_hi, IDESC, acc);
                        mma_tf32_pair(d_tmem, a_hi, b_lo, IDESC, 1u);
                        mma_tf32_pair(d_tmem, a_hi, b_hi, IDESC, 1u);
                    } else {
                        mma_tf32(d_tmem, a_lo, b_hi, IDESC, acc);
                        mma_tf32(d_tmem, a_hi, b_lo, IDESC, 1u);
                        mma_tf32(d_tmem, a_hi, b_hi, IDESC, 1u);
                    }
                }
                // Frees the stage (in both CTAs of a pair) once these MMAs are done.
                if (p.withhold != kWithholdRelease) {
                    if constexpr (PAIR) mma_commit_pair_mc(&empty[stage], 0x3);
                    else mma_commit(&empty[stage]);
                }
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            // Chunk ready for the epilogue (of both CTAs).
            if constexpr (PAIR) mma_commit_pair_mc(&tfull[ab], 0x3);
            else mma_commit(&tfull[ab]);
        };
        // Whole tiles, then the stream-K segments (the same order as the
        // producer and the epilogue walk).
        for (int t = tc_slot<PAIR>(); ok && t < p.sk_tile0; t += tc_slots<PAIR>())
            for (int kb0 = 0; ok && kb0 < p.k_blocks; kb0 += Cfg::CHUNK_KB)
                chunk(kb0, min(p.k_blocks, kb0 + Cfg::CHUNK_KB));
        TcWork<PAIR> w;
        w.begin(p);
        w.t = p.sk_tile0;                       // whole tiles done above
        TcSegment seg;
        while (ok && w.get(p, seg)) {
            for (int kb0 = seg.kb0; ok && kb0 < seg.kb1; kb0 += Cfg::CHUNK_KB)
                chunk(kb0, min(seg.kb1, kb0 + Cfg::CHUNK_KB));
            w.advance(p, seg);
        }
        // All MMAs this thread issued complete before the CTA tears down.
        if constexpr (PAIR) mma_commit_pair(drain);
        else mma_commit(drain);
        mbar_wait_bounded(drain, 0u, p.timeout_ns);
    } else if (warp >= 2) {
        // ---------------- epilogue: TMEM chunks -> FP32 sums -> C ----------------
        const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
        constexpr int SLAB = Cfg::SLAB;
        const int ew = warp - 2;                // epilogue warp index
        const int slab0 = (ew >> 2) * SLAB;     // first column of this warp's slab
        const float alpha = p.alpha, beta = p.beta;
        int gc = 0;
        bool ok = true;
        TcWork<PAIR> w;
        w.begin(p);
        TcSegment seg;
        while (ok && w.get(p, seg)) {
            float sum[SLAB];
#pragma unroll
            for (int c = 0; c < SLAB; ++c) sum[c] = 0.f;
            if constexpr (!BETA_ZERO) {
                // This segment ends by reading C: start pulling this lane's
                // row of the tile into L2 while the products are computed.
                if (seg.kb0 == 0) {
                    int bt, tm, tn;
                    tile_coords(seg.t, p.tiles_m, p.tiles_n, p.group_m, bt, tm, tn);
                    const int row = tm * TILE_M + (int)rank * BM + quarter * 32 + lane;
                    const int c0 = tn * BN + slab0;
                    if (row < p.M && c0 < p.N) {
                        const float *crow = p.C + (int64_t)bt * p.stride_c + (int64_t)row * p.ldc;
                        const int c1 = min(p.N, c0 + SLAB) - 1;
                        for (int c = c0; c < c1; c += 32) prefetch_l2(crow + c);
                        prefetch_l2(crow + c1);
                    }
                }
            }
            for (int kb0 = seg.kb0; kb0 < seg.kb1; kb0 += Cfg::CHUNK_KB, ++gc) {
                const int ab = gc & 1;
                const uint32_t use = (uint32_t)(gc >> 1);
                if (!mbar_wait_bounded<PAIR>(&tfull[ab], use & 1u, downstream_limit(p.timeout_ns))) {
                    record_error(p.err, kSiteConsumerFull);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                       (uint32_t)(ab * BN + slab0);
#pragma unroll
                for (int c0 = 0; c0 < SLAB; c0 += 16) {
                    float v[16];
                    tmem_ld_16cols(taddr + (uint32_t)c0, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) sum[c0 + i] += v[i];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR) mbar_arrive_cluster(cluster_addr(&tempty[ab], 0));
                    else mbar_arrive(&tempty[ab]);
                }
            }
            if (!ok) break;

            // ---------------- stream-K fixup ----------------
            if (seg.kb0 != 0 || seg.kb1 != p.k_blocks) {
                // Thread-major slot layout: the same (warp, lane) holds the
                // same rows and columns in every CTA, so stores and loads of
                // a slot are contiguous across the warp.
                if (seg.kb0 != 0) {
                    // Not the tile's first slice: hand the partial sums to the
                    // CTA that finishes the tile, then go on.
                    float4 *mine = reinterpret_cast<float4 *>(p.partials + (size_t)blockIdx.x * (BM * BN));
#pragma unroll
                    for (int q = 0; q < SLAB / 4; ++q)
                        __stcg(&mine[(ew * (SLAB / 4) + q) * 32 + lane],
                               make_float4(sum[4 * q], sum[4 * q + 1], sum[4 * q + 2], sum[4 * q + 3]));
                    __threadfence();
                    __syncwarp();
                    if (lane == 0 && p.withhold != kWithholdStreamKFlag)
                        st_release_gpu(&p.flags[blockIdx.x * Cfg::EPI_WARPS + ew], sk_tag);
                    w.advance(p, seg);
                    continue;
                }
                // The tile's first slice: add the partial tiles of the slots
                // that hold its other slices, in slot order (deterministic);
                // in a pair, those of the CTA of the same rank.
                const int tile_u0 = seg.t * p.k_blocks;
                const int c_first = tc_slot_of_unit<PAIR>(tile_u0 + seg.kb1, p);
                const int c_last = tc_slot_of_unit<PAIR>(tile_u0 + p.k_blocks - 1, p);
                if (lane == 0) {
                    for (int c = c_first; c <= c_last; ++c) {
                        const int cta = PAIR ? 2 * c + (int)rank : c;
                        if (!tag_wait_bounded(&p.flags[cta * Cfg::EPI_WARPS + ew], sk_tag, p.timeout_ns))
                            record_error(p.err, kSiteStreamKFlag);
                    }
                }
                __syncwarp();
                for (int c = c_first; c <= c_last; ++c) {
                    const int cta = PAIR ? 2 * c + (int)rank : c;
                    const float4 *other = reinterpret_cast<const float4 *>(p.partials + (size_t)cta * (BM * BN));
#pragma unroll
                    for (int q = 0; q < SLAB / 4; ++q) {
                        const float4 v = __ldcg(&other[(ew * (SLAB / 4) + q) * 32 + lane]);
                        sum[4 * q] += v.x;
                        sum[4 * q + 1] += v.y;
                        sum[4 * q + 2] += v.z;
                        sum[4 * q + 3] += v.w;
                    }
                }
            }

            int bt, tm, tn;
            tile_coords(seg.t, p.tiles_m, p.tiles_n, p.group_m, bt, tm, tn);
            float *cbase = p.C + (int64_t)bt * p.stride_c;
            if constexpr (C_VEC) {
                // Direct: each lane reads and writes its own row, 16 bytes at
                // a time; the loads of a group of 16 columns are issued
                // before its stores so that their latencies overlap.
                const int row = tm * TILE_M + (int)rank * BM + quarter * 32 + lane;
                if (row < p.M) {
                    float *crow = cbase + (int64_t)row * p.ldc;
                    constexpr int G = 4;             // float4 columns per group
#pragma unroll
                    for (int q0 = 0; q0 < SLAB / 4; q0 += G) {
                        float4 cin[G];
                        if constexpr (!BETA_ZERO) {
#pragma unroll
                            for (int j = 0; j < G; ++j) {
                                const int col = tn * BN + slab0 + 4 * (q0 + j);
                                if (col + 3 < p.N) {
                                    cin[j] = *reinterpret_cast<const float4 *>(crow + col);
                                } else {
                                    cin[j].x = col < p.N ? crow[col] : 0.f;
                                    cin[j].y = col + 1 < p.N ? crow[col + 1] : 0.f;
                                    cin[j].z = col + 2 < p.N ? crow[col + 2] : 0.f;
                                    cin[j].w = 0.f;
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < G; ++j) {
                            const int q = q0 + j;
                            const int col = tn * BN + slab0 + 4 * q;
                            float o[4] = {alpha * sum[4 * q], alpha * sum[4 * q + 1], alpha * sum[4 * q + 2],
                                          alpha * sum[4 * q + 3]};
                            if constexpr (!BETA_ZERO) {
                                o[0] = fmaf(beta, cin[j].x, o[0]);
                                o[1] = fmaf(beta, cin[j].y, o[1]);
                                o[2] = fmaf(beta, cin[j].z, o[2]);
                                o[3] = fmaf(beta, cin[j].w, o[3]);
                            }
                            if (col + 3 < p.N) {
                                *reinterpret_cast<float4 *>(crow + col) = make_float4(o[0], o[1], o[2], o[3]);
                            } else {
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    if (col + e < p.N) crow[col + e] = o[e];
                            }
                        }
                    }
                }
            } else {
                // Staged (C rows not 16-byte aligned): with 4-byte accesses
                // one lane per row would touch 32 rows per instruction.  Each 32 x 32 block of the warp's rows goes
                // through shared memory instead, so that lane l handles
                // column l of one row at a time: 128-byte row segments.
                float *tb = xpose + ew * (32 * 33);
                const int row0 = tm * TILE_M + (int)rank * BM + quarter * 32;
#pragma unroll
                for (int b = 0; b < SLAB / 32; ++b) {
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 32; ++c) tb[lane * 33 + c] = sum[32 * b + c];
                    __syncwarp();
                    const int col = tn * BN + slab0 + 32 * b + lane;
                    const bool col_ok = col < p.N;
#pragma unroll
                    for (int r0 = 0; r0 < 32; r0 += 16) {
                        float cin[16];
                        if constexpr (!BETA_ZERO) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int row = row0 + r0 + j;
                                cin[j] = (col_ok && row < p.M) ? cbase[(int64_t)row * p.ldc + col] : 0.f;
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int row = row0 + r0 + j;
                            if (col_ok && row < p.M) {
                                const float v = alpha * tb[(r0 + j) * 33 + lane];
                                float *dst = cbase + (int64_t)row * p.ldc + col;
                                if constexpr (BETA_ZERO) *dst = v;
                                else *dst = fmaf(beta, cin[j], v);
                            }
                        }
                    }
                }
            }
            w.advance(p, seg);
        }
    }

    // ---------------- teardown ----------------
    // In a pair, neither CTA leaves while the other's MMAs, copies or
    // arrivals may still touch its shared memory or barriers.
    tc_fence_before();
    if constexpr (PAIR) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
        else tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
    if (threadIdx.x == 32 && stream_k) sk_launch_done(p.sk_seq, sk_tag);
}

// ---------------------------------------------------------------- launches

namespace {
template <class Cfg>
Tf32x3Info make_info() {
    Tf32x3Info info;
    info.fn[0] = reinterpret_cast<const void *>(&sgemm_tf32x3_kernel<Cfg, true, true>);
    info.fn[1] = reinterpret_cast<const void *>(&sgemm_tf32x3_kernel<Cfg, true, false>);
    info.fn[2] = reinterpret_cast<const void *>(&sgemm_tf32x3_kernel<Cfg, false, true>);
    info.fn[3] = reinterpret_cast<const void *>(&sgemm_tf32x3_kernel<Cfg, false, false>);
    info.threads = Cfg::THREADS;
    info.smem = Cfg::SMEM_BYTES;
    info.bm = Cfg::TILE_M;
    info.bn = Cfg::BN;
    info.pair = Cfg::PAIR ? 1 : 0;
    info.box_a = Cfg::BM;
    info.box_b = Cfg::B_ROWS;
    info.bk = Cfg::BK;
    info.stages = Cfg::STAGES;
    info.chunk_kb = Cfg::CHUNK_KB;
    return info;
}
}  // namespace

// Tensor-core tile configurations: 1: 128 x 128 (3 stages, 4 epilogue
// warps), 2: 128 x 192 (2 stages, 8), 3: 128 x 256 (2 stages, 8), 4: 256 x
// 256 on an SM pair (each CTA 128 rows of A and 128 columns of B per stage,
// 3 stages, 8 epilogue warps).  Wider tiles read fewer shared-memory bytes
// per MMA FLOP; the pair halves B's bytes per SM.  Accumulator chunks of 8
// K slices (256 K) in every configuration: each chunk hands a TMEM buffer
// from the MMA issuer to the epilogue warps and back, and fewer hand-overs
// ran faster (4096^3 per call, chunks of 64 / 128 / 256 K: 508.0 / 468.7 /
// 457.7 us; 4095 x 4097 x 1023: 238.6 / 211.6 / 193.6 us) while the error
// grew with the chunk length (worst error over the acceptance bound at
// 512 x 512 x 16384: 0.037 / 0.058 / 0.132; mean error over sum |a b| at
// 1024^3: 1.8e-8 / 3.3e-8 / 6.4e-8).
Tf32x3Info tf32x3_info(int config) {
    static const Tf32x3Info infos[kNumTf32x3Configs] = {
        make_info<Tf32x3Config<128, 3, 8, 4>>(),
        make_info<Tf32x3Config<192, 2, 8, 8>>(),
        make_info<Tf32x3Config<256, 2, 8, 8>>(),
        make_info<Tf32x3Config<256, 3, 8, 8, true>>(),
    };
    if (config < 1 || config > kNumTf32x3Configs) config = 1;
    return infos[config - 1];
}

}  // namespace sg
