// FP32 SGEMM main kernel for sm_103a: C = alpha * A.B + beta * C, row major.
//
// Structure (persistent CTAs, one per SM slot; tiles taken round robin,
// then stream-K units):
//   * a producer: thread 0 (one of the consumers) streams the K slices of A
//     and B into an S-stage shared-memory ring with TMA tile loads; each
//     stage has a
//     "full" mbarrier (TMA transaction bytes) and an "empty" mbarrier (one
//     arrival per consumer warp).  Out-of-range rows/columns of partial tiles
//     arrive as zeros (TMA out-of-bounds fill), so M, N, K need not be tile
//     multiples.
//   * WARPS_M x WARPS_N consumer warps: each lane keeps an 8 x 16 register
//     tile of FP32 accumulators and, for every k, forms the outer product of
//     8 values of A and 16 values of B with packed two-wide FP32 FMAs
//     (fma.rn.f32x2: each lane issues one instruction per two products).
//   * epilogue straight from registers: alpha*acc (+ beta*C, and C is not
//     read when beta == 0), 16-byte stores when C's alignment allows; or, in
//     the STORE_TMA configurations (the automatic choice wherever C is not
//     read, and wherever C is not 16-byte aligned), each warp writes its
//     alpha*acc block to its own shared-memory staging area, and then either
//     one lane hands it to TMA tile stores, so that C drains to memory while
//     the next tile computes, or (C not 16-byte aligned) the warp writes it
//     back in 64-byte row runs.
//
// What the pages contribute, and what changed for this chip:
//   * the per-thread outer-product register tile and the K loop over staged
//     shared-memory slices ("2D Register Tiling: The Outer Product",
//     maxxfuu article4/page8; easonhuang.dev/blog/gpu_matmul, "2D
//     Blocktiling" and "Kernel 8: Warptiling");
//   * loading the next slice while this one is computed, one sync per slice
//     (easonhuang.dev, "Kernel 9 & 10: Staging"; "The Final Kernel",
//     maxxfuu article4/page14), here as a TMA + mbarrier ring of S stages
//     instead of register-staged double buffering;
//   * the thread tile's A values read as 16-byte vectors (the pages transpose
//     A in shared memory for this; TMA cannot transpose 4-byte elements, so
//     A stays k-contiguous and each 16-byte read carries 4 consecutive k of
//     one row, used over 4 k steps; the next group is read one k step ahead,
//     while each k's B values are read just before its FMAs, which is what
//     fits 255 registers -- some configurations keep 8-byte A reads with
//     both fragments double buffered); bank conflicts between the rows a warp
//     reads together are removed by the TMA 32/64/128-byte swizzle instead
//     of padding, which keeps every vector read 16-byte aligned ("The Final
//     Kernel", "The Padding Has To Go");
//   * rows of a lane are interleaved with stride WR and its columns with
//     stride 4*WC, so that the lanes of a warp read consecutive 16-byte
//     chunks of B (one wavefront, as in the pages' warptiling argument) and
//     distinct swizzled chunks of A;
//   * beta == 0 selects a kernel that never reads C ("The Final Kernel",
//     "Skipping The Read Of C"); __launch_bounds__(threads, 1) lets the
//     compiler spend registers on the 128 accumulators ("The Declaration
//     That Was Worth More Than Any Of It").
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace sg {

struct GemmArgs {
    int M, N, K;
    float alpha, beta;
    float *C;
    int64_t ldc;
    int64_t stride_c;     // elements between the C matrices of consecutive batches
    int tiles_m, tiles_n, num_tiles;   // num_tiles = batch * tiles_m * tiles_n
    int k_blocks;
    int group_m;          // rasterisation: tile rows per band
    int sk_tile0;         // tiles [0, sk_tile0) whole, round robin; [sk_tile0, num_tiles) stream-K
    float *partials;      // stream-K: one BM x BN partial tile per CTA
    uint32_t *flags;      // stream-K: per CTA and consumer warp, the launch tag of the part it stored
    uint32_t *sk_seq;     // stream-K: {tag of the last completed launch, CTAs finished in this one}
    uint32_t *err;        // device error word (bounded waits)
    uint64_t timeout_ns;
    int withhold;         // test hook (Withhold): a signal left out on purpose
};

template <int KA> struct AVecT;
template <> struct AVecT<4> { using type = float4; };
template <> struct AVecT<2> { using type = float2; };

__device__ __forceinline__ float vec_get(const float4 &v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}
__device__ __forceinline__ float vec_get(const float2 &v, int k) { return k == 0 ? v.x : v.y; }

// Tile configuration.
//   BM x BN output tile, BK-wide K slices, STAGES-deep shared-memory ring;
//   WARPS_M x WARPS_N consumer warps, each lane an 8 x 16 register tile
//   (lane grid WR x (32/WR) inside a warp); thread 0 also issues the TMA
//   loads;
//   KA: k values per vector read of A (4 -> 16 B, 2 -> 8 B);
//   PIPE_B: the next A group is always read one k step ahead of need
//   (register double buffering); 1 = the B values of the next k are read
//   while this k's FMAs run as well, 0 = each k's B values are read just
//   before its FMAs (which frees 16 registers for 16-byte A reads);
//   KQ_UNROLL: A-vector groups per loop iteration (even);
//   STORE_TMA: 1 = beta == 0 tiles leave through a per-warp shared-memory
//   staging area and TMA tile stores (64 x 16 boxes) instead of st.global;
//   REFILL_LAG (inline producer): after consuming slice g, thread 0 refills
//   the stage of slice g - REFILL_LAG.  1 never waits for a slower warp; 0
//   waits for all warps to release slice g but keeps STAGES - 1 slices in
//   flight instead of STAGES - 2 (what a 2-stage ring needs).
template <int BM_, int BN_, int BK_, int STAGES_, int WARPS_M_, int WARPS_N_,
          int WR_, int KQ_UNROLL_, int MIN_CTAS_, int KA_, int PIPE_B_, int STORE_TMA_ = 0,
          int REFILL_LAG_ = 1>
struct FfmaConfig {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_;
    static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_;
    static constexpr int WR = WR_, WC = 32 / WR_;
    static constexpr int TM = 8, TN = 16;
    static constexpr int WTM = WR * TM, WTN = WC * TN;
    static constexpr int KQ_UNROLL = KQ_UNROLL_;
    static constexpr int MIN_CTAS = MIN_CTAS_;
    static constexpr int KA = KA_;
    static constexpr bool PIPE_B = PIPE_B_ != 0;   // B fragments double buffered too
    static constexpr bool STORE_TMA = STORE_TMA_ != 0;
    static constexpr int REFILL_LAG = REFILL_LAG_;
    static constexpr int CONSUMER_WARPS = WARPS_M * WARPS_N;
    static constexpr int THREADS = CONSUMER_WARPS * 32;
    static constexpr int ROW_BYTES_A = BK * 4;                 // one row of the A slice
    static constexpr int A_STAGE_BYTES = BM * BK * 4;
    static constexpr int B_STAGE_BYTES = BK * BN * 4;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    // TMA swizzle span equals the A row: 128 B (BK=32), 64 B (BK=16), 32 B (BK=8).
    static constexpr int SWZ_MASK = ROW_BYTES_A / 16 - 1;      // 7, 3, 1
    // C staging for TMA stores: one WTM x WTN block per consumer warp, kept
    // as NJ boxes of WTM rows x 4*WC columns (box j = the lane columns of j).
    static constexpr int C_BOX_COLS = 4 * WC, C_BOX_BYTES = WTM * C_BOX_COLS * 4;
    static constexpr int STORE_BYTES = STORE_TMA ? CONSUMER_WARPS * WTM * WTN * 4 : 0;
    // Barriers, then 128 bytes for the TMA issuer's slice cursor and the
    // stream-K launch tag, then 1024 for aligning the stages.
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STORE_BYTES + 2 * STAGES * 8 + 128 + 1024;
    static constexpr int NKQ = BK / KA;                        // A-vector groups per slice
    // TMA boxes are at most 256 elements a side: wider tiles take several.
    // A's boxes stack rows (the stage layout is unchanged); B's boxes sit one
    // after another, each BK rows of BOX_N columns.
    static constexpr int BOX_M = BM < 256 ? BM : 256, A_BOXES = BM / BOX_M;
    static constexpr int BOX_N = BN < 256 ? BN : 256, B_BOXES = BN / BOX_N;

    static_assert(BK == 8 || BK == 16 || BK == 32, "A slice row must match a TMA swizzle span");
    static_assert(WR == 1 || WR == 2 || WR == 4 || WR == 8 || WR == 16 || WR == 32, "WR");
    static_assert(BM == WARPS_M * WTM && BN == WARPS_N * WTN, "tile / warp grid mismatch");
    static_assert(WTM * ROW_BYTES_A >= 1024, "warp row block must cover a swizzle period");
    static_assert(BM <= 1024 && BN <= 1024 && BM % BOX_M == 0 && BN % BOX_N == 0, "TMA boxes per tile");
    static_assert(BOX_N % WTN == 0, "a warp's columns lie in one B box");
    static_assert(A_STAGE_BYTES % 1024 == 0 && B_STAGE_BYTES % 1024 == 0, "stage alignment");
    static_assert(KA == 2 || KA == 4, "A vector width");
    static_assert(NKQ % KQ_UNROLL == 0, "unroll must divide the slice");
    static_assert(KQ_UNROLL % 2 == 0, "pipelined fragments alternate two buffers");
    static_assert(STAGES >= 2, "ring depth");
    static_assert(REFILL_LAG == 0 || REFILL_LAG == 1, "refill lag");
    // Staging writes are conflict-free when the 8 lanes of a quarter warp
    // cover two rows 64 bytes apart and four consecutive 16-byte chunks.
    static_assert(!STORE_TMA || (WR == 8 && WC == 4), "TMA store staging layout");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// Tile t -> (batch b, tile row tm, tile column tn).  Inside a batch, tiles
// are walked in bands of group_m tile rows, column by column, so that the
// tiles running at the same time share rows of A and columns of B in L2.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m,
                                            int &b, int &tm, int &tn) {
    const int per_batch = tiles_m * tiles_n;
    b = t / per_batch;
    t -= b * per_batch;
    const int per_group = group_m * tiles_n;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int rows = min(tiles_m - first_m, group_m);
    const int local = t - g * per_group;
    tm = first_m + local % rows;
    tn = local / rows;
}

// Work of one CTA, as segments: a run of K slices [kb0, kb1) of tile t.
//   Tiles [0, sk_tile0): whole tiles blockIdx.x, blockIdx.x + gridDim.x, ...
//     (consecutive tile numbers run concurrently, a compact band of C).
//   Tiles [sk_tile0, num_tiles): their (tile, slice) units, tile major, are
//     cut into gridDim.x equal contiguous ranges, one per CTA ("stream-K"),
//     so every CTA ends up with the same number of FMAs.  A tile cut between
//     CTAs is finished by the CTA holding its first slice (the last segment
//     of that CTA); the others store partial sums.
// Units are counted in 32 bits: the host enables stream-K only when
// num_tiles * k_blocks < 2^31.
struct Segment {
    int t, kb0, kb1;
};

struct WorkIter {
    int t;          // next whole tile
    int u, u_end;   // stream-K units (absolute: tile * k_blocks + slice)

    __device__ __forceinline__ void begin(const GemmArgs &p) {
        t = blockIdx.x;
        const int64_t base = (int64_t)p.sk_tile0 * p.k_blocks;
        const int64_t W = (int64_t)(p.num_tiles - p.sk_tile0) * p.k_blocks;
        u = (int)(base + (int64_t)blockIdx.x * W / gridDim.x);
        u_end = (int)(base + (int64_t)(blockIdx.x + 1) * W / gridDim.x);
    }
    __device__ __forceinline__ bool get(const GemmArgs &p, Segment &s) const {
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
    __device__ __forceinline__ void advance(const GemmArgs &p, const Segment &s) {
        if (t < p.sk_tile0) t += gridDim.x;
        else u += s.kb1 - s.kb0;
    }
};

// Stream-K: the CTA whose unit range contains unit u.
__device__ __forceinline__ int cta_of_unit(int u, const GemmArgs &p) {
    const int64_t base = (int64_t)p.sk_tile0 * p.k_blocks;
    const int64_t W = (int64_t)(p.num_tiles - p.sk_tile0) * p.k_blocks;
    return (int)((((int64_t)u - base + 1) * gridDim.x - 1) / W);
}

// The sequence of K slices a CTA loads, in consumption order.  Slice number
// g (counted from 0 across segments) goes to stage g % STAGES and completes
// phase (g / STAGES) & 1 of that stage's barriers.  Only the issuing thread
// uses the cursor; it lives in shared memory and is read and written once
// per issued slice, so that it holds no registers across the FMA loop.
struct SliceCursor {
    WorkIter it;
    Segment seg;
    int valid;
    int kb, bt, tm, tn;
    int stage;
    uint32_t phase;
    int issued;
};
constexpr int kCursorWords = sizeof(SliceCursor) / 4;
static_assert(sizeof(SliceCursor) % 4 == 0, "cursor is a block of 32-bit words");

__device__ __forceinline__ SliceCursor cursor_load(const SliceCursor *sc) {
    SliceCursor c;
    const volatile int *src = reinterpret_cast<const volatile int *>(sc);
    int *dst = reinterpret_cast<int *>(&c);
#pragma unroll
    for (int i = 0; i < kCursorWords; ++i) dst[i] = src[i];
    return c;
}

__device__ __forceinline__ void cursor_store(SliceCursor *sc, const SliceCursor &c) {
    volatile int *dst = reinterpret_cast<volatile int *>(sc);
    const int *src = reinterpret_cast<const int *>(&c);
#pragma unroll
    for (int i = 0; i < kCursorWords; ++i) dst[i] = src[i];
}

__device__ __forceinline__ void cursor_begin(SliceCursor *sc, const GemmArgs &p) {
    SliceCursor c;
    c.it.begin(p);
    c.valid = c.it.get(p, c.seg) ? 1 : 0;
    c.kb = c.seg.kb0;
    c.bt = c.tm = c.tn = 0;
    if (c.valid) tile_coords(c.seg.t, p.tiles_m, p.tiles_n, p.group_m, c.bt, c.tm, c.tn);
    c.stage = 0;
    c.phase = 0;
    c.issued = 0;
    cursor_store(sc, c);
}

__device__ __forceinline__ bool cursor_valid(const SliceCursor *sc) {
    return reinterpret_cast<const volatile SliceCursor *>(sc)->valid != 0;
}
__device__ __forceinline__ int cursor_issued(const SliceCursor *sc) {
    return reinterpret_cast<const volatile SliceCursor *>(sc)->issued;
}

// Issue the cursor's next slice (waiting, bounded, for its stage to be free).
template <class Cfg>
__device__ __forceinline__ bool issue_slice(SliceCursor *sc, const GemmArgs &p,
                                         const CUtensorMap *tmA, const CUtensorMap *tmB,
                                         unsigned char *sA, unsigned char *sB,
                                         uint64_t *full, uint64_t *empty) {
    SliceCursor c = cursor_load(sc);
    if (!mbar_wait_bounded(&empty[c.stage], c.phase ^ 1u, p.timeout_ns)) return false;
    mbar_arrive_expect_tx(&full[c.stage], Cfg::STAGE_BYTES);
#pragma unroll
    for (int q = 0; q < Cfg::A_BOXES; ++q)
        tma_load_3d(sA + c.stage * Cfg::A_STAGE_BYTES + q * (Cfg::BOX_M * Cfg::BK * 4), tmA, &full[c.stage],
                    c.kb * Cfg::BK, c.tm * Cfg::BM + q * Cfg::BOX_M, c.bt);
#pragma unroll
    for (int q = 0; q < Cfg::B_BOXES; ++q)
        tma_load_3d(sB + c.stage * Cfg::B_STAGE_BYTES + q * (Cfg::BK * Cfg::BOX_N * 4), tmB, &full[c.stage],
                    c.tn * Cfg::BN + q * Cfg::BOX_N, c.kb * Cfg::BK, c.bt);
    ++c.issued;
    if (++c.stage == Cfg::STAGES) { c.stage = 0; c.phase ^= 1u; }
    if (++c.kb == c.seg.kb1) {
        c.it.advance(p, c.seg);
        c.valid = c.it.get(p, c.seg) ? 1 : 0;
        if (c.valid) {
            c.kb = c.seg.kb0;
            tile_coords(c.seg.t, p.tiles_m, p.tiles_n, p.group_m, c.bt, c.tm, c.tn);
        }
    }
    cursor_store(sc, c);
    return true;
}

// Wait (bounded) until slices [from, to) have landed, so that a CTA that
// gives up never exits with its own TMA copies still in flight.
template <class Cfg>
__device__ __forceinline__ void drain_slices(int from, int to, uint64_t *full, uint64_t timeout_ns) {
    if (from < to - Cfg::STAGES) from = to - Cfg::STAGES;
    for (int g = from; g < to; ++g)
        mbar_wait_bounded(&full[g % Cfg::STAGES], (uint32_t)(g / Cfg::STAGES) & 1u, timeout_ns);
}

// TMA tile store of a shared-memory box to C (3-D map {N, M, batch});
// elements outside the map's extent are not written.  The stores of one
// thread form bulk groups: commit after issuing, wait before the source is
// reused (".read": the box has been read out of shared memory) or before
// the CTA exits (all writes done).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src,
                                             int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 :: "l"(map), "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Generic-proxy writes to shared memory, made visible to the TMA engine.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <class Cfg, bool BETA_ZERO, bool C_VEC>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_CTAS)
sgemm_ffma_tma_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC,
                      const GemmArgs p)
{
    // tmC is read only by configurations with STORE_TMA, for beta == 0 and
    // a 16-byte aligned C (the host encodes it then; otherwise it is unused).
    constexpr bool TMA_EPILOGUE = Cfg::STORE_TMA && BETA_ZERO && C_VEC;
    // Same configurations, C not 16-byte aligned: the block still goes
    // through the staging area, then leaves in row runs (plain stores).
    constexpr bool STAGED_EPILOGUE = Cfg::STORE_TMA && !C_VEC;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int TM = Cfg::TM, TN = Cfg::TN, WR = Cfg::WR, WC = Cfg::WC;
    constexpr int NJ = TN / 4;   // 16-byte column groups per lane
    constexpr int KA = Cfg::KA;  // k values per vector read of A (4: 16 B, 2: 8 B)
    constexpr int NKQ = Cfg::NKQ;
    constexpr int CONSUMER_THREADS = Cfg::CONSUMER_WARPS * 32;
    using AVec = typename AVecT<KA>::type;

    extern __shared__ unsigned char smem_raw[];
    // TMA 128-byte swizzle wants 1024-byte aligned destinations.  Offsetting
    // the __shared__ array itself keeps the pointer in the shared window.
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    unsigned char *smem = smem_raw + pad;
    unsigned char *sA = smem;
    unsigned char *sB = smem + STAGES * Cfg::A_STAGE_BYTES;
    unsigned char *sC = smem + STAGES * Cfg::STAGE_BYTES;   // STORE_BYTES of C staging
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * Cfg::STAGE_BYTES + Cfg::STORE_BYTES);
    uint64_t *empty = full + STAGES;
    SliceCursor *cursor = reinterpret_cast<SliceCursor *>(empty + STAGES);
    volatile uint32_t *sk_tag_s = reinterpret_cast<volatile uint32_t *>(cursor + 1);
    static_assert(sizeof(SliceCursor) + 4 <= 128, "cursor and tag fit their 128 bytes");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool stream_k = p.sk_tile0 < p.num_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], Cfg::CONSUMER_WARPS);
        }
        fence_barrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        // While the kernel before this one finishes: pull this CTA's first
        // slices into L2 (a hint; nothing is read before the wait below).
        WorkIter it0;
        it0.begin(p);
        Segment s0;
        if (it0.get(p, s0)) {
            int bt, tm, tn;
            tile_coords(s0.t, p.tiles_m, p.tiles_n, p.group_m, bt, tm, tn);
            for (int kb = s0.kb0; kb < s0.kb1 && kb < s0.kb0 + STAGES; ++kb) {
#pragma unroll
                for (int q = 0; q < Cfg::A_BOXES; ++q)
                    tma_prefetch_3d(&tmA, kb * BK, tm * BM + q * Cfg::BOX_M, bt);
#pragma unroll
                for (int q = 0; q < Cfg::B_BOXES; ++q)
                    tma_prefetch_3d(&tmB, tn * BN + q * Cfg::BOX_N, kb * BK, bt);
            }
        }
    }
    // Only shared memory, kernel parameters and L2 prefetches so far; from
    // here on global memory is read and written.
    griddep_launch_dependents();
    griddep_wait();
    if (threadIdx.x == 0 && stream_k) *sk_tag_s = sk_launch_tag(p.sk_seq);
    __syncthreads();
    // (The tag is read back from shared memory where it is used: a value
    // kept live across the FMA loop would compete for its registers.)

    // Thread 0 reports the end of its CTA's part of a stream-K launch at
    // whichever of its exits it takes (the normal end, or a wait that gave
    // up), so that the next launch gets a fresh tag in every case.
    auto cta_done = [&]() {
        if (threadIdx.x == 0 && p.sk_tile0 < p.num_tiles) sk_launch_done(p.sk_seq, *sk_tag_s);
    };
    // ---------------- consumers ----------------
    // Producer: thread 0 issues the first STAGES slices up front, then after
    // consuming slice g (g >= 1) refills the stage of slice g - 1, which
    // every warp has released by the time thread 0 is done with slice g (with
    // REFILL_LAG 0: the stage of slice g itself, once every warp released it).
    const bool producer = threadIdx.x == 0;
    if (producer) {
        if constexpr (TMA_EPILOGUE) prefetch_tensormap(&tmC);
        cursor_begin(cursor, p);
        while (cursor_valid(cursor) && cursor_issued(cursor) < STAGES)
            issue_slice<Cfg>(cursor, p, &tmA, &tmB, sA, sB, full, empty);   // fresh stages: never waits
    }

    const int wm = warp / Cfg::WARPS_N;
    const int wn = warp % Cfg::WARPS_N;
    const int lr = lane / WC;          // lane row in the warp grid
    const int lc = lane % WC;          // lane column
    // Rows of this lane inside the CTA tile: m_i = row0 + WR*i.
    const int row0 = wm * Cfg::WTM + lr;
    // Columns: n_j = col0 + 4*WC*j (+0..3).
    const int col0 = wn * Cfg::WTN + lc * 4;
    // This lane's first column inside the stage's B boxes.
    int b_off = col0;
    if constexpr (Cfg::B_BOXES > 1) b_off = (col0 / Cfg::BOX_N) * (Cfg::BK * Cfg::BOX_N) + col0 % Cfg::BOX_N;
    // Swizzle term of row0's A row; rows of other i differ by a compile-time
    // constant d_i because lr*ROW_BYTES_A and WR*i*ROW_BYTES_A occupy disjoint bits.
    const uint32_t a_x0 = ((uint32_t)(lr * Cfg::ROW_BYTES_A) >> 7) & Cfg::SWZ_MASK;
    const uint32_t a_row0_off = (uint32_t)row0 * Cfg::ROW_BYTES_A;

    // A: KA consecutive k of each of the lane's 8 rows, one vector read per
    // row.  Row m_i's 16-byte chunk c is stored at chunk c ^ swz(m_i).
    auto load_a = [&](const unsigned char *As, int kq, AVec (&a)[TM]) {
        const uint32_t chunk = (uint32_t)(kq * KA) >> 2;
        const uint32_t within = (uint32_t)(kq * KA * 4) & 15u;
        const uint32_t kx = chunk ^ a_x0;
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const uint32_t d_i = ((uint32_t)(WR * i * Cfg::ROW_BYTES_A) >> 7) & Cfg::SWZ_MASK;
            a[i] = *reinterpret_cast<const AVec *>(
                As + WR * i * Cfg::ROW_BYTES_A + (((kx ^ d_i) << 4) | within));
        }
    };
    // B: 16 values of row k, in 4 groups of 4 consecutive columns.
    auto load_b = [&](const float *Bs, int k, float4 (&b)[NJ]) {
        const float *brow = Bs + k * Cfg::BOX_N;
#pragma unroll
        for (int j = 0; j < NJ; ++j) b[j] = *reinterpret_cast<const float4 *>(brow + j * 4 * WC);
    };

    float2 acc[TM][TN / 2];
    // One k step of the outer product.  One CTA per SM: each B pair meets
    // all TM rows in turn (measured at 4096^3: 2127.6 -> 2121.5 us against
    // rows outermost); two CTAs per SM (configuration 10): rows outermost
    // (the other order measured 72.8 -> 74.5 us at 300 x 300 x 4096).
    auto fma_k = [&](const AVec (&a)[TM], int kr, const float4 (&b)[NJ]) {
        if constexpr (Cfg::MIN_CTAS == 1) {
            float2 a2[TM];
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const float av = vec_get(a[i], kr);
                a2[i] = make_float2(av, av);
            }
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const float2 b0 = make_float2(b[j].x, b[j].y), b1 = make_float2(b[j].z, b[j].w);
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    acc[i][2 * j] = __ffma2_rn(a2[i], b0, acc[i][2 * j]);
                    acc[i][2 * j + 1] = __ffma2_rn(a2[i], b1, acc[i][2 * j + 1]);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const float av = vec_get(a[i], kr);
                const float2 a2 = make_float2(av, av);
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    acc[i][2 * j] = __ffma2_rn(a2, make_float2(b[j].x, b[j].y), acc[i][2 * j]);
                    acc[i][2 * j + 1] = __ffma2_rn(a2, make_float2(b[j].z, b[j].w), acc[i][2 * j + 1]);
                }
            }
        }
    };

    WorkIter it;
    it.begin(p);
    Segment seg;
    int g = 0;             // slice number being consumed
    int stage = 0;
    uint32_t phase = 0;
    while (it.get(p, seg)) {
        int bt, tm, tn;
        tile_coords(seg.t, p.tiles_m, p.tiles_n, p.group_m, bt, tm, tn);

        if constexpr (!BETA_ZERO) {
            // This segment finishes its tile (its first slice) and reads C:
            // pull the tile's C rows into L2 while the products run.  Thread
            // r of the consumers takes row r (all rows once, BM <= threads
            // x 2), one prefetch per 128-byte line.
            if (seg.kb0 == 0) {
                for (int r = threadIdx.x; r < BM; r += CONSUMER_THREADS) {
                    const int row = tm * BM + r;
                    const int c0 = tn * BN;
                    if (row < p.M && c0 < p.N) {
                        const float *crow = p.C + (int64_t)bt * p.stride_c + (int64_t)row * p.ldc;
                        const int c1 = min(p.N, c0 + BN) - 1;
                        for (int c = c0; c < c1; c += 32)
                            asm volatile("prefetch.global.L2 [%0];" :: "l"(crow + c));
                        asm volatile("prefetch.global.L2 [%0];" :: "l"(crow + c1));
                    }
                }
            }
        }

#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);

        for (int kb = seg.kb0; kb < seg.kb1; ++kb, ++g) {
            if (!mbar_wait_bounded(&full[stage], phase, downstream_limit(p.timeout_ns))) {
                record_error(p.err, kSiteConsumerFull);
                if (producer) drain_slices<Cfg>(g, cursor_issued(cursor), full, p.timeout_ns);
                if constexpr (TMA_EPILOGUE) { if (lane == 0) bulk_wait_all(); }
                cta_done();
                return;
            }
            const unsigned char *As = sA + stage * Cfg::A_STAGE_BYTES + a_row0_off;
            const float *Bs = reinterpret_cast<const float *>(sB + stage * Cfg::B_STAGE_BYTES) + b_off;

            // Register double buffering: while the FMAs of k run, the B
            // values of k+1 (and, one k ahead of need, the next A group)
            // are read into the other buffer.  Loop iterations cover
            // KQ_UNROLL groups so the buffer roles are compile-time.
            AVec a0[TM], a1[TM];
            float4 b0[NJ], b1[NJ];
            load_a(As, 0, a0);
            if constexpr (Cfg::PIPE_B) load_b(Bs, 0, b0);
            constexpr int KSTEPS = Cfg::KQ_UNROLL * KA;
#pragma unroll 1
            for (int kq0 = 0; kq0 < NKQ; kq0 += Cfg::KQ_UNROLL) {
                const bool more = kq0 + Cfg::KQ_UNROLL < NKQ;
#pragma unroll
                for (int u = 0; u < Cfg::KQ_UNROLL; ++u) {
                    AVec (&ac)[TM] = (u & 1) ? a1 : a0;
                    AVec (&an)[TM] = (u & 1) ? a0 : a1;
#pragma unroll
                    for (int kr = 0; kr < KA; ++kr) {
                        const int ks = u * KA + kr;                 // k step inside the iteration
                        float4 (&bc)[NJ] = (Cfg::PIPE_B && (ks & 1)) ? b1 : b0;
                        float4 (&bn)[NJ] = (ks & 1) ? b0 : b1;
                        const bool last = ks == KSTEPS - 1;
                        if constexpr (Cfg::PIPE_B) {
                            if (!last || more) load_b(Bs, kq0 * KA + ks + 1, bn);
                        } else {
                            // Keep each k's B reads in place: hoisted
                            // reads of later k would need registers.
                            asm volatile("" ::: "memory");
                            load_b(Bs, kq0 * KA + ks, bc);
                        }
                        if (kr == KA - 2 && (u + 1 < Cfg::KQ_UNROLL || more))
                            load_a(As, kq0 + u + 1, an);
                        fma_k(ac, kr, bc);
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && p.withhold != kWithholdRelease) mbar_arrive(&empty[stage]);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            if (producer && g >= Cfg::REFILL_LAG && cursor_valid(cursor) && p.withhold != kWithholdRefill) {
                if (!issue_slice<Cfg>(cursor, p, &tmA, &tmB, sA, sB, full, empty)) {
                    record_error(p.err, kSiteProducerEmpty);
                    drain_slices<Cfg>(g + 1, cursor_issued(cursor), full, p.timeout_ns);
                    if constexpr (TMA_EPILOGUE) bulk_wait_all();
                    cta_done();
                    return;
                }
            }
        }

        // ---------------- stream-K fixup ----------------
        // Warp by warp: the same (warp, lane) holds the same elements of the
        // tile in every CTA, so each warp hands over and collects its own
        // part with no CTA-wide rendezvous; the flag of (CTA, warp) holds
        // this launch's tag once that warp's part is stored.
        if (seg.kb0 != 0 || seg.kb1 != p.k_blocks) {
            float4 *mine = reinterpret_cast<float4 *>(p.partials + (size_t)blockIdx.x * (BM * BN));
            if (seg.kb0 != 0) {
                // Not the first slice of the tile: hand the partial sums to
                // the CTA that finishes it, then go on with the next segment.
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < NJ; ++j)
                        __stcg(&mine[(i * NJ + j) * CONSUMER_THREADS + threadIdx.x],
                               make_float4(acc[i][2 * j].x, acc[i][2 * j].y,
                                           acc[i][2 * j + 1].x, acc[i][2 * j + 1].y));
                __threadfence();
                __syncwarp();
                if (lane == 0 && p.withhold != kWithholdStreamKFlag)
                    st_release_gpu(&p.flags[blockIdx.x * Cfg::CONSUMER_WARPS + warp], *sk_tag_s);
                it.advance(p, seg);
                continue;
            }
            // First slice of a tile cut between CTAs: add the partial sums of
            // the CTAs holding its other slices, in CTA order (deterministic).
            const int tile_u0 = seg.t * p.k_blocks;
            const int c_first = cta_of_unit(tile_u0 + seg.kb1, p);
            const int c_last = cta_of_unit(tile_u0 + p.k_blocks - 1, p);
            if (lane == 0) {
                for (int c = c_first; c <= c_last; ++c)
                    if (!tag_wait_bounded(&p.flags[c * Cfg::CONSUMER_WARPS + warp], *sk_tag_s, p.timeout_ns))
                        record_error(p.err, kSiteStreamKFlag);
            }
            __syncwarp();
            for (int c = c_first; c <= c_last; ++c) {
                const float4 *other = reinterpret_cast<const float4 *>(p.partials + (size_t)c * (BM * BN));
#pragma unroll
                for (int i = 0; i < TM; ++i) {
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        const float4 v = __ldcg(&other[(i * NJ + j) * CONSUMER_THREADS + threadIdx.x]);
                        acc[i][2 * j].x += v.x;
                        acc[i][2 * j].y += v.y;
                        acc[i][2 * j + 1].x += v.z;
                        acc[i][2 * j + 1].y += v.w;
                    }
                    // Keep the compiler from hoisting all 32 loads at once:
                    // registers are already full with the accumulators.
                    asm volatile("" ::: "memory");
                }
            }
        }

        // ---------------- epilogue ----------------
        const float alpha = p.alpha;
        const float beta = p.beta;
        // The warp's WTM x WTN block (alpha * acc) into its staging area as
        // NJ boxes of WTM rows x 16 columns (row pitch 64 bytes).  Lane
        // (lr, lc) writes row lr + 8i, chunk lc of box j: a quarter warp
        // covers two rows and four chunks, eight distinct bank groups.
        // alpha * acc is formed with packed multiplies (one instruction per
        // two products; with short K the scaling is a noticeable share of the
        // FMA pipe's work on a tile).
        unsigned char *stg = sC + warp * (Cfg::WTM * Cfg::WTN * 4);
        auto stage_block = [&]() {
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int cw = lc * 4 + 4 * WC * j;   // column inside the warp tile
                    const float2 v0 = __fmul2_rn(a2, acc[i][2 * j]);
                    const float2 v1 = __fmul2_rn(a2, acc[i][2 * j + 1]);
                    *reinterpret_cast<float4 *>(stg + (cw / Cfg::C_BOX_COLS) * Cfg::C_BOX_BYTES +
                                                (lr + WR * i) * (Cfg::C_BOX_COLS * 4) + (cw % Cfg::C_BOX_COLS) * 4) =
                        make_float4(v0.x, v0.y, v1.x, v1.y);
                }
        };
        if constexpr (TMA_EPILOGUE) {
            // Lane 0 then issues one TMA store per box.  Before overwriting,
            // lane 0 waits until its previous tile's boxes have been read.
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            stage_block();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // Boxes that start past the last row or column hold nothing
                // of C and are not issued; the others are clipped by TMA.
                const int y = tm * BM + wm * Cfg::WTM;
                const int x = tn * BN + wn * Cfg::WTN;
                if (y < p.M) {
#pragma unroll
                    for (int j = 0; j < Cfg::WTN / Cfg::C_BOX_COLS; ++j)
                        if (x + j * Cfg::C_BOX_COLS < p.N)
                            tma_store_3d(&tmC, stg + j * Cfg::C_BOX_BYTES, x + j * Cfg::C_BOX_COLS, y, bt);
                }
                bulk_commit();
            }
        } else if constexpr (STAGED_EPILOGUE) {
            // C not 16-byte aligned: after staging, each instruction covers
            // two rows x 16 columns (lanes 0-15 a run of one row, 16-31 the
            // next; conflict-free reads of one box), so a warp touches
            // 64-byte runs of C instead of 16-byte pieces of eight rows.
            // With beta != 0 the C values of a whole box (32 loads per
            // thread; the accumulators are in the staging area by now, so the
            // registers are free) are loaded before any is used: reading C
            // eight loads at a time cost a memory round trip per eight.
            __syncwarp();
            stage_block();
            __syncwarp();
            const float *stf = reinterpret_cast<const float *>(stg);
            const int half = lane >> 4, c16 = lane & 15;
            const int row_w = tm * BM + wm * Cfg::WTM;
            const int col_w = tn * BN + wn * Cfg::WTN;
            float *cb = p.C + (int64_t)bt * p.stride_c;
            constexpr int PAIRS = Cfg::WTM / 2;                    // row pairs of a box
            constexpr int NBOX = Cfg::WTN / Cfg::C_BOX_COLS;
            constexpr int BOXES = 1;                               // boxes per round
#pragma unroll 1
            for (int j0 = 0; j0 < NBOX; j0 += BOXES) {
                float cin[BOXES][PAIRS];
                if constexpr (!BETA_ZERO) {
#pragma unroll
                    for (int jj = 0; jj < BOXES; ++jj) {
                        const int col = col_w + Cfg::C_BOX_COLS * (j0 + jj) + c16;
#pragma unroll
                        for (int u = 0; u < PAIRS; ++u) {
                            const int row = row_w + 2 * u + half;
                            cin[jj][u] = (col < p.N && row < p.M) ? cb[(int64_t)row * p.ldc + col] : 0.f;
                        }
                    }
                }
#pragma unroll
                for (int jj = 0; jj < BOXES; ++jj) {
                    const int col = col_w + Cfg::C_BOX_COLS * (j0 + jj) + c16;
#pragma unroll
                    for (int u = 0; u < PAIRS; ++u) {
                        const int r = 2 * u + half;
                        const int row = row_w + r;
                        float v = stf[(j0 + jj) * (Cfg::C_BOX_BYTES / 4) + r * Cfg::C_BOX_COLS + c16];
                        if constexpr (!BETA_ZERO) v = fmaf(beta, cin[jj][u], v);
                        if (col < p.N && row < p.M) cb[(int64_t)row * p.ldc + col] = v;
                    }
                }
            }
            __syncwarp();   // the staging area is read before the next tile refills it
        } else {
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int row = tm * BM + row0 + WR * i;
                if (row >= p.M) continue;
                float *crow = p.C + (int64_t)bt * p.stride_c + (int64_t)row * p.ldc;
                if constexpr (BETA_ZERO) {
                    // C is only written: alpha * acc, 16 bytes at a time when allowed.
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        const int col = tn * BN + col0 + 4 * WC * j;
                        float v[4] = {acc[i][2 * j].x, acc[i][2 * j].y, acc[i][2 * j + 1].x, acc[i][2 * j + 1].y};
                        if (C_VEC && col + 3 < p.N) {
                            *reinterpret_cast<float4 *>(crow + col) =
                                make_float4(alpha * v[0], alpha * v[1], alpha * v[2], alpha * v[3]);
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (col + q < p.N) crow[col + q] = alpha * v[q];
                        }
                    }
                } else {
                    // Reading C: all of this row's loads are issued before its
                    // stores, so that their latencies overlap (a store followed
                    // by the next load of the same thread would serialise them).
                    float cin[NJ][4];
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        const int col = tn * BN + col0 + 4 * WC * j;
                        if (C_VEC && col + 3 < p.N) {
                            const float4 c = *reinterpret_cast<const float4 *>(crow + col);
                            cin[j][0] = c.x; cin[j][1] = c.y; cin[j][2] = c.z; cin[j][3] = c.w;
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q) cin[j][q] = col + q < p.N ? crow[col + q] : 0.f;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        const int col = tn * BN + col0 + 4 * WC * j;
                        float v[4] = {acc[i][2 * j].x, acc[i][2 * j].y, acc[i][2 * j + 1].x, acc[i][2 * j + 1].y};
#pragma unroll
                        for (int q = 0; q < 4; ++q) v[q] = fmaf(beta, cin[j][q], alpha * v[q]);
                        if (C_VEC && col + 3 < p.N) {
                            *reinterpret_cast<float4 *>(crow + col) = make_float4(v[0], v[1], v[2], v[3]);
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (col + q < p.N) crow[col + q] = v[q];
                        }
                    }
                }
            }
        }
        it.advance(p, seg);
    }
    cta_done();
    if constexpr (TMA_EPILOGUE) {
        if (lane == 0) bulk_wait_all();
    }
}

}  // namespace sg
