// Small products (every matrix of the call at most a few hundred rows and
// columns, little work in total): the persistent, TMA-fed main kernel
// spends most of its time there on start-up latency (tensor-map fetch, the
// first loads, a stream-K fixup chain), and a 128 x 128 tile leaves most
// SMs idle.  This kernel gives every 32 x 32 block of C a CTA of two warps
// instead, with plain loads:
//   * K is walked in 32-deep pieces; the next piece of A and B (with few
//     CTAs per SM, the next two) is loaded into registers (16 + 16 values a
//     thread per piece) while the current one is multiplied out of shared
//     memory, so global latency overlaps the FMAs;
//   * both pieces are kept k-major in shared memory ([k][m] and [k][n], row
//     pitch 40 floats): thread (ty, tx) of the 8 x 8 thread grid owns rows
//     4ty..4ty+3 and columns 4tx..4tx+3 of the block and reads one 16-byte
//     vector of each per k (a warp: four broadcast A vectors and 128
//     contiguous bytes of B), then issues 8 packed two-wide FMAs;
//   * a warp loads 8 contiguous elements x 4 rows (whole 32-byte sectors)
//     of a piece that shared memory keeps in its memory order, and 4 x 8 of
//     one it keeps transposed: with the pitch of 40 (8 banks per row) both
//     stores are conflict-free.  Transposed operands are read in place,
//     and batches are extra CTAs;
//   * when there are few blocks and K is long, a thread-block cluster of S
//     CTAs (S <= 8) shares one block: CTA r of the cluster takes the r-th
//     of S contiguous K ranges, leaves its 32 x 32 partial sums in its own
//     shared memory, and after a cluster barrier each CTA adds the S
//     partials of its 32/S rows through distributed shared memory in rank
//     order (deterministic) and writes them to C.
// Arithmetic: FP32 FMAs, K ascending within each range, ranges added in
// order; then alpha * acc (+ beta * C, and C is not read when beta == 0).
// The blocking is the pages' shared-memory tiling with a 2-D register tile
// per thread (easonhuang.dev/blog/gpu_matmul, "SMEM Caching" and "2D
// Blocktiling"), sized for latency rather than throughput.
#include "kernel_table.h"

namespace sg {

namespace {

constexpr int kTile = kSmallTile;     // C block per CTA (kTile x kTile)
constexpr int kPiece = kSmallPiece;   // K piece per shared-memory fill
constexpr int kPitch = 40;            // floats per k row: 8 banks apart, 16-byte rows
constexpr int kThreads = 64;
constexpr int kPerThread = kTile * kPiece / kThreads;   // 16 loads of A and of B

__device__ __forceinline__ float ld_cluster(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

template <bool TRANS_A, bool TRANS_B, bool BETA_ZERO, bool DEEP>
__global__ void __launch_bounds__(kThreads)
sgemm_small_kernel(const SmallArgs p) {
    __shared__ __align__(16) float sA[kPiece][kPitch];   // [k][m]; later the partial tile
    __shared__ __align__(16) float sB[kPiece][kPitch];   // [k][n]
    const int S = p.splits;
    const int blk = blockIdx.x / S;                 // block of C (batch major)
    const int rank = S > 1 ? (int)cluster_rank() : 0;
    const int per_batch = p.tiles_m * p.tiles_n;
    const int bt = blk / per_batch;
    const int t = blk - bt * per_batch;
    const int m0 = (t / p.tiles_n) * kTile;
    const int n0 = (t % p.tiles_n) * kTile;
    const float *A = p.A + (int64_t)bt * p.sa;
    const float *B = p.B + (int64_t)bt * p.sb;
    const int tid = threadIdx.x;
    const int tx = tid & 7, ty = tid >> 3;
    // This CTA's K range: pieces [rank P / S, (rank + 1) P / S).
    const int pieces = (p.K + kPiece - 1) / kPiece;
    const int kbeg = (int)((int64_t)rank * pieces / S) * kPiece;
    const int kend = min(p.K, (int)((int64_t)(rank + 1) * pieces / S) * kPiece);

    // Element r of this thread in a 32 x 32 piece, as stored in memory
    // (row = the non-contiguous index, col = the contiguous one).  A warp
    // covers 4 rows x 8 columns where the piece is stored in shared memory
    // as it lies in memory (banks 8 row + col: all 32 distinct), and 8 rows
    // x 4 columns where it is stored transposed (banks 8 col + row).
    auto coords = [&](bool transposing, int r, int &row, int &col) {
        const int idx = tid + kThreads * r;
        const int lane = idx & 31, w = idx >> 5;
        if (transposing) {
            col = (lane & 3) + 4 * (w & 7);
            row = (lane >> 2) + 8 * (w >> 3);
        } else {
            col = (lane & 7) + 8 * (w & 3);
            row = (lane >> 3) + 4 * (w >> 2);
        }
    };
    // Register sets of pieces in flight while one is multiplied: two with
    // DEEP (the next piece and the one after), else one.
    constexpr int kAhead = DEEP ? 2 : 1;
    float ra0[kPerThread], rb0[kPerThread], ra1[kPerThread], rb1[kPerThread];
    auto load = [&](float (&ra)[kPerThread], float (&rb)[kPerThread], int k0) {
#pragma unroll
        for (int r = 0; r < kPerThread; ++r) {
            int row, col;
            coords(!TRANS_A, r, row, col);
            {
                const int m = TRANS_A ? col : row, k = TRANS_A ? row : col;
                const int gm = m0 + m, gk = k0 + k;
                ra[r] = (gm < p.M && gk < kend)
                            ? (TRANS_A ? A[(int64_t)gk * p.lda + gm] : A[(int64_t)gm * p.lda + gk])
                            : 0.f;
            }
            coords(TRANS_B, r, row, col);
            {
                const int k = TRANS_B ? col : row, n = TRANS_B ? row : col;
                const int gk = k0 + k, gn = n0 + n;
                rb[r] = (gk < kend && gn < p.N)
                            ? (TRANS_B ? B[(int64_t)gn * p.ldb + gk] : B[(int64_t)gk * p.ldb + gn])
                            : 0.f;
            }
        }
    };
    auto stash = [&](const float (&ra)[kPerThread], const float (&rb)[kPerThread]) {
#pragma unroll
        for (int r = 0; r < kPerThread; ++r) {
            int row, col;
            coords(!TRANS_A, r, row, col);
            if (TRANS_A) sA[row][col] = ra[r]; else sA[col][row] = ra[r];
            coords(TRANS_B, r, row, col);
            if (TRANS_B) sB[col][row] = rb[r]; else sB[row][col] = rb[r];
        }
    };

    float2 acc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);

    // One piece: into shared memory from its register set, which then takes
    // the piece kAhead further on; then the FMAs.
    auto step = [&](float (&ra)[kPerThread], float (&rb)[kPerThread], int k0) {
        __syncthreads();   // the previous piece has been used
        stash(ra, rb);
        __syncthreads();
        if (k0 + kAhead * kPiece < kend) load(ra, rb, k0 + kAhead * kPiece);
        const int kn = min(kPiece, kend - k0);
#pragma unroll 8
        for (int k = 0; k < kn; ++k) {
            const float4 a = *reinterpret_cast<const float4 *>(&sA[k][4 * ty]);
            const float4 b = *reinterpret_cast<const float4 *>(&sB[k][4 * tx]);
            const float2 b01 = make_float2(b.x, b.y), b23 = make_float2(b.z, b.w);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 a2 = make_float2(av[i], av[i]);
                acc[i][0] = __ffma2_rn(a2, b01, acc[i][0]);
                acc[i][1] = __ffma2_rn(a2, b23, acc[i][1]);
            }
        }
    };
    if (kbeg < kend) load(ra0, rb0, kbeg);
    if constexpr (DEEP) {
        if (kbeg + kPiece < kend) load(ra1, rb1, kbeg + kPiece);
        for (int k0 = kbeg; k0 < kend; k0 += 2 * kPiece) {
            step(ra0, rb0, k0);
            if (k0 + kPiece < kend) step(ra1, rb1, k0 + kPiece);
        }
    } else {
        for (int k0 = kbeg; k0 < kend; k0 += kPiece) step(ra0, rb0, k0);
    }

    float *C = p.C + (int64_t)bt * p.sc;
    auto finish = [&](int row, int col, float v) {
        float *c = C + (int64_t)row * p.ldc + col;
        if (BETA_ZERO) *c = p.alpha * v;
        else *c = fmaf(p.beta, *c, p.alpha * v);
    };
    if (S == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = m0 + 4 * ty + i;
            if (row >= p.M) continue;
            const float v[4] = {acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (n0 + 4 * tx + j < p.N) finish(row, n0 + 4 * tx + j, v[j]);
        }
        return;
    }

    // Cluster: partial tile into this CTA's shared memory (sA, now free),
    // then CTA r sums rows [32 r / S, 32 (r + 1) / S) over ranks 0..S-1.
    float *part = &sA[0][0];   // 32 x 32, row pitch 32
    __syncthreads();           // every warp is done reading sA
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4 *>(part + (4 * ty + i) * kTile + 4 * tx) =
            make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
    cluster_sync();            // partials of every rank visible cluster-wide
    const int rows = kTile / S;
    for (int e = tid; e < rows * kTile; e += kThreads) {
        const int lr = rank * rows + e / kTile, lc = e % kTile;
        float v = 0.f;
        for (int q = 0; q < S; ++q) v += ld_cluster(cluster_addr(part + lr * kTile + lc, (uint32_t)q));
        const int row = m0 + lr, col = n0 + lc;
        if (row < p.M && col < p.N) finish(row, col, v);
    }
    cluster_sync();            // no CTA leaves while another still reads its partials
}

template <bool TA, bool TB, bool BZ, bool DEEP>
cudaError_t launch_small_t(const SmallArgs &p, int blocks, cudaStream_t s) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)blocks * (unsigned)p.splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    // Not chained to the kernel before it (programmatic stream
    // serialisation): measured 0.2-0.4 us faster per call at 128^3 / 256^3
    // but 24.7 -> 32.9 us at 512^3.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.splits > 1 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, sgemm_small_kernel<TA, TB, BZ, DEEP>, p);
}

// Few CTAs per SM (latency bound): two pieces in flight (216 registers a
// thread); more: one (up to 128 registers), so that more CTAs fit an SM.
template <bool TA, bool TB>
cudaError_t launch_small_b(const SmallArgs &p, int blocks, cudaStream_t s) {
    const bool deep = (int64_t)blocks * p.splits <= 2 * (int64_t)p.sms;
    if (p.beta == 0.0f)
        return deep ? launch_small_t<TA, TB, true, true>(p, blocks, s) : launch_small_t<TA, TB, true, false>(p, blocks, s);
    return deep ? launch_small_t<TA, TB, false, true>(p, blocks, s) : launch_small_t<TA, TB, false, false>(p, blocks, s);
}

}  // namespace

int small_blocks(int M, int N, int batch) {
    const int64_t b = (int64_t)batch * ((M + kTile - 1) / kTile) * ((N + kTile - 1) / kTile);
    return b > 0x7fffffff / kSmallMaxSplits ? 0 : (int)b;
}

int small_splits(int M, int N, int K, int batch, int sms) {
    const int64_t blocks = small_blocks(M, N, batch);
    const int pieces = (K + kPiece - 1) / kPiece;
    int s = 1;
    while (2 * s <= kSmallMaxSplits && 2 * s <= pieces && blocks * 2 * s <= 4 * (int64_t)sms) s *= 2;
    return s;
}

namespace {
template <bool TA, bool TB>
cudaError_t preload_small_ab() {
    const void *fns[] = {reinterpret_cast<const void *>(&sgemm_small_kernel<TA, TB, true, true>),
                         reinterpret_cast<const void *>(&sgemm_small_kernel<TA, TB, true, false>),
                         reinterpret_cast<const void *>(&sgemm_small_kernel<TA, TB, false, true>),
                         reinterpret_cast<const void *>(&sgemm_small_kernel<TA, TB, false, false>)};
    for (const void *fn : fns)
        if (cudaError_t e = load_kernel(fn); e != cudaSuccess) return e;
    return cudaSuccess;
}
}  // namespace

cudaError_t preload_small_kernels() {
    cudaError_t e = preload_small_ab<false, false>();
    if (e == cudaSuccess) e = preload_small_ab<false, true>();
    if (e == cudaSuccess) e = preload_small_ab<true, false>();
    if (e == cudaSuccess) e = preload_small_ab<true, true>();
    return e;
}

void launch_small(SmallArgs p, int trans_a, int trans_b, int batch, cudaStream_t s) {
    p.tiles_m = (p.M + kTile - 1) / kTile;
    p.tiles_n = (p.N + kTile - 1) / kTile;
    const int blocks = small_blocks(p.M, p.N, batch);
    if (blocks == 0 || p.splits < 1 || p.splits > kSmallMaxSplits) return;
    if (trans_a) {
        if (trans_b) launch_small_b<true, true>(p, blocks, s);
        else launch_small_b<true, false>(p, blocks, s);
    } else {
        if (trans_b) launch_small_b<false, true>(p, blocks, s);
        else launch_small_b<false, false>(p, blocks, s);
    }
}

}  // namespace sg
