// Small products (every matrix of the call at most a few hundred rows and
// columns, little work in total): the persistent, TMA-fed main kernel
// spends most of its time there on start-up latency (tensor-map fetch, the
// first loads, a stream-K fixup chain), and a 128 x 128 tile leaves most
// SMs idle.  This kernel gives every 32 x 32 block of C its own CTA of two
// warps instead, with plain loads and no cross-CTA exchange:
//   * K is walked in 32-deep pieces; the next piece of A and B is loaded
//     into registers (16 + 16 values a thread, coalesced along whichever
//     index is contiguous in memory) while the current one is multiplied
//     out of shared memory, so global latency overlaps the FMAs;
//   * thread (ty, tx) of the 8 x 8 thread grid owns rows ty + 8i and columns
//     tx + 8j (i, j < 4) of the block: the shared-memory reads of a warp are
//     four broadcast rows of A and eight consecutive columns of B, free of
//     bank conflicts with the 33-float row pitch;
//   * transposed operands are read in place (their index order only changes
//     which loads coalesce), and batches are extra CTAs.
// Arithmetic: one FP32 fmaf per product, K ascending, then alpha * acc
// (+ beta * C, and C is not read when beta == 0).  The blocking is the
// pages' shared-memory tiling with a 2-D register tile per thread
// (easonhuang.dev/blog/gpu_matmul, "SMEM Caching" and "2D Blocktiling"),
// sized for latency rather than throughput.
#include "kernel_table.h"

namespace sg {

namespace {

constexpr int kTile = kSmallTile;     // C block per CTA (kTile x kTile)
constexpr int kPiece = kSmallPiece;   // K piece per shared-memory fill
constexpr int kPitch = kTile + 1;
constexpr int kThreads = 64;
constexpr int kPerThread = kTile * kPiece / kThreads;   // 16 loads of A and of B

template <bool TRANS_A, bool TRANS_B, bool BETA_ZERO>
__global__ void __launch_bounds__(kThreads)
sgemm_small_kernel(const SmallArgs p) {
    __shared__ float sA[kTile][kPitch];    // [m][k]
    __shared__ float sB[kPiece][kPitch];   // [k][n]
    const int per_batch = p.tiles_m * p.tiles_n;
    const int bt = blockIdx.x / per_batch;
    const int t = blockIdx.x - bt * per_batch;
    const int m0 = (t / p.tiles_n) * kTile;
    const int n0 = (t % p.tiles_n) * kTile;
    const float *A = p.A + (int64_t)bt * p.sa;
    const float *B = p.B + (int64_t)bt * p.sb;
    const int tid = threadIdx.x;
    const int tx = tid & 7, ty = tid >> 3;

    // Element e = tid + 64 r of a 32 x 32 piece: (row, col) = (e / 32, e % 32)
    // of the piece as stored in memory, so that consecutive threads read
    // consecutive addresses.  For A stored [M][K] that is (m, k); for A
    // stored transposed ([K][M]) it is (k, m); likewise for B.
    float ra[kPerThread], rb[kPerThread];
    auto load = [&](int k0) {
#pragma unroll
        for (int r = 0; r < kPerThread; ++r) {
            const int e = tid + kThreads * r;
            const int hi = e >> 5, lo = e & 31;
            {
                const int m = TRANS_A ? lo : hi, k = TRANS_A ? hi : lo;
                const int gm = m0 + m, gk = k0 + k;
                ra[r] = (gm < p.M && gk < p.K)
                            ? (TRANS_A ? A[(int64_t)gk * p.lda + gm] : A[(int64_t)gm * p.lda + gk])
                            : 0.f;
            }
            {
                const int k = TRANS_B ? lo : hi, n = TRANS_B ? hi : lo;
                const int gk = k0 + k, gn = n0 + n;
                rb[r] = (gk < p.K && gn < p.N)
                            ? (TRANS_B ? B[(int64_t)gn * p.ldb + gk] : B[(int64_t)gk * p.ldb + gn])
                            : 0.f;
            }
        }
    };
    auto stash = [&]() {
#pragma unroll
        for (int r = 0; r < kPerThread; ++r) {
            const int e = tid + kThreads * r;
            const int hi = e >> 5, lo = e & 31;
            if (TRANS_A) sA[lo][hi] = ra[r]; else sA[hi][lo] = ra[r];
            if (TRANS_B) sB[lo][hi] = rb[r]; else sB[hi][lo] = rb[r];
        }
    };

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    load(0);
    for (int k0 = 0; k0 < p.K; k0 += kPiece) {
        __syncthreads();   // the previous piece has been used
        stash();
        __syncthreads();
        if (k0 + kPiece < p.K) load(k0 + kPiece);
        const int kn = min(kPiece, p.K - k0);
#pragma unroll 8
        for (int k = 0; k < kn; ++k) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = sA[ty + 8 * i][k];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = sB[k][tx + 8 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }

    float *C = p.C + (int64_t)bt * p.sc;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = m0 + ty + 8 * i;
        if (row >= p.M) continue;
        float *crow = C + (int64_t)row * p.ldc;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = n0 + tx + 8 * j;
            if (col >= p.N) continue;
            if (BETA_ZERO) crow[col] = p.alpha * acc[i][j];
            else crow[col] = fmaf(p.beta, crow[col], p.alpha * acc[i][j]);
        }
    }
}

template <bool TA, bool TB>
void launch_small_t(const SmallArgs &p, int blocks, cudaStream_t s) {
    if (p.beta == 0.0f) sgemm_small_kernel<TA, TB, true><<<blocks, kThreads, 0, s>>>(p);
    else sgemm_small_kernel<TA, TB, false><<<blocks, kThreads, 0, s>>>(p);
}

}  // namespace

int small_blocks(int M, int N, int batch) {
    const int64_t b = (int64_t)batch * ((M + kTile - 1) / kTile) * ((N + kTile - 1) / kTile);
    return b > 0x7fffffff ? 0 : (int)b;
}

void launch_small(SmallArgs p, int trans_a, int trans_b, int batch, cudaStream_t s) {
    p.tiles_m = (p.M + kTile - 1) / kTile;
    p.tiles_n = (p.N + kTile - 1) / kTile;
    const int blocks = small_blocks(p.M, p.N, batch);
    if (blocks == 0) return;
    if (trans_a) {
        if (trans_b) launch_small_t<true, true>(p, blocks, s);
        else launch_small_t<true, false>(p, blocks, s);
    } else {
        if (trans_b) launch_small_t<false, true>(p, blocks, s);
        else launch_small_t<false, false>(p, blocks, s);
    }
}

}  // namespace sg
