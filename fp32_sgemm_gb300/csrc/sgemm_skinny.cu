// Skinny products, bound by HBM rather than by the FMA pipes: few rows of
// C (M <= 32) or few columns (N <= 32).  The arithmetic intensity is about
// M/2 (or N/2) FLOP per byte of the large operand, so at M = 1 no kernel can
// beat streaming B once at HBM speed; the 128 x 128 tiles of the main kernel
// would waste up to 127/128 of their FMAs here.
//
//   small M: each thread owns 4 consecutive columns of C and walks them down
//     its K range with 16-byte loads of B (coalesced across the warp, eight
//     in flight per thread); the A values of the current K piece sit in
//     shared memory and are read as warp-wide broadcasts, each feeding 4
//     FMAs (packed two-wide).
//   small N: each thread owns 2 rows of C and walks them along K with four
//     16-byte loads per row (whole 32-byte sectors, eight loads in flight);
//     the K x N operand B sits in shared memory, and each broadcast B value
//     feeds 2 FMAs.
//   Both split K across CTAs until the chip is full: every split writes its
//   M x N partial sums to the workspace and a third kernel adds the splits in
//   order (deterministic) and applies alpha and beta.
//
// All arithmetic is FP32 (fmaf).  The pages have no skinny kernel; the
// coalescing argument of easonhuang.dev ("GMEM Coalesced") and the register
// reuse of "2D Register Tiling" are what these are built from.
#include <algorithm>

#include "kernel_table.h"

namespace sg {

constexpr int kSkinnyThreads = 256;
constexpr int kSkinnyKT = 128;      // K piece staged in shared memory

// ------------------------------------------------------------ small M

template <int MT>
__global__ void __launch_bounds__(kSkinnyThreads)
skinny_m_partial_kernel(int M, int N, int K, const float *__restrict__ A, int64_t lda,
                        const float *__restrict__ B, int64_t ldb, float *__restrict__ part,
                        int k_chunk, bool vec_b) {
    __shared__ float sA[MT][kSkinnyKT];
    const int split = blockIdx.y;
    const int kbeg = split * k_chunk;
    const int kend = min(K, kbeg + k_chunk);
    const int n = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    const bool active = n < N;
    const bool full4 = vec_b && n + 3 < N;
    float acc[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[m][e] = 0.f;
    for (int k0 = kbeg; k0 < kend; k0 += kSkinnyKT) {
        const int kn = min(kend - k0, kSkinnyKT);
        __syncthreads();
        for (int i = threadIdx.x; i < MT * kSkinnyKT; i += blockDim.x) {
            const int m = i / kSkinnyKT, k = i - m * kSkinnyKT;
            sA[m][k] = (m < M && k < kn) ? A[(int64_t)m * lda + k0 + k] : 0.f;
        }
        __syncthreads();
        if (!active) continue;
        const float *bcol = B + (int64_t)k0 * ldb + n;
        // Eight independent 16-byte loads in flight per thread, then the
        // FMAs (packed two-wide, a broadcast from shared memory).
        int k = 0;
        if (full4) {
            for (; k + 8 <= kn; k += 8) {
                float4 b[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    b[q] = __ldcs(reinterpret_cast<const float4 *>(bcol + (int64_t)(k + q) * ldb));
#pragma unroll
                for (int q = 0; q < 8; ++q)
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const float a = sA[m][k + q];
                        const float2 a2 = make_float2(a, a);
                        float2 lo = make_float2(acc[m][0], acc[m][1]);
                        float2 hi = make_float2(acc[m][2], acc[m][3]);
                        lo = __ffma2_rn(a2, make_float2(b[q].x, b[q].y), lo);
                        hi = __ffma2_rn(a2, make_float2(b[q].z, b[q].w), hi);
                        acc[m][0] = lo.x; acc[m][1] = lo.y; acc[m][2] = hi.x; acc[m][3] = hi.y;
                    }
            }
        }
        for (; k < kn; ++k) {
            float4 b;
            const float *bp = bcol + (int64_t)k * ldb;
            if (full4) {
                b = __ldcs(reinterpret_cast<const float4 *>(bp));
            } else {
                b.x = bp[0];
                b.y = n + 1 < N ? bp[1] : 0.f;
                b.z = n + 2 < N ? bp[2] : 0.f;
                b.w = n + 3 < N ? bp[3] : 0.f;
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float a = sA[m][k];
                acc[m][0] = fmaf(a, b.x, acc[m][0]);
                acc[m][1] = fmaf(a, b.y, acc[m][1]);
                acc[m][2] = fmaf(a, b.z, acc[m][2]);
                acc[m][3] = fmaf(a, b.w, acc[m][3]);
            }
        }
    }
    if (!active) return;
    float *out = part + (int64_t)split * M * N;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m >= M) break;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (n + e < N) out[(int64_t)m * N + n + e] = acc[m][e];
    }
}

// ------------------------------------------------------------ small N

constexpr int kRowsPerThread = 2;

template <int NT>
__global__ void __launch_bounds__(kSkinnyThreads)
skinny_n_partial_kernel(int M, int N, int K, const float *__restrict__ A, int64_t lda,
                        const float *__restrict__ B, int64_t ldb, float *__restrict__ part,
                        int k_chunk, bool vec_a) {
    constexpr int NP = (NT + 3) / 4 * 4;          // B row padded to whole float4s
    constexpr int R = kRowsPerThread;
    __shared__ __align__(16) float sB[kSkinnyKT][NP];
    const int split = blockIdx.y;
    const int kbeg = split * k_chunk;
    const int kend = min(K, kbeg + k_chunk);
    const int r0 = (blockIdx.x * blockDim.x + threadIdx.x) * R;
    float acc[R][NP];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < NP; ++j) acc[i][j] = 0.f;
    for (int k0 = kbeg; k0 < kend; k0 += kSkinnyKT) {
        const int kn = min(kend - k0, kSkinnyKT);
        __syncthreads();
        for (int i = threadIdx.x; i < kSkinnyKT * NP; i += blockDim.x) {
            const int k = i / NP, j = i - k * NP;
            sB[k][j] = (k < kn && j < N) ? B[(int64_t)(k0 + k) * ldb + j] : 0.f;
        }
        __syncthreads();
        if (r0 >= M) continue;
        // 16-byte row reads need the K piece to start 16-byte aligned too.
        const bool vec = vec_a && ((k0 & 3) == 0) && (kn & 15) == 0;
        if (vec) {
            for (int k = 0; k < kn; k += 16) {
                float4 a[R][4];                   // 16 consecutive k of each row
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    if (r0 + i < M) {
                        const float4 *ap = reinterpret_cast<const float4 *>(A + (int64_t)(r0 + i) * lda + k0 + k);
#pragma unroll
                        for (int v = 0; v < 4; ++v) a[i][v] = __ldcs(ap + v);
                    } else {
#pragma unroll
                        for (int v = 0; v < 4; ++v) a[i][v] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int q = 0; q < 16; ++q) {
#pragma unroll
                    for (int g = 0; g < NP / 4; ++g) {
                        const float4 b = *reinterpret_cast<const float4 *>(&sB[k + q][4 * g]);
#pragma unroll
                        for (int i = 0; i < R; ++i) {
                            const float4 &av = a[i][q >> 2];
                            const float x = (q & 3) == 0 ? av.x : (q & 3) == 1 ? av.y : (q & 3) == 2 ? av.z : av.w;
                            acc[i][4 * g] = fmaf(x, b.x, acc[i][4 * g]);
                            acc[i][4 * g + 1] = fmaf(x, b.y, acc[i][4 * g + 1]);
                            acc[i][4 * g + 2] = fmaf(x, b.z, acc[i][4 * g + 2]);
                            acc[i][4 * g + 3] = fmaf(x, b.w, acc[i][4 * g + 3]);
                        }
                    }
                }
            }
        } else {
            for (int k = 0; k < kn; ++k) {
                float a[R];
#pragma unroll
                for (int i = 0; i < R; ++i)
                    a[i] = (r0 + i < M) ? A[(int64_t)(r0 + i) * lda + k0 + k] : 0.f;
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    const float b = sB[k][j];
#pragma unroll
                    for (int i = 0; i < R; ++i) acc[i][j] = fmaf(a[i], b, acc[i][j]);
                }
            }
        }
    }
    if (r0 >= M) return;
    float *out = part + (int64_t)split * M * N;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        if (r0 + i >= M) break;
#pragma unroll
        for (int j = 0; j < NP; ++j)
            if (j < N) out[(int64_t)(r0 + i) * N + j] = acc[i][j];
    }
}

// C = alpha * (sum over splits, in split order) + beta * C; C not read when beta == 0.
__global__ void skinny_reduce_kernel(int M, int N, int splits, const float *__restrict__ part,
                                     float alpha, float beta, float *__restrict__ C, int64_t ldc) {
    const int64_t total = (int64_t)M * N;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int z = 0; z < splits; ++z) s += __ldcs(&part[(int64_t)z * total + i]);
        const int64_t m = i / N, n = i - m * N;
        float *c = C + m * ldc + n;
        *c = beta == 0.0f ? alpha * s : fmaf(beta, *c, alpha * s);
    }
}

// ------------------------------------------------------------ launches

namespace {
inline int64_t cdiv(int64_t x, int64_t a) { return (x + a - 1) / a; }
}  // namespace

// Splits of K: about 8 CTAs per SM in total, each at least 128 deep in K.
int skinny_splits(bool small_m, int M, int N, int K, int sms) {
    const int64_t blocks = small_m ? cdiv(N, 4 * kSkinnyThreads) : cdiv(M, kRowsPerThread * kSkinnyThreads);
    int64_t splits = cdiv(int64_t(sms) * 8, blocks);
    splits = std::min<int64_t>(splits, cdiv(K, kSkinnyKT));
    return int(std::max<int64_t>(1, std::min<int64_t>(splits, 65535)));
}

size_t skinny_workspace(int M, int N, int splits) {
    return size_t(splits) * size_t(M) * size_t(N) * 4;
}

template <int T>
void launch_m(int M, int N, int K, const float *A, int64_t lda, const float *B, int64_t ldb,
              float *part, int splits, int k_chunk, cudaStream_t s) {
    const bool vec_b = (reinterpret_cast<uintptr_t>(B) % 16 == 0) && ldb % 4 == 0;
    dim3 grid(unsigned(cdiv(N, 4 * kSkinnyThreads)), unsigned(splits));
    skinny_m_partial_kernel<T><<<grid, kSkinnyThreads, 0, s>>>(M, N, K, A, lda, B, ldb, part, k_chunk, vec_b);
}

template <int T>
void launch_n(int M, int N, int K, const float *A, int64_t lda, const float *B, int64_t ldb,
              float *part, int splits, int k_chunk, cudaStream_t s) {
    const bool vec_a = (reinterpret_cast<uintptr_t>(A) % 16 == 0) && lda % 4 == 0;
    dim3 grid(unsigned(cdiv(M, kRowsPerThread * kSkinnyThreads)), unsigned(splits));
    skinny_n_partial_kernel<T><<<grid, kSkinnyThreads, 0, s>>>(M, N, K, A, lda, B, ldb, part, k_chunk, vec_a);
}

cudaError_t preload_skinny_kernels() {
    const void *fns[] = {
        reinterpret_cast<const void *>(&skinny_m_partial_kernel<1>), reinterpret_cast<const void *>(&skinny_m_partial_kernel<2>),
        reinterpret_cast<const void *>(&skinny_m_partial_kernel<4>), reinterpret_cast<const void *>(&skinny_m_partial_kernel<8>),
        reinterpret_cast<const void *>(&skinny_m_partial_kernel<16>), reinterpret_cast<const void *>(&skinny_m_partial_kernel<32>),
        reinterpret_cast<const void *>(&skinny_n_partial_kernel<1>), reinterpret_cast<const void *>(&skinny_n_partial_kernel<2>),
        reinterpret_cast<const void *>(&skinny_n_partial_kernel<4>), reinterpret_cast<const void *>(&skinny_n_partial_kernel<8>),
        reinterpret_cast<const void *>(&skinny_n_partial_kernel<16>), reinterpret_cast<const void *>(&skinny_n_partial_kernel<32>),
        reinterpret_cast<const void *>(&skinny_reduce_kernel)};
    for (const void *fn : fns)
        if (cudaError_t e = load_kernel(fn); e != cudaSuccess) return e;
    return cudaSuccess;
}

void launch_skinny(bool small_m, int M, int N, int K, float alpha, const float *A, int64_t lda,
                   const float *B, int64_t ldb, float beta, float *C, int64_t ldc, float *part,
                   int splits, cudaStream_t s) {
    // k_chunk a multiple of 16 so that every split starts 64-byte aligned
    // along K (the small-N kernel reads 16 k per row at a time).
    const int k_chunk = int(cdiv(cdiv(K, splits), 16) * 16);
    const int small = small_m ? M : N;
    if (small_m) {
        if (small <= 1) launch_m<1>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
        else if (small <= 2) launch_m<2>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
        else if (small <= 4) launch_m<4>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
        else if (small <= 8) launch_m<8>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
        else if (small <= 16) launch_m<16>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
        else launch_m<32>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
    } else {
        if (small <= 1) launch_n<1>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
        else if (small <= 2) launch_n<2>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
        else if (small <= 4) launch_n<4>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
        else if (small <= 8) launch_n<8>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
        else if (small <= 16) launch_n<16>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
        else launch_n<32>(M, N, K, A, lda, B, ldb, part, splits, k_chunk, s);
    }
    const int64_t total = int64_t(M) * N;
    const unsigned blocks = unsigned(std::max<int64_t>(1, std::min<int64_t>(cdiv(total, 256), 65535)));
    skinny_reduce_kernel<<<blocks, 256, 0, s>>>(M, N, splits, part, alpha, beta, C, ldc);
}

}  // namespace sg
