// Skinny products fed by TMA: few rows of C (M <= 32) or few columns
// (N <= 32), with the large operand streamed from HBM through a six-stage
// shared-memory ring.  These shapes do M/2 (or N/2) FLOP per byte of the
// large operand, so the bound is HBM bandwidth; what a kernel must do is
// keep enough bytes in flight per SM (bandwidth x latency, ~60 KB at
// 44 GB/s per SM), which plain loads from registers do not reach at M = 8.
// Here one producer thread per CTA keeps five to six 34 KB stages in flight.
//
// Work decomposition.  The output is cut into blocks (small M: 1024 columns
// of all M rows; small N: 512 rows of all N columns) and K into k-blocks
// (8 or 16 deep); a unit is one (block, k-block) pair, and units are
// numbered block-major.  One persistent CTA per SM takes an equal
// contiguous range of units, so the load is even whatever the block count
// (the stream-K idea, applied to a K-split reduction).  A CTA's range spans
// one or a few blocks: for each block it touches it writes one partial tile
// (slot `seg` of its own) to the workspace, and a second kernel adds, for
// every output element, the partial tiles of the CTAs that touched its
// block in CTA order, so the result is deterministic.
//
//   small M: the CTA's 256 consumer threads own 4 consecutive columns each
//     (1024 columns).  A stage holds B[8 x 1024] (four 256-column TMA boxes)
//     and A[MT x 8]; each thread reads its 16-byte column group of the 8 B
//     rows (conflict-free, 512 contiguous bytes per warp) and broadcasts A.
//   small N: each consumer thread owns 2 rows (t and t + 256 of a 512-row
//     block).  A stage holds A[512 x 16] (two 256-row boxes, TMA 64-byte
//     swizzle, so that a warp's 16-byte reads of 32 different rows hit
//     distinct banks) and B[16 x NP]; B is read as broadcasts.
//
// All arithmetic is FP32 (packed two-wide FMAs).  The pages have no skinny
// kernel; this is built from the staging idea of "Kernel 9 & 10: Staging"
// (easonhuang.dev) and "The Final Kernel" double buffering, with TMA and
// mbarriers in place of cp.async.
#include <algorithm>

#include "kernel_table.h"
#include "ptx.cuh"

namespace sg {

namespace {

constexpr int kStages = 6;
constexpr int kConsumers = 256;
constexpr int kThreads = kConsumers + 32;        // + one producer warp
constexpr int kStageBytes = 34816;               // 32 KB of the big operand + 2 KB

// small M
constexpr int kMBK = 8;                          // k per stage
constexpr int kMBoxN = 256;                      // columns per B box
constexpr int kMCols = 4 * kConsumers;           // 1024 columns per block
constexpr int kMBoxes = kMCols / kMBoxN;         // 4
constexpr int kMBBytes = kMBK * kMCols * 4;      // 32768

// small N
constexpr int kNBK = 16;
constexpr int kNBoxM = 256;
constexpr int kNRows = 2 * kNBoxM;               // 512 rows per block
constexpr int kNABoxBytes = kNBoxM * kNBK * 4;   // 16384

constexpr int kSmemBytes = kStages * kStageBytes + 2 * kStages * 8 + 1024;

__host__ __device__ constexpr int pad4(int n) { return (n + 3) / 4 * 4; }

__device__ __forceinline__ int64_t unit_begin(int c, const SkinnyTmaArgs &p) {
    return (int64_t)c * p.units / p.ctas;
}

// The producer: one thread issues every stage of this CTA's unit range.
// Returns after the last issue, or (a consumer having stopped) after a
// bounded wait ran out and the copies it issued have landed.
template <class Issue>
__device__ __forceinline__ void produce(int n_units, uint64_t *full, uint64_t *empty,
                                        uint32_t tx_bytes, const SkinnyTmaArgs &p, Issue issue) {
    for (int i = 0; i < n_units; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.timeout_ns)) {
            record_error(p.err, kSiteProducerEmpty);
            for (int g = i > kStages ? i - kStages : 0; g < i; ++g)
                mbar_wait_bounded(&full[g % kStages], (uint32_t)(g / kStages) & 1u, p.timeout_ns);
            return;
        }
        mbar_arrive_expect_tx(&full[s], tx_bytes);
        issue(i, s);
    }
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
skinny_m_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const SkinnyTmaArgs p) {
    static_assert(MT * kMBK * 4 <= kStageBytes - kMBBytes, "A tile must fit the stage");
    extern __shared__ unsigned char smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    unsigned char *smem = smem_raw + pad;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;

    const int64_t u0 = unit_begin(blockIdx.x, p);
    const int n_units = int(unit_begin(blockIdx.x + 1, p) - u0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers / 32);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) {
            prefetch_tensormap(&tmA);
            prefetch_tensormap(&tmB);
            produce(n_units, full, empty, kMBBytes + MT * kMBK * 4, p, [&](int i, int s) {
                const int64_t u = u0 + i;
                const int j = int(u / p.kb), kb = int(u % p.kb);
                unsigned char *st = smem + s * kStageBytes;
#pragma unroll
                for (int q = 0; q < kMBoxes; ++q)
                    tma_load_2d(st + q * (kMBK * kMBoxN * 4), &tmB, &full[s], j * kMCols + q * kMBoxN,
                                kb * kMBK);
                tma_load_2d(st + kMBBytes, &tmA, &full[s], kb * kMBK, 0);
            });
        }
        return;
    }

    const int t = threadIdx.x, lane = t & 31;
    // Thread t: columns 4t .. 4t+3 of the block = box t/64, box column 4(t%64).
    const int b_off = (t >> 6) * (kMBK * kMBoxN) + 4 * (t & 63);
    float2 lo[MT], hi[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) lo[m] = hi[m] = make_float2(0.f, 0.f);
    int cur_j = n_units > 0 ? int(u0 / p.kb) : 0, seg = 0;

    auto flush = [&]() {
        float *out = p.part + ((int64_t)blockIdx.x * p.segs + seg) * p.tile_elems + 4 * t;
#pragma unroll
        for (int m = 0; m < MT; ++m)
            if (m < p.M)
                *reinterpret_cast<float4 *>(out + (int64_t)m * kMCols) =
                    make_float4(lo[m].x, lo[m].y, hi[m].x, hi[m].y);
    };

    for (int i = 0; i < n_units; ++i) {
        const int j = int((u0 + i) / p.kb);
        if (j != cur_j) {
            flush();
#pragma unroll
            for (int m = 0; m < MT; ++m) lo[m] = hi[m] = make_float2(0.f, 0.f);
            cur_j = j;
            ++seg;
        }
        const int s = i % kStages;
        if (!mbar_wait_bounded(&full[s], (uint32_t)(i / kStages) & 1u, p.timeout_ns)) {
            record_error(p.err, kSiteConsumerFull);
            return;
        }
        const unsigned char *st = smem + s * kStageBytes;
        const float *sB = reinterpret_cast<const float *>(st) + b_off;
        const float *sA = reinterpret_cast<const float *>(st + kMBBytes);
        // Two halves of 4 k each: 4 B rows in registers at a time.
#pragma unroll
        for (int kh = 0; kh < kMBK; kh += 4) {
            float4 b[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) b[k] = *reinterpret_cast<const float4 *>(sB + (kh + k) * kMBoxN);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float4 a = *reinterpret_cast<const float4 *>(sA + m * kMBK + kh);
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 a2 = make_float2(av[k], av[k]);
                    lo[m] = __ffma2_rn(a2, make_float2(b[k].x, b[k].y), lo[m]);
                    hi[m] = __ffma2_rn(a2, make_float2(b[k].z, b[k].w), hi[m]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (n_units > 0) flush();
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
skinny_n_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const SkinnyTmaArgs p) {
    constexpr int NP = pad4(NT);
    static_assert(2 * kNABoxBytes + kNBK * NP * 4 <= kStageBytes, "B tile must fit the stage");
    extern __shared__ unsigned char smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    unsigned char *smem = smem_raw + pad;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;

    const int64_t u0 = unit_begin(blockIdx.x, p);
    const int n_units = int(unit_begin(blockIdx.x + 1, p) - u0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers / 32);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) {
            prefetch_tensormap(&tmA);
            prefetch_tensormap(&tmB);
            produce(n_units, full, empty, 2 * kNABoxBytes + kNBK * NP * 4, p, [&](int i, int s) {
                const int64_t u = u0 + i;
                const int j = int(u / p.kb), kb = int(u % p.kb);
                unsigned char *st = smem + s * kStageBytes;
                tma_load_2d(st, &tmA, &full[s], kb * kNBK, j * kNRows);
                tma_load_2d(st + kNABoxBytes, &tmA, &full[s], kb * kNBK, j * kNRows + kNBoxM);
                tma_load_2d(st + 2 * kNABoxBytes, &tmB, &full[s], 0, kb * kNBK);
            });
        }
        return;
    }

    const int t = threadIdx.x, lane = t & 31;
    // Row t of each box is 64 bytes; with the 64-byte swizzle its 16-byte
    // chunk c sits at chunk c ^ ((t >> 1) & 3).
    const int a_row = t * (kNBK * 4);
    const int a_swz = (t >> 1) & 3;
    float2 acc[2][NP / 2];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int g = 0; g < NP / 2; ++g) acc[r][g] = make_float2(0.f, 0.f);
    int cur_j = n_units > 0 ? int(u0 / p.kb) : 0, seg = 0;

    auto flush = [&]() {
        float *out = p.part + ((int64_t)blockIdx.x * p.segs + seg) * p.tile_elems;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float *row = out + (int64_t)(r * kNBoxM + t) * NP;
#pragma unroll
            for (int g = 0; g < NP / 4; ++g)
                *reinterpret_cast<float4 *>(row + 4 * g) =
                    make_float4(acc[r][2 * g].x, acc[r][2 * g].y, acc[r][2 * g + 1].x, acc[r][2 * g + 1].y);
        }
    };

    for (int i = 0; i < n_units; ++i) {
        const int j = int((u0 + i) / p.kb);
        if (j != cur_j) {
            flush();
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int g = 0; g < NP / 2; ++g) acc[r][g] = make_float2(0.f, 0.f);
            cur_j = j;
            ++seg;
        }
        const int s = i % kStages;
        if (!mbar_wait_bounded(&full[s], (uint32_t)(i / kStages) & 1u, p.timeout_ns)) {
            record_error(p.err, kSiteConsumerFull);
            return;
        }
        const unsigned char *st = smem + s * kStageBytes;
        const float *sB = reinterpret_cast<const float *>(st + 2 * kNABoxBytes);
#pragma unroll
        for (int kq = 0; kq < kNBK / 4; ++kq) {
            const int chunk = (kq ^ a_swz) * 16;
            const float4 a0 = *reinterpret_cast<const float4 *>(st + a_row + chunk);
            const float4 a1 = *reinterpret_cast<const float4 *>(st + kNABoxBytes + a_row + chunk);
            const float x0[4] = {a0.x, a0.y, a0.z, a0.w};
            const float x1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float2 p0 = make_float2(x0[kk], x0[kk]);
                const float2 p1 = make_float2(x1[kk], x1[kk]);
#pragma unroll
                for (int g = 0; g < NP / 4; ++g) {
                    const float4 b = *reinterpret_cast<const float4 *>(sB + (kq * 4 + kk) * NP + 4 * g);
                    const float2 bl = make_float2(b.x, b.y), bh = make_float2(b.z, b.w);
                    acc[0][2 * g] = __ffma2_rn(p0, bl, acc[0][2 * g]);
                    acc[0][2 * g + 1] = __ffma2_rn(p0, bh, acc[0][2 * g + 1]);
                    acc[1][2 * g] = __ffma2_rn(p1, bl, acc[1][2 * g]);
                    acc[1][2 * g + 1] = __ffma2_rn(p1, bh, acc[1][2 * g + 1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (n_units > 0) flush();
}

// C = alpha * (sum of the partial tiles of the block, in CTA order) + beta * C;
// C is not read when beta == 0.
__global__ void skinny_tma_reduce_kernel(const SkinnyTmaArgs p, int small_m, int np, float alpha,
                                         float beta, float *__restrict__ C, int64_t ldc) {
    const int64_t total = (int64_t)p.M * p.N;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int m = int(idx / p.N), n = int(idx - (int64_t)m * p.N);
        int j, off;
        if (small_m) {
            j = n / kMCols;
            off = m * kMCols + (n - j * kMCols);
        } else {
            j = m / kNRows;
            off = (m - j * kNRows) * np + n;
        }
        // CTAs whose unit ranges meet block j: owners of its first and last unit.
        const int64_t first = (int64_t)j * p.kb, last = first + p.kb - 1;
        const int c_lo = int(((first + 1) * p.ctas + p.units - 1) / p.units - 1);
        const int c_hi = int(((last + 1) * p.ctas + p.units - 1) / p.units - 1);
        float s = 0.f;
        for (int c = c_lo; c <= c_hi; ++c) {
            const int seg = j - int(((int64_t)c * p.units / p.ctas) / p.kb);
            s += __ldcs(&p.part[((int64_t)c * p.segs + seg) * p.tile_elems + off]);
        }
        float *cp = C + (int64_t)m * ldc + n;
        *cp = beta == 0.0f ? alpha * s : fmaf(beta, *cp, alpha * s);
    }
}

// The shared-memory opt-in is set once per instantiation (each launcher
// below is its own function, so each has its own static).
template <int T>
void launch_m_tma(const CUtensorMap &a, const CUtensorMap &b, const SkinnyTmaArgs &p, cudaStream_t s) {
    static const bool opted_in = cudaFuncSetAttribute(skinny_m_tma_kernel<T>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                      kSmemBytes) == cudaSuccess;
    (void)opted_in;
    skinny_m_tma_kernel<T><<<p.ctas, kThreads, kSmemBytes, s>>>(a, b, p);
}

template <int T>
void launch_n_tma(const CUtensorMap &a, const CUtensorMap &b, const SkinnyTmaArgs &p, cudaStream_t s) {
    static const bool opted_in = cudaFuncSetAttribute(skinny_n_tma_kernel<T>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                      kSmemBytes) == cudaSuccess;
    (void)opted_in;
    skinny_n_tma_kernel<T><<<p.ctas, kThreads, kSmemBytes, s>>>(a, b, p);
}

template <int T>
cudaError_t preload_tma_t() {
    // The same opt-in the launchers make at their first call.
    cudaError_t e = cudaFuncSetAttribute(skinny_m_tma_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(skinny_n_tma_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess) e = load_kernel(reinterpret_cast<const void *>(&skinny_m_tma_kernel<T>));
    if (e == cudaSuccess) e = load_kernel(reinterpret_cast<const void *>(&skinny_n_tma_kernel<T>));
    return e;
}

inline int round_small(int n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : n <= 8 ? 8 : n <= 16 ? 16 : 32; }

}  // namespace

cudaError_t preload_skinny_tma_kernels() {
    cudaError_t e = preload_tma_t<1>();
    if (e == cudaSuccess) e = preload_tma_t<2>();
    if (e == cudaSuccess) e = preload_tma_t<4>();
    if (e == cudaSuccess) e = preload_tma_t<8>();
    if (e == cudaSuccess) e = preload_tma_t<16>();
    if (e == cudaSuccess) e = preload_tma_t<32>();
    if (e == cudaSuccess) e = load_kernel(reinterpret_cast<const void *>(&skinny_tma_reduce_kernel));
    return e;
}

SkinnyTmaGeom skinny_tma_geometry(bool small_m, int M, int N, int K, int sms) {
    SkinnyTmaGeom g;
    const int small = small_m ? M : N;
    g.rows = round_small(small);
    const int64_t blocks = small_m ? (N + kMCols - 1) / kMCols : (M + kNRows - 1) / kNRows;
    const int bk = small_m ? kMBK : kNBK;
    g.kb = (K + bk - 1) / bk;
    g.units = blocks * g.kb;
    g.ctas = int(std::max<int64_t>(1, std::min<int64_t>(sms, g.units)));
    g.segs = 1;
    for (int c = 0; c < g.ctas; ++c) {
        const int64_t u0 = (int64_t)c * g.units / g.ctas, u1 = (int64_t)(c + 1) * g.units / g.ctas;
        if (u1 > u0) g.segs = std::max<int>(g.segs, int((u1 - 1) / g.kb - u0 / g.kb + 1));
    }
    g.tile_elems = small_m ? M * kMCols : kNRows * pad4(g.rows);
    g.ws_bytes = size_t(g.ctas) * g.segs * size_t(g.tile_elems) * 4;
    if (small_m) {
        g.a_box[0] = kMBK;  g.a_box[1] = g.rows;
        g.b_box[0] = kMBoxN; g.b_box[1] = kMBK;
        g.a_swizzle64 = false;
    } else {
        g.a_box[0] = kNBK;  g.a_box[1] = kNBoxM;
        g.b_box[0] = pad4(g.rows); g.b_box[1] = kNBK;
        g.a_swizzle64 = true;
    }
    return g;
}

void launch_skinny_tma(bool small_m, const CUtensorMap &tmA, const CUtensorMap &tmB,
                       const SkinnyTmaGeom &g, int M, int N, int K, float alpha, float beta,
                       float *C, int64_t ldc, float *part, uint32_t *err, uint64_t timeout_ns,
                       cudaStream_t s) {
    SkinnyTmaArgs p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.kb = g.kb;
    p.units = g.units;
    p.ctas = g.ctas;
    p.segs = g.segs;
    p.tile_elems = g.tile_elems;
    p.part = part;
    p.err = err;
    p.timeout_ns = timeout_ns;
    if (small_m) {
        switch (g.rows) {
            case 1: launch_m_tma<1>(tmA, tmB, p, s); break;
            case 2: launch_m_tma<2>(tmA, tmB, p, s); break;
            case 4: launch_m_tma<4>(tmA, tmB, p, s); break;
            case 8: launch_m_tma<8>(tmA, tmB, p, s); break;
            case 16: launch_m_tma<16>(tmA, tmB, p, s); break;
            default: launch_m_tma<32>(tmA, tmB, p, s); break;
        }
    } else {
        switch (g.rows) {
            case 1: launch_n_tma<1>(tmA, tmB, p, s); break;
            case 2: launch_n_tma<2>(tmA, tmB, p, s); break;
            case 4: launch_n_tma<4>(tmA, tmB, p, s); break;
            case 8: launch_n_tma<8>(tmA, tmB, p, s); break;
            case 16: launch_n_tma<16>(tmA, tmB, p, s); break;
            default: launch_n_tma<32>(tmA, tmB, p, s); break;
        }
    }
    const int64_t total = int64_t(M) * N;
    const unsigned blocks = unsigned(std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, 65535)));
    skinny_tma_reduce_kernel<<<blocks, 256, 0, s>>>(p, small_m ? 1 : 0, pad4(g.rows), alpha, beta, C, ldc);
}

}  // namespace sg
