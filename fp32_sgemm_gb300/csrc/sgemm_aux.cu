// Auxiliary kernels of the SGEMM library: the scale-only path (K == 0 or
// alpha == 0), operand preparation (repacking for TMA, transposing
// operands given transposed, splitting into TF32 hi / lo parts for the
// 3xTF32 path) and the bounded-wait self test.
#include <algorithm>

#include "kernel_table.h"

namespace sg {

// Every kernel here takes a batch of matrices: matrix z starts at base +
// z * stride, and blockIdx.z walks the batch (looping past 65535).

// C = beta * C (or 0 when beta == 0, without reading C): the K == 0 and
// alpha == 0 cases, where A and B must not be read.
__global__ void sgemm_scale_c_kernel(int M, int N, float beta, float *C, int64_t ldc,
                                     int64_t stride_c, int batch) {
    for (int64_t z = blockIdx.z; z < batch; z += gridDim.z)
        for (int64_t r = blockIdx.y; r < M; r += gridDim.y) {
            float *row = C + z * stride_c + r * ldc;
            for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < N; c += gridDim.x * blockDim.x)
                row[c] = beta == 0.0f ? 0.0f : beta * row[c];
        }
}

// Asynchronous 4-byte copy global -> shared (no registers held while it is
// in flight); completion is awaited with cp_async_wait_all.
__device__ __forceinline__ void cp_async_4(float *dst_smem, const float *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_u32(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Quads (16-byte groups of 4 columns) per lane in one repack unit: a unit is
// 32 * kPackQuads groups of one row, all its loads issued before any store.
constexpr int kPackQuads = 8;
constexpr int kPackGroups = 32 * kPackQuads;

// One repack unit: columns [4 gbase, 4 (gbase + kPackGroups)) of one row,
// copied into a destination row whose start is 16-byte aligned.  The source is read
// once, with evict-first loads (measured: 598.5 -> 595.5 us per call at
// 4095 x 4097 x 1023, where this launch pays for the previous product's C
// leaving L2).  The source row may
// start at any 4-byte offset (odd pitch): lane l reads the 16-byte aligned
// quad that holds the start of its 4-column group and takes the rest from
// lane l + 1's quad by a shuffle (lane 31 from lane 0's next quad), so the
// row is read with 16-byte loads; a
// quad that reaches outside the row (its first or last) is read element by
// element, so nothing outside the row is touched.  The padding of the last
// group is written as zeros.  DOT: also add this lane's columns times the
// staged B columns (bstrip[jj * K + k]) into s[jj], k in ascending order.
template <bool DOT>
__device__ __forceinline__ void repack_chunk(const PackJob &j, const float *src, float *dst, int gbase, int lane,
                                             const float *bstrip, int K, int r, float (&s)[kEdgeMaxCols]) {
    const int ph = (int)((reinterpret_cast<uintptr_t>(src) >> 2) & 3u);   // floats past a 16-byte boundary
    const float *ab = src - ph;                                              // 16-byte aligned
    const int cols = j.cols;
    // Quad m of the aligned row holds row elements 4m - ph .. 4m - ph + 3.
    auto quad = [&](int m) {
        const int e0 = 4 * m - ph;
        if (e0 >= 0 && e0 + 3 < cols) return __ldcs(reinterpret_cast<const float4 *>(ab + 4 * m));
        float4 q;
        q.x = (e0 >= 0 && e0 < cols) ? __ldcs(ab + 4 * m) : 0.f;
        q.y = (e0 + 1 >= 0 && e0 + 1 < cols) ? __ldcs(ab + 4 * m + 1) : 0.f;
        q.z = (e0 + 2 >= 0 && e0 + 2 < cols) ? __ldcs(ab + 4 * m + 2) : 0.f;
        q.w = (e0 + 3 >= 0 && e0 + 3 < cols) ? __ldcs(ab + 4 * m + 3) : 0.f;
        return q;
    };
    float4 q4[kPackQuads];
#pragma unroll
    for (int q = 0; q < kPackQuads; ++q) {
        const int g = gbase + 32 * q + lane;     // this lane's group: row elements 4g .. 4g + 3
        // (With ph != 0 the quad after the last group may still hold the
        // last elements of the row.)
        q4[q] = (g < j.groups || (ph != 0 && g == j.groups)) ? quad(g) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // The quad after the unit's last one, for lane 31 (the others take it from lane 0).
    const int g_last = gbase + 32 * (kPackQuads - 1) + 31;
    const float4 after = (lane == 31 && ph != 0 && g_last < j.groups) ? quad(g_last + 1)
                                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kPackQuads; ++q) {
        const int g = gbase + 32 * q + lane;
        // The next quad: lane + 1's; for lane 31, lane 0's next one (or the
        // one loaded above).
        float4 nx, wrap = after;
        nx.x = __shfl_down_sync(0xffffffffu, q4[q].x, 1);
        nx.y = __shfl_down_sync(0xffffffffu, q4[q].y, 1);
        nx.z = __shfl_down_sync(0xffffffffu, q4[q].z, 1);
        if (q + 1 < kPackQuads) {
            wrap.x = __shfl_sync(0xffffffffu, q4[q + 1].x, 0);
            wrap.y = __shfl_sync(0xffffffffu, q4[q + 1].y, 0);
            wrap.z = __shfl_sync(0xffffffffu, q4[q + 1].z, 0);
        }
        if (lane == 31) nx = wrap;
        float4 o;
        if (ph == 0) o = q4[q];
        else if (ph == 1) o = make_float4(q4[q].y, q4[q].z, q4[q].w, nx.x);
        else if (ph == 2) o = make_float4(q4[q].z, q4[q].w, nx.x, nx.y);
        else o = make_float4(q4[q].w, nx.x, nx.y, nx.z);
        if (g < j.groups) {
            *reinterpret_cast<float4 *>(dst + 4 * g) = o;
            if constexpr (DOT) {
                const int k0 = 4 * g;                // < K; the group's later columns may pass K
#pragma unroll
                for (int jj = 0; jj < kEdgeMaxCols; ++jj) {
                    if (jj < r) {
                        const float *b = bstrip + jj * K + k0;
                        s[jj] = fmaf(o.x, b[0], s[jj]);
                        if (k0 + 1 < K) s[jj] = fmaf(o.y, b[1], s[jj]);
                        if (k0 + 2 < K) s[jj] = fmaf(o.z, b[2], s[jj]);
                        if (k0 + 3 < K) s[jj] = fmaf(o.w, b[3], s[jj]);
                    }
                }
            }
        }
    }
}

// C[row][n0 + jj] = alpha * s[jj] (+ beta * C) for jj < r, after summing s
// across the warp by a fixed butterfly (the same result every run).
__device__ __forceinline__ void edge_finish(const EdgeJob &e, int64_t row, int lane, float (&s)[kEdgeMaxCols]) {
#pragma unroll
    for (int jj = 0; jj < kEdgeMaxCols; ++jj)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s[jj] += __shfl_xor_sync(0xffffffffu, s[jj], o);
    if (lane == 0) {
        float *c = e.C + row * e.ldc + e.n0;
#pragma unroll
        for (int jj = 0; jj < kEdgeMaxCols; ++jj)
            if (jj < e.r) c[jj] = e.beta == 0.0f ? e.alpha * s[jj] : fmaf(e.beta, c[jj], e.alpha * s[jj]);
    }
}

// Operand preparation in one launch (launched with programmatic stream
// serialisation: it waits for the kernel before it, and lets the main kernel
// after it be placed as its CTAs finish), one persistent wave of CTAs:
//   * up to two repack jobs: rows x cols row-major matrices copied into
//     buffers whose row pitch is a multiple of 4 floats (16-byte aligned
//     rows), so that TMA can address them; a warp per (row, 1024 columns);
//   * the edge job: the last r <= kEdgeMaxCols columns of C when the main
//     kernel leaves them out (a last tile column that thin would multiply
//     mostly padding): C = alpha * A . B[:, n0 : n0 + r] (+ beta * C, C not
//     read when beta == 0).  B's r columns are a strided gather (one cache
//     line per k): every block stages them in shared memory once, by
//     asynchronous copies issued first and awaited only after the repacks
//     that do not need them.  When A is repacked in the same launch
//     (edge_pack), the products are taken from A's values as the repack
//     moves them: a warp per row of A, each lane summing its own columns in
//     ascending order with FP32 FMAs, then a fixed butterfly sum across the
//     warp; A is read once.  Otherwise a pass of its own over A, a warp per
//     row, lanes striding over k.
// Every role is bound by the latency of its loads, so each keeps many loads
// in flight with short chains: a repack unit's 8 quads per lane are all
// loaded before any is stored, in two CTAs per SM of up to 128 registers a
// thread (measured per call, 2048 x 2051 x 1100 with odd pitches: 177.9 us,
// against 183.5 with 4 quads per lane and four CTAs per SM; 8 quads in 64
// registers spilled, 190.7).
__global__ void __launch_bounds__(256, 2) sgemm_prep_kernel(const __grid_constant__ PrepArgs p) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;                  // warp in block
    const int wpb = blockDim.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * wpb + wib;
    const int64_t warps = (int64_t)gridDim.x * wpb;
    extern __shared__ float bstrip[];                  // [r][K], the edge job's columns of B
    const EdgeJob &e = p.edge;
    const bool edge = e.r > 0;
    if (edge) {
        // Column by column, so that lanes reading consecutive k hit
        // consecutive banks.
        for (int t = threadIdx.x; t < e.K * e.r; t += blockDim.x) {
            const int kk = t / e.r, jj = t - kk * e.r;
            cp_async_4(&bstrip[jj * e.K + kk], &e.B[(int64_t)kk * e.ldb + e.n0 + jj]);
        }
        cp_async_commit();
    }
    float s[kEdgeMaxCols];

    // The repack units of the jobs the edge job does not ride on, rows of
    // all batch entries in turn.
    const int fused = edge ? p.edge_pack : -1;
    const int64_t u0 = fused == 0 ? 0 : p.pack[0].units;
    const int64_t u1 = fused == 1 ? 0 : p.pack[1].units;
    for (int64_t w = gw; w < u0 + u1; w += warps) {
        const bool second = w >= u0;
        const PackJob &j = second ? p.pack[1] : p.pack[0];
        const int64_t v = second ? w - u0 : w;
        const int64_t chunks = (j.groups + kPackGroups - 1) / kPackGroups;
        const int64_t zr = v / chunks;
        const int gbase = (int)(v - zr * chunks) * kPackGroups;
        const int64_t z = zr / j.rows, r = zr - z * j.rows;
        repack_chunk<false>(j, j.src + z * j.s_src + r * j.ld_src, j.dst + z * j.s_dst + r * j.ld_dst, gbase,
                            lane, nullptr, 0, 0, s);
    }
    if (!edge) return;

    cp_async_wait_all();
    __syncthreads();
    if (fused >= 0) {
        // A's repack carrying the edge products (one batch entry): a warp per row.
        const PackJob &j = p.pack[fused];
        for (int64_t row = gw; row < j.rows; row += warps) {
#pragma unroll
            for (int jj = 0; jj < kEdgeMaxCols; ++jj) s[jj] = 0.f;
            const float *src = j.src + row * j.ld_src;
            float *dst = j.dst + row * j.ld_dst;
            for (int gbase = 0; gbase < j.groups; gbase += kPackGroups)
                repack_chunk<true>(j, src, dst, gbase, lane, bstrip, e.K, e.r, s);
            edge_finish(e, row, lane, s);
        }
        return;
    }
    for (int64_t row = gw; row < e.M; row += warps) {
#pragma unroll
        for (int jj = 0; jj < kEdgeMaxCols; ++jj) s[jj] = 0.f;
        const float *a = e.A + row * e.lda;
        // Sixteen k steps' loads of A in flight per lane; every sum takes k
        // in ascending order.
        int k = lane;
        for (; k + 15 * 32 < e.K; k += 16 * 32) {
            float av[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) av[u] = a[k + 32 * u];
#pragma unroll
            for (int u = 0; u < 16; ++u)
#pragma unroll
                for (int jj = 0; jj < kEdgeMaxCols; ++jj)
                    if (jj < e.r) s[jj] = fmaf(av[u], bstrip[jj * e.K + k + 32 * u], s[jj]);
        }
        for (; k < e.K; k += 32) {
            const float av = a[k];
#pragma unroll
            for (int jj = 0; jj < kEdgeMaxCols; ++jj)
                if (jj < e.r) s[jj] = fmaf(av, bstrip[jj * e.K + k], s[jj]);
        }
        edge_finish(e, row, lane, s);
    }
}

// Transpose rows x cols matrices src[r][c] -> dst[c][r] through 64 x 64
// tiles in shared memory: 16-byte reads along source rows (VEC_SRC, when the
// source allows; else 4-byte reads) and 16-byte writes of 256-byte
// destination row segments (VEC_DST).  Row pitch 65 keeps shared-memory
// accesses at most two-way conflicted.
//   SPLIT = false: plain copy (operands given transposed, for the FFMA path);
//   SPLIT = true : dst gets tf32_trunc(x) (the TF32 part the MMA would read
//                  of x), dst2 the residual tf32_rna(x - tf32_trunc(x))
//                  (3xTF32 path).  The high part is stored with its low bits
//                  cleared: the same products, but the tensor cores ran
//                  slower on operands whose dropped bits were not zero
//                  (8192^3 main kernel 3369 us against 3412-3430).
template <bool SPLIT, bool VEC_SRC, bool VEC_DST>
__global__ void __launch_bounds__(256)
sgemm_transpose_kernel(const float *__restrict__ src, int64_t ld_src, int64_t s_src,
                       float *__restrict__ dst, float *__restrict__ dst2, int64_t ld_dst,
                       int64_t s_dst, int rows, int cols, int batch) {
    __shared__ float t0[64][65];
    __shared__ float t1[SPLIT ? 64 : 1][SPLIT ? 65 : 1];
    griddep_launch_dependents();
    griddep_wait();              // the previous kernel may still read dst
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;     // 16 x 16
    const int c0 = blockIdx.x * 64;      // source columns
    const int r0 = blockIdx.y * 64;      // source rows
    for (int64_t z = blockIdx.z; z < batch; z += gridDim.z) {
        const float *sb = src + z * s_src;
        float x[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r0 + ty + 16 * i;
            const int c = c0 + 4 * tx;
            const float *sp = sb + (int64_t)r * ld_src + c;
            if (VEC_SRC && r < rows && c + 3 < cols) {
                const float4 v = __ldcs(reinterpret_cast<const float4 *>(sp));
                x[i][0] = v.x; x[i][1] = v.y; x[i][2] = v.z; x[i][3] = v.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) x[i][e] = (r < rows && c + e < cols) ? __ldcs(sp + e) : 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if constexpr (SPLIT) {
                    t0[ty + 16 * i][4 * tx + e] = tf32_trunc(x[i][e]);
                    t1[ty + 16 * i][4 * tx + e] = tf32_rna(x[i][e] - tf32_trunc(x[i][e]));
                } else {
                    t0[ty + 16 * i][4 * tx + e] = x[i][e];
                }
            }
        __syncthreads();
        float *db = dst + z * s_dst;
        float *db2 = SPLIT ? dst2 + z * s_dst : nullptr;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int cl = ty + 16 * j;
            const int c = c0 + cl;                   // destination row
            const int r = r0 + 4 * tx;               // destination columns r .. r+3
            if (c < cols) {
                float *dp = db + (int64_t)c * ld_dst + r;
                const float v[4] = {t0[4 * tx][cl], t0[4 * tx + 1][cl], t0[4 * tx + 2][cl], t0[4 * tx + 3][cl]};
                if (VEC_DST && r + 3 < rows) {
                    *reinterpret_cast<float4 *>(dp) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (r + e < rows) dp[e] = v[e];
                }
                if constexpr (SPLIT) {
                    float *dp2 = db2 + (int64_t)c * ld_dst + r;
                    const float w[4] = {t1[4 * tx][cl], t1[4 * tx + 1][cl], t1[4 * tx + 2][cl],
                                        t1[4 * tx + 3][cl]};
                    if (VEC_DST && r + 3 < rows) {
                        *reinterpret_cast<float4 *>(dp2) = make_float4(w[0], w[1], w[2], w[3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (r + e < rows) dp2[e] = w[e];
                    }
                }
            }
        }
        __syncthreads();
    }
}

// Row-major split into hi / lo parts (3xTF32 path), scalar: hi =
// tf32_trunc(x), lo = tf32_rna(x - tf32_trunc(x)).  hi == nullptr: only lo
// is written (the MMA reads hi from the operand in place).  A block takes
// 1024 columns of two rows at a time, each thread issuing its eight loads
// before any store (4095 x 1023, lda 1023: 8.7 us under ncu, against 19.4
// with one element per thread and row).
__global__ void __launch_bounds__(256)
sgemm_split_rows_kernel(const float *__restrict__ src, int64_t ld_src, int64_t s_src,
                        float *__restrict__ hi, float *__restrict__ lo, int64_t ld_dst,
                        int64_t s_dst, int rows, int cols, int batch) {
    griddep_launch_dependents();
    griddep_wait();
    constexpr int R = 2, U = 4;                  // rows and columns per thread and step
    for (int64_t z = blockIdx.z; z < batch; z += gridDim.z)
        for (int64_t r0 = (int64_t)blockIdx.y * R; r0 < rows; r0 += (int64_t)gridDim.y * R)
            for (int c0 = blockIdx.x * 256 * U; c0 < cols; c0 += gridDim.x * 256 * U) {
                float x[R][U];
#pragma unroll
                for (int i = 0; i < R; ++i)
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int c = c0 + 256 * u + (int)threadIdx.x;
                        x[i][u] = (r0 + i < rows && c < cols) ? src[z * s_src + (r0 + i) * ld_src + c] : 0.f;
                    }
#pragma unroll
                for (int i = 0; i < R; ++i)
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int c = c0 + 256 * u + (int)threadIdx.x;
                        if (r0 + i < rows && c < cols) {
                            const int64_t o = z * s_dst + (r0 + i) * ld_dst + c;
                            if (hi != nullptr) hi[o] = tf32_trunc(x[i][u]);
                            lo[o] = tf32_rna(x[i][u] - tf32_trunc(x[i][u]));
                        }
                    }
            }
}

// Same, 16 bytes at a time (src and dst 16-byte aligned; pitches, batch
// strides and cols multiples of 4 floats).  A block covers 1024 float4 of a
// row; each thread issues its four loads before any store.  The source is
// read evict-first unless the main kernel reads it again (hi == nullptr).
__global__ void __launch_bounds__(256)
sgemm_split_rows_vec4_kernel(const float4 *__restrict__ src, int64_t ld4, int64_t s4,
                             float4 *__restrict__ hi, float4 *__restrict__ lo, int64_t ldd4,
                             int64_t sd4, int rows, int cols4, int batch) {
    griddep_launch_dependents();
    griddep_wait();
    for (int64_t z = blockIdx.z; z < batch; z += gridDim.z)
        for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
            const float4 *sr = src + z * s4 + r * ld4;
            float4 *h = hi != nullptr ? hi + z * sd4 + r * ldd4 : nullptr;
            float4 *l = lo + z * sd4 + r * ldd4;
            const int c = blockIdx.x * 1024 + threadIdx.x;
            float4 x[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (c + 256 * i < cols4) x[i] = hi != nullptr ? __ldcs(&sr[c + 256 * i]) : sr[c + 256 * i];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (c + 256 * i < cols4) {
                    float4 xl;
                    xl.x = tf32_rna(x[i].x - tf32_trunc(x[i].x));
                    xl.y = tf32_rna(x[i].y - tf32_trunc(x[i].y));
                    xl.z = tf32_rna(x[i].z - tf32_trunc(x[i].z));
                    xl.w = tf32_rna(x[i].w - tf32_trunc(x[i].w));
                    if (hi != nullptr) h[c + 256 * i] = make_float4(tf32_trunc(x[i].x), tf32_trunc(x[i].y), tf32_trunc(x[i].z), tf32_trunc(x[i].w));
                    l[c + 256 * i] = xl;
                }
            }
        }
}

// Self test of the bounded wait: waits on a barrier that nothing completes.
__global__ void sgemm_wait_selftest_kernel(uint32_t *err, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait_bounded(&bar, 0, timeout_ns)) record_error(err, kSiteSelfTest);
    }
}


namespace {
inline int64_t cdiv(int64_t x, int64_t a) { return (x + a - 1) / a; }
}  // namespace

namespace {
unsigned zdim(int batch) { return unsigned(std::min(std::max(batch, 1), 65535)); }
// Launch with programmatic stream serialisation, as the main kernels are:
// the kernel's CTAs may be placed while the kernel before it finishes, and
// wait for it (griddepcontrol.wait) before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
}  // namespace

void launch_scale_c(int M, int N, float beta, float *C, int64_t ldc, int64_t stride_c, int batch,
                    cudaStream_t s) {
    dim3 grid(unsigned(std::min<int64_t>(cdiv(N, 256), 8)), unsigned(std::min<int64_t>(M, 65535)), zdim(batch));
    sgemm_scale_c_kernel<<<grid, 256, 0, s>>>(M, N, beta, C, ldc, stride_c, batch);
}

cudaError_t launch_prep(PrepArgs p, int sms, cudaStream_t s) {
    int64_t units = 0;
    if (p.edge.r == 0 || p.edge_pack >= p.npack) p.edge_pack = -1;
    for (int i = 0; i < 2; ++i) {
        PackJob &j = p.pack[i];
        if (i >= p.npack) j = PackJob{};
        j.groups = (j.cols + 3) / 4;
        if (i == p.edge_pack) {
            j.units = j.rows;                                         // rows (one batch entry)
        } else {
            j.units = (int64_t)j.batch * j.rows * cdiv(j.groups, kPackGroups);   // (row, chunk)
            units += j.units;
        }
    }
    // One persistent wave: two CTAs of eight warps per SM, every warp takes
    // repack units and then edge rows in turn.
    const int64_t warps_needed = std::max<int64_t>(units, p.edge.r > 0 ? p.edge.M : 0);
    const int blocks = (int)std::min<int64_t>(cdiv(warps_needed, 8), 2 * (int64_t)sms);
    if (blocks == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = p.edge.r > 0 ? size_t(p.edge.r) * size_t(p.edge.K) * 4 : 0;   // <= kEdgeMaxStrip floats
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sgemm_prep_kernel, p);
}

void launch_transpose(const float *src, int64_t ld_src, int64_t s_src, float *dst, float *dst2,
                      int64_t ld_dst, int64_t s_dst, int rows, int cols, int batch, cudaStream_t s) {
    dim3 grid(unsigned(cdiv(cols, 64)), unsigned(cdiv(rows, 64)), zdim(batch));
    const bool vs = reinterpret_cast<uintptr_t>(src) % 16 == 0 && ld_src % 4 == 0 &&
                    (batch == 1 || s_src % 4 == 0);
    const bool vd = reinterpret_cast<uintptr_t>(dst) % 16 == 0 && ld_dst % 4 == 0 &&
                    (batch == 1 || s_dst % 4 == 0) &&
                    (dst2 == nullptr || reinterpret_cast<uintptr_t>(dst2) % 16 == 0);
    auto go = [&](auto kernel) {
        launch_chained(kernel, grid, s, src, ld_src, s_src, dst, dst2, ld_dst, s_dst, rows, cols, batch);
    };
    if (dst2 != nullptr) {
        if (vs && vd) go(sgemm_transpose_kernel<true, true, true>);
        else if (vd) go(sgemm_transpose_kernel<true, false, true>);
        else go(sgemm_transpose_kernel<true, false, false>);
    } else {
        if (vs && vd) go(sgemm_transpose_kernel<false, true, true>);
        else if (vd) go(sgemm_transpose_kernel<false, false, true>);
        else go(sgemm_transpose_kernel<false, false, false>);
    }
}

void launch_split_rows(const float *src, int64_t ld_src, int64_t s_src, float *hi, float *lo,
                       int64_t ld_dst, int64_t s_dst, int rows, int cols, int batch, cudaStream_t s) {
    const bool vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && ld_src % 4 == 0 && cols % 4 == 0 &&
                     ld_dst % 4 == 0 && (batch == 1 || (s_src % 4 == 0 && s_dst % 4 == 0));
    if (vec && reinterpret_cast<uintptr_t>(hi) % 16 == 0 && reinterpret_cast<uintptr_t>(lo) % 16 == 0) {   // (hi may be null)
        dim3 grid(unsigned(std::max<int64_t>(1, cdiv(cols / 4, 1024))), unsigned(std::min<int64_t>(rows, 65535)),
                  zdim(batch));
        launch_chained(sgemm_split_rows_vec4_kernel, grid, s, reinterpret_cast<const float4 *>(src), ld_src / 4,
                       s_src / 4, reinterpret_cast<float4 *>(hi), reinterpret_cast<float4 *>(lo), ld_dst / 4,
                       s_dst / 4, rows, cols / 4, batch);
        return;
    }
    dim3 grid(unsigned(std::min<int64_t>(cdiv(cols, 1024), 8)), unsigned(std::min<int64_t>(cdiv(rows, 2), 65535)),
              zdim(batch));
    launch_chained(sgemm_split_rows_kernel, grid, s, src, ld_src, s_src, hi, lo, ld_dst, s_dst, rows, cols, batch);
}

cudaError_t preload_aux_kernels() {
    const void *fns[] = {
        reinterpret_cast<const void *>(&sgemm_scale_c_kernel),
        reinterpret_cast<const void *>(&sgemm_prep_kernel),
        reinterpret_cast<const void *>(&sgemm_transpose_kernel<true, true, true>),
        reinterpret_cast<const void *>(&sgemm_transpose_kernel<true, false, true>),
        reinterpret_cast<const void *>(&sgemm_transpose_kernel<true, false, false>),
        reinterpret_cast<const void *>(&sgemm_transpose_kernel<false, true, true>),
        reinterpret_cast<const void *>(&sgemm_transpose_kernel<false, false, true>),
        reinterpret_cast<const void *>(&sgemm_transpose_kernel<false, false, false>),
        reinterpret_cast<const void *>(&sgemm_split_rows_kernel),
        reinterpret_cast<const void *>(&sgemm_split_rows_vec4_kernel),
        reinterpret_cast<const void *>(&sgemm_wait_selftest_kernel)};
    for (const void *fn : fns)
        if (cudaError_t e = load_kernel(fn); e != cudaSuccess) return e;
    return cudaSuccess;
}

void launch_wait_selftest(uint32_t *err, uint64_t timeout_ns, cudaStream_t s) {
    sgemm_wait_selftest_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
}

}  // namespace sg
