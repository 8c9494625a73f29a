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

// Copy rows x cols row-major matrices into buffers with row pitch ld_dst (a
// multiple of 4 floats), so that TMA can address them.
__global__ void sgemm_pack_rows_kernel(const float *src, int64_t ld_src, int64_t s_src, float *dst,
                                       int64_t ld_dst, int64_t s_dst, int rows, int cols, int batch) {
    for (int64_t z = blockIdx.z; z < batch; z += gridDim.z)
        for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
            const float *sr = src + z * s_src + r * ld_src;
            float *d = dst + z * s_dst + r * ld_dst;
            for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < cols; c += gridDim.x * blockDim.x)
                d[c] = sr[c];
        }
}

// Transpose rows x cols matrices src[r][c] -> dst[c][r] through 32 x 128
// tiles in shared memory (128-byte coalesced reads and writes; the tile's
// row pitch of 129 words keeps both phases free of bank conflicts).
//   SPLIT = false: plain copy (operands given transposed, for the FFMA path);
//   SPLIT = true : dst gets tf32(x), dst2 gets tf32(x - tf32(x)) (3xTF32 path).
template <bool SPLIT>
__global__ void __launch_bounds__(256)
sgemm_transpose_kernel(const float *__restrict__ src, int64_t ld_src, int64_t s_src,
                       float *__restrict__ dst, float *__restrict__ dst2, int64_t ld_dst,
                       int64_t s_dst, int rows, int cols, int batch) {
    __shared__ float t0[32][129];
    __shared__ float t1[SPLIT ? 32 : 1][SPLIT ? 129 : 1];
    const int c0 = blockIdx.x * 128;     // source columns
    const int r0 = blockIdx.y * 32;      // source rows
    const int tx = threadIdx.x, ty = threadIdx.y;   // 32 x 8
    for (int64_t z = blockIdx.z; z < batch; z += gridDim.z) {
        const float *sb = src + z * s_src;
        float x[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r0 + ty + 8 * i;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = c0 + tx + 32 * e;
                x[i][e] = (r < rows && c < cols) ? __ldcs(&sb[(int64_t)r * ld_src + c]) : 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if constexpr (SPLIT) {
                    const float xh = tf32_rna(x[i][e]);
                    t0[ty + 8 * i][tx + 32 * e] = xh;
                    t1[ty + 8 * i][tx + 32 * e] = tf32_rna(x[i][e] - xh);
                } else {
                    t0[ty + 8 * i][tx + 32 * e] = x[i][e];
                }
            }
        __syncthreads();
        const int r = r0 + tx;
        float *db = dst + z * s_dst;
        float *db2 = SPLIT ? dst2 + z * s_dst : nullptr;
#pragma unroll 4
        for (int j = 0; j < 16; ++j) {
            const int cl = ty + 8 * j;
            const int c = c0 + cl;
            if (c < cols && r < rows) {
                db[(int64_t)c * ld_dst + r] = t0[tx][cl];
                if constexpr (SPLIT) db2[(int64_t)c * ld_dst + r] = t1[tx][cl];
            }
        }
        __syncthreads();
    }
}

// Row-major split into TF32 hi / lo parts (3xTF32 path), scalar.
__global__ void sgemm_split_rows_kernel(const float *__restrict__ src, int64_t ld_src, int64_t s_src,
                                        float *__restrict__ hi, float *__restrict__ lo, int64_t ld_dst,
                                        int64_t s_dst, int rows, int cols, int batch) {
    for (int64_t z = blockIdx.z; z < batch; z += gridDim.z)
        for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
            const float *sr = src + z * s_src + r * ld_src;
            float *h = hi + z * s_dst + r * ld_dst;
            float *l = lo + z * s_dst + r * ld_dst;
            for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < cols; c += gridDim.x * blockDim.x) {
                const float x = sr[c];
                const float xh = tf32_rna(x);
                h[c] = xh;
                l[c] = tf32_rna(x - xh);
            }
        }
}

// Same, 16 bytes at a time over the whole batch (src 16-byte aligned; the
// pitches, batch strides and cols multiples of 4 floats).
__global__ void sgemm_split_rows_vec4_kernel(const float4 *__restrict__ src, int64_t ld4, int64_t s4,
                                             float4 *__restrict__ hi, float4 *__restrict__ lo,
                                             int64_t ldd4, int64_t sd4, int64_t rows, int64_t cols4,
                                             int64_t batch) {
    const int64_t per = rows * cols4;
    const int64_t total = per * batch;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t z = i / per;
        const int64_t rem = i - z * per;
        const int64_t r = rem / cols4, c = rem - r * cols4;
        const float4 x = __ldcs(&src[z * s4 + r * ld4 + c]);
        float4 xh, xl;
        xh.x = tf32_rna(x.x); xl.x = tf32_rna(x.x - xh.x);
        xh.y = tf32_rna(x.y); xl.y = tf32_rna(x.y - xh.y);
        xh.z = tf32_rna(x.z); xl.z = tf32_rna(x.z - xh.z);
        xh.w = tf32_rna(x.w); xl.w = tf32_rna(x.w - xh.w);
        hi[z * sd4 + r * ldd4 + c] = xh;
        lo[z * sd4 + r * ldd4 + c] = xl;
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
int num_sms() {
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}
}  // namespace

void launch_scale_c(int M, int N, float beta, float *C, int64_t ldc, int64_t stride_c, int batch,
                    cudaStream_t s) {
    dim3 grid(unsigned(std::min<int64_t>(cdiv(N, 256), 8)), unsigned(std::min<int64_t>(M, 65535)), zdim(batch));
    sgemm_scale_c_kernel<<<grid, 256, 0, s>>>(M, N, beta, C, ldc, stride_c, batch);
}

void launch_pack_rows(const float *src, int64_t ld_src, int64_t s_src, float *dst, int64_t ld_dst,
                      int64_t s_dst, int rows, int cols, int batch, cudaStream_t s) {
    dim3 grid(unsigned(std::min<int64_t>(cdiv(cols, 256), 8)), unsigned(std::min<int64_t>(rows, 65535)), zdim(batch));
    sgemm_pack_rows_kernel<<<grid, 256, 0, s>>>(src, ld_src, s_src, dst, ld_dst, s_dst, rows, cols, batch);
}

void launch_transpose(const float *src, int64_t ld_src, int64_t s_src, float *dst, float *dst2,
                      int64_t ld_dst, int64_t s_dst, int rows, int cols, int batch, cudaStream_t s) {
    dim3 grid(unsigned(cdiv(cols, 128)), unsigned(cdiv(rows, 32)), zdim(batch));
    if (dst2 != nullptr)
        sgemm_transpose_kernel<true><<<grid, dim3(32, 8), 0, s>>>(src, ld_src, s_src, dst, dst2, ld_dst,
                                                                 s_dst, rows, cols, batch);
    else
        sgemm_transpose_kernel<false><<<grid, dim3(32, 8), 0, s>>>(src, ld_src, s_src, dst, nullptr, ld_dst,
                                                                  s_dst, rows, cols, batch);
}

void launch_split_rows(const float *src, int64_t ld_src, int64_t s_src, float *hi, float *lo,
                       int64_t ld_dst, int64_t s_dst, int rows, int cols, int batch, cudaStream_t s) {
    const bool vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && ld_src % 4 == 0 && cols % 4 == 0 &&
                     ld_dst % 4 == 0 && (batch == 1 || (s_src % 4 == 0 && s_dst % 4 == 0));
    if (vec) {
        const int64_t total = int64_t(rows) * (cols / 4) * batch;
        const int64_t blocks = std::min<int64_t>(cdiv(total, 256), int64_t(num_sms()) * 8);
        sgemm_split_rows_vec4_kernel<<<unsigned(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(
            reinterpret_cast<const float4 *>(src), ld_src / 4, s_src / 4, reinterpret_cast<float4 *>(hi),
            reinterpret_cast<float4 *>(lo), ld_dst / 4, s_dst / 4, rows, cols / 4, batch);
        return;
    }
    dim3 grid(unsigned(std::min<int64_t>(cdiv(cols, 256), 8)), unsigned(std::min<int64_t>(rows, 65535)), zdim(batch));
    sgemm_split_rows_kernel<<<grid, 256, 0, s>>>(src, ld_src, s_src, hi, lo, ld_dst, s_dst, rows, cols, batch);
}

void launch_wait_selftest(uint32_t *err, uint64_t timeout_ns, cudaStream_t s) {
    sgemm_wait_selftest_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
}

}  // namespace sg
