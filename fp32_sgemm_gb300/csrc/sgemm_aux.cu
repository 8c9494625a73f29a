// Auxiliary kernels of the SGEMM library: the scale-only path (K == 0 or
// alpha == 0), operand repacking for TMA, and the bounded-wait self test.
#include <algorithm>

#include "kernel_table.h"

namespace sg {

// C = beta * C (or 0 when beta == 0, without reading C): the K == 0 and
// alpha == 0 cases, where A and B must not be read.
__global__ void sgemm_scale_c_kernel(int M, int N, float beta, float *C, int64_t ldc) {
    for (int64_t r = blockIdx.y; r < M; r += gridDim.y) {
        float *row = C + r * ldc;
        for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < N; c += gridDim.x * blockDim.x)
            row[c] = beta == 0.0f ? 0.0f : beta * row[c];
    }
}

// Copy a rows x cols row-major matrix into a buffer with row pitch ld_dst
// (a multiple of 4 floats), so that TMA can address it.
__global__ void sgemm_pack_rows_kernel(const float *src, int64_t ld_src, float *dst,
                                       int64_t ld_dst, int rows, int cols) {
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const float *s = src + r * ld_src;
        float *d = dst + r * ld_dst;
        for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < cols; c += gridDim.x * blockDim.x)
            d[c] = s[c];
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

void launch_scale_c(int M, int N, float beta, float *C, int64_t ldc, cudaStream_t s) {
    dim3 grid(unsigned(std::min<int64_t>(cdiv(N, 256), 8)), unsigned(std::min<int64_t>(M, 65535)));
    sgemm_scale_c_kernel<<<grid, 256, 0, s>>>(M, N, beta, C, ldc);
}

void launch_pack_rows(const float *src, int64_t ld_src, float *dst, int64_t ld_dst,
                      int rows, int cols, cudaStream_t s) {
    dim3 grid(unsigned(std::min<int64_t>(cdiv(cols, 256), 8)), unsigned(std::min<int64_t>(rows, 65535)));
    sgemm_pack_rows_kernel<<<grid, 256, 0, s>>>(src, ld_src, dst, ld_dst, rows, cols);
}

void launch_wait_selftest(uint32_t *err, uint64_t timeout_ns, cudaStream_t s) {
    sgemm_wait_selftest_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
}

}  // namespace sg
