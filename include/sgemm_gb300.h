/*
 * sgemm_gb300.h: C ABI of the FP32 general matrix multiply for NVIDIA GB300
 * (sm_103a).
 *
 *   C = alpha * A . B + beta * C        (FP32 in, FP32 FMA, FP32 out)
 *
 * A is M x K, B is K x N, C is M x N, all ROW MAJOR with leading dimensions
 * (row pitches, in elements) lda >= max(1, K), ldb >= max(1, N),
 * ldc >= max(1, N).  The operation and its 2MNK FLOP count are the problem
 * statement of "Matmul I: tiling and shared memory" (notes.ybc.sh cap-07,
 * section 1); alpha and beta enter in the epilogue as in "2D Register Tiling:
 * The Outer Product" (maxxfuu article4/page8, "The Kernel"); with beta == 0 C
 * is not read, as in "The Final Kernel" (maxxfuu article4/page14, "Skipping
 * The Read Of C").  Those pages give the kernel signature as
 * (M, N, K, alpha, A, B, beta, C) with the leading dimensions implied by the
 * shapes; this ABI adds explicit leading dimensions and a stream.
 *
 * Conventions shared by every entry point
 *   - Pointers A, B, C are DEVICE pointers owned by the caller, 4-byte
 *     aligned.  Unless stated otherwise a call only enqueues work on `stream`
 *     (0 = legacy default stream) and returns; it neither synchronises nor
 *     allocates device memory.
 *   - Quick returns (BLAS conventions; the pages do not discuss them):
 *       M == 0 or N == 0       -> nothing is done, SUCCESS.
 *       K == 0 or alpha == 0   -> C = beta * C; A and B are not read.
 *       beta == 0              -> C is write-only: NaN/Inf already in C never
 *                                 reach the result.
 *     Entries of C beyond column N (the ldc padding) are never touched.
 *   - Results are rounded FP32 sums of FP32 products; the summation order over
 *     k is fixed for a given shape, so repeated calls give identical bits.
 *   - Errors are returned, never printed or raised; see sgemmStatus_t.
 *   - Thread safety: a handle may be used from one host thread at a time.
 *     Calls on one handle share its workspace and its device control block
 *     (stream-K flags), so calls on one handle must not run concurrently on
 *     the GPU: order them on one stream, or use one handle per stream.
 *   - Main kernels are launched with programmatic stream serialisation:
 *     they may be placed on SMs while the previous kernel in the stream
 *     finishes, and wait for it before touching any memory.
 *   - CUDA graphs: sgemmEx(), sgemm() and sgemmStridedBatched() enqueue only
 *     kernels on `stream`, so they can be captured, provided the workspace
 *     they need is attached and the same shape was run once before the
 *     capture (the first call of a kernel variant sets its attributes).
 *     Replays stay correct: the stream-K flags carry a launch tag kept in
 *     device memory, fresh for every launch.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef __CUDA_RUNTIME_API_H__
typedef struct CUstream_st *cudaStream_t;
typedef struct CUevent_st *cudaEvent_t;
#endif

typedef enum sgemmStatus {
    SGEMM_STATUS_SUCCESS = 0,
    SGEMM_STATUS_INVALID_VALUE = 1,      /* bad size, leading dimension, NULL pointer or handle */
    SGEMM_STATUS_MISALIGNED = 2,         /* A, B or C not 4-byte aligned */
    SGEMM_STATUS_ARCH_MISMATCH = 3,      /* current device is not compute capability 10.3 */
    SGEMM_STATUS_WORKSPACE_REQUIRED = 4, /* operands need packing and no (or too small a) workspace is set */
    SGEMM_STATUS_LAUNCH_FAILED = 5,      /* a CUDA call or kernel launch failed */
    SGEMM_STATUS_DEVICE_TIMEOUT = 6,     /* a kernel's bounded wait expired (sgemmGetDeviceError) */
    SGEMM_STATUS_NOT_SUPPORTED = 7,      /* sizes beyond what the kernels address (see sgemmEx) */
    SGEMM_STATUS_INTERNAL_ERROR = 8
} sgemmStatus_t;

typedef struct sgemmContext *sgemmHandle_t;

/* Operand form for sgemmStridedBatched: the operand as stored (N) or its
 * transpose (T), both row major. */
typedef enum sgemmOperation {
    SGEMM_OP_N = 0,
    SGEMM_OP_T = 1
} sgemmOperation_t;

/* Human-readable name of a status code (static storage, never NULL). */
const char *sgemmGetStatusString(sgemmStatus_t status);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
sgemmStatus_t sgemmGetVersion(int *version);

/*
 * Create a handle bound to the CURRENT device.  Checks that the device is
 * compute capability 10.3 (ARCH_MISMATCH otherwise), reads its SM count,
 * creates the two copy streams and the events of sgemmHostEx, and allocates
 * the handle's 32 KiB device control block (the error word, and the flags
 * and launch sequence through which stream-K CTAs hand over partial tiles):
 * the only device allocation the library makes, done here and never on the
 * compute path.
 */
sgemmStatus_t sgemmCreate(sgemmHandle_t *handle);

/* Release a handle (synchronises its device first).  NULL is a no-op. */
sgemmStatus_t sgemmDestroy(sgemmHandle_t handle);

/*
 * Per-device default handle used by sgemm(); created on first use for the
 * current device and kept until process exit.  Callers may attach a
 * workspace to it with sgemmSetWorkspace().
 */
sgemmStatus_t sgemmGetDefaultHandle(sgemmHandle_t *handle);

/*
 * Bytes of device workspace sgemmEx() can use for these operands, under the
 * handle's current math mode and schedule:
 *   - room to repack A and/or B when an operand cannot be read in place (base
 *     not 16-byte aligned or row pitch not a multiple of 16 bytes) into rows
 *     padded to a multiple of 4 floats: REQUIRED for such operands;
 *   - math mode 1 (3xTF32): the TF32 hi / lo parts of A and B: REQUIRED;
 *   - stream-K scratch (one BM x BN FP32 partial tile per CTA of the
 *     launch) when the output tiles do not divide evenly over the SMs or are
 *     too few to fill them (their K ranges are then split):
 *     OPTIONAL; with less workspace the call runs whole tiles per CTA instead
 *     (same result up to summation order, less even load);
 *   - skinny products (M or N <= 32): the partial sums of their K splits:
 *     OPTIONAL; without them the main kernel runs.
 * Same validation as sgemmEx().  Calls that share a workspace must be
 * ordered on one stream.
 */
sgemmStatus_t sgemmGetWorkspaceSize(sgemmHandle_t handle, int64_t M, int64_t N,
                                    int64_t K, const float *A, int64_t lda,
                                    const float *B, int64_t ldb, size_t *bytes);

/*
 * Attach caller-owned device memory (256-byte aligned, `bytes` long) as the
 * handle's workspace; ptr == NULL detaches.  The library reads and writes it
 * during calls enqueued afterwards; the caller must keep it alive until that
 * work has finished.
 */
sgemmStatus_t sgemmSetWorkspace(sgemmHandle_t handle, void *ptr, size_t bytes);

/*
 * C = alpha * A . B + beta * C on `stream`, using `handle`'s device,
 * workspace and error word.  A, B, C: device pointers, row major, leading
 * dimensions as above.  Returns INVALID_VALUE for negative sizes, leading
 * dimensions below the minimum, a NULL pointer with nonzero extent, or a
 * NULL handle; MISALIGNED for pointers that are not 4-byte aligned;
 * NOT_SUPPORTED for M, N or K >= 2^31 or an operand span of 2^40 bytes or
 * more; WORKSPACE_REQUIRED when packing is needed (see
 * sgemmGetWorkspaceSize) and the attached workspace is missing or too small;
 * LAUNCH_FAILED if a launch is rejected.  Operands may not overlap C.
 */
sgemmStatus_t sgemmEx(sgemmHandle_t handle, int64_t M, int64_t N, int64_t K,
                      float alpha, const float *A, int64_t lda, const float *B,
                      int64_t ldb, float beta, float *C, int64_t ldc,
                      cudaStream_t stream);

/* sgemmEx() with the current device's default handle. */
sgemmStatus_t sgemm(int64_t M, int64_t N, int64_t K, float alpha,
                    const float *A, int64_t lda, const float *B, int64_t ldb,
                    float beta, float *C, int64_t ldc, cudaStream_t stream);

/*
 * Strided-batched product with optional transposed operands:
 *
 *   C_z = alpha * op(A_z) . op(B_z) + beta * C_z,   z = 0 .. batchCount-1
 *
 * all matrices ROW MAJOR.  op(A) is M x K: opA == SGEMM_OP_N reads A stored
 * M x K (lda >= K), SGEMM_OP_T reads A stored K x M (lda >= M) as its
 * transpose.  op(B) is K x N: opB == SGEMM_OP_N reads B stored K x N
 * (ldb >= N), SGEMM_OP_T reads B stored N x K (ldb >= K).  C_z is M x N
 * (ldc >= N).  Matrix z of an operand starts at base + z * stride (elements;
 * strides >= 0, a zero stride reuses one matrix for every z).  The C
 * matrices of different z must not overlap.  batchCount == 0 is a no-op.
 * With (N, N, batchCount 1) this is sgemmEx().
 *
 * FFMA path: operands given transposed, or whose base, row pitch or batch
 * stride TMA cannot address (16-byte multiples), are first copied into the
 * workspace in M x K / K x N row-major form; all output tiles of all batch
 * entries share one persistent grid (and one stream-K split).  3xTF32 path
 * (sgemmSetMathMode 1): the split pre-pass reads either form directly.
 * Workspace needs: sgemmStridedBatchedWorkspaceSize().  Errors as for
 * sgemmEx(); INVALID_VALUE also for an unknown op, a negative batchCount or
 * stride; NOT_SUPPORTED when batchCount * output tiles reaches 2^31.
 * These forms are not on the pages (which fix row-major NN); the transposed
 * forms follow the BLAS convention that "Matmul I" cites for cuBLAS.
 */
sgemmStatus_t sgemmStridedBatched(sgemmHandle_t handle, sgemmOperation_t opA,
                                  sgemmOperation_t opB, int64_t M, int64_t N,
                                  int64_t K, float alpha, const float *A,
                                  int64_t lda, int64_t strideA, const float *B,
                                  int64_t ldb, int64_t strideB, float beta,
                                  float *C, int64_t ldc, int64_t strideC,
                                  int64_t batchCount, cudaStream_t stream);

/* Workspace sgemmStridedBatched() can use for these operands (same meaning
 * as sgemmGetWorkspaceSize(): repacking is required, stream-K scratch
 * optional, the 3xTF32 split parts required in math mode 1). */
sgemmStatus_t sgemmStridedBatchedWorkspaceSize(
    sgemmHandle_t handle, sgemmOperation_t opA, sgemmOperation_t opB, int64_t M,
    int64_t N, int64_t K, const float *A, int64_t lda, int64_t strideA,
    const float *B, int64_t ldb, int64_t strideB, int64_t batchCount,
    size_t *bytes);

/*
 * Bytes of device workspace sgemmHostEx() needs: device copies of A, B and C
 * with rows padded to a multiple of 4 floats.
 */
sgemmStatus_t sgemmHostWorkspaceSize(int64_t M, int64_t N, int64_t K,
                                     size_t *bytes);

/*
 * The same product with A, B and C in HOST memory (pinned memory gives full
 * copy bandwidth; pageable memory works but is staged by the driver).  The
 * operands are copied into `dev_workspace` (device memory of at least
 * sgemmHostWorkspaceSize() bytes, owned by the caller), the product runs
 * there, and the M x N result is copied back into C.  The copies overlap the
 * arithmetic: C is computed in pieces (a first block of 1024 rows cut into
 * up to four column pieces when M is at least 2048, then up to three row
 * blocks, the last at most 512 rows high), each
 * multiplied on `stream` as soon as its parts of A and B are up, while the
 * next parts are copied in and finished pieces copied out (on two streams
 * the handle owns).  The call returns before
 * the work finishes; everything it enqueued is ordered before later work on
 * `stream`, so synchronising `stream` makes C valid, and the host buffers
 * must stay untouched until then.  C is read (copied up) only when
 * beta != 0.  The multiplication itself uses the handle's own workspace as
 * sgemmEx() does (3xTF32 operand splits, stream-K scratch): its size is
 * sgemmGetWorkspaceSize() for 256-byte aligned A and B with
 * lda = K and ldb = N rounded up to multiples of 4; WORKSPACE_REQUIRED when
 * a required part is missing.
 */
sgemmStatus_t sgemmHostEx(sgemmHandle_t handle, int64_t M, int64_t N, int64_t K,
                          float alpha, const float *A_host, int64_t lda,
                          const float *B_host, int64_t ldb, float beta,
                          float *C_host, int64_t ldc, void *dev_workspace,
                          size_t workspace_bytes, cudaStream_t stream);

/*
 * Description of what sgemmEx() would launch for these arguments (no work
 * is enqueued): the number of kernel launches, the output tile (BM x BN),
 * the number of CTAs of the main kernel and whether operands are repacked.
 */
typedef struct sgemmPlan {
    int launches;       /* kernels one call enqueues (0 for M == 0 or N == 0); repacks of A and
                           B and the edge columns share one preparation launch */
    int tile_m, tile_n; /* output tile of the main kernel (0 if none) */
    int tile_k;         /* K slice staged per pipeline step */
    int stages;         /* shared-memory pipeline depth (kind 4: 6 when the TMA-fed
                           streaming kernels run, 0 for the plain-load ones) */
    int ctas;           /* CTAs of the main kernel (persistent grid) */
    int packs_a, packs_b; /* 1 if the operand is repacked into the workspace */
    int vector_epilogue;  /* 1 if C is written with 16-byte stores */
    int kind;           /* 0 none, 1 FFMA main kernel, 2 scale-only (K == 0 or alpha == 0),
                           3 3xTF32 tensor-core kernel (after the split pre-pass),
                           4 skinny streaming kernel + split reduction (M or N <= 32),
                           5 small-product kernel: one CTA (or a cluster of up to 8
                           sharing K) per 32 x 32 block of C, for matrices of at most
                           1024 rows and columns, K <= 8192 and at most 2^27
                           multiply-adds in the call (2^28 while the blocks fill at
                           most two CTAs per SM; any number for matrices of at most
                           64 x 64; FFMA, automatic tile choice only) */
    int stream_k;       /* 1 if K slices of some tiles are split between CTAs (stream-K) */
    int raster_group;   /* tile rows per band of the tile order (tiles running together
                           share rows of A and columns of B in L2); 0 if no tiles */
    int edge_cols;      /* kind 1: the last edge_cols (<= 8) columns of C are computed in the
                           preparation launch (a warp per row) instead of by a last tile column
                           that thin; the main kernel covers whole tiles.  Only in the automatic
                           setting, for NN products of one matrix with M * K >= 2^21 */
} sgemmPlan_t;

sgemmStatus_t sgemmQueryPlan(sgemmHandle_t handle, int64_t M, int64_t N,
                             int64_t K, float alpha, const float *A,
                             int64_t lda, const float *B, int64_t ldb,
                             float beta, const float *C, int64_t ldc,
                             sgemmPlan_t *plan);

/*
 * Pin the main kernel's tile configuration for calls on this handle:
 * 0 = automatic choice by shape (default: 10 when both sides are at most
 * 128, 18 / 19 for large products of 17 to 32 rows / columns, 16 for at
 * most 64 rows, 17 for at most 64 columns; otherwise the tile shape with
 * the least padded area per element of C over its relative speed (256 x 128
 * and 128 x 256: 1, 128 x 128 of configuration 10: 0.88, not for the short
 * K below), a tie between the first two going to 128 x 256 under 256 rows
 * or for products more than twice as wide as tall; then, when beta == 0 and
 * C is 16-byte aligned or when C is not 16-byte aligned (C through a
 * shared-memory staging area), 27 for 128 x 256, 23 / 24 for K of at most
 * 64 that is a multiple of 16 / not a multiple of 16 (multiples of 32
 * excepted), else 28; otherwise 30 for 128 x 256, 20 / 21 for K of at most
 * 64 that is not a multiple of 32, else 29).  Fixed configurations (every one
 * but 10 is eight warps in one CTA per SM; fp32_sgemm_gb300/csrc/
 * sgemm_algo*.cu):
 *   10 = 128 x 128, four warps, two CTAs per SM;
 *   16 = 64 x 512, 17 = 512 x 64, 18 = 32 x 1024, 19 = 1024 x 32;
 *   20 / 21 = 256 x 128 with K slices of 16 / 8 (6 / 8 stages);
 *   23 / 24 = 256 x 128 with K slices of 16 / 8 (4 / 8 stages) and C
 *   through shared memory;
 *   27 / 28 = 128 x 256 / 256 x 128, K slices of 32, 2 stages, C through
 *   shared memory (by TMA when beta == 0 and C is 16-byte aligned, in row
 *   runs of plain stores when C is not 16-byte aligned);
 *   29 / 30 = 256 x 128 / 128 x 256, K slices of 32, 4 stages, C from
 *   registers.
 * Other numbers up to 30 (configurations measured slower and no longer
 * built) return INVALID_VALUE, here or, for 1..4 set in math mode 0, from
 * the product call.  In math mode 1
 * (3xTF32) the values 1..4 pick the tensor-core tile instead: 128 x 128,
 * 128 x 192 or 128 x 256 on one SM, or 256 x 256 on an SM pair (a cluster
 * of two CTAs sharing each MMA).  Every configuration computes the same
 * result up to summation order.
 */
sgemmStatus_t sgemmSetAlgo(sgemmHandle_t handle, int algo);

/*
 * Arithmetic of the main kernel for calls on this handle:
 * 0 = FP32 FFMA on the CUDA cores (default): every product and sum in FP32.
 * 1 = error-compensated 3xTF32 on the 5th-generation tensor cores
 *     (tcgen05): each operand is split into a TF32 part and a TF32 residual
 *     (x = hi + lo: hi is x with its low 13 mantissa bits dropped, which is
 *     what the tensor core reads of an FP32 operand, lo = x - hi rounded to
 *     nearest TF32) and C = alpha * (A_hi.B_hi + A_hi.B_lo + A_lo.B_hi) +
 *     beta * C with FP32 accumulation.  The omitted A_lo.B_lo term and the
 *     rounding of lo bound the extra relative error per product near 2^-21;
 *     integer-valued inputs of magnitude < 2^11 give bit-exact results.
 *     Needs a workspace of 2 * (M + N) * round_up(K, 32) floats (rounded
 *     up to 256 bytes per part; B stored N x K or K x N alike) for the
 *     split operands, plus the stream-K partial tiles when they are used
 *     (sgemmGetWorkspaceSize gives the exact figure); the split runs as two
 *     extra kernels before the product (an operand of at most 64 MB stored
 *     K contiguous, 16-byte aligned, is read in place as its own high part
 *     and only its residual is written).
 * The pages treat TF32 only as a different contest; the splitting follows
 * Ootomo & Yokota, "Recovering single precision accuracy from Tensor Cores
 * while surpassing the FP32 theoretical peak performance" (2022).
 */
sgemmStatus_t sgemmSetMathMode(sgemmHandle_t handle, int mode);

/*
 * How output tiles are shared among the persistent CTAs of the main kernel:
 * 0 = automatic (default): stream-K when whole tiles would leave the SMs
 *     unevenly loaded and the workspace has room for its scratch;
 * 1 = whole tiles only, round robin;
 * 2 = stream-K whenever the workspace has room (every CTA gets the same
 *     number of (tile, K slice) units; tiles cut between CTAs are summed in
 *     a fixed order, so results stay deterministic).
 */
sgemmStatus_t sgemmSetSchedule(sgemmHandle_t handle, int schedule);

/*
 * Measurement hook: when both events are non-NULL, every later call on this
 * handle records `start` on its stream immediately before the main kernel
 * launch and `stop` immediately after it (the repack, split and flag-reset
 * work of the call falls outside), so cudaEventElapsedTime gives the main
 * kernel's own duration.  The events are the caller's (created, and kept
 * alive while calls may record them); NULL, NULL turns the hook off.  One
 * of the two NULL is INVALID_VALUE.  The pages time whole programs with
 * nvbench or averaged repetitions (easonhuang.dev "Results"; the HuajingLin
 * wiki's benchmark table); this hook times the main kernel alone through the
 * C ABI.
 */
sgemmStatus_t sgemmSetKernelEvents(sgemmHandle_t handle, cudaEvent_t start,
                                   cudaEvent_t stop);

/*
 * Limit, in nanoseconds, on every wait a kernel of this handle performs
 * (default 2e9, minimum 1e6).  A wait that runs out records an error in the
 * handle's error word and lets the kernel return instead of hanging.
 */
sgemmStatus_t sgemmSetWaitTimeout(sgemmHandle_t handle, uint64_t timeout_ns);


/*
 * Synchronise the handle's device, read and clear its error word.  *code is
 * 0 when no kernel recorded an error; otherwise the return value is
 * DEVICE_TIMEOUT and *code holds the raw word of the FIRST expiry since the
 * last read: bits 24..31 say which wait expired (1 a consumer's wait for
 * operand data, 2 the TMA issuer's wait for a free pipeline stage, 3 the
 * self test, 4 the wait for another CTA's stream-K partial tile, 5 the
 * consumer warps' rendezvous around that exchange), bits 0..23 the CTA
 * index.  A call during which a wait expired has left C undefined.
 */
sgemmStatus_t sgemmGetDeviceError(sgemmHandle_t handle, int *code);

/*
 * TEST HOOK for failure detection, not for production use: calls on this
 * handle leave out one signal inside the kernels on purpose, so that the
 * bounded wait for it runs out and its give-up path runs (record the site
 * in the error word, let the CTA's own copies land, free tensor memory,
 * return); no kernel faults or hangs.  The C these calls write is
 * undefined.  `which`:
 *   0 = none (default);
 *   1 = CTAs holding a stream-K partial tile never announce it (site 4
 *       expires, in both math modes, on launches that use stream-K);
 *   2 = the TMA issuer stops after filling the pipeline once (site 1
 *       expires, on launches whose CTAs take more K slices than stages);
 *   3 = consumers never release a pipeline stage (site 2 expires, same
 *       launches).
 * Only the main kernels (FFMA and 3xTF32) honour it.  Use a short limit
 * (sgemmSetWaitTimeout) so that the expiries come quickly.  INVALID_VALUE
 * for other values or a NULL handle.
 */
sgemmStatus_t sgemmSetTestWithheldSignal(sgemmHandle_t handle, int which);

/*
 * Health check of the bounded-wait machinery: enqueue one single-CTA kernel
 * that waits on a shared-memory barrier no one ever arrives on, with limit
 * timeout_ns.  The wait must run out and record code 3 in the error word;
 * the kernel then returns normally, so the context stays usable.
 */
sgemmStatus_t sgemmSelfTestWaitTimeout(sgemmHandle_t handle,
                                       uint64_t timeout_ns,
                                       cudaStream_t stream);

/*
 * sgemmNoAlloc: the same product as sgemm(), for callers that cannot
 * allocate device memory at all -- code running where the allocator is off
 * limits (inside an allocator hook or memory pool, under a framework that
 * owns all device memory, or with a device-memory budget fixed up front).
 * The paper (the SGEMM pages this library follows) has no counterpart of it.
 *
 * It calls no cudaMalloc, cudaFree or allocating library routine.  Its
 * scratch (error word, stream-K flags and partial tiles, repacked operands)
 * lives in one file-scope device array of SGEMM_NOALLOC_SCRATCH_BYTES
 * (32 MiB) that every GPU loading this library holds until process exit.
 * The caller passes A, B and C as for sgemm().
 *   - The first call on a device does one-time set-up on the current device:
 *     it checks the architecture, reads the SM count, looks up the array's
 *     device address (which loads the library module holding the array and
 *     so commits its 32 MiB), and loads every kernel this entry point can
 *     launch, with each one's shared-memory opt-in and occupancy, so that
 *     no later call loads code or commits memory.  Make that first call
 *     before any stream capture and outside any allocator hook.
 *   - Every call shares the one array per device and the array keeps the
 *     last call's contents; the stream-K partial-tile flags carry a tag per
 *     launch, kept in the array's control block (zero when the module
 *     loads), so nothing is cleared between calls.  Calls whose work overlaps
 *     on the GPU (different streams, or different host threads without
 *     ordering) race on the array: order them on one stream.
 *   - Operands that need repacking (base not 16-byte aligned or row pitch not
 *     a multiple of 4 floats) must fit in the array: M * round_up(K, 4) and
 *     K * round_up(N, 4) floats together at most 32 MiB minus 32 KiB (the
 *     array's first 32 KiB are the control block a handle has of its own);
 *     larger ones return SGEMM_STATUS_NOT_SUPPORTED before anything is
 *     enqueued.  Stream-K is used only when its scratch fits as well.
 *   - Every wait inside these kernels is bounded (2 s by default, see
 *     sgemmNoAllocSetWaitTimeout); an expiry is recorded in the array's own
 *     error word, which sgemmNoAllocGetDeviceError reads and clears.
 * Other status codes as for sgemm().
 */
#define SGEMM_NOALLOC_SCRATCH_BYTES (32u << 20)
sgemmStatus_t sgemmNoAlloc(int64_t M, int64_t N, int64_t K, float alpha,
                           const float *A, int64_t lda, const float *B,
                           int64_t ldb, float beta, float *C, int64_t ldc,
                           cudaStream_t stream);

/*
 * Synchronise the CURRENT device, then read and clear the error word that
 * sgemmNoAlloc's kernels on this device record bounded-wait expiries in
 * (the first expiry since the last read is kept).  *code and the return
 * value as for sgemmGetDeviceError(): 0 and SUCCESS when nothing expired
 * (also before the first sgemmNoAlloc call on the device, which is then
 * not touched), otherwise the raw word and DEVICE_TIMEOUT.  Allocates
 * nothing.  Like sgemmNoAlloc, the pages have no counterpart of it.
 */
sgemmStatus_t sgemmNoAllocGetDeviceError(int *code);

/*
 * Wait limit, in nanoseconds, of sgemmNoAlloc's kernels on the CURRENT
 * device (default 2e9, minimum 1e6; INVALID_VALUE below).  Host setting
 * only: nothing is enqueued or allocated.
 */
sgemmStatus_t sgemmNoAllocSetWaitTimeout(uint64_t timeout_ns);

/*
 * sgemmSetTestWithheldSignal() for sgemmNoAlloc's calls on the CURRENT
 * device (same values and meaning; TEST HOOK, not for production use).
 */
sgemmStatus_t sgemmNoAllocSetTestWithheldSignal(int which);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
