// C ABI of the GB300 FP32 SGEMM library (declared in include/sgemm_gb300.h).
//
// Host side of the hot path: argument validation, BLAS quick returns, the
// choice between reading A/B in place through TMA or repacking them into the
// caller's workspace first, tensor-map encoding, tile-configuration choice
// and the persistent launch.  The launch shape follows the pages' host
// launcher (a grid of output tiles, one kernel instantiation per beta == 0 /
// beta != 0; "The Final Kernel", maxxfuu article4/page14, launch_sgemm_final),
// made persistent: at most one CTA per SM slot, tiles taken round robin.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/sgemm_gb300.h"
#include "kernel_table.h"

namespace {

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr uint64_t kMinTimeoutNs = 1000000ull;
// Device control block: error word and stream-K sequence in the first 256
// bytes, then one flag word per CTA and warp of a stream-K launch (up to
// 1016 CTAs of 8 warps: more than two CTAs on every SM of the part).
constexpr size_t kCtlBytes = 32768;
constexpr int kCtlFlagsOffset = 64;                         // words
constexpr int kCtlFlagWords = int(kCtlBytes / 4) - kCtlFlagsOffset;

using sg::KernelEntry;
using sg::kMaxDevices;
using sg::kNumAlgos;

KernelEntry g_kernels[kNumAlgos][4];
std::once_flag g_kernels_once;
std::mutex g_occ_mutex;

void init_kernel_table() {
    sg::fill_algo10(g_kernels[9]);
    sg::fill_algo16(g_kernels[15]);
    sg::fill_algo17(g_kernels[16]);
    sg::fill_algo18(g_kernels[17]);
    sg::fill_algo19(g_kernels[18]);
    sg::fill_algo20(g_kernels[19]);
    sg::fill_algo21(g_kernels[20]);
    sg::fill_algo23(g_kernels[22]);
    sg::fill_algo24(g_kernels[23]);
    sg::fill_algo27(g_kernels[26]);
    sg::fill_algo28(g_kernels[27]);
    sg::fill_algo29(g_kernels[28]);
    sg::fill_algo30(g_kernels[29]);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

}  // namespace

struct sgemmContext {
    int device = -1;
    int sm_count = 0;
    // Device control block (allocated with the handle): word 0 the error
    // word, words 1-2 the stream-K launch sequence {tag, CTAs finished},
    // from word kCtlFlagsOffset the stream-K flags (kCtlFlagWords words: one
    // per CTA and warp of a launch).
    uint32_t *d_err = nullptr;
    uint32_t *d_flags = nullptr;
    uint32_t *d_sk_seq = nullptr;
    int flag_words = 0;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    uint64_t timeout_ns = kDefaultTimeoutNs;
    int algo = 0;
    int schedule = 0;   // 0 automatic, 1 whole tiles only, 2 stream-K whenever it applies
    int math = 0;       // 0 FP32 FFMA, 1 error-compensated 3xTF32 on the tensor cores
    int withhold = 0;   // test hook: signal the kernels leave out (sg::Withhold)
    cudaEvent_t ev_start = nullptr, ev_stop = nullptr;   // around the main kernel, if set
    // sgemmHostEx pipeline: copy-in and copy-out streams and their events,
    // created with the handle.
    static constexpr int kHostChunks = 8;     // pieces of one sgemmHostEx call (at most 7)
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_begin = nullptr, ev_end = nullptr;
    cudaEvent_t ev_in[kHostChunks] = {}, ev_done[kHostChunks] = {};
};

namespace {

sgemmHandle_t g_default[kMaxDevices] = {};
std::mutex g_default_mutex;

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
inline int64_t ceil_div(int64_t x, int64_t a) { return (x + a - 1) / a; }

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
constexpr int64_t kMaxBytes = int64_t(1) << 40;

// One call in its general form: C_z = alpha * op(A_z) . op(B_z) + beta * C_z
// for z < batch, every matrix row major; op(A) is M x K (opA == N: A stored
// M x K; opA == T: A stored K x M), op(B) is K x N (opB == N: B stored
// K x N; opB == T: B stored N x K); matrix z of an operand starts at
// base + z * stride (elements).
struct Problem {
    int opA = 0, opB = 0;
    int64_t M = 0, N = 0, K = 0;
    float alpha = 1.f, beta = 0.f;
    const float *A = nullptr;
    int64_t lda = 0, sa = 0;
    const float *B = nullptr;
    int64_t ldb = 0, sb = 0;
    float *C = nullptr;
    int64_t ldc = 0, sc = 0;
    int64_t batch = 1;

    int64_t a_cols() const { return opA ? M : K; }   // stored A: columns
    int64_t b_cols() const { return opB ? K : N; }   // stored B: columns
    bool empty() const { return M == 0 || N == 0 || batch == 0; }
};

Problem nn_problem(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                   const float *B, int64_t ldb, float beta, const float *C, int64_t ldc) {
    Problem q;
    q.M = M; q.N = N; q.K = K;
    q.alpha = alpha; q.beta = beta;
    q.A = A; q.lda = lda;
    q.B = B; q.ldb = ldb;
    q.C = const_cast<float *>(C); q.ldc = ldc;
    return q;
}

// Validation shared by every entry point.  Pure host logic: no CUDA calls.
sgemmStatus_t validate(const Problem &q, bool need_c = true) {
    if (q.opA < 0 || q.opA > 1 || q.opB < 0 || q.opB > 1) return SGEMM_STATUS_INVALID_VALUE;
    if (q.M < 0 || q.N < 0 || q.K < 0 || q.batch < 0) return SGEMM_STATUS_INVALID_VALUE;
    if (q.sa < 0 || q.sb < 0 || q.sc < 0) return SGEMM_STATUS_INVALID_VALUE;
    if (q.lda < std::max<int64_t>(1, q.a_cols()) || q.ldb < std::max<int64_t>(1, q.b_cols()) ||
        q.ldc < std::max<int64_t>(1, q.N))
        return SGEMM_STATUS_INVALID_VALUE;
    if (q.empty()) return SGEMM_STATUS_SUCCESS;
    const bool need_ab = q.alpha != 0.0f && q.K > 0;
    if (need_c && q.C == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    if (need_ab && (q.A == nullptr || q.B == nullptr)) return SGEMM_STATUS_INVALID_VALUE;
    if (need_c && !aligned(q.C, 4)) return SGEMM_STATUS_MISALIGNED;
    if (need_ab && (!aligned(q.A, 4) || !aligned(q.B, 4))) return SGEMM_STATUS_MISALIGNED;
    if (q.M > kMaxDim || q.N > kMaxDim || q.K > kMaxDim || q.batch > kMaxDim)
        return SGEMM_STATUS_NOT_SUPPORTED;
    if (q.lda > kMaxBytes / 4 || q.ldb > kMaxBytes / 4 || q.ldc > kMaxBytes / 4 ||
        q.sa > kMaxBytes / 4 || q.sb > kMaxBytes / 4 || q.sc > kMaxBytes / 4)
        return SGEMM_STATUS_NOT_SUPPORTED;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t validate(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                       const void *B, int64_t ldb, const void *C, int64_t ldc, bool need_ab) {
    Problem q = nn_problem(M, N, K, need_ab ? 1.f : 0.f, static_cast<const float *>(A), lda,
                           static_cast<const float *>(B), ldb, 0.f, static_cast<const float *>(C), ldc);
    return validate(q);
}

inline bool tma_ok(const void *p, int64_t ld) { return aligned(p, 16) && (ld % 4) == 0; }
// Operand readable in place by 3-D TMA: base 16-byte aligned, row pitch and
// (for a real batch) batch stride multiples of 16 bytes.
inline bool tma_ok_batched(const void *p, int64_t ld, int64_t stride, int64_t batch) {
    return tma_ok(p, ld) && (batch == 1 || (stride % 4 == 0 && stride > 0));
}

// The TMA-fed skinny kernels read A and B in place: both 16-byte aligned
// with row pitches of whole 16-byte units; below a 256-wide large dimension
// or K < 16 the plain-load kernels serve.
inline bool skinny_tma_eligible(const Problem &q, bool small_m) {
    return tma_ok(q.A, q.lda) && tma_ok(q.B, q.ldb) && q.K >= 16 && (small_m ? q.N : q.M) >= 256;
}

struct Plan {
    sgemmPlan_t pub{};
    int algo_index = -1;   // row of g_kernels
    int variant = 0;       // column of g_kernels
    // FFMA path: how each operand reaches TMA (0 in place, 1 repacked rows,
    // 2 transposed into the workspace) and its pitch / batch stride there.
    int prep_a = 0, prep_b = 0;
    int64_t lda_p = 0, ldb_p = 0, sa_p = 0, sb_p = 0;
    size_t ws_a = 0, ws_b = 0;      // repacked A / B
    size_t ws_partials = 0;         // stream-K partial tiles (0 when not used)
    int tiles_m = 0, tiles_n = 0, num_tiles = 0, group_m = 16;
    int k_blocks = 0;
    int dp_ctas = 0, sk_ctas = 0;   // persistent grid for whole tiles / stream-K
    int sk_tile0 = 0;               // first tile of the stream-K part
    int64_t kp = 0;                 // 3xTF32: row pitch of the split operands
    size_t ws_split_a = 0, ws_split_b = 0;   // 3xTF32: bytes of one part (hi or lo)
    size_t ws_split = 0;            // 3xTF32: A_hi, A_lo, B_hi^T, B_lo^T
    int tf32_cfg = 0;               // 3xTF32: tile configuration (1-based)
    // Skinny path (kind 4): which side is small, K splits, partial sums.
    bool skinny_m = false;
    int skinny_split = 0;
    size_t ws_skinny = 0;
    bool skinny_tma = false;        // TMA-fed skinny kernels (operands read in place)
    sg::SkinnyTmaGeom skinny_geom;
    int small_splits = 1;           // small-product kernel (kind 5): CTAs per block of C
    // FFMA path: columns [n_main, N) of C are computed by the edge job of
    // the preparation launch instead of a last tile column that thin.
    int64_t n_main = 0;
    int edge_cols = 0;
};

// Configuration 29 (256 x 128 tile, eight consumer warps, one CTA per SM,
// BK = 32, 4 stages, TMA issued by a compute thread, 16-byte A reads (four
// k per read) double buffered one k ahead, each k's B read just before its
// FMAs) measured fastest from 1024^3 to 8192^3 where C is 16-byte aligned
// and read (beta != 0); otherwise configuration 28 (the same tile and loop,
// a 2-stage ring, C through a shared-memory staging area: TMA stores when
// beta == 0 and C is aligned, else row runs).  Their loop beat the earlier
// one (8-byte A and 16-byte B reads both double buffered, since removed) by
// 1-2% (4096^3: 2160 -> 2134 us; 8192^3: 17293 -> 17023 us; beta = 0.5:
// 2197 -> 2148 us).
constexpr int kDefaultAlgo = 29;     // beta != 0, C 16-byte aligned
constexpr int kStoreTmaAlgo = 28;    // beta == 0 or C not 16-byte aligned
constexpr int kWideStoreTmaAlgo = 27;   // the same, 128 x 256, for wide products
constexpr int kWideAlgo = 30;           // 128 x 256 reading C from registers

// 17 to 32 rows (columns), large enough to give every SM at least 8 K slices
// of 32 x 1024 (1024 x 32) tiles: there the FFMA kernel with those tiles runs
// at ~70% of the FMA peak and the streaming kernel's 32-row variant at ~50%
// (measured at 16384-long K and N: 310 vs 408-416 us).  Smaller products
// stay on the streaming kernel, which spreads them over every SM.
bool thin_ffma_preferred(const sgemmContext *h, const Problem &q) {
    if (h->algo != 0 || h->math != 0) return false;
    const int64_t small = std::min(q.M, q.N), big = std::max(q.M, q.N);
    if (small <= 16 || small > 32) return false;
    return ceil_div(big, 1024) * ceil_div(q.K, 16) >= 8 * int64_t(h->sm_count);
}

// Small products take the 32 x 32 block kernel (one CTA, or a cluster of
// CTAs sharing K, per block; no persistent grid, no TMA, no stream-K
// exchange): matrices of at most kSmallMaxDim rows and columns, K at most
// kSmallMaxK, and at most 2^27 multiply-adds in the call (2^28 while the
// blocks fill at most two CTAs per SM; any number for matrices of at most
// 64 x 64, e.g. 1000 x 64^3: 61.1 -> 28.2 us).  There the tile kernel is bound by
// its start-up latency and leaves SMs idle; measured per call (CUDA graph
// replay): 128^3 16.4 -> 4.6 us, 256^3 20.5 -> 5.4, 512^3 36.9 -> 19.6,
// 128 x 128 x 8192 81.9 -> 41.7, 1000 x 64^3 61.3 -> 28.2; beyond, e.g.
// 128 x 128^3 (2^28) 22.7 vs 27.4 us, the tile kernel wins.  Only in the
// automatic FFMA setting (a pinned tile configuration or schedule, or math
// mode 1, keeps the kernel asked for).
// Edge columns are split off only when M x K is at least this (below, the
// saved padding is worth less than the work of the edge job).
constexpr double kEdgeMinMK = double(1 << 21);

constexpr int64_t kSmallMaxDim = 1024;
constexpr int64_t kSmallMaxK = 8192;
constexpr int64_t kSmallMaxWork = int64_t(1) << 27;   // batch x M x N x K multiply-adds

bool small_preferred(const sgemmContext *h, const Problem &q) {
    if (h->algo != 0 || h->schedule != 0 || h->math != 0) return false;
    if (q.M > kSmallMaxDim || q.N > kSmallMaxDim || q.K > kSmallMaxK) return false;
    const int64_t blocks = sg::small_blocks(int(q.M), int(q.N), int(q.batch));
    if (blocks == 0) return false;
    // Matrices of at most 64 x 64 would leave 3/4 of a 128 x 128 tile idle.
    if (q.M <= 64 && q.N <= 64) return true;
    const int64_t work = q.batch * q.M * q.N * q.K;
    return work <= kSmallMaxWork || (work <= 2 * kSmallMaxWork && blocks <= 2 * int64_t(h->sm_count));
}

// Tile configuration by shape (for the main kernel; the small-product
// kernel above takes the smallest calls first).  Products with at most 64
// rows (columns) take the 64 x 512 (512 x 64) tile, which computes no
// padding rows (columns) beyond 64; 17 to 32, the 32 x 1024 (1024 x 32)
// tile.  Everything else takes 256 x 128, or 128 x 256 when the product is
// under 256 rows or more than twice as wide as tall.  All of these are one
// CTA of eight consumer warps per SM: two CTAs of four warps per SM run
// mostly one at a time (measured: the warp scheduler favours the older
// CTA, whose inline TMA issuer keeps it fed while the other CTA's ring
// starves), whereas warps of one CTA are held together by the shared ring.
// Matrices with both sides <= 128 that reach the main kernel (large
// batches of them) take the 128 x 128 tile, which wastes the least of its
// lanes.
//
// When beta == 0 and C is 16-byte aligned, the 256 x 128 and 128 x 256 tiles
// come in a form whose warps hand C to TMA stores through shared memory, so
// that C drains while the next tile computes; there the ring has only two
// stages (the staging area takes the room) and each is refilled as soon as
// every warp released it (measured at 4096^3: 2184 -> 2159 us; 16384^2 with
// K = 8 / 16 / 32 / 64: 213 / 278 / 389 / 686 -> 173 / 224 / 346 / 593 us).
// Short K takes the 16- or 8-deep slices (configurations 23, 24): the slice
// depth that divides K multiplies no zero padding.
bool c_vector_ok(const Problem &q) {
    return tma_ok(q.C, q.ldc) && (q.batch == 1 || q.sc % 4 == 0);
}

int choose_algo(const sgemmContext *h, const Problem &q) {
    if (h->algo != 0) return sg::algo_shipped(h->algo) ? h->algo - 1 : -1;
    if (q.M <= 128 && q.N <= 128) return 10 - 1;
    if (q.M <= 32 && q.M <= q.N) return 18 - 1;
    if (q.N <= 32) return 19 - 1;
    if (q.M <= 64 && q.M <= q.N) return 16 - 1;
    if (q.N <= 64) return 17 - 1;
    // Tile shape: the least padded area per element of C over the tile's
    // relative speed, 256 x 128 and 128 x 256 1.0, 128 x 128 (configuration
    // 10: four warps, two CTAs per SM) 0.88 (measured on batches: 100 x
    // 200 x 300 x 400, equal padding, 129.7 / 148.5 us; 40 x 300 x 300 x
    // 1024, padding 2.18 / 1.64: 257.2 / 215.5 us).  Between the first two,
    // equal padding goes to 128 x 256 under 256 rows or for products more
    // than twice as wide as tall.
    const int64_t tall_area = ceil_div(q.M, 256) * 256 * ceil_div(q.N, 128) * 128;
    const int64_t wide_area = ceil_div(q.M, 128) * 128 * ceil_div(q.N, 256) * 256;
    const int64_t square_area = ceil_div(q.M, 128) * 128 * ceil_div(q.N, 128) * 128;
    const bool wide = tall_area == wide_area ? (q.M < 256 || q.N > 2 * q.M) : wide_area < tall_area;
    const bool short_k = q.K <= 64 && q.K % 32 != 0;   // slices no deeper than needed (below)
    if (!short_k && double(square_area) / 0.88 < double(std::min(tall_area, wide_area))) return 10 - 1;
    // Staging-area epilogues: TMA stores (beta == 0, aligned C) or row runs
    // (C not 16-byte aligned; 4095 x 4097 x 1023 with beta = 0.25:
    // 669 -> 617 us).  Aligned C with beta != 0 keeps the register epilogue.
    if (c_vector_ok(q) ? q.beta == 0.0f : true) {
        if (wide) return kWideStoreTmaAlgo - 1;
        // Short K: the K slice that divides K (32, 16, else 8 deep).
        if (short_k) return (q.K % 16 == 0 ? 23 : 24) - 1;
        return kStoreTmaAlgo - 1;
    }
    if (wide) return kWideAlgo - 1;
    // Short K (writing C bounds the product): slices no deeper than needed,
    // so that little zero padding is multiplied (measured at 16384^2: K = 8
    // 393 -> 213 us with 8-deep slices, K = 16 393 -> 278 us with 16-deep).
    if (short_k) return (q.K % 16 == 0 || q.K > 32 ? 20 : 21) - 1;
    return kDefaultAlgo - 1;
}

// CTAs of a main-kernel configuration per SM of device `dev` (queried once
// per device, after the shared-memory opt-in); -1 if the query fails.
int occupancy_on(int dev, KernelEntry &e) {
    std::lock_guard<std::mutex> lk(g_occ_mutex);
    int &occ = e.occupancy[dev];
    if (occ == 0) {
        if (cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, e.smem) != cudaSuccess)
            return -1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, e.fn, e.threads, e.smem) != cudaSuccess || n < 1)
            return -1;
        occ = n;
    }
    return occ;
}

int occupancy_for(const sgemmContext *h, KernelEntry &e) { return occupancy_on(h->device, e); }

size_t align256(size_t x) { return (x + 255) / 256 * 256; }


// 3xTF32 plan: operands are always split into the workspace (TF32 hi and lo
// parts, K contiguous), so any layout, pitch and alignment of A and B works.
// Automatic tensor-core tile choice: the one with the least estimated time,
// waves (whole tiles per SM, rounded up) times the time of one tile, which
// grows with its width over the tensor-pipe efficiency measured at 8192^3
// (128 x 128: 0.86, shared-memory bound; 128 x 256: 0.91).  128 x 192 was
// slower than both everywhere and is only used when asked for.
// CTAs of a stream-K launch (0: none).  At least half a wave of tiles:
// every resident CTA.  Fewer: each tile's K range is cut into s pieces, s as
// large as the slots allow but at most 16 (the CTA that finishes a tile
// adds the other pieces' partial tiles one after another).
//   even_deep: with at least 6 K slices per slot and at most 16 pieces per
//   tile, spread the units evenly over every slot instead (no slot idle).
//   Measured (automatic vs even, us per call): 1024^3 52.6 / 51.3 and
//   2048 x 1024 x 512 48.1 / 46.9 (6.7 slices per slot) go even;
//   1024^2 x 768 43.1 / 44.1, 768^2 x 1024 43.1 / 45.0 and 1024^2 x 512
//   33.9 / 37.9 (3.8-5 slices per slot) keep the pieces.
int64_t stream_k_ctas(int64_t tiles, int64_t k_blocks, int64_t slots, bool even_deep = false) {
    if (2 * tiles > slots) return tiles * k_blocks >= slots ? slots : 0;
    if (even_deep && 16 * tiles >= slots && tiles * k_blocks >= 6 * slots) return slots;
    const int64_t s = std::min<int64_t>({slots / std::max<int64_t>(tiles, 1), 16, k_blocks});
    return s >= 2 ? tiles * s : 0;
}

int choose_tf32x3_config(const sgemmContext *h, const Problem &q) {
    if (h->algo >= 1 && h->algo <= sg::kNumTf32x3Configs) return h->algo;
    // Among the tiles whose count fills the chip (with stream-K evening out
    // the last wave), the least padded tile area per element of C over the
    // tile's relative speed wins.  Speeds from the measured main kernels:
    // 128 x 128 0.86, 128 x 256 0.91 (fewer shared-memory bytes per MMA,
    // the resource this kernel is bound by), 256 x 256 on an SM pair 1.04
    // (4096^3: 516.5 us for 128 x 256, 450.8 us for the pair tile).  The
    // padding matters for batches of small matrices (300 x 64 x 64 x 512:
    // 81.0 us with 128 x 128 tiles, 95.8 with 128 x 256, 121.0 with the pair
    // tile).  The pair tile counts as filling the chip at half of the pairs
    // (2048^3, 64 tiles: 71.3 us against 76.2 for 128 x 256; 1024^3, 16
    // tiles: 36.4 against 32.4).
    const int64_t sms = h->sm_count;
    const bool deep = ceil_div(q.K, 32) >= 4;
    auto tiles = [&](int64_t bm, int64_t bn) { return ceil_div(q.M, bm) * ceil_div(q.N, bn) * q.batch; };
    auto cost = [&](int64_t bm, int64_t bn, double speed) {
        return double(ceil_div(q.M, bm) * bm) * double(ceil_div(q.N, bn) * bn) /
               (double(q.M) * double(q.N) * speed);
    };
    int pick = 0;
    double pick_cost = 0.0;
    auto consider = [&](int cfg, double c) {
        if (pick == 0 || c < pick_cost) { pick = cfg; pick_cost = c; }
    };
    if (deep && 4 * tiles(256, 256) >= sms) consider(4, cost(256, 256, 1.04));
    if (deep && h->schedule != 1 && tiles(128, 256) >= sms) consider(3, cost(128, 256, 0.91));
    if (pick != 0) {
        if (tiles(128, 128) >= sms) consider(1, cost(128, 128, 0.86));
        return pick;
    }
    const double width[2] = {128.0, 256.0};
    const double eff[2] = {0.86, 0.91};
    const int cfg[2] = {1, 3};
    int best = 1;
    double best_t = 0.0;
    for (int i = 0; i < 2; ++i) {
        const int64_t t_i = ceil_div(q.M, 128) * ceil_div(q.N, int64_t(width[i])) * q.batch;
        const double t = double(ceil_div(t_i, sms)) * width[i] / eff[i];
        if (i == 0 || t < best_t) { best_t = t; best = cfg[i]; }
    }
    return best;
}

sgemmStatus_t make_plan_tf32x3(const sgemmContext *h, const Problem &q, Plan &pl) {
    pl.tf32_cfg = choose_tf32x3_config(h, q);
    const sg::Tf32x3Info info = sg::tf32x3_info(pl.tf32_cfg);
    pl.pub.kind = 3;
    pl.pub.vector_epilogue = c_vector_ok(q) ? 1 : 0;
    pl.variant = (q.beta == 0.0f ? 0 : 2) + (pl.pub.vector_epilogue ? 0 : 1);
    pl.kp = round_up(q.K, 32);     // split rows start on 128-byte lines
    if (ceil_div(q.K, 32) > 65535 || ceil_div(q.M, 32) > 65535) return SGEMM_STATUS_NOT_SUPPORTED;
    pl.ws_split_a = align256(size_t(q.batch) * size_t(q.M) * size_t(pl.kp) * 4);
    pl.ws_split_b = align256(size_t(q.batch) * size_t(q.N) * size_t(pl.kp) * 4);
    pl.ws_split = 2 * pl.ws_split_a + 2 * pl.ws_split_b;
    pl.tiles_m = int(ceil_div(q.M, info.bm));
    pl.tiles_n = int(ceil_div(q.N, info.bn));
    const int64_t tiles = int64_t(pl.tiles_m) * pl.tiles_n * q.batch;
    if (tiles > kMaxDim) return SGEMM_STATUS_NOT_SUPPORTED;
    pl.num_tiles = int(tiles);
    pl.k_blocks = int(ceil_div(q.K, info.bk));
    // Slots: CTAs resident at once, or for the SM-pair tile, clusters of 2.
    static std::mutex occ_mutex;
    static int slot_cache[kMaxDevices][sg::kNumTf32x3Configs][4] = {};
    int64_t slots = 0;
    {
        std::lock_guard<std::mutex> lk(occ_mutex);
        int &o = slot_cache[h->device][pl.tf32_cfg - 1][pl.variant];
        if (o == 0) {
            const void *fn = info.fn[pl.variant];
            int n = 0;
            if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, info.smem) != cudaSuccess)
                return SGEMM_STATUS_LAUNCH_FAILED;
            if (info.pair) {
                cudaLaunchConfig_t cfg{};
                cfg.gridDim = dim3(2 * h->sm_count);
                cfg.blockDim = dim3(info.threads);
                cfg.dynamicSmemBytes = size_t(info.smem);
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = 2;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
            } else {
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, info.threads, info.smem) != cudaSuccess)
                    n = 0;
                n *= h->sm_count;
            }
            if (n < 1) return SGEMM_STATUS_LAUNCH_FAILED;
            o = n;
        }
        slots = o;
    }
    const int per_slot = info.pair ? 2 : 1;     // CTAs per slot
    pl.dp_ctas = int(std::min<int64_t>(pl.num_tiles, slots)) * per_slot;
    // Stream-K for a partial last wave, as for the FFMA kernel, where it
    // pays: cutting tiles costs this kernel about a fifth of a tile's time
    // (measured: partial-tile stores and loads, the counter handshake), so
    // whole tiles stay when the last wave is more than 3/4 full; few tiles
    // (at most half a wave) are split along K when K is deep (>= 1024;
    // below that the split measured slower than one CTA per tile).
    // For the SM-pair tile the cut pays only up to a half-full last wave
    // (measured per call, cut against whole: 4096^3, 3.37 waves, 516.6 /
    // 560.4 us; 8192^3, 13.47 waves, 3624 / 3690 us; 6144^3, 7.58 waves,
    // 1651 / 1614 us).
    const double per_sm = double(pl.num_tiles) / double(slots);
    const double frac = per_sm - std::floor(per_sm);
    const int64_t units = int64_t(pl.num_tiles) * pl.k_blocks;
    const double frac_max = info.pair ? 0.5 : 0.75;
    const bool sk_pays = (per_sm >= 1.0 && frac > 0.0 && frac < frac_max) ||
                         (2 * pl.num_tiles <= slots && pl.k_blocks >= 32);
    const bool want_sk = h->schedule == 2 || (h->schedule == 0 && sk_pays);
    const int64_t sk_ctas = stream_k_ctas(pl.num_tiles, pl.k_blocks, slots);
    if (want_sk && pl.k_blocks >= 2 && units < kMaxDim && sk_ctas > 0) {
        // Only the tiles past the last full wave are cut, when they give
        // every CTA at least 8 K slices: CTAs working at different K offsets
        // of many tiles at once would need all of those tiles' operands in
        // L2 (four hi/lo streams), so the cut region is kept small.  With a
        // thinner remainder, the last full wave joins it.
        const int64_t waves = pl.num_tiles / slots;
        const int64_t rem_units = (pl.num_tiles - waves * slots) * pl.k_blocks;
        int64_t first = waves * slots;
        if (rem_units < 8 * slots) first = waves >= 1 ? (waves - 1) * slots : 0;
        pl.sk_tile0 = int(first);
        pl.sk_ctas = int(sk_ctas) * per_slot;
        // One partial tile per CTA: its box_a rows of the tile.
        pl.ws_partials = size_t(pl.sk_ctas) * size_t(info.box_a) * size_t(info.bn) * 4;
    }
    pl.pub.tile_m = info.bm;
    pl.pub.tile_n = info.bn;
    pl.pub.tile_k = info.bk;
    pl.pub.stages = info.stages;
    pl.pub.packs_a = 1;
    pl.pub.packs_b = 1;
    pl.pub.launches = 3;
    return SGEMM_STATUS_SUCCESS;
}

// Plan of one call: operand preparation, kernel variant, grid and stream-K
// split.  Queries the kernel's occupancy once per device (a CUDA call);
// everything else is host arithmetic.
sgemmStatus_t make_plan(const sgemmContext *h, const Problem &q, Plan &pl) {
    pl = Plan{};
    if (q.empty()) return SGEMM_STATUS_SUCCESS;
    if (q.K == 0 || q.alpha == 0.0f) {
        pl.pub.kind = 2;
        pl.pub.launches = 1;
        return SGEMM_STATUS_SUCCESS;
    }
    std::call_once(g_kernels_once, init_kernel_table);
    // Few rows or few columns: streaming kernels bound by HBM (either math
    // mode; their FMAs are FP32), when the workspace holds their partial sums.
    if (q.opA == 0 && q.opB == 0 && q.batch == 1 && (q.M <= sg::kSkinnyMax || q.N <= sg::kSkinnyMax) &&
        !thin_ffma_preferred(h, q)) {
        const bool small_m = q.M <= sg::kSkinnyMax && (q.M <= q.N || q.N > sg::kSkinnyMax);
        if (skinny_tma_eligible(q, small_m)) {
            const sg::SkinnyTmaGeom g = sg::skinny_tma_geometry(small_m, int(q.M), int(q.N), int(q.K),
                                                               h->sm_count);
            const size_t need = align256(g.ws_bytes);
            if (h->ws != nullptr && h->ws_bytes >= need) {
                pl.pub.kind = 4;
                pl.pub.launches = 2;
                pl.pub.vector_epilogue = 0;
                pl.pub.stages = 6;
                pl.pub.tile_k = small_m ? 8 : 16;
                pl.skinny_m = small_m;
                pl.skinny_tma = true;
                pl.skinny_geom = g;
                pl.ws_skinny = need;
                pl.pub.ctas = g.ctas;
                return SGEMM_STATUS_SUCCESS;
            }
        }
        const int splits = sg::skinny_splits(small_m, int(q.M), int(q.N), int(q.K), h->sm_count);
        const size_t need = align256(sg::skinny_workspace(int(q.M), int(q.N), splits));
        if (h->ws != nullptr && h->ws_bytes >= need) {
            pl.pub.kind = 4;
            pl.pub.launches = 2;
            pl.pub.vector_epilogue = 0;
            pl.skinny_m = small_m;
            pl.skinny_split = splits;
            pl.ws_skinny = need;
            pl.pub.ctas = int(ceil_div(small_m ? q.N : q.M, 1024) * splits);
            return SGEMM_STATUS_SUCCESS;
        }
    }
    if (small_preferred(h, q)) {
        pl.pub.kind = 5;
        pl.pub.launches = 1;
        pl.pub.tile_m = pl.pub.tile_n = sg::kSmallTile;
        pl.pub.tile_k = sg::kSmallPiece;
        pl.pub.stages = 1;
        pl.small_splits = sg::small_splits(int(q.M), int(q.N), int(q.K), int(q.batch), h->sm_count);
        pl.pub.ctas = sg::small_blocks(int(q.M), int(q.N), int(q.batch)) * pl.small_splits;
        return SGEMM_STATUS_SUCCESS;
    }
    if (h->math == 1) return make_plan_tf32x3(h, q, pl);
    pl.pub.kind = 1;
    // A as TMA reads it: [batch][M][K] rows of K.
    if (q.opA == 0 && tma_ok_batched(q.A, q.lda, q.sa, q.batch)) {
        pl.prep_a = 0;
        pl.lda_p = q.lda;
        pl.sa_p = q.batch == 1 ? round_up(q.M * q.lda, 4) : q.sa;
    } else {
        pl.prep_a = q.opA == 0 ? 1 : 2;
        pl.lda_p = round_up(q.K, 4);
        pl.sa_p = q.M * pl.lda_p;
        pl.ws_a = align256(size_t(q.batch) * size_t(pl.sa_p) * 4);
    }
    // B as TMA reads it: [batch][K][N] rows of N.
    if (q.opB == 0 && tma_ok_batched(q.B, q.ldb, q.sb, q.batch)) {
        pl.prep_b = 0;
        pl.ldb_p = q.ldb;
        pl.sb_p = q.batch == 1 ? round_up(q.K * q.ldb, 4) : q.sb;
    } else {
        pl.prep_b = q.opB == 0 ? 1 : 2;
        pl.ldb_p = round_up(q.N, 4);
        pl.sb_p = q.K * pl.ldb_p;
        pl.ws_b = align256(size_t(q.batch) * size_t(pl.sb_p) * 4);
    }
    if ((pl.prep_a == 2 && ceil_div(q.K, 32) > 65535) || (pl.prep_b == 2 && ceil_div(q.N, 32) > 65535))
        return SGEMM_STATUS_NOT_SUPPORTED;   // transpose grid
    pl.pub.packs_a = pl.prep_a != 0;
    pl.pub.packs_b = pl.prep_b != 0;
    pl.pub.vector_epilogue = c_vector_ok(q) ? 1 : 0;
    pl.algo_index = choose_algo(h, q);
    if (pl.algo_index < 0) return SGEMM_STATUS_INVALID_VALUE;   // a configuration that is not built
    pl.variant = (q.beta == 0.0f ? 0 : 2) + (pl.pub.vector_epilogue ? 0 : 1);
    KernelEntry &e = g_kernels[pl.algo_index][pl.variant];
    // A last tile column of at most kEdgeMaxCols columns would multiply
    // mostly zero padding (4095 x 4097 x 1023: 16 tiles of 256 x 128 for one
    // column, 3% of the launch); in the automatic setting, when there is
    // enough work for that to matter, those columns go to the edge job of
    // the preparation launch, and the main kernel covers whole tiles only.
    pl.n_main = q.N;
    const int64_t edge = q.N % e.bn;
    if (h->algo == 0 && q.opA == 0 && q.opB == 0 && q.batch == 1 && edge >= 1 && edge <= sg::kEdgeMaxCols &&
        q.N > e.bn && double(q.M) * double(q.K) >= kEdgeMinMK && q.K * edge <= sg::kEdgeMaxStrip) {
        pl.edge_cols = int(edge);
        pl.n_main = q.N - edge;
    }
    pl.tiles_m = int(ceil_div(q.M, e.bm));
    pl.tiles_n = int(ceil_div(pl.n_main, e.bn));
    const int64_t tiles = int64_t(pl.tiles_m) * pl.tiles_n * q.batch;
    if (tiles > kMaxDim) return SGEMM_STATUS_NOT_SUPPORTED;
    pl.num_tiles = int(tiles);
    pl.k_blocks = int(ceil_div(q.K, e.bk));
    const int occ = occupancy_for(h, e);
    if (occ < 1) return SGEMM_STATUS_LAUNCH_FAILED;
    const int64_t slots = int64_t(h->sm_count) * occ;
    pl.dp_ctas = int(std::min<int64_t>(pl.num_tiles, slots));
    // Whole tiles leave the SMs unevenly loaded when the tile count is not a
    // multiple of the SM count (the last wave is partial).  Stream-K gives
    // every resident CTA the same number of (tile, K slice) units instead.
    const double per_sm = double(pl.num_tiles) / h->sm_count;
    const double dp_eff = per_sm / std::ceil(per_sm);
    const int64_t units = int64_t(pl.num_tiles) * pl.k_blocks;
    const bool want_sk = h->schedule == 2 || (h->schedule == 0 && dp_eff < 0.985);
    // Schedule 2 spreads the units evenly over every CTA slot; the automatic
    // schedule may use fewer CTAs for few tiles (each tile cut into pieces).
    const int64_t sk_ctas = h->schedule == 2 ? std::min(units, slots)
                                             : stream_k_ctas(pl.num_tiles, pl.k_blocks, slots, true);
    if (want_sk && pl.k_blocks >= 2 && units < kMaxDim && sk_ctas > 0) {
        // All but the last full wave of tiles run whole (their concurrent
        // tiles form a compact band, friendly to L2); the last wave plus the
        // remainder is split evenly in (tile, K slice) units.
        const int64_t waves = pl.num_tiles / slots;
        pl.sk_tile0 = waves >= 2 ? int((waves - 1) * slots) : 0;
        pl.sk_ctas = int(sk_ctas);
        pl.ws_partials = size_t(sk_ctas) * size_t(e.bm) * size_t(e.bn) * 4;
    }
    pl.pub.tile_m = e.bm;
    pl.pub.tile_n = e.bn;
    pl.pub.tile_k = e.bk;
    pl.pub.stages = e.stages;
    pl.pub.edge_cols = pl.edge_cols;
    // Transposes are launches of their own; repacks and the edge job share
    // one preparation launch.
    pl.pub.launches = 1 + (pl.prep_a == 2) + (pl.prep_b == 2) +
                      ((pl.prep_a == 1 || pl.prep_b == 1 || pl.edge_cols > 0) ? 1 : 0);
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t make_plan(const sgemmContext *h, int64_t M, int64_t N, int64_t K, float alpha,
                        const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                        const float *C, int64_t ldc, Plan &pl) {
    return make_plan(h, nn_problem(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc), pl);
}

// 3-D tiled tensor map over FP32 data: dims {inner, outer, batch}, row pitch
// ld and batch stride in elements (both multiples of 4), box {bi, bo, 1}.
sgemmStatus_t encode_3d(CUtensorMap *map, const float *ptr, int64_t inner, int64_t outer,
                        int64_t batch, int64_t ld, int64_t bstride, int box_inner, int box_outer,
                        CUtensorMapSwizzle swz) {
    auto enc = encode_fn();
    if (enc == nullptr) return SGEMM_STATUS_LAUNCH_FAILED;
    cuuint64_t dims[3] = {cuuint64_t(inner), cuuint64_t(outer), cuuint64_t(batch)};
    cuuint64_t strides[2] = {cuuint64_t(ld) * 4, cuuint64_t(bstride) * 4};
    cuuint32_t box[3] = {cuuint32_t(box_inner), cuuint32_t(box_outer), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SGEMM_STATUS_SUCCESS : SGEMM_STATUS_LAUNCH_FAILED;
}

sgemmStatus_t encode_2d(CUtensorMap *map, const float *ptr, int64_t inner, int64_t outer, int64_t ld,
                        int box_inner, int box_outer, CUtensorMapSwizzle swz) {
    auto enc = encode_fn();
    if (enc == nullptr) return SGEMM_STATUS_LAUNCH_FAILED;
    cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    cuuint64_t strides[1] = {cuuint64_t(ld) * 4};
    cuuint32_t box[2] = {cuuint32_t(box_inner), cuuint32_t(box_outer)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SGEMM_STATUS_SUCCESS : SGEMM_STATUS_LAUNCH_FAILED;
}

CUtensorMapSwizzle swizzle_for_bk(int bk) {
    return bk == 32 ? CU_TENSOR_MAP_SWIZZLE_128B
                    : bk == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
}

inline sgemmStatus_t last_launch() {
    return cudaGetLastError() == cudaSuccess ? SGEMM_STATUS_SUCCESS : SGEMM_STATUS_LAUNCH_FAILED;
}

// Main kernels are launched with programmatic stream serialisation: their
// CTAs may be placed (and set up their barriers) while the previous kernel
// in the stream finishes; they wait for it (griddepcontrol.wait) before
// touching global memory.  cluster = 2: CTAs in pairs (SM-pair tiles).
sgemmStatus_t launch_main(sgemmContext *h, const void *fn, int ctas, int threads, int smem,
                          void **kargs, cudaStream_t stream, int cluster = 1) {
    if (h->ev_start != nullptr && cudaEventRecord(h->ev_start, stream) != cudaSuccess)
        return SGEMM_STATUS_LAUNCH_FAILED;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = unsigned(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 2 : 1;
    cudaError_t err = cudaLaunchKernelExC(&cfg, fn, kargs);
    if (err == cudaSuccess && h->ev_stop != nullptr) err = cudaEventRecord(h->ev_stop, stream);
    return err == cudaSuccess ? SGEMM_STATUS_SUCCESS : SGEMM_STATUS_LAUNCH_FAILED;
}

// Stream-K needs its partial tiles in the workspace (after `used` bytes)
// and one flag word per CTA and warp in the handle's control block.
bool sk_usable(const sgemmContext *h, const Plan &pl, size_t used, int warps) {
    return pl.sk_ctas > 0 && h->ws != nullptr && h->ws_bytes >= used + pl.ws_partials &&
           int64_t(pl.sk_ctas) * warps <= h->flag_words;
}

sgemmStatus_t run_tf32x3(sgemmContext *h, const Plan &pl, const Problem &q, cudaStream_t stream) {
    if (h->ws == nullptr || h->ws_bytes < pl.ws_split) return SGEMM_STATUS_WORKSPACE_REQUIRED;
    const sg::Tf32x3Info info = sg::tf32x3_info(pl.tf32_cfg);
    char *ws = static_cast<char *>(h->ws);
    float *a_hi = reinterpret_cast<float *>(ws);
    float *a_lo = reinterpret_cast<float *>(ws + pl.ws_split_a);
    float *b_hi = reinterpret_cast<float *>(ws + 2 * pl.ws_split_a);
    float *b_lo = reinterpret_cast<float *>(ws + 2 * pl.ws_split_a + pl.ws_split_b);
    const int M = int(q.M), N = int(q.N), K = int(q.K), batch = int(q.batch);
    const int64_t sa_d = q.M * pl.kp, sb_d = q.N * pl.kp;
    // A_hi / A_lo as [batch][M][kp] and B_hi / B_lo as [batch][N][kp]: K
    // contiguous for both, whatever the stored layout.  The high part is the
    // operand itself (the MMA reads its TF32 bits), so an operand stored K
    // contiguous that TMA can address is read in place as its high part and
    // only its residual is written: the split of A moves 128 instead of 192
    // MB at 4096^3 (516.0 -> 504.5 us per call).  Only up to 64 MB of
    // operand: a larger one read in place did not pay (8192^3: 3577 -> 3608
    // us per call; 6144^3 no gain).
    const int64_t kDirectMaxBytes = int64_t(64) << 20;
    const bool a_direct = q.opA == 0 && tma_ok_batched(q.A, q.lda, q.sa, q.batch) &&
                          q.batch * q.M * q.K * 4 <= kDirectMaxBytes;
    const bool b_direct = q.opB == 1 && tma_ok_batched(q.B, q.ldb, q.sb, q.batch) &&
                          q.batch * q.N * q.K * 4 <= kDirectMaxBytes;
    if (q.opA == 0)
        sg::launch_split_rows(q.A, q.lda, q.sa, a_direct ? nullptr : a_hi, a_lo, pl.kp, sa_d, M, K, batch, stream);
    else sg::launch_transpose(q.A, q.lda, q.sa, a_hi, a_lo, pl.kp, sa_d, K, M, batch, stream);
    if (q.opB == 0) sg::launch_transpose(q.B, q.ldb, q.sb, b_hi, b_lo, pl.kp, sb_d, K, N, batch, stream);
    else sg::launch_split_rows(q.B, q.ldb, q.sb, b_direct ? nullptr : b_hi, b_lo, pl.kp, sb_d, N, K, batch, stream);
    if (last_launch() != SGEMM_STATUS_SUCCESS) return SGEMM_STATUS_LAUNCH_FAILED;

    CUtensorMap tm[4];
    const float *ptrs[4] = {a_direct ? q.A : a_hi, a_lo, b_direct ? q.B : b_hi, b_lo};
    for (int i = 0; i < 4; ++i) {
        const bool is_a = i < 2;
        const bool direct = i == 0 ? a_direct : i == 2 ? b_direct : false;
        int64_t ld = pl.kp, bstride = is_a ? sa_d : sb_d;
        if (direct) {
            ld = is_a ? q.lda : q.ldb;
            bstride = q.batch == 1 ? ld * (is_a ? q.M : q.N) : (is_a ? q.sa : q.sb);
        }
        sgemmStatus_t st = encode_3d(&tm[i], ptrs[i], q.K, is_a ? q.M : q.N, q.batch, ld, bstride, info.bk,
                                     is_a ? info.box_a : info.box_b, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != SGEMM_STATUS_SUCCESS) return st;
    }
    sg::Tf32x3Args args{};
    args.M = M;
    args.N = N;
    args.K = K;
    args.alpha = q.alpha;
    args.beta = q.beta;
    args.C = q.C;
    args.ldc = q.ldc;
    args.stride_c = q.sc;
    args.tiles_m = pl.tiles_m;
    args.tiles_n = pl.tiles_n;
    args.num_tiles = pl.num_tiles;
    args.k_blocks = pl.k_blocks;
    args.group_m = pl.group_m;
    args.err = h->d_err;
    args.timeout_ns = h->timeout_ns;
    args.withhold = h->withhold;
    args.sk_tile0 = pl.num_tiles;
    int ctas = pl.dp_ctas;
    if (sk_usable(h, pl, pl.ws_split, info.threads / 32 - 2)) {
        args.sk_tile0 = pl.sk_tile0;
        args.flags = h->d_flags;
        args.sk_seq = h->d_sk_seq;
        args.partials = reinterpret_cast<float *>(ws + pl.ws_split);
        ctas = pl.sk_ctas;
    }
    void *kargs[] = {&tm[0], &tm[1], &tm[2], &tm[3], &args};
    return launch_main(h, info.fn[pl.variant], ctas, info.threads, info.smem, kargs, stream,
                       info.pair ? 2 : 1);
}

sgemmStatus_t run(sgemmContext *h, const Problem &q, cudaStream_t stream) {
    sgemmStatus_t st = validate(q);
    if (st != SGEMM_STATUS_SUCCESS || q.empty()) return st;
    if (h == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    Plan pl;
    st = make_plan(h, q, pl);
    if (st != SGEMM_STATUS_SUCCESS) return st;

    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return SGEMM_STATUS_LAUNCH_FAILED;
    if (cur != h->device) return SGEMM_STATUS_INVALID_VALUE;

    if (pl.pub.kind == 2) {
        sg::launch_scale_c(int(q.M), int(q.N), q.beta, q.C, q.ldc, q.sc, int(q.batch), stream);
        return last_launch();
    }
    if (pl.pub.kind == 3) return run_tf32x3(h, pl, q, stream);
    if (pl.pub.kind == 5) {
        sg::SmallArgs a{};
        a.M = int(q.M);
        a.N = int(q.N);
        a.K = int(q.K);
        a.alpha = q.alpha;
        a.beta = q.beta;
        a.A = q.A;
        a.lda = q.lda;
        a.sa = q.sa;
        a.B = q.B;
        a.ldb = q.ldb;
        a.sb = q.sb;
        a.C = q.C;
        a.ldc = q.ldc;
        a.sc = q.sc;
        a.splits = pl.small_splits;
        a.sms = h->sm_count;
        if (h->ev_start != nullptr && cudaEventRecord(h->ev_start, stream) != cudaSuccess)
            return SGEMM_STATUS_LAUNCH_FAILED;
        sg::launch_small(a, q.opA, q.opB, int(q.batch), stream);
        if (last_launch() != SGEMM_STATUS_SUCCESS) return SGEMM_STATUS_LAUNCH_FAILED;
        if (h->ev_stop != nullptr && cudaEventRecord(h->ev_stop, stream) != cudaSuccess)
            return SGEMM_STATUS_LAUNCH_FAILED;
        return SGEMM_STATUS_SUCCESS;
    }
    if (pl.pub.kind == 4) {
        if (h->ev_start != nullptr && cudaEventRecord(h->ev_start, stream) != cudaSuccess)
            return SGEMM_STATUS_LAUNCH_FAILED;
        bool done = false;
        if (pl.skinny_tma) {
            const sg::SkinnyTmaGeom &g = pl.skinny_geom;
            CUtensorMap tmA, tmB;
            if (encode_2d(&tmA, q.A, q.K, q.M, q.lda, g.a_box[0], g.a_box[1],
                          g.a_swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE) ==
                    SGEMM_STATUS_SUCCESS &&
                encode_2d(&tmB, q.B, q.N, q.K, q.ldb, g.b_box[0], g.b_box[1], CU_TENSOR_MAP_SWIZZLE_NONE) ==
                    SGEMM_STATUS_SUCCESS) {
                sg::launch_skinny_tma(pl.skinny_m, tmA, tmB, g, int(q.M), int(q.N), int(q.K), q.alpha, q.beta,
                                      q.C, q.ldc, static_cast<float *>(h->ws), h->d_err, h->timeout_ns, stream);
                done = true;
            }
        }
        if (!done) {
            // Plain-load kernels (also the fallback should a tensor map be refused).
            const int splits = sg::skinny_splits(pl.skinny_m, int(q.M), int(q.N), int(q.K), h->sm_count);
            if (h->ws == nullptr || h->ws_bytes < sg::skinny_workspace(int(q.M), int(q.N), splits))
                return SGEMM_STATUS_WORKSPACE_REQUIRED;
            sg::launch_skinny(pl.skinny_m, int(q.M), int(q.N), int(q.K), q.alpha, q.A, q.lda, q.B, q.ldb,
                              q.beta, q.C, q.ldc, static_cast<float *>(h->ws), splits, stream);
        }
        if (last_launch() != SGEMM_STATUS_SUCCESS) return SGEMM_STATUS_LAUNCH_FAILED;
        if (h->ev_stop != nullptr && cudaEventRecord(h->ev_stop, stream) != cudaSuccess)
            return SGEMM_STATUS_LAUNCH_FAILED;
        return SGEMM_STATUS_SUCCESS;
    }

    const float *Ause = q.A, *Buse = q.B;
    // Stream-K scratch is optional: without room for it, whole tiles are used.
    const bool use_sk = sk_usable(h, pl, pl.ws_a + pl.ws_b, g_kernels[pl.algo_index][pl.variant].threads / 32);
    // The main kernel covers columns [0, n_main) of C.
    const int M = int(q.M), N = int(pl.n_main), K = int(q.K), batch = int(q.batch);
    if (pl.prep_a || pl.prep_b || pl.edge_cols) {
        if ((pl.prep_a || pl.prep_b) && (h->ws == nullptr || h->ws_bytes < pl.ws_a + pl.ws_b))
            return SGEMM_STATUS_WORKSPACE_REQUIRED;
        char *ws = static_cast<char *>(h->ws);
        sg::PrepArgs prep{};
        prep.edge_pack = -1;
        if (pl.prep_a) {
            float *Ap = reinterpret_cast<float *>(ws);
            if (pl.prep_a == 1) {
                if (pl.edge_cols && batch == 1) prep.edge_pack = prep.npack;
                prep.pack[prep.npack++] = sg::PackJob{q.A, q.lda, q.sa, Ap, pl.lda_p, pl.sa_p, M, K, batch, 0, 0};
            }
            else
                sg::launch_transpose(q.A, q.lda, q.sa, Ap, nullptr, pl.lda_p, pl.sa_p, K, M, batch, stream);
            Ause = Ap;
        }
        if (pl.prep_b) {
            float *Bp = reinterpret_cast<float *>(ws + pl.ws_a);
            if (pl.prep_b == 1)
                prep.pack[prep.npack++] = sg::PackJob{q.B, q.ldb, q.sb, Bp, pl.ldb_p, pl.sb_p, K, N, batch, 0, 0};
            else
                sg::launch_transpose(q.B, q.ldb, q.sb, Bp, nullptr, pl.ldb_p, pl.sb_p, int(q.N), K, batch, stream);
            Buse = Bp;
        }
        if (pl.edge_cols)
            prep.edge = sg::EdgeJob{q.A, q.lda, q.B, q.ldb, q.C, q.ldc, M, K, N, pl.edge_cols, q.alpha, q.beta};
        if (last_launch() != SGEMM_STATUS_SUCCESS) return SGEMM_STATUS_LAUNCH_FAILED;
        if ((prep.npack > 0 || pl.edge_cols) && sg::launch_prep(prep, h->sm_count, stream) != cudaSuccess)
            return SGEMM_STATUS_LAUNCH_FAILED;
    }

    int variant = pl.variant;
    CUtensorMap tmA, tmB, tmC;
    std::memset(&tmC, 0, sizeof(tmC));
    if (g_kernels[pl.algo_index][variant].c_box_rows > 0) {
        // TMA-store epilogue: C as a 3-D map {N, M, batch}.  A C layout the
        // encoder rejects takes the st.global epilogue of the same tile.
        const KernelEntry &ec = g_kernels[pl.algo_index][variant];
        const int64_t sc = q.batch == 1 ? q.ldc * q.M : q.sc;
        if (encode_3d(&tmC, q.C, pl.n_main, q.M, q.batch, q.ldc, sc, ec.c_box_cols, ec.c_box_rows,
                      CU_TENSOR_MAP_SWIZZLE_NONE) != SGEMM_STATUS_SUCCESS)
            variant = 1;
    }
    KernelEntry &e = g_kernels[pl.algo_index][variant];

    // Boxes of at most 256 rows / columns; wider tiles load several.
    st = encode_3d(&tmA, Ause, q.K, q.M, q.batch, pl.lda_p, pl.sa_p, e.bk, std::min(e.bm, 256), swizzle_for_bk(e.bk));
    if (st != SGEMM_STATUS_SUCCESS) return st;
    st = encode_3d(&tmB, Buse, pl.n_main, q.K, q.batch, pl.ldb_p, pl.sb_p, std::min(e.bn, 256), e.bk,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != SGEMM_STATUS_SUCCESS) return st;

    sg::GemmArgs args{};
    args.M = M;
    args.N = N;
    args.K = K;
    args.alpha = q.alpha;
    args.beta = q.beta;
    args.C = q.C;
    args.ldc = q.ldc;
    args.stride_c = q.sc;
    args.tiles_m = pl.tiles_m;
    args.tiles_n = pl.tiles_n;
    args.num_tiles = pl.num_tiles;
    args.k_blocks = pl.k_blocks;
    args.group_m = pl.group_m;
    args.err = h->d_err;
    args.timeout_ns = h->timeout_ns;
    args.withhold = h->withhold;
    int ctas = pl.dp_ctas;
    args.sk_tile0 = pl.num_tiles;
    if (use_sk) {
        // Partial tiles in the workspace; flags and launch tags in the
        // handle's control block (no reset needed between launches).
        args.sk_tile0 = pl.sk_tile0;
        args.flags = h->d_flags;
        args.sk_seq = h->d_sk_seq;
        args.partials = reinterpret_cast<float *>(static_cast<char *>(h->ws) + pl.ws_a + pl.ws_b);
        ctas = pl.sk_ctas;
    }
    void *kargs[] = {&tmA, &tmB, &tmC, &args};
    return launch_main(h, e.fn, ctas, e.threads, e.smem, kargs, stream);
}

sgemmStatus_t run(sgemmContext *h, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                  int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                  cudaStream_t stream) {
    return run(h, nn_problem(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc), stream);
}

size_t workspace_bytes(const Plan &pl) {
    return pl.ws_a + pl.ws_b + pl.ws_partials + pl.ws_split;
}

// Skinny products use the workspace only when it is big enough; the size
// query reports what they would use so that callers can provide it.
size_t skinny_query_bytes(const sgemmContext *h, const Problem &q) {
    if (q.opA != 0 || q.opB != 0 || q.batch != 1 || q.empty() || q.K == 0 || q.alpha == 0.0f) return 0;
    if (thin_ffma_preferred(h, q)) return 0;
    if (q.M > sg::kSkinnyMax && q.N > sg::kSkinnyMax) return 0;
    const bool small_m = q.M <= sg::kSkinnyMax && (q.M <= q.N || q.N > sg::kSkinnyMax);
    const int splits = sg::skinny_splits(small_m, int(q.M), int(q.N), int(q.K), h->sm_count);
    size_t bytes = align256(sg::skinny_workspace(int(q.M), int(q.N), splits));
    if (skinny_tma_eligible(q, small_m))
        bytes = std::max(bytes, align256(sg::skinny_tma_geometry(small_m, int(q.M), int(q.N), int(q.K),
                                                                 h->sm_count).ws_bytes));
    return bytes;
}

// Workspace a call on these operands can use, whatever its beta and C: the
// tile configuration (and with it the stream-K scratch) depends on whether
// C is read (beta != 0) and whether C is 16-byte aligned with a pitch of
// whole 16-byte units, so the query plans each of those cases and keeps
// the largest need.  C's own address is never dereferenced by planning.
sgemmStatus_t workspace_query(const sgemmContext *h, Problem q, size_t *bytes) {
    static float *const kAlignedC = reinterpret_cast<float *>(uintptr_t(256));
    static float *const kOddC = reinterpret_cast<float *>(uintptr_t(260));
    const struct { float beta; float *c; int64_t ldc; } cases[3] = {
        {0.0f, kAlignedC, round_up(std::max<int64_t>(1, q.N), 4)},
        {1.0f, kAlignedC, round_up(std::max<int64_t>(1, q.N), 4)},
        {1.0f, kOddC, std::max<int64_t>(1, q.N)},
    };
    size_t need = 0;
    for (const auto &c : cases) {
        q.beta = c.beta;
        q.C = c.c;
        q.ldc = c.ldc;
        q.sc = q.batch == 1 ? 0 : c.ldc * q.M;
        Plan pl;
        sgemmStatus_t st = make_plan(h, q, pl);
        if (st != SGEMM_STATUS_SUCCESS) return st;
        need = std::max({need, workspace_bytes(pl), skinny_query_bytes(h, q)});
    }
    *bytes = need;
    return SGEMM_STATUS_SUCCESS;
}

void release_handle_resources(sgemmContext *h) {
    if (h->d_err) cudaFree(h->d_err);
    if (h->s_in) cudaStreamDestroy(h->s_in);
    if (h->s_out) cudaStreamDestroy(h->s_out);
    if (h->ev_begin) cudaEventDestroy(h->ev_begin);
    if (h->ev_end) cudaEventDestroy(h->ev_end);
    for (int i = 0; i < sgemmContext::kHostChunks; ++i) {
        if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
        if (h->ev_done[i]) cudaEventDestroy(h->ev_done[i]);
    }
    h->d_err = nullptr;
}

}  // namespace

extern "C" {

const char *sgemmGetStatusString(sgemmStatus_t s) {
    switch (s) {
        case SGEMM_STATUS_SUCCESS: return "SGEMM_STATUS_SUCCESS";
        case SGEMM_STATUS_INVALID_VALUE: return "SGEMM_STATUS_INVALID_VALUE";
        case SGEMM_STATUS_MISALIGNED: return "SGEMM_STATUS_MISALIGNED";
        case SGEMM_STATUS_ARCH_MISMATCH: return "SGEMM_STATUS_ARCH_MISMATCH";
        case SGEMM_STATUS_WORKSPACE_REQUIRED: return "SGEMM_STATUS_WORKSPACE_REQUIRED";
        case SGEMM_STATUS_LAUNCH_FAILED: return "SGEMM_STATUS_LAUNCH_FAILED";
        case SGEMM_STATUS_DEVICE_TIMEOUT: return "SGEMM_STATUS_DEVICE_TIMEOUT";
        case SGEMM_STATUS_NOT_SUPPORTED: return "SGEMM_STATUS_NOT_SUPPORTED";
        case SGEMM_STATUS_INTERNAL_ERROR: return "SGEMM_STATUS_INTERNAL_ERROR";
    }
    return "SGEMM_STATUS_UNKNOWN";
}

sgemmStatus_t sgemmGetVersion(int *version) {
    if (version == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    *version = kVersion;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmCreate(sgemmHandle_t *handle) {
    if (handle == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    *handle = nullptr;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_STATUS_LAUNCH_FAILED;
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_STATUS_NOT_SUPPORTED;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SGEMM_STATUS_LAUNCH_FAILED;
    if (major != 10 || minor != 3) return SGEMM_STATUS_ARCH_MISMATCH;
    auto *h = new (std::nothrow) sgemmContext();
    if (h == nullptr) return SGEMM_STATUS_INTERNAL_ERROR;
    h->device = dev;
    h->sm_count = sms;
    h->flag_words = kCtlFlagWords;
    bool ok = cudaMalloc(&h->d_err, kCtlBytes) == cudaSuccess &&
              cudaMemset(h->d_err, 0, kCtlBytes) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h->ev_begin, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&h->ev_end, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < sgemmContext::kHostChunks; ++i)
        ok = cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h->ev_done[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        release_handle_resources(h);
        delete h;
        return SGEMM_STATUS_LAUNCH_FAILED;
    }
    h->d_sk_seq = h->d_err + 1;
    h->d_flags = h->d_err + kCtlFlagsOffset;
    *handle = h;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmDestroy(sgemmHandle_t h) {
    if (h == nullptr) return SGEMM_STATUS_SUCCESS;
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    release_handle_resources(h);
    if (prev >= 0) cudaSetDevice(prev);
    delete h;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmGetDefaultHandle(sgemmHandle_t *handle) {
    if (handle == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_STATUS_LAUNCH_FAILED;
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_STATUS_NOT_SUPPORTED;
    std::lock_guard<std::mutex> lk(g_default_mutex);
    if (g_default[dev] == nullptr) {
        sgemmStatus_t st = sgemmCreate(&g_default[dev]);
        if (st != SGEMM_STATUS_SUCCESS) return st;
    }
    *handle = g_default[dev];
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmGetWorkspaceSize(sgemmHandle_t h, int64_t M, int64_t N, int64_t K,
                                    const float *A, int64_t lda, const float *B, int64_t ldb,
                                    size_t *bytes) {
    if (bytes == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    *bytes = 0;
    const float dummy_c = 0.f;
    sgemmStatus_t st = validate(M, N, K, A, lda, B, ldb, &dummy_c, std::max<int64_t>(1, N), true);
    if (st != SGEMM_STATUS_SUCCESS || M == 0 || N == 0 || K == 0) return st;
    if (h == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    return workspace_query(h, nn_problem(M, N, K, 1.0f, A, lda, B, ldb, 0.0f, nullptr, N), bytes);
}

sgemmStatus_t sgemmSetWorkspace(sgemmHandle_t h, void *ptr, size_t bytes) {
    if (h == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    if (ptr != nullptr && !aligned(ptr, 256)) return SGEMM_STATUS_MISALIGNED;
    h->ws = ptr;
    h->ws_bytes = ptr ? bytes : 0;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmEx(sgemmHandle_t h, int64_t M, int64_t N, int64_t K, float alpha,
                      const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                      float *C, int64_t ldc, cudaStream_t stream) {
    sgemmStatus_t st = validate(M, N, K, A, lda, B, ldb, C, ldc, alpha != 0.0f);
    if (st != SGEMM_STATUS_SUCCESS || M == 0 || N == 0) return st;
    if (h == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    return run(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

sgemmStatus_t sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                    const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                    cudaStream_t stream) {
    sgemmStatus_t st = validate(M, N, K, A, lda, B, ldb, C, ldc, alpha != 0.0f);
    if (st != SGEMM_STATUS_SUCCESS || M == 0 || N == 0) return st;
    sgemmHandle_t h = nullptr;
    st = sgemmGetDefaultHandle(&h);
    if (st != SGEMM_STATUS_SUCCESS) return st;
    return run(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

namespace {
Problem general_problem(int opA, int opB, int64_t M, int64_t N, int64_t K, float alpha,
                        const float *A, int64_t lda, int64_t sa, const float *B, int64_t ldb,
                        int64_t sb, float beta, float *C, int64_t ldc, int64_t sc, int64_t batch) {
    Problem q;
    q.opA = opA; q.opB = opB;
    q.M = M; q.N = N; q.K = K;
    q.alpha = alpha; q.beta = beta;
    q.A = A; q.lda = lda; q.sa = sa;
    q.B = B; q.ldb = ldb; q.sb = sb;
    q.C = C; q.ldc = ldc; q.sc = sc;
    q.batch = batch;
    return q;
}
}  // namespace

sgemmStatus_t sgemmStridedBatched(sgemmHandle_t h, sgemmOperation_t opA, sgemmOperation_t opB,
                                  int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                                  int64_t lda, int64_t strideA, const float *B, int64_t ldb,
                                  int64_t strideB, float beta, float *C, int64_t ldc, int64_t strideC,
                                  int64_t batchCount, cudaStream_t stream) {
    const Problem q = general_problem(int(opA), int(opB), M, N, K, alpha, A, lda, strideA, B, ldb,
                                      strideB, beta, C, ldc, strideC, batchCount);
    sgemmStatus_t st = validate(q);
    if (st != SGEMM_STATUS_SUCCESS || q.empty()) return st;
    if (h == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    return run(h, q, stream);
}

sgemmStatus_t sgemmStridedBatchedWorkspaceSize(sgemmHandle_t h, sgemmOperation_t opA,
                                               sgemmOperation_t opB, int64_t M, int64_t N, int64_t K,
                                               const float *A, int64_t lda, int64_t strideA,
                                               const float *B, int64_t ldb, int64_t strideB,
                                               int64_t batchCount, size_t *bytes) {
    if (bytes == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    *bytes = 0;
    const float dummy_c = 0.f;
    const Problem q = general_problem(int(opA), int(opB), M, N, K, 1.0f, A, lda, strideA, B, ldb,
                                      strideB, 0.0f, const_cast<float *>(&dummy_c),
                                      std::max<int64_t>(1, N), 0, batchCount);
    sgemmStatus_t st = validate(q);
    if (st != SGEMM_STATUS_SUCCESS || q.empty() || K == 0) return st;
    if (h == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    return workspace_query(h, q, bytes);
}

sgemmStatus_t sgemmHostWorkspaceSize(int64_t M, int64_t N, int64_t K, size_t *bytes) {
    if (bytes == nullptr || M < 0 || N < 0 || K < 0) return SGEMM_STATUS_INVALID_VALUE;
    *bytes = align256(size_t(M) * size_t(round_up(std::max<int64_t>(K, 1), 4)) * 4) +
             align256(size_t(K) * size_t(round_up(std::max<int64_t>(N, 1), 4)) * 4) +
             align256(size_t(M) * size_t(round_up(std::max<int64_t>(N, 1), 4)) * 4);
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmHostEx(sgemmHandle_t h, int64_t M, int64_t N, int64_t K, float alpha,
                          const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                          float *C, int64_t ldc, void *dws, size_t ws_bytes, cudaStream_t stream) {
    sgemmStatus_t st = validate(M, N, K, A, lda, B, ldb, C, ldc, alpha != 0.0f);
    if (st != SGEMM_STATUS_SUCCESS || M == 0 || N == 0) return st;
    if (h == nullptr || dws == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    if (!aligned(dws, 256)) return SGEMM_STATUS_MISALIGNED;
    size_t need = 0;
    sgemmHostWorkspaceSize(M, N, K, &need);
    if (ws_bytes < need) return SGEMM_STATUS_WORKSPACE_REQUIRED;
    const int64_t lda_p = round_up(std::max<int64_t>(K, 1), 4);
    const int64_t ldb_p = round_up(std::max<int64_t>(N, 1), 4);
    const int64_t ldc_p = ldb_p;
    char *base = static_cast<char *>(dws);
    float *dA = reinterpret_cast<float *>(base);
    float *dB = reinterpret_cast<float *>(base + align256(size_t(M) * lda_p * 4));
    float *dC = reinterpret_cast<float *>(base + align256(size_t(M) * lda_p * 4) +
                                          align256(size_t(K) * ldb_p * 4));
    const bool use_ab = K > 0 && alpha != 0.0f;
    // The product runs as a sequence of pieces of C, each multiplied on
    // `stream` as soon as its operands are up, while the next operands are
    // copied in on the handle's copy-in stream and finished pieces copied
    // out on its copy-out stream.  The first row block is cut into column
    // pieces, so that the first multiplication needs only part of B; the
    // copy-in order follows the pieces (B's first columns, A's first rows,
    // B's next columns, ..., then A's further row blocks, with C's matching
    // parts when beta != 0).
    struct Piece { int64_t r0, r1, c0, c1; };
    Piece pieces[sgemmContext::kHostChunks];
    int np = 0;
    // Measured at 4096^3 and 8192^3 among first blocks of 512 to 2048 rows
    // in 1 to 4 column pieces and last blocks of 256 to 1024 rows: a first
    // block of 1024 rows in four column pieces (the first product needs a
    // quarter of B) and a last block of 512 rows (a short drain) was fastest
    // at both sizes (4096^3: 2.58 ms, against 2.66 ms with two column halves
    // and a 1024-row last block).
    constexpr int64_t kFirstRows = 1024;   // rows of the first block
    constexpr int kFirstCols = 4;          // column pieces of the first block, at most
    constexpr int kMoreBlocks = 3;         // row blocks after the first, at most
    constexpr int64_t kLastRows = 512;     // the last block at most this high
    if (M >= 2 * kFirstRows) {
        const int cols = int(std::max<int64_t>(1, std::min<int64_t>(kFirstCols, N / 1024)));
        for (int j = 0; j < cols; ++j) {
            // Column cuts on 128-column (tile and 16-byte) boundaries.
            const int64_t c0 = j == 0 ? 0 : (N * j / cols) / 128 * 128;
            const int64_t c1 = j == cols - 1 ? N : (N * (j + 1) / cols) / 128 * 128;
            pieces[np++] = {0, kFirstRows, c0, c1};
        }
        // The rest: at most kMoreBlocks blocks, the last no higher than
        // kLastRows (a short drain), the others equal.
        const int64_t rest = M - kFirstRows;
        const int64_t last = std::min<int64_t>(kLastRows, rest);
        const int others = int(std::min<int64_t>(kMoreBlocks - 1, ceil_div(rest - last, 1024)));
        int64_t r = kFirstRows;
        for (int b = 0; b < others; ++b) {
            const int64_t r1 = kFirstRows + (rest - last) * (b + 1) / others;
            pieces[np++] = {r, r1, 0, N};
            r = r1;
        }
        pieces[np++] = {r, M, 0, N};
    } else {
        const int blocks = int(std::max<int64_t>(1, std::min<int64_t>(4, M / 1024)));
        for (int bi = 0; bi < blocks; ++bi) pieces[np++] = {M * bi / blocks, M * (bi + 1) / blocks, 0, N};
    }
    auto fail = [](cudaError_t e) { return e != cudaSuccess; };
    auto up = [&](float *dst, int64_t ldd, const float *src, int64_t lds, int64_t rows, int64_t cols) {
        return rows > 0 && cols > 0 &&
               fail(cudaMemcpy2DAsync(dst, ldd * 4, src, lds * 4, cols * 4, rows, cudaMemcpyHostToDevice, h->s_in));
    };
    if (fail(cudaEventRecord(h->ev_begin, stream)) || fail(cudaStreamWaitEvent(h->s_in, h->ev_begin, 0)) ||
        fail(cudaStreamWaitEvent(h->s_out, h->ev_begin, 0)))
        return SGEMM_STATUS_LAUNCH_FAILED;
    int64_t a_rows_up = 0, b_cols_up = 0;    // how much of A (rows) and B (columns) is up
    for (int i = 0; i < np; ++i) {
        const Piece &pc = pieces[i];
        if (use_ab) {
            if (pc.c1 > b_cols_up) {
                if (up(dB + b_cols_up, ldb_p, B + b_cols_up, ldb, K, pc.c1 - b_cols_up)) return SGEMM_STATUS_LAUNCH_FAILED;
                b_cols_up = pc.c1;
            }
            if (pc.r1 > a_rows_up) {
                if (up(dA + a_rows_up * lda_p, lda_p, A + a_rows_up * lda, lda, pc.r1 - a_rows_up, K))
                    return SGEMM_STATUS_LAUNCH_FAILED;
                a_rows_up = pc.r1;
            }
        }
        if (beta != 0.0f && up(dC + pc.r0 * ldc_p + pc.c0, ldc_p, C + pc.r0 * ldc + pc.c0, ldc, pc.r1 - pc.r0,
                               pc.c1 - pc.c0))
            return SGEMM_STATUS_LAUNCH_FAILED;
        if (fail(cudaEventRecord(h->ev_in[i], h->s_in)) || fail(cudaStreamWaitEvent(stream, h->ev_in[i], 0)))
            return SGEMM_STATUS_LAUNCH_FAILED;
        st = run(h, pc.r1 - pc.r0, pc.c1 - pc.c0, K, alpha, dA + pc.r0 * lda_p, lda_p, dB + pc.c0, ldb_p, beta,
                 dC + pc.r0 * ldc_p + pc.c0, ldc_p, stream);
        if (st != SGEMM_STATUS_SUCCESS) return st;
        if (fail(cudaEventRecord(h->ev_done[i], stream)) || fail(cudaStreamWaitEvent(h->s_out, h->ev_done[i], 0)) ||
            fail(cudaMemcpy2DAsync(C + pc.r0 * ldc + pc.c0, ldc * 4, dC + pc.r0 * ldc_p + pc.c0, ldc_p * 4,
                                   (pc.c1 - pc.c0) * 4, pc.r1 - pc.r0, cudaMemcpyDeviceToHost, h->s_out)))
            return SGEMM_STATUS_LAUNCH_FAILED;
    }
    // Join: work enqueued on `stream` after this call sees the result.
    if (fail(cudaEventRecord(h->ev_end, h->s_out)) || fail(cudaStreamWaitEvent(stream, h->ev_end, 0)))
        return SGEMM_STATUS_LAUNCH_FAILED;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmQueryPlan(sgemmHandle_t h, int64_t M, int64_t N, int64_t K, float alpha,
                             const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                             const float *C, int64_t ldc, sgemmPlan_t *plan) {
    if (plan == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    std::memset(plan, 0, sizeof(*plan));
    sgemmStatus_t st = validate(M, N, K, A, lda, B, ldb, C, ldc, alpha != 0.0f);
    if (st != SGEMM_STATUS_SUCCESS || M == 0 || N == 0) return st;
    if (h == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    Plan pl;
    st = make_plan(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, pl);
    if (st != SGEMM_STATUS_SUCCESS) return st;
    if (pl.pub.kind == 1 || pl.pub.kind == 3) pl.pub.raster_group = pl.group_m;
    if (pl.pub.kind == 3) {
        const bool use_sk = pl.sk_ctas > 0 && h->ws != nullptr &&
                            h->ws_bytes >= pl.ws_split + pl.ws_partials;
        pl.pub.ctas = use_sk ? pl.sk_ctas : pl.dp_ctas;
        pl.pub.stream_k = use_sk ? 1 : 0;
    }
    if (pl.pub.kind == 1) {
        const bool use_sk = pl.sk_ctas > 0 && h->ws != nullptr &&
                            h->ws_bytes >= pl.ws_a + pl.ws_b + pl.ws_partials;
        pl.pub.ctas = use_sk ? pl.sk_ctas : pl.dp_ctas;
        pl.pub.stream_k = use_sk ? 1 : 0;
    }
    *plan = pl.pub;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmSetAlgo(sgemmHandle_t h, int algo) {
    // 1..4 also name the tensor-core tiles of math mode 1.
    if (h == nullptr || algo < 0 || algo > kNumAlgos ||
        (algo > sg::kNumTf32x3Configs && !sg::algo_shipped(algo)))
        return SGEMM_STATUS_INVALID_VALUE;
    h->algo = algo;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmSetKernelEvents(sgemmHandle_t h, cudaEvent_t start, cudaEvent_t stop) {
    if (h == nullptr || ((start == nullptr) != (stop == nullptr))) return SGEMM_STATUS_INVALID_VALUE;
    h->ev_start = start;
    h->ev_stop = stop;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmSetMathMode(sgemmHandle_t h, int mode) {
    if (h == nullptr || mode < 0 || mode > 1) return SGEMM_STATUS_INVALID_VALUE;
    h->math = mode;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmSetSchedule(sgemmHandle_t h, int schedule) {
    if (h == nullptr || schedule < 0 || schedule > 2) return SGEMM_STATUS_INVALID_VALUE;
    h->schedule = schedule;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmSetWaitTimeout(sgemmHandle_t h, uint64_t timeout_ns) {
    if (h == nullptr || timeout_ns < kMinTimeoutNs) return SGEMM_STATUS_INVALID_VALUE;
    h->timeout_ns = timeout_ns;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmSetTestWithheldSignal(sgemmHandle_t h, int which) {
    if (h == nullptr || which < sg::kWithholdNone || which > sg::kWithholdRelease)
        return SGEMM_STATUS_INVALID_VALUE;
    h->withhold = which;
    return SGEMM_STATUS_SUCCESS;
}

sgemmStatus_t sgemmGetDeviceError(sgemmHandle_t h, int *code) {
    if (h == nullptr || code == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    *code = 0;
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return SGEMM_STATUS_LAUNCH_FAILED;
    uint32_t word = 0;
    sgemmStatus_t st = SGEMM_STATUS_SUCCESS;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&word, h->d_err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(h->d_err, 0, sizeof(uint32_t)) != cudaSuccess)
        st = SGEMM_STATUS_LAUNCH_FAILED;
    if (prev >= 0 && prev != h->device) cudaSetDevice(prev);
    if (st != SGEMM_STATUS_SUCCESS) return st;
    *code = int(word);
    return word == 0 ? SGEMM_STATUS_SUCCESS : SGEMM_STATUS_DEVICE_TIMEOUT;
}

sgemmStatus_t sgemmSelfTestWaitTimeout(sgemmHandle_t h, uint64_t timeout_ns, cudaStream_t stream) {
    if (h == nullptr || timeout_ns < kMinTimeoutNs || timeout_ns > 10 * kDefaultTimeoutNs)
        return SGEMM_STATUS_INVALID_VALUE;
    sg::launch_wait_selftest(h->d_err, timeout_ns, stream);
    return cudaGetLastError() == cudaSuccess ? SGEMM_STATUS_SUCCESS : SGEMM_STATUS_LAUNCH_FAILED;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point (sgemmNoAlloc).
//
// For callers that may not allocate device memory at all: code running where
// the allocator is off limits (inside a memory pool or allocator hook, under
// a framework that owns every byte of device memory, or in a process whose
// memory budget is fixed up front).  Its scratch (error word, stream-K flags
// and partial tiles, repacked operands) lives in one file-scope device array
// that every GPU loading this library holds until the process exits.

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;   // 32 MiB per device
constexpr size_t kStaticCtlBytes = kCtlBytes;               // control block (as a handle's)

}  // namespace

static __device__ __align__(256) unsigned char g_sgemm_static_scratch[kStaticScratchBytes];

namespace {

struct StaticScratchSlot {
    std::once_flag once;
    std::atomic<bool> ready{false};   // set-up ran (status below is final)
    sgemmStatus_t status = SGEMM_STATUS_INTERNAL_ERROR;
    unsigned char *ptr = nullptr;     // device address of g_sgemm_static_scratch
    int sm_count = 0;
    // Settings of this device's calls (host values; no device state).
    std::atomic<uint64_t> timeout_ns{kDefaultTimeoutNs};
    std::atomic<int> withhold{0};
};
StaticScratchSlot g_static_slots[kMaxDevices];

// Once per device, with that device current: the architecture check, the SM
// count, the array's device address (in host code its name is only a
// host-side stand-in), and every kernel this entry point can launch loaded
// up front -- each main-kernel configuration with its shared-memory opt-in
// and occupancy (cached per device), the small-product, skinny and
// auxiliary kernels -- so that no later call loads a module.  Looking up
// the address loads the module holding the array, which commits its memory.
void setup_static_scratch(StaticScratchSlot &slot, int dev) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        slot.status = SGEMM_STATUS_LAUNCH_FAILED;
        return;
    }
    if (major != 10 || minor != 3) {
        slot.status = SGEMM_STATUS_ARCH_MISMATCH;
        return;
    }
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_sgemm_static_scratch) != cudaSuccess || ptr == nullptr) {
        slot.status = SGEMM_STATUS_LAUNCH_FAILED;
        return;
    }
    std::call_once(g_kernels_once, init_kernel_table);
    for (auto &row : g_kernels)
        for (KernelEntry &e : row)
            if (e.fn != nullptr && occupancy_on(dev, e) < 1) {
                slot.status = SGEMM_STATUS_LAUNCH_FAILED;
                return;
            }
    if (sg::preload_small_kernels() != cudaSuccess || sg::preload_skinny_kernels() != cudaSuccess ||
        sg::preload_skinny_tma_kernels() != cudaSuccess || sg::preload_aux_kernels() != cudaSuccess ||
        encode_fn() == nullptr) {
        slot.status = SGEMM_STATUS_LAUNCH_FAILED;
        return;
    }
    slot.ptr = static_cast<unsigned char *>(ptr);
    slot.sm_count = sms;
    slot.status = SGEMM_STATUS_SUCCESS;
}

// The current device's slot, set up on first use.
sgemmStatus_t static_slot(StaticScratchSlot *&out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_STATUS_LAUNCH_FAILED;
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_STATUS_NOT_SUPPORTED;
    StaticScratchSlot &slot = g_static_slots[dev];
    std::call_once(slot.once, [&slot, dev] {
        setup_static_scratch(slot, dev);
        slot.ready.store(true);
    });
    out = &slot;
    return slot.status;
}

}  // namespace

extern "C" sgemmStatus_t sgemmNoAlloc(int64_t M, int64_t N, int64_t K, float alpha,
                                      const float *A, int64_t lda, const float *B, int64_t ldb,
                                      float beta, float *C, int64_t ldc, cudaStream_t stream) {
    sgemmStatus_t st = validate(M, N, K, A, lda, B, ldb, C, ldc, alpha != 0.0f);
    if (st != SGEMM_STATUS_SUCCESS || M == 0 || N == 0) return st;
    StaticScratchSlot *slot = nullptr;
    st = static_slot(slot);
    if (st != SGEMM_STATUS_SUCCESS) return st;
    int dev = -1;
    cudaGetDevice(&dev);

    // A context on the stack whose error word and workspace are carved out
    // of the static array.
    sgemmContext ctx;
    ctx.device = dev;
    ctx.sm_count = slot->sm_count;
    ctx.d_err = reinterpret_cast<uint32_t *>(slot->ptr);
    ctx.d_sk_seq = ctx.d_err + 1;
    ctx.d_flags = ctx.d_err + kCtlFlagsOffset;
    ctx.flag_words = kCtlFlagWords;
    ctx.ws = slot->ptr + kStaticCtlBytes;
    ctx.ws_bytes = kStaticScratchBytes - kStaticCtlBytes;
    ctx.timeout_ns = slot->timeout_ns.load();
    ctx.withhold = slot->withhold.load();

    Plan pl;
    st = make_plan(&ctx, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, pl);
    if (st != SGEMM_STATUS_SUCCESS) return st;
    // Operands that must be repacked have to fit in the static array;
    // stream-K scratch is used only when it fits as well.
    if (pl.ws_a + pl.ws_b > ctx.ws_bytes) return SGEMM_STATUS_NOT_SUPPORTED;
    return run(&ctx, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

extern "C" sgemmStatus_t sgemmNoAllocSetWaitTimeout(uint64_t timeout_ns) {
    if (timeout_ns < kMinTimeoutNs) return SGEMM_STATUS_INVALID_VALUE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_STATUS_LAUNCH_FAILED;
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_STATUS_NOT_SUPPORTED;
    g_static_slots[dev].timeout_ns.store(timeout_ns);
    return SGEMM_STATUS_SUCCESS;
}

extern "C" sgemmStatus_t sgemmNoAllocSetTestWithheldSignal(int which) {
    if (which < sg::kWithholdNone || which > sg::kWithholdRelease) return SGEMM_STATUS_INVALID_VALUE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_STATUS_LAUNCH_FAILED;
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_STATUS_NOT_SUPPORTED;
    g_static_slots[dev].withhold.store(which);
    return SGEMM_STATUS_SUCCESS;
}

extern "C" sgemmStatus_t sgemmNoAllocGetDeviceError(int *code) {
    if (code == nullptr) return SGEMM_STATUS_INVALID_VALUE;
    *code = 0;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_STATUS_LAUNCH_FAILED;
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_STATUS_NOT_SUPPORTED;
    StaticScratchSlot &slot = g_static_slots[dev];
    // No call has set up this device: no kernel of this path has run on it.
    if (!slot.ready.load()) return SGEMM_STATUS_SUCCESS;
    if (slot.status != SGEMM_STATUS_SUCCESS) return slot.status;
    uint32_t word = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&word, slot.ptr, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(slot.ptr, 0, sizeof(word)) != cudaSuccess)
        return SGEMM_STATUS_LAUNCH_FAILED;
    *code = int(word);
    return word == 0 ? SGEMM_STATUS_SUCCESS : SGEMM_STATUS_DEVICE_TIMEOUT;
}
