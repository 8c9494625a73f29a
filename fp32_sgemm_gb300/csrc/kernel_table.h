// Registry of compiled main-kernel instantiations.  Each sgemm_algo*.cu
// translation unit instantiates one tile configuration (all four
// beta == 0 / beta != 0 x vector / scalar epilogue variants) so that the
// configurations compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include "sgemm_ffma.cuh"

namespace sg {

constexpr int kMaxDevices = 64;

struct KernelEntry {
    const void *fn;
    int threads;
    int smem;
    int bm, bn, bk, stages;
    int c_box_rows, c_box_cols;   // > 0: beta == 0 vector variant stores C by TMA, boxes of this size
    int occupancy[kMaxDevices];   // CTAs per SM, 0 = not yet queried
};

// Variant index: (beta != 0) * 2 + (scalar epilogue).
template <class Cfg, bool BZ, bool CV>
KernelEntry make_entry() {
    KernelEntry e{};
    e.fn = reinterpret_cast<const void *>(&sgemm_ffma_tma_kernel<Cfg, BZ, CV>);
    e.threads = Cfg::THREADS;
    e.smem = Cfg::SMEM_BYTES;
    e.bm = Cfg::BM;
    e.bn = Cfg::BN;
    e.bk = Cfg::BK;
    e.stages = Cfg::STAGES;
    if (Cfg::STORE_TMA && BZ && CV) {
        e.c_box_rows = Cfg::WTM;
        e.c_box_cols = Cfg::C_BOX_COLS;
    }
    return e;
}

template <class Cfg>
void fill_variants(KernelEntry *v) {
    v[0] = make_entry<Cfg, true, true>();
    v[1] = make_entry<Cfg, true, false>();
    v[2] = make_entry<Cfg, false, true>();
    v[3] = make_entry<Cfg, false, false>();
}

// Tile configurations are numbered 1..kNumAlgos (sgemmSetAlgo); the
// numbers of configurations measured slower and no longer built stay
// unused, so the shipped ones keep their numbers.
constexpr int kNumAlgos = 30;
constexpr int kShippedAlgos[] = {10, 16, 17, 18, 19, 20, 21, 23, 24, 27, 28, 29, 30};
constexpr bool algo_shipped(int algo) {
    for (int a : kShippedAlgos)
        if (a == algo) return true;
    return false;
}
void fill_algo10(KernelEntry *v);
void fill_algo16(KernelEntry *v);
void fill_algo17(KernelEntry *v);
void fill_algo18(KernelEntry *v);
void fill_algo19(KernelEntry *v);
void fill_algo20(KernelEntry *v);
void fill_algo21(KernelEntry *v);
void fill_algo23(KernelEntry *v);
void fill_algo24(KernelEntry *v);
void fill_algo27(KernelEntry *v);
void fill_algo28(KernelEntry *v);
void fill_algo29(KernelEntry *v);
void fill_algo30(KernelEntry *v);

// Tensor-core 3xTF32 path (sgemm_tf32x3.cu).
struct Tf32x3Args {
    int M, N, K;
    float alpha, beta;
    float *C;
    int64_t ldc;
    int64_t stride_c;
    int tiles_m, tiles_n, num_tiles;
    int k_blocks;
    int group_m;
    // Stream-K (as for the FFMA kernel): tiles >= sk_tile0 are cut into
    // (tile, K slice) units shared evenly by the CTAs; partial tiles go to
    // `partials` (one BM x BN slot per CTA) and each epilogue warp announces
    // its part by writing the launch tag to its word of `flags` (one per
    // CTA and epilogue warp).  sk_tile0 == num_tiles: none.
    int sk_tile0;
    float *partials;
    uint32_t *flags;
    uint32_t *sk_seq;    // {tag of the last completed launch, CTAs finished in this one}
    uint32_t *err;
    uint64_t timeout_ns;
    int withhold;        // test hook (Withhold): a signal left out on purpose
};
struct Tf32x3Info {
    const void *fn[4];   // variant index as for the FFMA kernels
    int threads, smem, bm, bn, bk, stages, chunk_kb;   // bm x bn: the tile
    int pair;            // 1: a cluster of 2 CTAs (an SM pair) per tile
    int box_a, box_b;    // rows of A, of B^T one CTA loads per stage
};
constexpr int kNumTf32x3Configs = 4;
Tf32x3Info tf32x3_info(int config);   // 1-based tile configuration
// Skinny products, M <= 32 or N <= 32 (sgemm_skinny.cu).
constexpr int kSkinnyMax = 32;
int skinny_splits(bool small_m, int M, int N, int K, int sms);
size_t skinny_workspace(int M, int N, int splits);
void launch_skinny(bool small_m, int M, int N, int K, float alpha, const float *A, int64_t lda,
                   const float *B, int64_t ldb, float beta, float *C, int64_t ldc, float *part,
                   int splits, cudaStream_t s);

// Small products (sgemm_small.cu): one CTA of 64 threads (or a cluster of
// `splits` CTAs sharing K) per 32 x 32 block of each C matrix, plain loads,
// K in 32-deep pieces.  Operands may be
// stored transposed (trans_a: A stored K x M; trans_b: B stored N x K);
// matrix z of an operand starts at base + z * stride.
constexpr int kSmallTile = 32, kSmallPiece = 32, kSmallMaxSplits = 8;
struct SmallArgs {
    int M, N, K;
    float alpha, beta;
    const float *A;
    int64_t lda, sa;
    const float *B;
    int64_t ldb, sb;
    float *C;
    int64_t ldc, sc;
    int splits;             // CTAs per block of C (a cluster), 1..kSmallMaxSplits
    int sms;                // SMs of the device
    int tiles_m, tiles_n;   // set by launch_small
};
int small_blocks(int M, int N, int batch);   // blocks of C in one launch (0: too many)
// K ranges per block: doubled while the pieces last and the launch stays
// within 4 CTAs per SM.
int small_splits(int M, int N, int K, int batch, int sms);
void launch_small(SmallArgs p, int trans_a, int trans_b, int batch, cudaStream_t s);

// TMA-fed skinny kernels (sgemm_skinny_tma.cu), for operands TMA reads in
// place.  A unit is one (output block, k-block) pair; CTA c of `ctas` takes
// units [c * units / ctas, (c + 1) * units / ctas) and writes one partial
// tile per output block its range meets (at most `segs`).
struct SkinnyTmaArgs {
    int M, N, K;
    int kb;              // k-blocks per output block
    int64_t units;       // output blocks x kb
    int ctas, segs, tile_elems;
    float *part;         // [ctas][segs][tile_elems]
    uint32_t *err;
    uint64_t timeout_ns;
};
struct SkinnyTmaGeom {
    int rows = 0;        // the small dimension rounded up to 1, 2, 4, 8, 16 or 32
    int kb = 0;
    int64_t units = 0;
    int ctas = 0, segs = 0, tile_elems = 0;
    size_t ws_bytes = 0;
    int a_box[2] = {0, 0}, b_box[2] = {0, 0};   // TMA boxes {inner, outer}
    bool a_swizzle64 = false;                    // A box with the 64-byte swizzle
};
SkinnyTmaGeom skinny_tma_geometry(bool small_m, int M, int N, int K, int sms);
// tmA: 2-D map of A (dims {K, M}); tmB: 2-D map of B (dims {N, K}); boxes as
// the geometry gives.  Launches the streaming kernel and the reduction.
void launch_skinny_tma(bool small_m, const CUtensorMap &tmA, const CUtensorMap &tmB,
                       const SkinnyTmaGeom &g, int M, int N, int K, float alpha, float beta,
                       float *C, int64_t ldc, float *part, uint32_t *err, uint64_t timeout_ns,
                       cudaStream_t s);

// Auxiliary kernels (sgemm_aux.cu); all take a batch (matrix z at base + z * stride).
void launch_scale_c(int M, int N, float beta, float *C, int64_t ldc, int64_t stride_c, int batch,
                    cudaStream_t s);
// One launch of operand preparation before the main kernel: up to two
// repacks (rows x cols matrices, batch of them, into pitch ld_dst) and the
// edge job (C's last r columns, r <= kEdgeMaxCols, that the main kernel
// leaves out).  Unused parts: npack = 0 / 1, edge.r = 0.
constexpr int kEdgeMaxCols = 8;
// The edge job's B columns (K x r floats) are staged whole in shared memory.
constexpr int kEdgeMaxStrip = 12288;   // floats (48 KB)
struct PackJob {
    const float *src;
    int64_t ld_src, s_src;
    float *dst;
    int64_t ld_dst, s_dst;
    int rows, cols, batch;
    int64_t groups, units;   // set by launch_prep
};
struct EdgeJob {
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    float *C;
    int64_t ldc;
    int M, K, n0, r;        // columns [n0, n0 + r) of C
    float alpha, beta;
};
struct PrepArgs {
    PackJob pack[2];
    int npack;
    EdgeJob edge;
    int edge_pack;       // pack job that is A (one batch entry): the edge products ride on its repack; -1: none
};
cudaError_t launch_prep(PrepArgs p, int sms, cudaStream_t s);
// src[r][c] -> dst[c][r]; with dst2 != NULL the TF32 split: dst = hi, dst2 = lo.
void launch_transpose(const float *src, int64_t ld_src, int64_t s_src, float *dst, float *dst2,
                      int64_t ld_dst, int64_t s_dst, int rows, int cols, int batch, cudaStream_t s);
void launch_split_rows(const float *src, int64_t ld_src, int64_t s_src, float *hi, float *lo,
                       int64_t ld_dst, int64_t s_dst, int rows, int cols, int batch, cudaStream_t s);
void launch_wait_selftest(uint32_t *err, uint64_t timeout_ns, cudaStream_t s);

// Load a kernel's code now rather than at its first launch (with lazy module
// loading the first launch would load it, which can commit device memory).
inline cudaError_t load_kernel(const void *fn) {
    cudaFuncAttributes a;
    return cudaFuncGetAttributes(&a, fn);
}
// Every kernel each translation unit can launch, loaded on the current
// device (the skinny TMA kernels also get their shared-memory opt-in).
cudaError_t preload_small_kernels();
cudaError_t preload_skinny_kernels();
cudaError_t preload_skinny_tma_kernels();
cudaError_t preload_aux_kernels();

}  // namespace sg
