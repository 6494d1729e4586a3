// kernels.cuh -- launchers of the reduction kernels (host side).
//
// Every launcher enqueues one kernel on `stream` and returns the launch
// status.  Sizes are in inputs; x points to 16-bit patterns (dtype kF16,
// kBF16) or binary32 values (kF32).  `op` is kOpSum (the sum of the inputs)
// or kOpSquares (the sum of their squares).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "config.cuh"

namespace tcr {

// A call's first kernel is launched with programmatic stream serialization:
// it may become resident, and run the set-up before its griddepcontrol.wait,
// while the stream's previous kernel finishes (every kernel launched this
// way waits before its first global memory access, and the library's
// kernels let their dependents launch as they start).
inline cudaError_t launch_first(const void *k, dim3 grid, dim3 block, void **args, size_t smem,
                                cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, k, args);
}

// ---- FIXED_ORDER (balanced tree over index order)
// Chunked: CTA work unit u = (segment u / cps, chunk u % cps); the chunk of
// 2^chunk_log2 inputs is split evenly over the CTA's warps; dst[u] is the
// chunk's aligned subtree.  vrun = 2 or 3 (sums only): the blocked order
// with runs of 2^vrun inputs inside each vector (3: 16-bit inputs only).
cudaError_t launch_fixed_chunk(int dtype, int op, bool aligned, const void *x, size_t seg_len,
                               size_t units, size_t cps, int chunk_log2, float *dst, int grid,
                               int block, cudaStream_t stream, int vrun = 0);
// One warp per row, rows <= kRowsWarpMaxBytes long: out[r] = row tree.
cudaError_t launch_fixed_rows_warp(int dtype, int op, bool aligned, const void *x, size_t rows,
                                   size_t cols, float *out, int grid, int block,
                                   cudaStream_t stream, int vrun = 0);

// ---- FIXED_ORDER, blocked order with runs longer than a vector
// (2^run_log2 inputs, run_log2 > log2 of the inputs per vector): each lane
// owns one run of a round of 32 runs; dst[u] is the chunk's aligned subtree
// (chunk 2^chunk_log2 = warps x span, span a whole number of rounds).  CTAs
// of at most 256 threads.
cudaError_t launch_blocked_chunk(int dtype, bool aligned, const void *x, size_t seg_len,
                                 size_t units, size_t cps, int chunk_log2, int run_log2,
                                 float *dst, int grid, int block, cudaStream_t stream);
// Rows whose pieces (max(run, 8 vectors) inputs each), padded to 2^lpr,
// number at most 16 (lpr <= 4): 32 >> lpr whole rows to a warp's round,
// out[r] = row r's value; one launch, no partials.
cudaError_t launch_blocked_rows(int dtype, bool aligned, const void *x, size_t rows, size_t cols,
                                int run_log2, int lpr, float *out, int grid, int block, cudaStream_t stream);

// ---- SHUFFLE_TREE (declared grid-stride order)
// Block team: grid = segments * G CTAs of Bt threads; CTA (s, b) writes its
// block value to dst[s * G + b].
cudaError_t launch_shuffle_block(int dtype, int op, bool aligned, const void *x, size_t seg_len,
                                 size_t segments, int G, float *dst, int block,
                                 cudaStream_t stream);
// Warp team (Bt = 32, G = 1): one warp per row, out[r] = warp value.
cudaError_t launch_shuffle_rows_warp(int dtype, int op, bool aligned, const void *x, size_t rows,
                                     size_t cols, float *out, int grid, int block,
                                     cudaStream_t stream);

// ---- MMA_CHAIN (tensor-core chains of R MMAs against a ones matrix)
cudaError_t launch_mma_chunk(int dtype, int op, bool aligned, int R, const void *x, size_t seg_len,
                             size_t units, size_t cps, int chunk_log2, float *dst, int grid,
                             int block, cudaStream_t stream);
// One warp per row, rows <= kRowsWarpMaxBytes long.
cudaError_t launch_mma_rows(int dtype, int op, bool aligned, int R, const void *x, size_t rows,
                            size_t cols, float *out, int grid, int block, cudaStream_t stream);

// ---- short rows, several to a warp group (packed.cuh): family kPackedFixed
// (FIXED_ORDER), kPackedShuffle (SHUFFLE_TREE, one-warp team) or kPackedMma
// (MMA_CHAIN, 16-bit sums).  A row takes 2^vlog vector slots
// (packed_rows_vlog: -1 when the row is too long to pack); `aligned` as for
// the launch (x 16-byte aligned and rows whole vectors; other rows that all
// start on an 8-byte boundary are read with 8-byte loads, the rest as
// realigned 16-byte granules); CTAs of kRowsBlock threads, one warp per
// group of 256 >> vlog rows.
constexpr int kPackedFixed = 0, kPackedShuffle = 1, kPackedMma = 2;
// pair: the kernel of tcr_reduce_rows_moments / _mean_var (out_a, out_b
// as for launch_rows_pair; op ignored).
int packed_rows_vlog(int family, size_t cols, int vector_len);
bool packed_rows_supported(int family, int dtype, int op, size_t cols, int vector_len, bool aligned,
                           bool pair);
size_t packed_rows_groups(size_t rows, int vlog);
cudaError_t launch_packed_rows(int family, int dtype, int op, int R, bool aligned, const void *x,
                               size_t rows, size_t cols, int vlog, float *out, int grid, int block,
                               cudaStream_t stream);
cudaError_t launch_packed_rows_pair(int family, int dtype, int R, bool aligned, const void *x,
                                    size_t rows, size_t cols, int vlog, float *out_a, float *out_b,
                                    int mean_var, int grid, int block, cudaStream_t stream);
int occupancy_packed(int family, int dtype, int op, int R, int vlog, bool aligned, bool pair);

// ---- MMA_CHAIN on tcgen05 (bulk copies into shared memory, D in TMEM):
// grid = tmem_units(n), one CTA per work unit, two resident per SM taking
// over the units of those not yet launched; dst[u] is the partial of work
// unit u (2^16 inputs, fewer for small n: 2^tmem_unit_log2(n)); x must be
// 16-byte aligned.  inject_stall: withhold the publication of the chain the
// epilogue waits for first, so that a wait runs out its limit (tests of the
// failure path only).
cudaError_t launch_mma_tmem(int dtype, int R, const uint16_t *x, size_t n, float *dst, int grid,
                            bool inject_stall, cudaStream_t stream);
size_t tmem_units(size_t n);
int tmem_block_threads();
int tmem_unit_log2(size_t n);
// Rows: rows of 1024 k columns (k a divisor or a multiple of 16) as one
// flat array of 32 KiB bulk copies, each lane group taking 1024 inputs of
// one row (grid = the units, one CTA per unit, taken over as for sums);
// other rows with one MMA tile holding 16 rows (8 of D's lanes to a row)
// from 3-D tensor-map or per-row bulk copies (at most one CTA per SM; grid
// from tmem_rows_grid).  dst[row * chunks + c] is row `row`'s partial over
// column chunk c (tmem_rows_chunks(cols) chunks per row; one chunk: dst is
// the output).  x must be 16-byte aligned and cols a multiple of 8, rows
// and cols < 2^31.
cudaError_t launch_mma_tmem_rows(int dtype, int R, const uint16_t *x, size_t rows, size_t cols,
                                 float *dst, int grid, bool inject_stall, cudaStream_t stream);
// The device word the tcgen05 kernels set when a wait gave up (bit 0);
// synchronous; optionally cleared after reading.
cudaError_t read_device_faults(unsigned int *flags, bool clear);
size_t tmem_rows_chunks(size_t cols);
size_t tmem_rows_units(size_t rows, size_t cols);
// CTAs to launch for the rows: one per unit for rows of 1024 k columns (k a
// divisor or a multiple of 16, read as a flat array), else at most one per
// SM; 0 when there are too many units for one launch.
int tmem_rows_grid(size_t rows, size_t cols, size_t sms);

// ---- sums and sums of squares in one pass (rows; the mean/variance calls)
// family: which mode's policies run side by side
constexpr int kPairFixed = 0, kPairShuffle = 1, kPairMma = 2;
// One warp per row (rows <= kRowsWarpMaxBytes): out_a[r], out_b[r] = the
// row's sum and sum of squares, or (mean_var != 0) its mean and variance.
cudaError_t launch_rows_pair(int family, int dtype, bool aligned, int R, const void *x, size_t rows,
                             size_t cols, float *out_a, float *out_b, int mean_var, int grid,
                             int block, cudaStream_t stream);
cudaError_t launch_mma_rows_pair(int dtype, bool aligned, int R, const void *x, size_t rows,
                                 size_t cols, float *out_a, float *out_b, int mean_var, int grid,
                                 int block, cudaStream_t stream);
// Chunked (FIXED, MMA): dst_a[u], dst_b[u] = work unit u's two partials.
cudaError_t launch_chunk_pair(int family, int dtype, bool aligned, int R, const void *x,
                              size_t seg_len, size_t units, size_t cps, int chunk_log2,
                              float *dst_a, float *dst_b, int grid, int block, cudaStream_t stream);
cudaError_t launch_mma_chunk_pair(int dtype, bool aligned, int R, const void *x, size_t seg_len,
                                  size_t units, size_t cps, int chunk_log2, float *dst_a,
                                  float *dst_b, int grid, int block, cudaStream_t stream);
// SHUFFLE_TREE block team: CTA (s, b) writes its two block values.
cudaError_t launch_shuffle_block_pair(int dtype, bool aligned, const void *x, size_t seg_len,
                                      size_t segments, int G, float *dst_a, float *dst_b, int block,
                                      cudaStream_t stream);
// mean[r], var[r] from s1[r], s2[r] (waits for the producing launch).
cudaError_t launch_mean_var(const float *s1, const float *s2, size_t rows, size_t cols, float *mean,
                            float *var, cudaStream_t stream);

// ---- split-K GEMM, C = A * W^T (k_gemm.cu): A M x K, W N x K row-major
// 16-bit (16-byte aligned, K a multiple of 8), out = C (splits == 1) or the
// partials P (splits x M x N); split s covers 64-column boxes
// [s * kbps, min((s + 1) * kbps, ceil(K / 64))).  Persistent CTA pairs
// (clusters of two SMs, 256 x 256 tiles, tcgen05.mma.cta_group::2), or one
// CTA per SM with 128 x 256 tiles where a pair cannot be scheduled.
// inject_stall: withhold the first tile's publication so that a wait runs
// out its limit (tests of the failure path only).
cudaError_t launch_gemm_splitk(int dtype, const void *A, const void *W, size_t M, size_t N, size_t K,
                               int splits, int kbps, float *out, bool inject_stall, cudaStream_t stream);
// The grid launch_gemm_splitk uses, and the output tile it works in.
int gemm_launch_grid(size_t M, size_t N, int splits);
int gemm_tile_m_run();
int gemm_tile_n_run();
// C[i] = balanced tree over P[s * mn + i] in split order (waits for the GEMM).
cudaError_t launch_splitk_combine(const float *P, size_t mn, int splits, float *C, cudaStream_t stream);
cudaError_t read_gemm_faults(unsigned int *flags, bool clear);
int gemm_tile_m();
int gemm_tile_n();
int gemm_tile_k();
int gemm_block_threads();

// ---- combine: out[s] = balanced tree over partials[s*count .. s*count+count-1]
// padded with -0.0; one CTA of 1024 threads per segment, or one thread per
// segment when count is small (the same tree either way).
cudaError_t launch_combine(const float *partials, size_t segments, size_t count, float *out,
                           cudaStream_t stream);

// Make the driver load every variant of a kernel family now (one
// cudaFuncGetAttributes per variant), so that no later launch of them loads
// code: the chunk kernels' sums (FIXED_ORDER plain tree; MMA_CHAIN at every
// R), for every input type and alignment, and the two combine kernels.
cudaError_t preload_fixed_chunk_sums();
cudaError_t preload_mma_chunk_sums();
cudaError_t preload_combine();


}  // namespace tcr
