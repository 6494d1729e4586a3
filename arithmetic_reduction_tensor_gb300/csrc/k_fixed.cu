// k_fixed.cu -- FIXED_ORDER: the balanced binary32 tree over index order.
//
// The order is the one of "Taming Bitwise Behavior in GPU Kernels with
// Tensor Core" (arXiv 2609.11356), Abstract: a balanced-tree reduction, so
// that every launch configuration lands in one bit-equivalence class.  The
// tree is over the segment's inputs in index order, power-of-two aligned,
// padded with -0.0.  Because every piece of work here is an aligned subtree
// -- an 8-input vector, a 2048-input warp group, a warp span, a CTA chunk,
// the partials above them -- any split of the work computes the same nodes,
// and the result depends only on the inputs and the segment length.
//
// The leaves are placed for speed: a warp group holds 8 coalesced warp
// loads, and the reduce-scatter butterfly of group_tree (stream.cuh) forms
// the group's 11 tree levels with 12 shuffles -- the "data-layout
// optimisation" idea of the same Abstract applied inside a warp, so the
// fixed order costs few instructions over a free order.
#include "stream.cuh"

namespace tcr {

template <int DT, int OP, bool ALIGNED>
__global__ void __launch_bounds__(1024)
fixed_chunk_kernel(const uint16_t *__restrict__ x, size_t seg_len, size_t units, size_t cps,
                   int chunk_log2, float *__restrict__ dst)
{
    // a chunk of 2^13 inputs per warp: 4 groups per span, < 2^3
    chunk_body<FixedReducer<DT, OP, 3>, ALIGNED>(x, seg_len, units, cps, chunk_log2, dst);
}

template <int DT, int OP, bool ALIGNED>
__global__ void __launch_bounds__(kRowsBlock, kRowsMinCtas)
fixed_rows_warp_kernel(const uint16_t *__restrict__ x, size_t rows, size_t cols,
                       float *__restrict__ out)
{
    // rows of at most kRowsWarpMaxCols = 8 groups, < 2^4
    rows_body<FixedReducer<DT, OP, 4>, ALIGNED>(x, rows, cols, out);
}

// ---------------------------------------------------------------- host

template <template <int, int, bool> class K, typename F>
static F pick(int dtype, int op, bool aligned)
{
    if (dtype == kF16) {
        if (op == kOpSquares) return aligned ? (F)K<kF16, kOpSquares, true>::fn : (F)K<kF16, kOpSquares, false>::fn;
        return aligned ? (F)K<kF16, kOpSum, true>::fn : (F)K<kF16, kOpSum, false>::fn;
    }
    if (op == kOpSquares) return aligned ? (F)K<kBF16, kOpSquares, true>::fn : (F)K<kBF16, kOpSquares, false>::fn;
    return aligned ? (F)K<kBF16, kOpSum, true>::fn : (F)K<kBF16, kOpSum, false>::fn;
}

template <int DT, int OP, bool A>
struct ChunkK {
    static constexpr auto fn = fixed_chunk_kernel<DT, OP, A>;
};
template <int DT, int OP, bool A>
struct RowsK {
    static constexpr auto fn = fixed_rows_warp_kernel<DT, OP, A>;
};

using ChunkFn = void (*)(const uint16_t *, size_t, size_t, size_t, int, float *);
using RowsFn = void (*)(const uint16_t *, size_t, size_t, float *);

cudaError_t launch_fixed_chunk(int dtype, int op, bool aligned, const uint16_t *x, size_t seg_len,
                               size_t units, size_t cps, int chunk_log2, float *dst, int grid,
                               int block, cudaStream_t stream)
{
    ChunkFn k = pick<ChunkK, ChunkFn>(dtype, op, aligned);
    k<<<grid, block, 0, stream>>>(x, seg_len, units, cps, chunk_log2, dst);
    return cudaGetLastError();
}

cudaError_t launch_fixed_rows_warp(int dtype, int op, bool aligned, const uint16_t *x, size_t rows,
                                   size_t cols, float *out, int grid, int block,
                                   cudaStream_t stream)
{
    RowsFn k = pick<RowsK, RowsFn>(dtype, op, aligned);
    k<<<grid, block, 0, stream>>>(x, rows, cols, out);
    return cudaGetLastError();
}

int occupancy_fixed(bool rows, int dtype, int op, bool aligned, int block)
{
    int n = 0;
    cudaError_t e = rows ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                               &n, pick<RowsK, RowsFn>(dtype, op, aligned), block, 0)
                         : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                               &n, pick<ChunkK, ChunkFn>(dtype, op, aligned), block, 0);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace tcr
