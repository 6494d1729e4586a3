// k_fixed.cu -- FIXED_ORDER: the balanced binary32 tree over index order.
//
// The order is the one of "Taming Bitwise Behavior in GPU Kernels with
// Tensor Core" (arXiv 2609.11356), Abstract: a balanced-tree reduction, so
// that every launch configuration lands in one bit-equivalence class.  The
// tree is over the segment's inputs in index order, power-of-two aligned,
// padded with -0.0.  Because every piece of work here is an aligned subtree
// -- a 16-byte vector (8 or 4 inputs), a warp group of 256 vectors, a warp
// span, a CTA chunk, the partials above them -- any split of the work
// computes the same nodes, and the result depends only on the inputs and
// the segment length.
//
// The leaves are placed for speed: a warp group holds 8 coalesced warp
// loads, and the reduce-scatter butterfly of group_tree (stream.cuh) forms
// the group's 8 tree levels above the vectors with 12 shuffles -- the "data-layout
// optimisation" idea of the same Abstract applied inside a warp, so the
// fixed order costs few instructions over a free order.
#include "stream.cuh"

namespace tcr {

template <int DT, int OP, bool ALIGNED, int VRUN>
__global__ void __launch_bounds__(1024)
fixed_chunk_kernel(const void *__restrict__ x, size_t seg_len, size_t units, size_t cps,
                   int chunk_log2, float *__restrict__ dst)
{
    // a warp span of 4 groups, < 2^3
    chunk_body<FixedReducer<DT, OP, 3, VRUN>, ALIGNED>(x, seg_len, units, cps, chunk_log2, dst);
}

template <int DT, int OP, bool ALIGNED, int VRUN>
__global__ void __launch_bounds__(kRowsBlock, kRowsMinCtas)
fixed_rows_warp_kernel(const void *__restrict__ x, size_t rows, size_t cols,
                       float *__restrict__ out)
{
    // rows of at most kRowsWarpMaxBytes = 8 groups, < 2^4
    rows_body<FixedReducer<DT, OP, 4, VRUN>, ALIGNED>(x, rows, cols, out);
}

// ---------------------------------------------------------------- host

template <int DT, int OP, int VRUN>
static const void *pick_dov(bool rows, bool aligned)
{
    if (rows) return aligned ? (const void *)fixed_rows_warp_kernel<DT, OP, true, VRUN>
                             : (const void *)fixed_rows_warp_kernel<DT, OP, false, VRUN>;
    return aligned ? (const void *)fixed_chunk_kernel<DT, OP, true, VRUN>
                   : (const void *)fixed_chunk_kernel<DT, OP, false, VRUN>;
}

// vrun: 0 the balanced tree; 2 or 3 (sums only) runs of 4 or 8 inputs inside
// a vector (3 for 16-bit inputs only)
template <int DT>
static const void *pick_d(bool rows, int op, bool aligned, int vrun)
{
    if (vrun == 0)
        return op == kOpSquares ? pick_dov<DT, kOpSquares, 0>(rows, aligned)
                                : pick_dov<DT, kOpSum, 0>(rows, aligned);
    if (op != kOpSum) return nullptr;
    if (vrun == 2) return pick_dov<DT, kOpSum, 2>(rows, aligned);
    if constexpr (Elem<DT>::kPerVec == 8) {
        if (vrun == 3) return pick_dov<DT, kOpSum, 3>(rows, aligned);
    }
    return nullptr;
}

static const void *pick(bool rows, int dtype, int op, bool aligned, int vrun)
{
    switch (dtype) {
    case kF16: return pick_d<kF16>(rows, op, aligned, vrun);
    case kBF16: return pick_d<kBF16>(rows, op, aligned, vrun);
    case kF32: return pick_d<kF32>(rows, op, aligned, vrun);
    default: return nullptr;
    }
}

cudaError_t launch_fixed_chunk(int dtype, int op, bool aligned, const void *x, size_t seg_len,
                               size_t units, size_t cps, int chunk_log2, float *dst, int grid,
                               int block, cudaStream_t stream, int vrun)
{
    const void *k = pick(false, dtype, op, aligned, vrun);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&seg_len, (void *)&units, (void *)&cps,
                    (void *)&chunk_log2, (void *)&dst};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

cudaError_t launch_fixed_rows_warp(int dtype, int op, bool aligned, const void *x, size_t rows,
                                   size_t cols, float *out, int grid, int block,
                                   cudaStream_t stream, int vrun)
{
    const void *k = pick(true, dtype, op, aligned, vrun);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&rows, (void *)&cols, (void *)&out};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

cudaError_t preload_fixed_chunk_sums()
{
    for (int dt : {kF16, kBF16, kF32})
        for (bool aligned : {true, false}) {
            cudaFuncAttributes a;
            const cudaError_t e = cudaFuncGetAttributes(&a, pick(false, dt, kOpSum, aligned, 0));
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

}  // namespace tcr
