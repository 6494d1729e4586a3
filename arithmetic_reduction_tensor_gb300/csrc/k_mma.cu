// k_mma.cu -- MMA_CHAIN: the sum as chains of tensor-core multiply-
// accumulates against a ones matrix.
//
// "GPU Tensor Cores for fast Arithmetic Reductions" (arXiv 2001.05585),
// Abstract: the reduction of n numbers is encoded as chained m x m MMAs run
// in parallel on the tensor cores; each chain of R MMAs keeps its
// sub-result in 32-bit floating point, and the sub-results are then all
// reduced into a final 32-bit result; small thread blocks do best with
// R = 4 or 5, large ones with R = 1.
//
// Here m = 16 (mma.sync m16n8k16, fp16/bf16 in, fp32 accumulate), one MMA
// per coalesced 512-byte warp load, the lane's 16-byte vector used as its A
// fragment as loaded (MmaReducer in stream.cuh).  Chain sub-results are
// reduced in fp32: lane accumulators, the butterfly over row groups, the
// tree over a CTA's warps, and the combine kernel over CTA chunks.  Rows
// use one warp per row, so every load is a contiguous 512 bytes of the row.
// The sum of squares uses the same tiles with D = A * A^T (MmaSqReducer):
// a genuine contraction, two MMAs per tile.  Binary32 inputs are split
// exactly into three bfloat16 parts on the CUDA cores and the parts summed
// on the tensor cores, three MMAs per 256 inputs (MmaSplitReducer).
#include "stream.cuh"

namespace tcr {

template <int DT, int R, int OP, bool ALIGNED>
__global__ void __launch_bounds__(1024)
mma_chunk_kernel(const void *__restrict__ x, size_t seg_len, size_t units, size_t cps,
                 int chunk_log2, float *__restrict__ dst)
{
    chunk_body<MmaRed<DT, R, OP>, ALIGNED>(x, seg_len, units, cps, chunk_log2, dst);
}

template <int DT, int R, int OP, bool ALIGNED>
__global__ void __launch_bounds__(kRowsBlock, kRowsMinCtas)
mma_rows_warp_kernel(const void *__restrict__ x, size_t rows, size_t cols,
                     float *__restrict__ out)
{
    rows_body<MmaRed<DT, R, OP>, ALIGNED>(x, rows, cols, out);
}

// ---------------------------------------------------------------- host

template <int DT, int R, int OP>
static void *pick_dro(bool rows, bool aligned)
{
    if (rows) return aligned ? (void *)mma_rows_warp_kernel<DT, R, OP, true>
                             : (void *)mma_rows_warp_kernel<DT, R, OP, false>;
    return aligned ? (void *)mma_chunk_kernel<DT, R, OP, true>
                   : (void *)mma_chunk_kernel<DT, R, OP, false>;
}

template <int DT, int R>
static void *pick_dr(bool rows, int op, bool aligned)
{
    return op == kOpSquares ? pick_dro<DT, R, kOpSquares>(rows, aligned)
                            : pick_dro<DT, R, kOpSum>(rows, aligned);
}

template <int R>
static void *pick_r(bool rows, int dtype, int op, bool aligned)
{
    switch (dtype) {
    case kF16: return pick_dr<kF16, R>(rows, op, aligned);
    case kBF16: return pick_dr<kBF16, R>(rows, op, aligned);
    case kF32: return pick_dr<kF32, R>(rows, op, aligned);
    default: return nullptr;
    }
}

static void *pick(bool rows, int dtype, int op, bool aligned, int R)
{
    switch (R) {
    case 1: return pick_r<1>(rows, dtype, op, aligned);
    case 2: return pick_r<2>(rows, dtype, op, aligned);
    case 3: return pick_r<3>(rows, dtype, op, aligned);
    case 4: return pick_r<4>(rows, dtype, op, aligned);
    case 5: return pick_r<5>(rows, dtype, op, aligned);
    case 6: return pick_r<6>(rows, dtype, op, aligned);
    case 7: return pick_r<7>(rows, dtype, op, aligned);
    case 8: return pick_r<8>(rows, dtype, op, aligned);
    default: return nullptr;
    }
}

cudaError_t launch_mma_chunk(int dtype, int op, bool aligned, int R, const void *x,
                             size_t seg_len, size_t units, size_t cps, int chunk_log2, float *dst,
                             int grid, int block, cudaStream_t stream)
{
    void *k = pick(false, dtype, op, aligned, R);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&seg_len, (void *)&units, (void *)&cps,
                    (void *)&chunk_log2, (void *)&dst};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

cudaError_t launch_mma_rows(int dtype, int op, bool aligned, int R, const void *x, size_t rows,
                            size_t cols, float *out, int grid, int block, cudaStream_t stream)
{
    void *k = pick(true, dtype, op, aligned, R);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&rows, (void *)&cols, (void *)&out};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

cudaError_t preload_mma_chunk_sums()
{
    for (int R = 1; R <= 8; R++)
        for (int dt : {kF16, kBF16, kF32})
            for (bool aligned : {true, false}) {
                cudaFuncAttributes a;
                const cudaError_t e = cudaFuncGetAttributes(&a, pick(false, dt, kOpSum, aligned, R));
                if (e != cudaSuccess) return e;
            }
    return cudaSuccess;
}

}  // namespace tcr
