// k_moments_mma.cu -- MMA_CHAIN's sum and sum of squares of every row in
// one pass: the chains against ones (MmaReducer, or the binary32 split) and
// the A * A^T diagonal chains (MmaSqReducer) run on the same registers of
// every warp load (PairReducer in stream.cuh); see k_moments.cu.
#include "stream.cuh"

namespace tcr {

template <int DT, int R>
using MmaPair = PairReducer<MmaRed<DT, R, kOpSum>, MmaRed<DT, R, kOpSquares>>;

template <int DT, int R, bool ALIGNED>
__global__ void __launch_bounds__(kRowsBlock, kRowsMinCtas)
mma_rows_pair_kernel(const void *__restrict__ x, size_t rows, size_t cols,
                     float *__restrict__ out_a, float *__restrict__ out_b, int mean_var)
{
    rows_pair_body<MmaPair<DT, R>, ALIGNED>(x, rows, cols, out_a, out_b, mean_var);
}

template <int DT, int R, bool ALIGNED>
__global__ void __launch_bounds__(1024)
mma_chunk_pair_kernel(const void *__restrict__ x, size_t seg_len, size_t units, size_t cps,
                      int chunk_log2, float *__restrict__ dst_a, float *__restrict__ dst_b)
{
    chunk_pair_body<MmaPair<DT, R>, ALIGNED>(x, seg_len, units, cps, chunk_log2, dst_a, dst_b);
}

template <int DT, int R>
static const void *pick_dr(bool rows, bool aligned)
{
    if (rows) return aligned ? (const void *)mma_rows_pair_kernel<DT, R, true>
                             : (const void *)mma_rows_pair_kernel<DT, R, false>;
    return aligned ? (const void *)mma_chunk_pair_kernel<DT, R, true>
                   : (const void *)mma_chunk_pair_kernel<DT, R, false>;
}

template <int R>
static const void *pick_r(bool rows, int dtype, bool aligned)
{
    switch (dtype) {
    case kF16: return pick_dr<kF16, R>(rows, aligned);
    case kBF16: return pick_dr<kBF16, R>(rows, aligned);
    case kF32: return pick_dr<kF32, R>(rows, aligned);
    default: return nullptr;
    }
}

static const void *pick(bool rows, int dtype, bool aligned, int R)
{
    switch (R) {
    case 1: return pick_r<1>(rows, dtype, aligned);
    case 2: return pick_r<2>(rows, dtype, aligned);
    case 3: return pick_r<3>(rows, dtype, aligned);
    case 4: return pick_r<4>(rows, dtype, aligned);
    case 5: return pick_r<5>(rows, dtype, aligned);
    case 6: return pick_r<6>(rows, dtype, aligned);
    case 7: return pick_r<7>(rows, dtype, aligned);
    case 8: return pick_r<8>(rows, dtype, aligned);
    default: return nullptr;
    }
}

cudaError_t launch_mma_rows_pair(int dtype, bool aligned, int R, const void *x, size_t rows,
                                 size_t cols, float *out_a, float *out_b, int mean_var, int grid,
                                 int block, cudaStream_t stream)
{
    const void *k = pick(true, dtype, aligned, R);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&rows, (void *)&cols, (void *)&out_a, (void *)&out_b,
                    (void *)&mean_var};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

cudaError_t launch_mma_chunk_pair(int dtype, bool aligned, int R, const void *x, size_t seg_len,
                                  size_t units, size_t cps, int chunk_log2, float *dst_a,
                                  float *dst_b, int grid, int block, cudaStream_t stream)
{
    const void *k = pick(false, dtype, aligned, R);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&seg_len, (void *)&units, (void *)&cps,
                    (void *)&chunk_log2, (void *)&dst_a, (void *)&dst_b};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

}  // namespace tcr
