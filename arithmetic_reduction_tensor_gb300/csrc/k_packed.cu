// k_packed.cu -- launcher of the packed short-row kernels (packed.cuh).
#include <cstdint>

#include "packed.cuh"

namespace tcr {

static const void *pick(int family, int dtype, int op, int R, int vlog, int align, bool pair)
{
    switch (family) {
    case kPackedFixed: return packed_pick_fixed(dtype, op, vlog, align, pair);
    case kPackedShuffle: return packed_pick_shuffle(dtype, op, vlog, align, pair);
    case kPackedMma: return packed_pick_mma(dtype, op, vlog, R, align, pair);
    default: return nullptr;
    }
}

// Rows that are not 16-byte aligned but all start on a 4-byte boundary (x
// 4-byte aligned, a row a whole number of 4-byte words) are read with 8-byte
// loads (8-byte boundaries and words) or 4-byte loads instead of as
// realigned granules: the same vectors, the same bits.
static int align_class(int dtype, bool aligned, const void *x, size_t cols)
{
    if (aligned) return 1;
    const size_t eb = dtype == kF32 ? 4 : 2;
    return ((uintptr_t)x & 3u) == 0 && (cols * eb) % 4 == 0 ? 2 : 0;
}

int packed_rows_vlog(int family, size_t cols, int vector_len)
{
    const size_t nvec = (cols + (size_t)vector_len - 1) / (size_t)vector_len;
    int v = 0;
    while (((size_t)1 << v) < nvec) v++;
    if (family == kPackedMma && v < 2) v = 2;
    return v <= kPackedMaxVlog ? v : -1;
}

bool packed_rows_supported(int family, int dtype, int op, size_t cols, int vector_len, bool aligned,
                           bool pair)
{
    const int v = packed_rows_vlog(family, cols, vector_len);
    return cols > 0 && v >= 0 && pick(family, dtype, op, 1, v, aligned ? 1 : 0, pair) != nullptr;
}

size_t packed_rows_groups(size_t rows, int vlog)
{
    const size_t rpg = (size_t)256 >> vlog;
    return (rows + rpg - 1) / rpg;
}

cudaError_t launch_packed_rows(int family, int dtype, int op, int R, bool aligned, const void *x,
                               size_t rows, size_t cols, int vlog, float *out, int grid, int block,
                               cudaStream_t stream)
{
    const void *k = pick(family, dtype, op, R, vlog, align_class(dtype, aligned, x, cols), false);
    if (!k || block != kRowsBlock) return cudaErrorInvalidValue;
    float *none = nullptr;
    int mv = 0;
    void *args[] = {(void *)&x, (void *)&rows, (void *)&cols, (void *)&out, (void *)&none, (void *)&mv};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

cudaError_t launch_packed_rows_pair(int family, int dtype, int R, bool aligned, const void *x,
                                    size_t rows, size_t cols, int vlog, float *out_a, float *out_b,
                                    int mean_var, int grid, int block, cudaStream_t stream)
{
    const void *k = pick(family, dtype, kOpSum, R, vlog, align_class(dtype, aligned, x, cols), true);
    if (!k || block != kRowsBlock) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&rows, (void *)&cols, (void *)&out_a, (void *)&out_b,
                    (void *)&mean_var};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

int occupancy_packed(int family, int dtype, int op, int R, int vlog, bool aligned, bool pair)
{
    const void *k = pick(family, dtype, op, R, vlog, aligned ? 1 : 0, pair);
    int n = 0;
    if (!k || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kRowsBlock, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace tcr
