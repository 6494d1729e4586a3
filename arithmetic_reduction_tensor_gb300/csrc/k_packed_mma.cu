// k_packed_mma.cu -- MMA_CHAIN short rows, several to a warp group
// (packed.cuh): sums, sums of squares, and both in one pass, of 16-bit and
// binary32 inputs.
// A row of at most 256 inputs is one tile, so the chain length matters only
// for rows spanning 2 or 4 loads; a chain longer than the row is the row's
// one chain (R is clamped to the loads per row).
#include "packed.cuh"

namespace tcr {

template <int DT, int OP, bool AL, bool P>
static const void *pick(int vlog, int R)
{
    switch (vlog) {
    case 2: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 2, 1, AL, P>;
    case 3: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 3, 1, AL, P>;
    case 4: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 4, 1, AL, P>;
    case 5: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 5, 1, AL, P>;
    case 6:
        return R == 1 ? (const void *)packed_rows_kernel<DT, OP, kPackedMma, 6, 1, AL, P>
                      : (const void *)packed_rows_kernel<DT, OP, kPackedMma, 6, 2, AL, P>;
    case 7:
        switch (R) {
        case 1: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 7, 1, AL, P>;
        case 2: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 7, 2, AL, P>;
        case 3: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 7, 3, AL, P>;
        default: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 7, 4, AL, P>;
        }
    default: return nullptr;
    }
}

template <int DT>
static const void *by_pair(int op, int vlog, int R, bool aligned, bool pair)
{
    if (pair) return aligned ? pick<DT, kOpSum, true, true>(vlog, R) : pick<DT, kOpSum, false, true>(vlog, R);
    if (op == kOpSquares)
        return aligned ? pick<DT, kOpSquares, true, false>(vlog, R) : pick<DT, kOpSquares, false, false>(vlog, R);
    return aligned ? pick<DT, kOpSum, true, false>(vlog, R) : pick<DT, kOpSum, false, false>(vlog, R);
}

const void *packed_pick_mma(int dtype, int op, int vlog, int R, bool aligned, bool pair)
{
    if (R < 1 || R > 8) return nullptr;
    switch (dtype) {
    case kF16: return by_pair<kF16>(op, vlog, R, aligned, pair);
    case kBF16: return by_pair<kBF16>(op, vlog, R, aligned, pair);
    case kF32: return by_pair<kF32>(op, vlog, R, aligned, pair);
    default: return nullptr;
    }
}

}  // namespace tcr
