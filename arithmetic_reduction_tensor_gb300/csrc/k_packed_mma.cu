// k_packed_mma.cu -- MMA_CHAIN short rows, several to a warp group
// (packed.cuh): sums, sums of squares, and both in one pass, of 16-bit and
// binary32 inputs.
// A row of at most 256 inputs is one tile, so the chain length matters only
// for rows spanning 2 or 4 loads; a chain longer than the row is the row's
// one chain (R is clamped to the loads per row).
#include "packed.cuh"

namespace tcr {

template <int DT, int OP, int AL, bool P>
static const void *pick(int vlog, int R)
{
    switch (vlog) {
    case 2: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 2, 1, AL != 0, P, AL == 2>;
    case 3: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 3, 1, AL != 0, P, AL == 2>;
    case 4: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 4, 1, AL != 0, P, AL == 2>;
    case 5: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 5, 1, AL != 0, P, AL == 2>;
    case 6:
        return R == 1 ? (const void *)packed_rows_kernel<DT, OP, kPackedMma, 6, 1, AL != 0, P, AL == 2>
                      : (const void *)packed_rows_kernel<DT, OP, kPackedMma, 6, 2, AL != 0, P, AL == 2>;
    case 7:
        switch (R) {
        case 1: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 7, 1, AL != 0, P, AL == 2>;
        case 2: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 7, 2, AL != 0, P, AL == 2>;
        case 3: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 7, 3, AL != 0, P, AL == 2>;
        default: return (const void *)packed_rows_kernel<DT, OP, kPackedMma, 7, 4, AL != 0, P, AL == 2>;
        }
    default: return nullptr;
    }
}

template <int DT, int OP, bool P>
static const void *by_align(int vlog, int R, int align)
{
    switch (align) {
    case 0: return pick<DT, OP, 0, P>(vlog, R);
    case 1: return pick<DT, OP, 1, P>(vlog, R);
    default: return pick<DT, OP, 2, P>(vlog, R);
    }
}

template <int DT>
static const void *by_pair(int op, int vlog, int R, int align, bool pair)
{
    if (pair) return by_align<DT, kOpSum, true>(vlog, R, align);
    if (op == kOpSquares) return by_align<DT, kOpSquares, false>(vlog, R, align);
    return by_align<DT, kOpSum, false>(vlog, R, align);
}

const void *packed_pick_mma(int dtype, int op, int vlog, int R, int align, bool pair)
{
    if (R < 1 || R > 8 || align < 0 || align > 2) return nullptr;
    switch (dtype) {
    case kF16: return by_pair<kF16>(op, vlog, R, align, pair);
    case kBF16: return by_pair<kBF16>(op, vlog, R, align, pair);
    case kF32: return by_pair<kF32>(op, vlog, R, align, pair);
    default: return nullptr;
    }
}

}  // namespace tcr
