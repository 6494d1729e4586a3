// k_packed_mma.cu -- MMA_CHAIN short rows of 16-bit inputs, several to a
// warp group (packed.cuh).  A row of at most 256 inputs is one MMA, so the
// chain length matters only for rows spanning 2 or 4 loads; a chain longer
// than the row is the row's one chain (R is clamped to the loads per row).
#include "packed.cuh"

namespace tcr {

template <int DT, bool AL>
static const void *pick(int vlog, int R)
{
    switch (vlog) {
    case 2: return (const void *)packed_rows_kernel<DT, kOpSum, kPackedMma, 2, 1, AL>;
    case 3: return (const void *)packed_rows_kernel<DT, kOpSum, kPackedMma, 3, 1, AL>;
    case 4: return (const void *)packed_rows_kernel<DT, kOpSum, kPackedMma, 4, 1, AL>;
    case 5: return (const void *)packed_rows_kernel<DT, kOpSum, kPackedMma, 5, 1, AL>;
    case 6:
        return R == 1 ? (const void *)packed_rows_kernel<DT, kOpSum, kPackedMma, 6, 1, AL>
                      : (const void *)packed_rows_kernel<DT, kOpSum, kPackedMma, 6, 2, AL>;
    case 7:
        switch (R) {
        case 1: return (const void *)packed_rows_kernel<DT, kOpSum, kPackedMma, 7, 1, AL>;
        case 2: return (const void *)packed_rows_kernel<DT, kOpSum, kPackedMma, 7, 2, AL>;
        case 3: return (const void *)packed_rows_kernel<DT, kOpSum, kPackedMma, 7, 3, AL>;
        default: return (const void *)packed_rows_kernel<DT, kOpSum, kPackedMma, 7, 4, AL>;
        }
    default: return nullptr;
    }
}

const void *packed_pick_mma(int dtype, int vlog, int R, bool aligned)
{
    if (R < 1 || R > 8) return nullptr;
    switch (dtype) {
    case kF16: return aligned ? pick<kF16, true>(vlog, R) : pick<kF16, false>(vlog, R);
    case kBF16: return aligned ? pick<kBF16, true>(vlog, R) : pick<kBF16, false>(vlog, R);
    default: return nullptr;
    }
}

}  // namespace tcr
