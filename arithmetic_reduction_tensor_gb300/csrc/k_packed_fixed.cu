// k_packed_fixed.cu -- FIXED_ORDER short rows, several to a warp group
// (packed.cuh): sums, sums of squares, and both in one pass, of 16-bit and
// binary32 inputs.
#include <utility>

#include "packed.cuh"

#ifndef TCR_PACKED_MODE
#define TCR_PACKED_MODE kPackedFixed
#define TCR_PACKED_PICK packed_pick_fixed
#endif

namespace tcr {

template <int DT, int OP, bool AL, bool PAIR, int... VL>
static const void *by_vlog(int vlog, std::integer_sequence<int, VL...>)
{
    static const void *const k[] = {
        (const void *)packed_rows_kernel<DT, OP, TCR_PACKED_MODE, VL, 1, AL, PAIR>...};
    return k[vlog];
}

template <int DT, int OP, bool PAIR>
static const void *by_align(int vlog, bool aligned)
{
    using S = std::make_integer_sequence<int, kPackedMaxVlog + 1>;
    return aligned ? by_vlog<DT, OP, true, PAIR>(vlog, S{}) : by_vlog<DT, OP, false, PAIR>(vlog, S{});
}

template <int DT>
static const void *by_op(int op, int vlog, bool aligned, bool pair)
{
    if (pair) return by_align<DT, kOpSum, true>(vlog, aligned);
    return op == kOpSquares ? by_align<DT, kOpSquares, false>(vlog, aligned)
                            : by_align<DT, kOpSum, false>(vlog, aligned);
}

const void *TCR_PACKED_PICK(int dtype, int op, int vlog, bool aligned, bool pair)
{
    if (vlog < 0 || vlog > kPackedMaxVlog) return nullptr;
    switch (dtype) {
    case kF16: return by_op<kF16>(op, vlog, aligned, pair);
    case kBF16: return by_op<kBF16>(op, vlog, aligned, pair);
    case kF32: return by_op<kF32>(op, vlog, aligned, pair);
    default: return nullptr;
    }
}

}  // namespace tcr
