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

template <int DT, int OP, int AL, bool PAIR, int... VL>
static const void *by_vlog(int vlog, std::integer_sequence<int, VL...>)
{
    static const void *const k[] = {
        (const void *)packed_rows_kernel<DT, OP, TCR_PACKED_MODE, VL, 1, AL != 0, PAIR, AL == 2>...};
    return k[vlog];
}

template <int DT, int OP, bool PAIR>
static const void *by_align(int vlog, int align)
{
    using S = std::make_integer_sequence<int, kPackedMaxVlog + 1>;
    switch (align) {
    case 0: return by_vlog<DT, OP, 0, PAIR>(vlog, S{});
    case 1: return by_vlog<DT, OP, 1, PAIR>(vlog, S{});
    default: return by_vlog<DT, OP, 2, PAIR>(vlog, S{});
    }
}

template <int DT>
static const void *by_op(int op, int vlog, int align, bool pair)
{
    if (pair) return by_align<DT, kOpSum, true>(vlog, align);
    return op == kOpSquares ? by_align<DT, kOpSquares, false>(vlog, align)
                            : by_align<DT, kOpSum, false>(vlog, align);
}

const void *TCR_PACKED_PICK(int dtype, int op, int vlog, int align, bool pair)
{
    if (vlog < 0 || vlog > kPackedMaxVlog || align < 0 || align > 2) return nullptr;
    switch (dtype) {
    case kF16: return by_op<kF16>(op, vlog, align, pair);
    case kBF16: return by_op<kBF16>(op, vlog, align, pair);
    case kF32: return by_op<kF32>(op, vlog, align, pair);
    default: return nullptr;
    }
}

}  // namespace tcr
