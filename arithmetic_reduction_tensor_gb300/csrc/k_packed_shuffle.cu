// k_packed_shuffle.cu -- SHUFFLE_TREE short rows (one-warp team), several to a warp group
// (packed.cuh): sums and sums of squares of 16-bit and binary32 inputs.
#include <utility>

#include "packed.cuh"

namespace tcr {

template <int DT, int OP, bool AL, int... VL>
static const void *by_vlog(int vlog, std::integer_sequence<int, VL...>)
{
    static const void *const k[] = {(const void *)packed_rows_kernel<DT, OP, kPackedShuffle, VL, 1, AL>...};
    return k[vlog];
}

template <int DT, int OP>
static const void *by_align(int vlog, bool aligned)
{
    using S = std::make_integer_sequence<int, kPackedMaxVlog + 1>;
    return aligned ? by_vlog<DT, OP, true>(vlog, S{}) : by_vlog<DT, OP, false>(vlog, S{});
}

template <int DT>
static const void *by_op(int op, int vlog, bool aligned)
{
    return op == kOpSquares ? by_align<DT, kOpSquares>(vlog, aligned) : by_align<DT, kOpSum>(vlog, aligned);
}

const void *packed_pick_shuffle(int dtype, int op, int vlog, bool aligned)
{
    if (vlog < 0 || vlog > kPackedMaxVlog) return nullptr;
    switch (dtype) {
    case kF16: return by_op<kF16>(op, vlog, aligned);
    case kBF16: return by_op<kBF16>(op, vlog, aligned);
    case kF32: return by_op<kF32>(op, vlog, aligned);
    default: return nullptr;
    }
}

}  // namespace tcr
