// k_shuffle.cu -- SHUFFLE_TREE: the conventional GPU reduction, with its
// order declared.
//
// "GPU Tensor Cores for fast Arithmetic Reductions" (arXiv 2001.05585),
// Abstract, measures its method against a conventional GPU reduction; this
// is that reduction, written so that its order is a descriptor ("Taming
// Bitwise Behavior in GPU Kernels with Tensor Core", arXiv 2609.11356,
// Abstract): a team of G blocks of Bt threads reduces one segment;
//   thread g = b*Bt + t accumulates, starting from -0.0, the 8-input trees
//   of vectors g, g + G*Bt, g + 2*G*Bt, ... in that order;
//   a warp combines its lanes by the butterfly with offsets 16, 8, 4, 2, 1;
//   a block is the balanced tree over its warps; the segment is the
//   balanced tree over its G blocks (the combine kernel, when G > 1).
#include "stream.cuh"

namespace tcr {

constexpr int kShuffleUnroll = 8;    // vectors in flight per thread

// Block team: thread value = -0.0 + vector(first) + vector(first + stride)
// + ... in order, a vector being its 8-input tree; vectors past the
// segment are -0.0, the identity.  Software-pipelined: the next 8 vectors
// are loaded before the current 8 are added.  While every vector of a batch
// is whole (and the segment 16-byte aligned) the loads walk a pointer with
// no bounds checks; the ragged end continues, in the same order, with the
// checked loads.
template <int DT, int OP, bool ALIGNED>
__device__ __forceinline__ float grid_stride_acc(const uint16_t *seg, size_t len, size_t first,
                                                 size_t stride)
{
    constexpr int U = kShuffleUnroll;
    const size_t nvec = (len + 7) / 8;
    const uint4 pad = make_uint4(kNegZero2, kNegZero2, kNegZero2, kNegZero2);
    float acc = -0.0f;
    size_t v0 = first;
    if (ALIGNED) {
        const size_t nfull = len / 8;               // whole vectors
        if (v0 + (size_t)(U - 1) * stride < nfull) {
            const size_t step = 8 * stride;
            const uint16_t *p = seg + 8 * v0;
            uint4 q[U];
#pragma unroll
            for (int u = 0; u < U; u++) q[u] = ld_stream(p + (size_t)u * step);
            for (;;) {
                float t[U];
#pragma unroll
                for (int u = 0; u < U; u++) t[u] = tree8<DT, OP>(q[u]);
                v0 += (size_t)U * stride;
                p += (size_t)U * step;
                const bool more = v0 + (size_t)(U - 1) * stride < nfull;
                if (more) {
#pragma unroll
                    for (int u = 0; u < U; u++) q[u] = ld_stream(p + (size_t)u * step);
                }
#pragma unroll
                for (int u = 0; u < U; u++) acc = __fadd_rn(acc, t[u]);
                if (!more) break;
            }
        }
    }
    if (v0 >= nvec) return acc;
    uint4 q[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
        const size_t v = v0 + (size_t)u * stride;
        q[u] = v < nvec ? ld_vec<ALIGNED>(seg, len, v, 0x8000u) : pad;
    }
    for (; v0 < nvec; v0 += (size_t)U * stride) {
        float t[U];
#pragma unroll
        for (int u = 0; u < U; u++) t[u] = tree8<DT, OP>(q[u]);
        const size_t n0 = v0 + (size_t)U * stride;
#pragma unroll
        for (int u = 0; u < U; u++) {
            const size_t v = n0 + (size_t)u * stride;
            q[u] = v < nvec ? ld_vec<ALIGNED>(seg, len, v, 0x8000u) : pad;
        }
#pragma unroll
        for (int u = 0; u < U; u++) acc = __fadd_rn(acc, t[u]);
    }
    return acc;
}

template <int DT, int OP, bool ALIGNED>
__global__ void __launch_bounds__(1024)
shuffle_block_kernel(const uint16_t *__restrict__ x, size_t seg_len, int G,
                     float *__restrict__ dst)
{
    __shared__ float warp_val[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const size_t s = blockIdx.x / (unsigned)G;
    const size_t b = blockIdx.x - s * (unsigned)G;
    const uint16_t *seg = x + s * seg_len;
    const size_t stride = (size_t)G * blockDim.x;
    float acc = grid_stride_acc<DT, OP, ALIGNED>(seg, seg_len, b * blockDim.x + threadIdx.x, stride);
    pdl_launch_dependents();
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, off));
    if (lane == 0) warp_val[warp] = acc;
    __syncthreads();
    if (warp == 0) {
        float w = warp_tree_lane_order(lane < nwarps ? warp_val[lane] : -0.0f);
        if (lane == 0) dst[blockIdx.x] = w;
    }
}

// Warp team (Bt = 32, G = 1): one warp per segment; the warp stream's
// group order visits lane j's vectors j, j+32, j+64, ... in order.
template <int DT, int OP, bool ALIGNED>
__global__ void __launch_bounds__(kRowsBlock, kRowsMinCtas)
shuffle_rows_warp_kernel(const uint16_t *__restrict__ x, size_t rows, size_t cols,
                         float *__restrict__ out)
{
    rows_body<ShuffleReducer<DT, OP>, ALIGNED>(x, rows, cols, out);
}

// ---------------------------------------------------------------- host

template <template <int, int, bool> class K, typename F>
static F pick(int dtype, int op, bool aligned)
{
    if (dtype == kF16) {
        if (op == kOpSquares) return aligned ? (F)K<kF16, kOpSquares, true>::fn : (F)K<kF16, kOpSquares, false>::fn;
        return aligned ? (F)K<kF16, kOpSum, true>::fn : (F)K<kF16, kOpSum, false>::fn;
    }
    if (op == kOpSquares) return aligned ? (F)K<kBF16, kOpSquares, true>::fn : (F)K<kBF16, kOpSquares, false>::fn;
    return aligned ? (F)K<kBF16, kOpSum, true>::fn : (F)K<kBF16, kOpSum, false>::fn;
}

template <int DT, int OP, bool A>
struct BlockK {
    static constexpr auto fn = shuffle_block_kernel<DT, OP, A>;
};
template <int DT, int OP, bool A>
struct RowsK {
    static constexpr auto fn = shuffle_rows_warp_kernel<DT, OP, A>;
};

using BlockFn = void (*)(const uint16_t *, size_t, int, float *);
using RowsFn = void (*)(const uint16_t *, size_t, size_t, float *);

cudaError_t launch_shuffle_block(int dtype, int op, bool aligned, const uint16_t *x, size_t seg_len,
                                 size_t segments, int G, float *dst, int block,
                                 cudaStream_t stream)
{
    BlockFn k = pick<BlockK, BlockFn>(dtype, op, aligned);
    k<<<(unsigned)(segments * (size_t)G), block, 0, stream>>>(x, seg_len, G, dst);
    return cudaGetLastError();
}

cudaError_t launch_shuffle_rows_warp(int dtype, int op, bool aligned, const uint16_t *x, size_t rows,
                                     size_t cols, float *out, int grid, int block,
                                     cudaStream_t stream)
{
    RowsFn k = pick<RowsK, RowsFn>(dtype, op, aligned);
    k<<<grid, block, 0, stream>>>(x, rows, cols, out);
    return cudaGetLastError();
}

int occupancy_shuffle(bool rows, int dtype, int op, bool aligned, int block)
{
    int n = 0;
    cudaError_t e = rows ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                               &n, pick<RowsK, RowsFn>(dtype, op, aligned), block, 0)
                         : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                               &n, pick<BlockK, BlockFn>(dtype, op, aligned), block, 0);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace tcr
