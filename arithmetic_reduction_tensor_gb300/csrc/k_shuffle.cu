// k_shuffle.cu -- SHUFFLE_TREE: the conventional GPU reduction, with its
// order declared.
//
// "GPU Tensor Cores for fast Arithmetic Reductions" (arXiv 2001.05585),
// Abstract, measures its method against a conventional GPU reduction; this
// is that reduction, written so that its order is a descriptor ("Taming
// Bitwise Behavior in GPU Kernels with Tensor Core", arXiv 2609.11356,
// Abstract): a team of G blocks of Bt threads reduces one segment;
//   thread g = b*Bt + t accumulates, starting from -0.0, the trees of the
//   16-byte vectors (8 inputs of 16 bits, 4 of binary32) g, g + G*Bt,
//   g + 2*G*Bt, ... in that order;
//   a warp combines its lanes by the butterfly with offsets 16, 8, 4, 2, 1;
//   a block is the balanced tree over its warps; the segment is the
//   balanced tree over its G blocks (the combine kernel, when G > 1).
#include "stream.cuh"

namespace tcr {

constexpr int kShuffleUnroll = 8;    // vectors in flight per thread

// Block team: thread value = -0.0 + vector(first) + vector(first + stride)
// + ... in order, a vector being the tree over its 16 bytes of inputs;
// vectors past the segment are -0.0, the identity.  Software-pipelined:
// the next 8 vectors are loaded before the current 8 are added.  While
// every vector of a batch is whole (and the segment 16-byte aligned) the
// loads walk a pointer with no bounds checks; the ragged end continues, in
// the same order, with the checked loads.
template <int DT, int OP, bool ALIGNED>
__device__ __forceinline__ float grid_stride_acc(const typename Elem<DT>::T *seg, size_t len,
                                                 size_t first, size_t stride)
{
    constexpr int U = kShuffleUnroll;
    constexpr int V = Elem<DT>::kPerVec;
    const size_t nvec = (len + V - 1) / V;
    const uint32_t nz = Elem<DT>::kNegZeroWord;
    const uint4 pad = make_uint4(nz, nz, nz, nz);
    float acc = -0.0f;
    size_t v0 = first;
    if (ALIGNED) {
        const size_t nfull = len / V;               // whole vectors
        if (v0 + (size_t)(U - 1) * stride < nfull) {
            const size_t step = V * stride;
            const typename Elem<DT>::T *p = seg + V * v0;
            uint4 q[U];
#pragma unroll
            for (int u = 0; u < U; u++) q[u] = ld_stream(p + (size_t)u * step);
            for (;;) {
                float t[U];
#pragma unroll
                for (int u = 0; u < U; u++) t[u] = vec_tree<DT, OP>(q[u]);
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
        q[u] = v < nvec ? ld_vec<DT, ALIGNED, true>(seg, len, v) : pad;
    }
    for (; v0 < nvec; v0 += (size_t)U * stride) {
        float t[U];
#pragma unroll
        for (int u = 0; u < U; u++) t[u] = vec_tree<DT, OP>(q[u]);
        const size_t n0 = v0 + (size_t)U * stride;
#pragma unroll
        for (int u = 0; u < U; u++) {
            const size_t v = n0 + (size_t)u * stride;
            q[u] = v < nvec ? ld_vec<DT, ALIGNED, true>(seg, len, v) : pad;
        }
#pragma unroll
        for (int u = 0; u < U; u++) acc = __fadd_rn(acc, t[u]);
    }
    return acc;
}

// The same accumulation for a segment that does not start 16-byte aligned
// (see the unaligned segments of stream.cuh): thread g loads the 16-byte
// granule holding the first input of each of its vectors, lane 31 also the
// granule after it (the next vector belongs to the next warp's lane 0), and
// the vector is shifted out of its two granules by the segment's byte
// offset, P words then hs bits -- the same in every thread.  Four vectors
// in flight (their granules take the registers of eight vectors).  The loop
// runs while any lane of the warp has a vector, so every lane takes part
// in the shuffles; vectors past the segment are -0.0.
template <int DT, int OP, int P>
__device__ __forceinline__ float grid_stride_acc_unaligned(const typename Elem<DT>::T *seg, size_t len,
                                                           size_t first, size_t stride, uint32_t hs)
{
    constexpr int U = kShuffleUnroll / 2;
    constexpr int V = Elem<DT>::kPerVec;
    constexpr size_t EB = sizeof(typename Elem<DT>::T);
    const int lane = threadIdx.x & 31;
    const uintptr_t a = (uintptr_t)seg;
    const uint4 *g0 = reinterpret_cast<const uint4 *>(a & ~(uintptr_t)15);
    const size_t glim = ((size_t)(a & 15) + len * EB - 1) >> 4;      // last granule
    const size_t nvec = (len + V - 1) / V;
    const uint32_t f = Elem<DT>::kNegZeroWord;
    const uint4 pad = make_uint4(f, f, f, f);
    auto load = [&](size_t v0, uint4 (&q)[U], uint4 (&qt)[U]) {
#pragma unroll
        for (int u = 0; u < U; u++) {
            const size_t v = v0 + (size_t)u * stride;
            q[u] = v <= glim ? ld_stream(g0 + v) : pad;
            qt[u] = (lane == 31 && v + 1 <= glim) ? ld_stream(g0 + v + 1) : pad;
        }
    };
    float acc = -0.0f;
    size_t v0 = first;
    if (v0 - (size_t)lane >= nvec) return acc;
    uint4 q[U], qt[U];
    load(v0, q, qt);
    for (;;) {
        // the warp's last vector of this batch lies past a whole vector:
        // mask the inputs past the segment
        const bool tail = (v0 - (size_t)lane + 31 + (size_t)(U - 1) * stride + 1) * V > len;
        float t[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            uint4 hi;
            hi.x = __shfl_down_sync(kFull, q[u].x, 1);
            hi.y = __shfl_down_sync(kFull, q[u].y, 1);
            hi.z = __shfl_down_sync(kFull, q[u].z, 1);
            hi.w = __shfl_down_sync(kFull, q[u].w, 1);
            if (lane == 31) hi = qt[u];
            const uint32_t w[8] = {q[u].x, q[u].y, q[u].z, q[u].w, hi.x, hi.y, hi.z, hi.w};
            uint32_t o[4] = {__funnelshift_r(w[P], w[P + 1], hs), __funnelshift_r(w[P + 1], w[P + 2], hs),
                             __funnelshift_r(w[P + 2], w[P + 3], hs), __funnelshift_r(w[P + 3], w[P + 4], hs)};
            if (tail) {
                const long long left = (long long)len - (long long)(V * (v0 + (size_t)u * stride));
                const int cnt = left <= 0 ? 0 : (left >= V ? V : (int)left);
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int kb = cnt * 8 * (int)EB - 32 * i;
                    const uint32_t m = __funnelshift_lc(0xffffffffu, 0u, (uint32_t)(kb < 0 ? 0 : kb));
                    o[i] = (o[i] & m) | (f & ~m);
                }
            }
            t[u] = vec_tree<DT, OP>(make_uint4(o[0], o[1], o[2], o[3]));
        }
        v0 += (size_t)U * stride;
        const bool more = v0 - (size_t)lane < nvec;      // the same in every lane
        if (more) load(v0, q, qt);
#pragma unroll
        for (int u = 0; u < U; u++) acc = __fadd_rn(acc, t[u]);
        if (!more) break;
    }
    return acc;
}

template <int DT, int OP, bool ALIGNED>
__global__ void __launch_bounds__(1024)
shuffle_block_kernel(const void *__restrict__ xv, size_t seg_len, int G, float *__restrict__ dst)
{
    pdl_launch_dependents();   // the combine may launch now; it waits for this grid to finish
    pdl_wait_primary();        // the stream's previous kernel has finished
    using T = typename Elem<DT>::T;
    __shared__ float warp_val[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const size_t s = blockIdx.x / (unsigned)G;
    const size_t b = blockIdx.x - s * (unsigned)G;
    const T *seg = static_cast<const T *>(xv) + s * seg_len;
    const size_t stride = (size_t)G * blockDim.x;
    const size_t first = b * blockDim.x + threadIdx.x;
    float acc;
    if constexpr (ALIGNED) {
        acc = grid_stride_acc<DT, OP, true>(seg, seg_len, first, stride);
    } else {
        const uint32_t sb = (uint32_t)((uintptr_t)seg & 15), hs = (sb & 3u) * 8u;
        switch (sb >> 2) {                               // the same in every thread
        case 0: acc = grid_stride_acc_unaligned<DT, OP, 0>(seg, seg_len, first, stride, hs); break;
        case 1: acc = grid_stride_acc_unaligned<DT, OP, 1>(seg, seg_len, first, stride, hs); break;
        case 2: acc = grid_stride_acc_unaligned<DT, OP, 2>(seg, seg_len, first, stride, hs); break;
        default: acc = grid_stride_acc_unaligned<DT, OP, 3>(seg, seg_len, first, stride, hs); break;
        }
    }
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
shuffle_rows_warp_kernel(const void *__restrict__ x, size_t rows, size_t cols,
                         float *__restrict__ out)
{
    rows_body<ShuffleReducer<DT, OP>, ALIGNED>(x, rows, cols, out);
}

// ---------------------------------------------------------------- host

template <int DT, int OP>
static const void *pick_do(bool rows, bool aligned)
{
    if (rows) return aligned ? (const void *)shuffle_rows_warp_kernel<DT, OP, true>
                             : (const void *)shuffle_rows_warp_kernel<DT, OP, false>;
    return aligned ? (const void *)shuffle_block_kernel<DT, OP, true>
                   : (const void *)shuffle_block_kernel<DT, OP, false>;
}

template <int DT>
static const void *pick_d(bool rows, int op, bool aligned)
{
    return op == kOpSquares ? pick_do<DT, kOpSquares>(rows, aligned)
                            : pick_do<DT, kOpSum>(rows, aligned);
}

static const void *pick(bool rows, int dtype, int op, bool aligned)
{
    switch (dtype) {
    case kF16: return pick_d<kF16>(rows, op, aligned);
    case kBF16: return pick_d<kBF16>(rows, op, aligned);
    case kF32: return pick_d<kF32>(rows, op, aligned);
    default: return nullptr;
    }
}

cudaError_t launch_shuffle_block(int dtype, int op, bool aligned, const void *x, size_t seg_len,
                                 size_t segments, int G, float *dst, int block,
                                 cudaStream_t stream)
{
    const void *k = pick(false, dtype, op, aligned);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&seg_len, (void *)&G, (void *)&dst};
    return launch_first(k, dim3((unsigned)(segments * (size_t)G)), dim3(block), args, 0, stream);
}

cudaError_t launch_shuffle_rows_warp(int dtype, int op, bool aligned, const void *x, size_t rows,
                                     size_t cols, float *out, int grid, int block,
                                     cudaStream_t stream)
{
    const void *k = pick(true, dtype, op, aligned);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&rows, (void *)&cols, (void *)&out};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

}  // namespace tcr
