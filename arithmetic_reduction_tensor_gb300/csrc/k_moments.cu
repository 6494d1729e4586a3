// k_moments.cu -- the sum and the sum of squares of every row in one pass,
// and the rows' mean and variance from them.
//
// Two reductions of one input, fused so that the input is read once: the
// cascaded reductions named by the "RedFuser" title in the list of work
// built on "GPU Tensor Cores for fast Arithmetic Reductions" (arXiv
// 2001.05585).  Each of the two values is the one the single reduction of
// the same mode gives -- the same kernels' policies (PairReducer in
// stream.cuh) run side by side on every group of loads -- so FIXED_ORDER and
// SHUFFLE_TREE stay bit-exact to their declared orders.  The mean and
// variance follow from the two sums by a declared binary32 formula
// (mean_var_of in common.cuh).  This file holds the ordered modes and the
// mean/variance epilogue; k_moments_mma.cu the tensor-core pairs.
#include <cstring>

#include "stream.cuh"

namespace tcr {

template <int DT>
using FixedPair = FixedPairReducer<DT, 4>;
template <int DT>
using FixedChunkPair = FixedPairReducer<DT, 3>;
template <int DT>
using ShufflePair = ShufflePairReducer<DT>;

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kRowsBlock, kRowsMinCtas)
fixed_rows_pair_kernel(const void *__restrict__ x, size_t rows, size_t cols,
                       float *__restrict__ out_a, float *__restrict__ out_b, int mean_var)
{
    rows_pair_body<FixedPair<DT>, ALIGNED>(x, rows, cols, out_a, out_b, mean_var);
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kRowsBlock, kRowsMinCtas)
shuffle_rows_pair_kernel(const void *__restrict__ x, size_t rows, size_t cols,
                         float *__restrict__ out_a, float *__restrict__ out_b, int mean_var)
{
    rows_pair_body<ShufflePair<DT>, ALIGNED>(x, rows, cols, out_a, out_b, mean_var);
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(1024)
fixed_chunk_pair_kernel(const void *__restrict__ x, size_t seg_len, size_t units, size_t cps,
                        int chunk_log2, float *__restrict__ dst_a, float *__restrict__ dst_b)
{
    chunk_pair_body<FixedChunkPair<DT>, ALIGNED>(x, seg_len, units, cps, chunk_log2, dst_a, dst_b);
}

// SHUFFLE_TREE block team, both sums: thread g accumulates the vector trees
// of the leaves and of their squares over vectors g, g + stride, ... in
// order (the declared order of each, side by side).
template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(1024)
shuffle_block_pair_kernel(const void *__restrict__ xv, size_t seg_len, int G,
                          float *__restrict__ dst_a, float *__restrict__ dst_b)
{
    pdl_launch_dependents();   // the combine may launch now; it waits for this grid to finish
    pdl_wait_primary();        // the stream's previous kernel has finished
    using T = typename Elem<DT>::T;
    constexpr int V = Elem<DT>::kPerVec;
    constexpr int U = 4;
    __shared__ float warp_val[2][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const size_t s = blockIdx.x / (unsigned)G;
    const size_t b = blockIdx.x - s * (unsigned)G;
    const T *seg = static_cast<const T *>(xv) + s * seg_len;
    const size_t stride = (size_t)G * blockDim.x;
    const size_t nvec = (seg_len + V - 1) / V;
    const uint32_t nz = Elem<DT>::kNegZeroWord;
    float acc_a = -0.0f, acc_b = -0.0f;
    uint4 q[U];
    size_t v0 = b * blockDim.x + threadIdx.x;
#pragma unroll
    for (int u = 0; u < U; u++) {
        const size_t v = v0 + (size_t)u * stride;
        q[u] = v < nvec ? ld_vec<DT, ALIGNED, true>(seg, seg_len, v) : make_uint4(nz, nz, nz, nz);
    }
    for (; v0 < nvec; v0 += (size_t)U * stride) {
        float ta[U], tb[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            ta[u] = vec_tree<DT, kOpSum>(q[u]);
            tb[u] = vec_tree<DT, kOpSquares>(q[u]);
        }
        const size_t n0 = v0 + (size_t)U * stride;
#pragma unroll
        for (int u = 0; u < U; u++) {
            const size_t v = n0 + (size_t)u * stride;
            q[u] = v < nvec ? ld_vec<DT, ALIGNED, true>(seg, seg_len, v) : make_uint4(nz, nz, nz, nz);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            acc_a = __fadd_rn(acc_a, ta[u]);
            acc_b = __fadd_rn(acc_b, tb[u]);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        acc_a = __fadd_rn(acc_a, __shfl_xor_sync(kFull, acc_a, off));
        acc_b = __fadd_rn(acc_b, __shfl_xor_sync(kFull, acc_b, off));
    }
    if (lane == 0) {
        warp_val[0][warp] = acc_a;
        warp_val[1][warp] = acc_b;
    }
    __syncthreads();
    if (warp == 0) {
        const float a = warp_tree_lane_order(lane < nwarps ? warp_val[0][lane] : -0.0f);
        const float c = warp_tree_lane_order(lane < nwarps ? warp_val[1][lane] : -0.0f);
        if (lane == 0) {
            dst_a[blockIdx.x] = a;
            dst_b[blockIdx.x] = c;
        }
    }
}

// mean[r], var[r] from s1[r], s2[r] (the chunked paths' epilogue).
__global__ void mean_var_kernel(const float *__restrict__ s1, const float *__restrict__ s2,
                                size_t rows, size_t cols, float *__restrict__ mean,
                                float *__restrict__ var)
{
    pdl_launch_dependents();
    pdl_wait_primary();
    for (size_t r = (size_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
         r += (size_t)gridDim.x * blockDim.x) {
        float m, v;
        mean_var_of(s1[r], s2[r], cols, m, v);
        mean[r] = m;
        var[r] = v;
    }
}

// ---------------------------------------------------------------- host

template <int DT>
static const void *pick_d(int which, bool aligned)
{
    switch (which) {
    case 0: return aligned ? (const void *)fixed_rows_pair_kernel<DT, true>
                           : (const void *)fixed_rows_pair_kernel<DT, false>;
    case 1: return aligned ? (const void *)shuffle_rows_pair_kernel<DT, true>
                           : (const void *)shuffle_rows_pair_kernel<DT, false>;
    case 2: return aligned ? (const void *)fixed_chunk_pair_kernel<DT, true>
                           : (const void *)fixed_chunk_pair_kernel<DT, false>;
    case 3: return aligned ? (const void *)shuffle_block_pair_kernel<DT, true>
                           : (const void *)shuffle_block_pair_kernel<DT, false>;
    default: return nullptr;
    }
}

static const void *pick(int which, int dtype, bool aligned)
{
    switch (dtype) {
    case kF16: return pick_d<kF16>(which, aligned);
    case kBF16: return pick_d<kBF16>(which, aligned);
    case kF32: return pick_d<kF32>(which, aligned);
    default: return nullptr;
    }
}

cudaError_t launch_rows_pair(int family, int dtype, bool aligned, int R, const void *x, size_t rows,
                             size_t cols, float *out_a, float *out_b, int mean_var, int grid,
                             int block, cudaStream_t stream)
{
    if (family == kPairMma)
        return launch_mma_rows_pair(dtype, aligned, R, x, rows, cols, out_a, out_b, mean_var, grid,
                                    block, stream);
    const void *k = pick(family == kPairFixed ? 0 : 1, dtype, aligned);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&rows, (void *)&cols, (void *)&out_a, (void *)&out_b,
                    (void *)&mean_var};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

cudaError_t launch_chunk_pair(int family, int dtype, bool aligned, int R, const void *x,
                              size_t seg_len, size_t units, size_t cps, int chunk_log2,
                              float *dst_a, float *dst_b, int grid, int block, cudaStream_t stream)
{
    if (family == kPairMma)
        return launch_mma_chunk_pair(dtype, aligned, R, x, seg_len, units, cps, chunk_log2, dst_a,
                                     dst_b, grid, block, stream);
    const void *k = family == kPairFixed ? pick(2, dtype, aligned) : nullptr;
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&seg_len, (void *)&units, (void *)&cps,
                    (void *)&chunk_log2, (void *)&dst_a, (void *)&dst_b};
    return launch_first(k, dim3(grid), dim3(block), args, 0, stream);
}

cudaError_t launch_shuffle_block_pair(int dtype, bool aligned, const void *x, size_t seg_len,
                                      size_t segments, int G, float *dst_a, float *dst_b, int block,
                                      cudaStream_t stream)
{
    const void *k = pick(3, dtype, aligned);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&seg_len, (void *)&G, (void *)&dst_a, (void *)&dst_b};
    return launch_first(k, dim3((unsigned)(segments * (size_t)G)), dim3(block), args, 0, stream);
}

cudaError_t launch_mean_var(const float *s1, const float *s2, size_t rows, size_t cols, float *mean,
                            float *var, cudaStream_t stream)
{
    if (rows == 0) return cudaSuccess;
    const size_t blocks = (rows + 255) / 256;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)(blocks < 1184 ? blocks : 1184));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mean_var_kernel, s1, s2, rows, cols, mean, var);
}

}  // namespace tcr
