// k_combine.cu -- deterministic combine of per-CTA partials.
//
// "GPU Tensor Cores for fast Arithmetic Reductions" (arXiv 2001.05585),
// Abstract: all chain sub-results are reduced into a final 32-bit result.
// Here the partials of one segment are combined by the balanced binary32
// tree over partial index, padded with -0.0 -- the upper levels of the
// FIXED_ORDER tree, the grid level of the declared SHUFFLE_TREE order, and
// the final fp32 reduction of the MMA_CHAIN sub-results.  No atomics: the
// order is fixed by the tree alone.
#include "common.cuh"
#include "kernels.cuh"

namespace tcr {

__global__ void __launch_bounds__(1024)
combine_kernel(const float *__restrict__ partials, size_t count, float *__restrict__ out)
{
    __shared__ float warp_val[32];
    const float *p = partials + (size_t)blockIdx.x * count;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    // 1024 threads; thread t owns the aligned subtree of leaves
    // [t*M, t*M + M), M = 2^max(0, ceil(log2 count) - 10)
    const int h = ceil_log2_sz(count);
    const size_t M = (size_t)1 << (h > 10 ? h - 10 : 0);
    const size_t lo = (size_t)t * M;
    TreeCounter<24> tc;
    for (size_t i = 0; i < M; i++) {
        if (lo + i >= count) break;
        tc.push(__ldg(p + lo + i));
    }
    float v = warp_tree_lane_order(tc.finish());
    if (lane == 0) warp_val[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float w = warp_tree_lane_order(warp_val[lane]);
        if (lane == 0) out[blockIdx.x] = w;
    }
}

cudaError_t launch_combine(const float *partials, size_t segments, size_t count, float *out,
                           cudaStream_t stream)
{
    combine_kernel<<<(unsigned)segments, 1024, 0, stream>>>(partials, count, out);
    return cudaGetLastError();
}

}  // namespace tcr
