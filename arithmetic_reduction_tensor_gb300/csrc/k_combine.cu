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

// Aligned subtree of the W partials p[lo .. lo+W) (those past count are
// -0.0), all loaded before any is added.
template <int W>
__device__ __forceinline__ float leaf_tree(const float *__restrict__ p, size_t lo, size_t count)
{
    float v[W];
    if (W >= 4 && lo + W <= count && (((uintptr_t)(p + lo)) & 15u) == 0) {
#pragma unroll
        for (int i = 0; i < W / 4; i++) {
            const float4 f = __ldg(reinterpret_cast<const float4 *>(p + lo) + i);
            v[4 * i] = f.x;
            v[4 * i + 1] = f.y;
            v[4 * i + 2] = f.z;
            v[4 * i + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < W; i++) v[i] = lo + i < count ? __ldg(p + lo + i) : -0.0f;
    }
#pragma unroll
    for (int w = 1; w < W; w <<= 1)
#pragma unroll
        for (int i = 0; i < W; i += 2 * w) v[i] = __fadd_rn(v[i], v[i + w]);
    return v[0];
}

__global__ void __launch_bounds__(1024)
combine_kernel(const float *__restrict__ partials, size_t count, float *__restrict__ out)
{
    __shared__ float warp_val[32];
    // the partials are written by the kernel launched just before this one
    pdl_launch_dependents();   // the next call's first kernel may launch; it waits for this one
    pdl_wait_primary();
    const float *p = partials + (size_t)blockIdx.x * count;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    // 1024 threads; thread t owns the aligned subtree of leaves
    // [t*M, t*M + M), M = 2^max(0, ceil(log2 count) - 10)
    const int h = ceil_log2_sz(count);
    const size_t M = (size_t)1 << (h > 10 ? h - 10 : 0);
    const size_t lo = (size_t)t * M;
    float v;
    switch (M) {
    case 1: v = leaf_tree<1>(p, lo, count); break;
    case 2: v = leaf_tree<2>(p, lo, count); break;
    case 4: v = leaf_tree<4>(p, lo, count); break;
    case 8: v = leaf_tree<8>(p, lo, count); break;
    default: {
        // 16 leaves at a time, merged in a binary counter
        TreeCounter<24> tc;
        for (size_t i = 0; i < M && lo + i < count; i += 16) tc.push(leaf_tree<16>(p, lo + i, count));
        v = tc.finish();
        break;
    }
    }
    v = warp_tree_lane_order(v);
    if (lane == 0) warp_val[warp] = v;
    __syncthreads();
    if (warp == 0) {
        const float w = warp_tree_lane_order(warp_val[lane]);
        if (lane == 0) out[blockIdx.x] = w;
    }
}

// Many segments with few partials each (long rows): one thread per segment
// pushes its partials into a binary counter -- the same balanced tree,
// padded with -0.0, as combine_kernel forms.
constexpr size_t kCombineRowsMaxCount = 64;

__global__ void __launch_bounds__(256)
combine_rows_kernel(const float *__restrict__ partials, size_t segments, size_t count,
                    float *__restrict__ out)
{
    pdl_launch_dependents();   // the next call's first kernel may launch; it waits for this one
    pdl_wait_primary();
    const size_t r = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= segments) return;
    const float *p = partials + r * count;
    TreeCounter<7> tc;
    for (size_t i = 0; i < count; i++) tc.push(__ldg(p + i));
    out[r] = tc.finish();
}

// Launched with programmatic stream serialization: the combine's launch
// overlaps the end of the kernel before it, and pdl_wait_primary() holds
// its threads until that kernel's partials are complete and visible.
cudaError_t launch_combine(const float *partials, size_t segments, size_t count, float *out,
                           cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (count <= kCombineRowsMaxCount && segments > 1) {
        cfg.gridDim = dim3((unsigned)((segments + 255) / 256));
        cfg.blockDim = dim3(256);
        return cudaLaunchKernelEx(&cfg, combine_rows_kernel, partials, segments, count, out);
    }
    cfg.gridDim = dim3((unsigned)segments);
    cfg.blockDim = dim3(1024);
    return cudaLaunchKernelEx(&cfg, combine_kernel, partials, count, out);
}

cudaError_t preload_combine()
{
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, combine_kernel);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, combine_rows_kernel);
    return e;
}

}  // namespace tcr
