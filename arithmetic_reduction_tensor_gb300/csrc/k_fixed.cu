// k_fixed.cu -- FIXED_ORDER: the balanced binary32 tree over index order.
//
// The order is the one of "Taming Bitwise Behavior in GPU Kernels with
// Tensor Core" (arXiv 2609.11356), Abstract: a balanced-tree reduction, so
// that every launch configuration lands in one bit-equivalence class.  The
// tree is over the segment's inputs in index order, power-of-two aligned,
// padded with -0.0.  Because every subtree here is aligned, any split of
// the work into aligned pieces (vectors, warp loads, warp groups, CTA
// chunks, partials) computes the same nodes, and the result depends only
// on the inputs and the segment length.
//
// Data layout of one warp group (2048 inputs = 8 warp loads of 256): lane
// j of warp load k holds vector k*32 + j (inputs 8 apart per lane, so each
// load instruction is one fully coalesced 512-byte transaction).  The
// in-lane 8-input tree gives level 3; levels 4..8 (within a warp load) and
// 9..11 (across the 8 loads) are formed by a reduce-scatter butterfly that
// halves the number of values each lane carries at each of the first
// three steps, 12 shuffles per group instead of 8 * 5 + 3.  This is the
// "data layout optimisation" idea of the same Abstract applied to a warp:
// the leaves are placed so that a fixed order costs few extra instructions.
#include "common.cuh"
#include "kernels.cuh"

namespace tcr {

// t[k]: lane's 8-input subtree of warp load k (k = 0..7) of one group.
// Returns the aligned subtree of the whole group (2048 inputs) in every
// lane.  Additions are commutative bit for bit, so which lane of a pair
// forms a node does not matter; which children it adds is fixed.
__device__ __forceinline__ float group_tree(const float t[8], int lane)
{
    const bool b0 = lane & 1, b1 = lane & 2, b2 = lane & 4;
    // level 4 (16 inputs: lanes j, j^1): even lanes keep loads 0..3,
    // odd lanes keep loads 4..7.  Afterwards u[i] is load i + 4*b0.
    float u[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float keep = b0 ? t[i + 4] : t[i];
        float send = b0 ? t[i] : t[i + 4];
        u[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 1));
    }
    // level 5 (32 inputs: lanes j, j^2): v[i] is load i + 2*b1 + 4*b0.
    float v[2];
#pragma unroll
    for (int i = 0; i < 2; i++) {
        float keep = b1 ? u[i + 2] : u[i];
        float send = b1 ? u[i] : u[i + 2];
        v[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 2));
    }
    // level 6 (64 inputs: lanes j, j^4): w is load b2 + 2*b1 + 4*b0.
    float keep = b2 ? v[1] : v[0];
    float send = b2 ? v[0] : v[1];
    float w = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 4));
    // levels 7, 8 (128, 256 inputs): the rest of the warp load.
    w = __fadd_rn(w, __shfl_xor_sync(kFull, w, 8));
    w = __fadd_rn(w, __shfl_xor_sync(kFull, w, 16));
    // levels 9..11: loads k, k^1 differ in lane bit 2; k, k^2 in lane bit 1;
    // k, k^4 in lane bit 0.
    w = __fadd_rn(w, __shfl_xor_sync(kFull, w, 4));
    w = __fadd_rn(w, __shfl_xor_sync(kFull, w, 2));
    w = __fadd_rn(w, __shfl_xor_sync(kFull, w, 1));
    return w;
}

// Aligned subtree of the group of 2048 inputs starting at gbase of a
// segment of len inputs (inputs past len are -0.0).
template <int DT, bool ALIGNED>
__device__ __forceinline__ float group_value(const uint16_t *seg, size_t len, size_t gbase,
                                             int lane)
{
    float t[8];
    if (ALIGNED && gbase + kGroup <= len) {
        uint4 q[8];
#pragma unroll
        for (int k = 0; k < 8; k++) q[k] = ld_stream(seg + gbase + 256 * k + 8 * lane);
#pragma unroll
        for (int k = 0; k < 8; k++) t[k] = tree8<DT>(q[k]);
    } else {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            size_t vec = (gbase + 256 * k) / 8 + (size_t)lane;
            t[k] = 8 * vec < len ? tree8<DT>(ld_vec<ALIGNED>(seg, len, vec, 0x8000u)) : -0.0f;
        }
    }
    return group_tree(t, lane);
}

// Aligned subtree of ngroups * 2048 inputs starting at base (ngroups a
// power of two, base a multiple of ngroups * 2048).  Groups past len are
// wholly padding (-0.0) and are not visited.
template <int DT, bool ALIGNED>
__device__ __forceinline__ float warp_span_tree(const uint16_t *seg, size_t len, size_t base,
                                                size_t ngroups, int lane)
{
    TreeCounter<8> tc;
    for (size_t g = 0; g < ngroups; g++) {
        size_t gbase = base + g * kGroup;
        if (gbase >= len) break;
        tc.push(group_value<DT, ALIGNED>(seg, len, gbase, lane));
    }
    return tc.finish();
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(1024)
fixed_chunk_kernel(const uint16_t *__restrict__ x, size_t seg_len, size_t units, size_t cps,
                   int chunk_log2, float *__restrict__ dst)
{
    __shared__ float warp_val[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const size_t span = ((size_t)1 << chunk_log2) / (size_t)nwarps;
    const size_t ngroups = span / kGroup;
    for (size_t u = blockIdx.x; u < units; u += gridDim.x) {
        const size_t s = u / cps, c = u - s * cps;
        const uint16_t *seg = x + s * seg_len;
        const size_t base = (c << chunk_log2) + (size_t)warp * span;
        float v = warp_span_tree<DT, ALIGNED>(seg, seg_len, base, ngroups, lane);
        if (lane == 0) warp_val[warp] = v;
        __syncthreads();
        if (warp == 0) {
            // tree over the CTA's warps in warp order; lanes past nwarps pad
            float w = warp_tree_lane_order(lane < nwarps ? warp_val[lane] : -0.0f);
            if (lane == 0) dst[u] = w;
        }
        __syncthreads();
    }
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(1024)
fixed_rows_warp_kernel(const uint16_t *__restrict__ x, size_t rows, size_t cols,
                       float *__restrict__ out)
{
    const int lane = threadIdx.x & 31;
    const size_t gw = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
    size_t ngroups = 1;
    while (ngroups * kGroup < cols) ngroups <<= 1;
    for (size_t r = gw; r < rows; r += nw) {
        float v = warp_span_tree<DT, ALIGNED>(x + r * cols, cols, 0, ngroups, lane);
        if (lane == 0) out[r] = v;
    }
}

// ---------------------------------------------------------------- host

template <typename K>
static int occupancy_of(K kernel, int block)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, block, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

#define TCR_PICK(KERNEL, dtype, aligned)                                                   \
    ((dtype) == kF16 ? ((aligned) ? KERNEL<kF16, true> : KERNEL<kF16, false>)              \
                     : ((aligned) ? KERNEL<kBF16, true> : KERNEL<kBF16, false>))

cudaError_t launch_fixed_chunk(int dtype, bool aligned, const uint16_t *x, size_t seg_len,
                               size_t units, size_t cps, int chunk_log2, float *dst, int grid,
                               int block, cudaStream_t stream)
{
    auto k = TCR_PICK(fixed_chunk_kernel, dtype, aligned);
    k<<<grid, block, 0, stream>>>(x, seg_len, units, cps, chunk_log2, dst);
    return cudaGetLastError();
}

cudaError_t launch_fixed_rows_warp(int dtype, bool aligned, const uint16_t *x, size_t rows,
                                   size_t cols, float *out, int grid, int block,
                                   cudaStream_t stream)
{
    auto k = TCR_PICK(fixed_rows_warp_kernel, dtype, aligned);
    k<<<grid, block, 0, stream>>>(x, rows, cols, out);
    return cudaGetLastError();
}

int occupancy_fixed(bool rows, int dtype, bool aligned, int block)
{
    if (rows) return occupancy_of(TCR_PICK(fixed_rows_warp_kernel, dtype, aligned), block);
    return occupancy_of(TCR_PICK(fixed_chunk_kernel, dtype, aligned), block);
}

}  // namespace tcr
