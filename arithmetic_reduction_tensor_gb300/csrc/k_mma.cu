// k_mma.cu -- MMA_CHAIN: the sum as chains of tensor-core multiply-
// accumulates against a ones matrix.
//
// "GPU Tensor Cores for fast Arithmetic Reductions" (arXiv 2001.05585),
// Abstract: the reduction of n numbers is encoded as chained m x m MMAs run
// in parallel on the tensor cores; each chain of R MMAs keeps its
// sub-result in 32-bit floating point, and the sub-results are then all
// reduced into a final 32-bit result; small thread blocks do best with
// R = 4 or 5, large ones with R = 1.
//
// Here m = 16 (mma.sync m16n8k16, fp16/bf16 in, fp32 accumulate).  With
// B = ones, D[i][j] = sum_k A[i][k] for every column j, so the sum of all
// 256 A elements is the sum of D's column over its 16 rows -- whatever
// element sits in whatever A slot.  A lane's 16-byte load is therefore its
// A fragment as it stands (no shuffles, no ldmatrix): one coalesced warp
// load of 512 bytes is one MMA.  A chain is R MMAs into the same fp32 D;
// then each lane adds d0 + d2 (its two rows) into its fp32 accumulator and
// D restarts from zero.  The fp32 accumulators are combined across the
// warp (lanes of equal lane%4 hold the same column: offsets 4, 8, 16),
// across warps (balanced tree in smem) and across CTA chunks (combine).
#include "common.cuh"
#include "kernels.cuh"

namespace tcr {

// One chain step: D += A*ones, and after every R-th MMA fold D into the
// lane accumulator.
template <int DT, int R>
struct Chain {
    float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
    int cnt = 0;

    __device__ __forceinline__ void flush(float &acc_lo, float &acc_hi)
    {
        acc_lo = __fadd_rn(acc_lo, d0);
        acc_hi = __fadd_rn(acc_hi, d2);
        d0 = d1 = d2 = d3 = 0.f;
        cnt = 0;
    }

    __device__ __forceinline__ void step(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         float &acc_lo, float &acc_hi)
    {
        mma_ones<DT>(d0, d1, d2, d3, a0, a1, a2, a3);
        if (++cnt == R) flush(acc_lo, acc_hi);
    }

    __device__ __forceinline__ void finish(float &acc_lo, float &acc_hi)
    {
        if (cnt) flush(acc_lo, acc_hi);
    }
};

template <int DT, int R, bool ALIGNED>
__global__ void __launch_bounds__(1024)
mma_chunk_kernel(const uint16_t *__restrict__ x, size_t seg_len, size_t units, size_t cps,
                 int chunk_log2, float *__restrict__ dst)
{
    __shared__ float warp_val[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const size_t span = ((size_t)1 << chunk_log2) / (size_t)nwarps;
    for (size_t u = blockIdx.x; u < units; u += gridDim.x) {
        const size_t s = u / cps, c = u - s * cps;
        const uint16_t *seg = x + s * seg_len;
        const size_t base = (c << chunk_log2) + (size_t)warp * span;
        size_t end = base + span;
        if (end > seg_len) end = seg_len;
        float acc_lo = 0.f, acc_hi = 0.f;
        Chain<DT, R> ch;
        for (size_t gb = base; gb < end; gb += kGroup) {
            uint4 q[8];
            if (ALIGNED && gb + kGroup <= seg_len) {
#pragma unroll
                for (int k = 0; k < 8; k++) q[k] = ld_stream(seg + gb + 256 * k + 8 * lane);
            } else {
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    size_t vec = (gb + 256 * k) / 8 + (size_t)lane;
                    q[k] = 8 * vec < seg_len ? ld_vec<ALIGNED>(seg, seg_len, vec, 0)
                                             : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int k = 0; k < 8; k++) ch.step(q[k].x, q[k].y, q[k].z, q[k].w, acc_lo, acc_hi);
        }
        ch.finish(acc_lo, acc_hi);
        float acc = __fadd_rn(acc_lo, acc_hi);
        acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, 4));
        acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, 8));
        acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, 16));
        if (lane == 0) warp_val[warp] = acc;
        __syncthreads();
        if (warp == 0) {
            float w = warp_tree_lane_order(lane < nwarps ? warp_val[lane] : 0.f);
            if (lane == 0) dst[u] = w;
        }
        __syncthreads();
    }
}

// Rows: a warp owns 16 consecutive rows.  Lane (g = lane/4, t = lane%4)
// loads 8 inputs of row g and 8 of row g+8 at the same columns; the low
// and high halves of the two 16-byte vectors form the A fragments of two
// MMAs (registers a0a1, a4a5 from row g; a2a3, a6a7 from row g+8), so D's
// rows are the 16 row sums.  Every lane of a quad holds the same row sums.
constexpr int kRowsUnroll = 4;    // 32-column blocks in flight per warp

template <int DT, int R, bool ALIGNED>
__global__ void __launch_bounds__(1024)
mma_rows_kernel(const uint16_t *__restrict__ x, size_t rows, size_t cols,
                float *__restrict__ out)
{
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const size_t gw = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
    const size_t tiles = (rows + 15) / 16;
    const size_t nvec = (cols + 7) / 8;
    for (size_t tile = gw; tile < tiles; tile += nw) {
        const size_t ra = tile * 16 + (size_t)g, rb = ra + 8;
        const bool va = ra < rows, vb = rb < rows;
        const uint16_t *pa = x + (va ? ra : 0) * cols;
        const uint16_t *pb = x + (vb ? rb : 0) * cols;
        float acc_a = 0.f, acc_b = 0.f;
        Chain<DT, R> ch;
        for (size_t c0 = 0; c0 < cols; c0 += 32 * kRowsUnroll) {
            uint4 qa[kRowsUnroll], qb[kRowsUnroll];
#pragma unroll
            for (int u = 0; u < kRowsUnroll; u++) {
                const size_t vec = (c0 + 32 * (size_t)u) / 8 + (size_t)t;
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                qa[u] = (va && vec < nvec) ? ld_vec<ALIGNED>(pa, cols, vec, 0) : z;
                qb[u] = (vb && vec < nvec) ? ld_vec<ALIGNED>(pb, cols, vec, 0) : z;
            }
#pragma unroll
            for (int u = 0; u < kRowsUnroll; u++) {
                if (c0 + 32 * (size_t)u < cols) {       // warp-uniform
                    ch.step(qa[u].x, qb[u].x, qa[u].y, qb[u].y, acc_a, acc_b);
                    ch.step(qa[u].z, qb[u].z, qa[u].w, qb[u].w, acc_a, acc_b);
                }
            }
        }
        ch.finish(acc_a, acc_b);
        if (t == 0) {
            if (va) out[ra] = acc_a;
            if (vb) out[rb] = acc_b;
        }
    }
}

// ---------------------------------------------------------------- host

template <int R>
static void *pick_chunk(int dtype, bool aligned)
{
    if (dtype == kF16) return aligned ? (void *)mma_chunk_kernel<kF16, R, true>
                                      : (void *)mma_chunk_kernel<kF16, R, false>;
    return aligned ? (void *)mma_chunk_kernel<kBF16, R, true>
                   : (void *)mma_chunk_kernel<kBF16, R, false>;
}

template <int R>
static void *pick_rows(int dtype, bool aligned)
{
    if (dtype == kF16) return aligned ? (void *)mma_rows_kernel<kF16, R, true>
                                      : (void *)mma_rows_kernel<kF16, R, false>;
    return aligned ? (void *)mma_rows_kernel<kBF16, R, true>
                   : (void *)mma_rows_kernel<kBF16, R, false>;
}

static void *pick(bool rows, int dtype, bool aligned, int R)
{
    switch (R) {
    case 1: return rows ? pick_rows<1>(dtype, aligned) : pick_chunk<1>(dtype, aligned);
    case 2: return rows ? pick_rows<2>(dtype, aligned) : pick_chunk<2>(dtype, aligned);
    case 3: return rows ? pick_rows<3>(dtype, aligned) : pick_chunk<3>(dtype, aligned);
    case 4: return rows ? pick_rows<4>(dtype, aligned) : pick_chunk<4>(dtype, aligned);
    case 5: return rows ? pick_rows<5>(dtype, aligned) : pick_chunk<5>(dtype, aligned);
    case 6: return rows ? pick_rows<6>(dtype, aligned) : pick_chunk<6>(dtype, aligned);
    case 7: return rows ? pick_rows<7>(dtype, aligned) : pick_chunk<7>(dtype, aligned);
    case 8: return rows ? pick_rows<8>(dtype, aligned) : pick_chunk<8>(dtype, aligned);
    default: return nullptr;
    }
}

cudaError_t launch_mma_chunk(int dtype, bool aligned, int R, const uint16_t *x, size_t seg_len,
                             size_t units, size_t cps, int chunk_log2, float *dst, int grid,
                             int block, cudaStream_t stream)
{
    void *k = pick(false, dtype, aligned, R);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&seg_len, (void *)&units, (void *)&cps,
                    (void *)&chunk_log2, (void *)&dst};
    return cudaLaunchKernel(k, dim3(grid), dim3(block), args, 0, stream);
}

cudaError_t launch_mma_rows(int dtype, bool aligned, int R, const uint16_t *x, size_t rows,
                            size_t cols, float *out, int grid, int block, cudaStream_t stream)
{
    void *k = pick(true, dtype, aligned, R);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&rows, (void *)&cols, (void *)&out};
    return cudaLaunchKernel(k, dim3(grid), dim3(block), args, 0, stream);
}

int occupancy_mma(bool rows, int dtype, bool aligned, int R, int block)
{
    void *k = pick(rows, dtype, aligned, R);
    int n = 0;
    if (!k || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, block, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace tcr
