// stream.cuh -- the warp stream shared by the chunked and per-row kernels.
//
// A warp walks its inputs in groups of 2048 (8 warp loads of 256): lane j
// of warp load k of a group holds vector 32*k + j of the group, so each
// load instruction is one coalesced 512-byte transaction.  The loop is
// software-pipelined: the 8 loads of the next group (of the same span, or
// of the warp's next work unit) are issued before the current group's
// dependent arithmetic runs, so a warp keeps 4 KiB of loads in flight
// while it shuffles.  A reducer policy turns groups into the mode's result:
//
//   FixedReducer    balanced tree over index order (FIXED_ORDER)
//   ShuffleReducer  grid-stride accumulation of one warp team (SHUFFLE_TREE)
//   MmaReducer      tensor-core chains of R MMAs against ones (MMA_CHAIN)
//
// Each policy splits a group into take() -- which consumes the 8 loaded
// vectors into registers -- and reduce(), the dependent part that runs while
// the next group's loads are in flight.
#pragma once

#include "common.cuh"
#include "kernels.cuh"

namespace tcr {

// The 8 vectors of the group starting at input gbase of a segment of len
// inputs; inputs past len read as the 16-bit pattern FILL.
template <bool ALIGNED, uint16_t FILL>
__device__ __forceinline__ void load_group(uint4 (&q)[8], const uint16_t *seg, size_t len,
                                           size_t gbase, int lane)
{
    if (ALIGNED && gbase + kGroup <= len) {
#pragma unroll
        for (int k = 0; k < 8; k++) q[k] = ld_stream(seg + gbase + 256 * k + 8 * lane);
    } else {
        const uint32_t f2 = (uint32_t)FILL * 0x10001u;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const size_t vec = gbase / 8 + 32 * (size_t)k + (size_t)lane;
            q[k] = 8 * vec < len ? ld_vec<ALIGNED>(seg, len, vec, FILL) : make_uint4(f2, f2, f2, f2);
        }
    }
}

// ---------------------------------------------------------------- trees

// t[k]: the lane's 8-input subtree of warp load k (k = 0..7) of a group.
// Returns the aligned subtree of the whole group (2048 inputs) in every
// lane.  Levels 4..6 are a reduce-scatter butterfly that halves the values
// each lane carries (12 shuffles per group instead of 43).  Additions are
// commutative bit for bit, so which lane of a pair forms a node does not
// matter; which two children it adds is fixed.
__device__ __forceinline__ float group_tree(const float (&t)[8], int lane)
{
    const bool b0 = lane & 1, b1 = lane & 2, b2 = lane & 4;
    // level 4 (16 inputs: lanes j, j^1): even lanes keep loads 0..3, odd
    // lanes loads 4..7; afterwards u[i] is load i + 4*b0
    float u[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float keep = b0 ? t[i + 4] : t[i];
        const float send = b0 ? t[i] : t[i + 4];
        u[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 1));
    }
    // level 5 (32 inputs: lanes j, j^2): v[i] is load i + 2*b1 + 4*b0
    float v[2];
#pragma unroll
    for (int i = 0; i < 2; i++) {
        const float keep = b1 ? u[i + 2] : u[i];
        const float send = b1 ? u[i] : u[i + 2];
        v[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 2));
    }
    // level 6 (64 inputs: lanes j, j^4): w is load b2 + 2*b1 + 4*b0
    const float keep = b2 ? v[1] : v[0];
    const float send = b2 ? v[0] : v[1];
    float w = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 4));
    // levels 7, 8 (128, 256 inputs): the rest of the warp load
    w = __fadd_rn(w, __shfl_xor_sync(kFull, w, 8));
    w = __fadd_rn(w, __shfl_xor_sync(kFull, w, 16));
    // levels 9..11: loads k, k^1 differ in lane bit 2; k, k^2 in lane bit 1;
    // k, k^4 in lane bit 0
    w = __fadd_rn(w, __shfl_xor_sync(kFull, w, 4));
    w = __fadd_rn(w, __shfl_xor_sync(kFull, w, 2));
    w = __fadd_rn(w, __shfl_xor_sync(kFull, w, 1));
    return w;
}

// ---------------------------------------------------------------- policies

// FIXED_ORDER: the groups of a span are consecutive aligned subtrees; they
// merge in a binary counter, so any count of groups gives the balanced tree
// padded with -0.0.  LEVELS bounds the groups per span (< 2^LEVELS).  For
// sums of squares the pad's leaf is (-0.0)^2 = +0.0, which is the identity
// too, since every leaf is then at least +0.0.
template <int DT, int OP, int LEVELS>
struct FixedReducer {
    static constexpr uint16_t kFill = 0x8000;    // -0.0
    TreeCounter<LEVELS> tc;
    float t[8];

    __device__ __forceinline__ void take(const uint4 (&q)[8])
    {
#pragma unroll
        for (int k = 0; k < 8; k++) t[k] = tree8<DT, OP>(q[k]);
    }
    __device__ __forceinline__ void reduce(int lane) { tc.push(group_tree(t, lane)); }
    __device__ __forceinline__ float value(int) const { return tc.finish(); }
};

// SHUFFLE_TREE, one-warp team: lane j adds the 8-input trees of vectors
// j, j+32, j+64, ... in that order (group after group, load k after load
// k-1), starting from -0.0; the warp value is the butterfly with offsets
// 16, 8, 4, 2, 1.  Vectors past the segment are -0.0, the identity.
template <int DT, int OP>
struct ShuffleReducer {
    static constexpr uint16_t kFill = 0x8000;
    float acc = -0.0f;
    float t[8];

    __device__ __forceinline__ void take(const uint4 (&q)[8])
    {
#pragma unroll
        for (int k = 0; k < 8; k++) t[k] = tree8<DT, OP>(q[k]);
    }
    __device__ __forceinline__ void reduce(int)
    {
#pragma unroll
        for (int k = 0; k < 8; k++) acc = __fadd_rn(acc, t[k]);
    }
    __device__ __forceinline__ float value(int) const
    {
        float a = acc;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) a = __fadd_rn(a, __shfl_xor_sync(kFull, a, off));
        return a;
    }
};

// MMA_CHAIN: one m16n8k16 MMA per warp load -- the lane's 16-byte vector is
// its A fragment as it stands, since with B = ones the sum of D's column
// over its 16 rows is the sum of all 256 A elements whatever their slots.
// R MMAs chain into one fp32 D; then d0 (row lane/4) and d2 (row lane/4+8)
// are added into the lane's fp32 accumulators and D restarts from zero.
// The warp value sums the accumulators over the 8 row groups (lanes of
// equal lane%4 hold the same column: offsets 4, 8, 16).
template <int DT, int R>
struct MmaReducer {
    static constexpr uint16_t kFill = 0x0000;
    float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
    float acc_lo = 0.f, acc_hi = 0.f;
    int cnt = 0;

    __device__ __forceinline__ void flush()
    {
        acc_lo = __fadd_rn(acc_lo, d0);
        acc_hi = __fadd_rn(acc_hi, d2);
        d0 = d1 = d2 = d3 = 0.f;
        cnt = 0;
    }
    __device__ __forceinline__ void take(const uint4 (&q)[8])
    {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            mma_ones<DT>(d0, d1, d2, d3, q[k].x, q[k].y, q[k].z, q[k].w);
            if (++cnt == R) flush();
        }
    }
    __device__ __forceinline__ void reduce(int) {}
    __device__ __forceinline__ float value(int)
    {
        if (cnt) flush();
        float a = __fadd_rn(acc_lo, acc_hi);
        a = __fadd_rn(a, __shfl_xor_sync(kFull, a, 4));
        a = __fadd_rn(a, __shfl_xor_sync(kFull, a, 8));
        a = __fadd_rn(a, __shfl_xor_sync(kFull, a, 16));
        return a;
    }
};

// MMA_CHAIN, sum of squares: a dense contraction on the tensor cores.  For
// a 16 x 16 tile A, D = A * A^T has the row sums of squares on its diagonal.
// In the m16n8k16 fragments the B operand of A^T's first 8 columns
// (B[k][n] = A[n][k], n < 8) is exactly the lane's own A registers a0a1 and
// a4a5, and that of the last 8 columns is a2a3 and a6a7: two MMAs per tile,
// no data movement.  The diagonal D[g][g] (rows 0..7) lands in d0 / d1 and
// D[g+8][g] (rows 8..15) in d2 / d3 of lane (g, t = g/2).  Chains of R tiles
// flush those two values into the lane's fp32 accumulator; the warp value is
// the sum over all lanes (eight of them hold values).
template <int DT, int R>
struct MmaSqReducer {
    static constexpr uint16_t kFill = 0x0000;
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;    // A * (rows 0..7)^T
    float q0 = 0.f, q1 = 0.f, q2 = 0.f, q3 = 0.f;    // A * (rows 8..15)^T
    float acc = 0.f;
    int cnt = 0;

    __device__ __forceinline__ void flush()
    {
        const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
        if (t == (g >> 1)) acc = __fadd_rn(acc, (g & 1) ? __fadd_rn(p1, q3) : __fadd_rn(p0, q2));
        p0 = p1 = p2 = p3 = q0 = q1 = q2 = q3 = 0.f;
        cnt = 0;
    }
    __device__ __forceinline__ void take(const uint4 (&q)[8])
    {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            mma_ab<DT>(p0, p1, p2, p3, q[k].x, q[k].y, q[k].z, q[k].w, q[k].x, q[k].z);
            mma_ab<DT>(q0, q1, q2, q3, q[k].x, q[k].y, q[k].z, q[k].w, q[k].y, q[k].w);
            if (++cnt == R) flush();
        }
    }
    __device__ __forceinline__ void reduce(int) {}
    __device__ __forceinline__ float value(int)
    {
        if (cnt) flush();
        float a = acc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) a = __fadd_rn(a, __shfl_xor_sync(kFull, a, off));
        return a;
    }
};

// ---------------------------------------------------------------- kernels

// Chunked: CTA work unit u = (segment u / cps, chunk u % cps); the chunk of
// 2^chunk_log2 inputs is split into one aligned span per warp; dst[u] is
// the balanced tree over the CTA's warp values (warp order, -0.0 pad).
// Persistent: CTA b takes units b, b + grid, b + 2*grid, ...
template <class Red, bool ALIGNED>
__device__ __forceinline__ void chunk_body(const uint16_t *__restrict__ x, size_t seg_len,
                                           size_t units, size_t cps, int chunk_log2,
                                           float *__restrict__ dst)
{
    __shared__ float warp_val[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    // every warp span is 2^kWarpSpanLog2 inputs (chunk_log2 = kWarpSpanLog2
    // + log2 warps), so the groups per span are a compile-time constant
    constexpr size_t span = (size_t)1 << kWarpSpanLog2;
    constexpr int ngroups = (int)(span / kGroup);
    size_t u = blockIdx.x;
    if (u < units) {
        size_t s = u / cps;
        const uint16_t *seg = x + s * seg_len;
        size_t base = ((u - s * cps) << chunk_log2) + (size_t)warp * span;
        uint4 q[8];
        load_group<ALIGNED, Red::kFill>(q, seg, seg_len, base, lane);
        for (;;) {
            const size_t nu = u + gridDim.x;
            const bool has_next = nu < units;
            const uint16_t *nseg = seg;
            size_t nbase = 0;
            if (has_next) {
                const size_t ns = nu / cps;
                nseg = x + ns * seg_len;
                nbase = ((nu - ns * cps) << chunk_log2) + (size_t)warp * span;
            }
            Red red;
            // not unrolled: one group of loads in flight ahead, no more, so
            // the loop fits the 64 registers a 1024-thread CTA allows
#pragma unroll 1
            for (int g = 0; g < ngroups; g++) {
                red.take(q);
                if (g + 1 < ngroups)
                    load_group<ALIGNED, Red::kFill>(q, seg, seg_len, base + (size_t)(g + 1) * kGroup,
                                                    lane);
                else if (has_next)
                    load_group<ALIGNED, Red::kFill>(q, nseg, seg_len, nbase, lane);
                red.reduce(lane);
            }
            const float v = red.value(lane);
            if (lane == 0) warp_val[warp] = v;
            __syncthreads();
            if (warp == 0) {
                const float w = warp_tree_lane_order(lane < nwarps ? warp_val[lane] : -0.0f);
                if (lane == 0) dst[u] = w;
            }
            __syncthreads();
            if (!has_next) break;
            u = nu;
            seg = nseg;
            base = nbase;
        }
    }
    pdl_launch_dependents();
}

// One warp per row (rows of at most 2^LEVELS groups): out[r] is the row's
// value.  Persistent: warp w takes rows w, w + warps, w + 2*warps, ...
template <class Red, bool ALIGNED>
__device__ __forceinline__ void rows_body(const uint16_t *__restrict__ x, size_t rows,
                                          size_t cols, float *__restrict__ out)
{
    const int lane = threadIdx.x & 31;
    const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
    size_t r = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t ngroups = (cols + kGroup - 1) / kGroup;
    if (r < rows && ngroups > 0) {
        uint4 q[8];
        load_group<ALIGNED, Red::kFill>(q, x + r * cols, cols, 0, lane);
        for (;;) {
            const size_t nr = r + nw;
            const bool has_next = nr < rows;
            Red red;
#pragma unroll 1
            for (size_t g = 0; g < ngroups; g++) {
                red.take(q);
                if (g + 1 < ngroups)
                    load_group<ALIGNED, Red::kFill>(q, x + r * cols, cols, (g + 1) * kGroup, lane);
                else if (has_next)
                    load_group<ALIGNED, Red::kFill>(q, x + nr * cols, cols, 0, lane);
                red.reduce(lane);
            }
            const float v = red.value(lane);
            if (lane == 0) out[r] = v;
            if (!has_next) break;
            r = nr;
        }
    }
}

}  // namespace tcr
