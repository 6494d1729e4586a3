// stream.cuh -- the warp stream shared by the chunked and per-row kernels.
//
// A warp walks its inputs in groups of 8 warp loads of 32 vectors (4 KiB:
// 2048 16-bit inputs, 1024 binary32 inputs): lane j of warp load k of a
// group holds vector 32*k + j of the group, so each load instruction is one
// coalesced 512-byte transaction.  The loop is software-pipelined: the 8
// loads of the next group (of the same span, or of the warp's next work
// unit) are issued before the current group's dependent arithmetic runs,
// so a warp keeps 4 KiB of loads in flight while it shuffles.  A reducer policy turns groups into the mode's result:
//
//   FixedReducer    balanced tree over index order (FIXED_ORDER)
//   ShuffleReducer  grid-stride accumulation of one warp team (SHUFFLE_TREE)
//   MmaReducer      tensor-core chains of R MMAs against ones (MMA_CHAIN)
//   MmaSqReducer    tensor-core A * A^T diagonals (MMA_CHAIN, squares)
//   MmaSplitReducer binary32 inputs split exactly into three bfloat16
//                   parts, then chains against ones (MMA_CHAIN)
//
// Each policy splits a group into take() -- which consumes the 8 loaded
// vectors into registers -- and reduce(), the dependent part that runs while
// the next group's loads are in flight.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "kernels.cuh"

namespace tcr {

// The 8 vectors of the group starting at input gbase of a segment of len
// inputs; inputs past len read as -0.0 (NEGZERO) or zero bits.
template <int DT, bool ALIGNED, bool NEGZERO>
__device__ __forceinline__ void load_group(uint4 (&q)[8], const typename Elem<DT>::T *seg,
                                           size_t len, size_t gbase, int lane)
{
    constexpr int V = Elem<DT>::kPerVec;
    if (ALIGNED && gbase + group_len<DT>() <= len) {
#pragma unroll
        for (int k = 0; k < 8; k++) q[k] = ld_stream(seg + gbase + 32 * V * k + V * lane);
    } else {
        const uint32_t f = fill_word<DT, NEGZERO>();
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const size_t vec = gbase / V + 32 * (size_t)k + (size_t)lane;
            q[k] = V * vec < len ? ld_vec<DT, ALIGNED, NEGZERO>(seg, len, vec)
                                 : make_uint4(f, f, f, f);
        }
    }
}

// ---------------------------------------------------------------- unaligned segments
//
// A segment that does not start 16-byte aligned (a misaligned x, or rows
// whose stride is not whole vectors) is read in whole 16-byte aligned
// granules, numbered from the one holding the segment's first byte: vector
// v (inputs V v .. V v + V - 1) starts in granule v, at the segment's byte
// offset sb in its granule (the same for every vector), and ends in granule
// v + 1.  Lane j of load k loads granule v of its vector; the next granule
// is lane j + 1's (lane 0's of load k + 1 for lane 31, one extra load by
// lane 31 after load 7).  A granule is loaded only when it holds a byte of
// the segment, so the loads stay inside the 16-byte granules the data
// touches.  The vectors are shifted out of the granules (realign_group)
// when the group is reduced, while the next group's loads are in flight.

template <int DT, bool NEGZERO>
__device__ __forceinline__ void load_group_raw(uint4 (&q)[8], uint4 &qt, const typename Elem<DT>::T *seg,
                                               size_t len, size_t gbase, int lane)
{
    constexpr int V = Elem<DT>::kPerVec;
    constexpr size_t EB = sizeof(typename Elem<DT>::T);
    const uintptr_t a = (uintptr_t)seg;
    const uint4 *g0 = reinterpret_cast<const uint4 *>(a & ~(uintptr_t)15);
    const size_t glim = ((size_t)(a & 15) + len * EB - 1) >> 4;     // last granule
    const size_t v0 = gbase / V + (size_t)lane;
    const uint32_t f = fill_word<DT, NEGZERO>();
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const size_t v = v0 + 32 * (size_t)k;
        q[k] = v <= glim ? ld_stream(g0 + v) : make_uint4(f, f, f, f);
    }
    qt = make_uint4(f, f, f, f);
    if (lane == 31 && gbase / V + 256 <= glim) qt = ld_stream(g0 + gbase / V + 256);
}

// Shift every vector of a group out of its two granules: P whole words,
// then hs bits (0 or 16; always 0 for binary32) -- P and hs are the same
// for the whole warp.
template <int DT, int P>
__device__ __forceinline__ void shift_group(uint4 (&q)[8], const uint4 &qt, uint32_t hs, int lane)
{
    const int src = (lane + 1) & 31;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const uint4 lo = q[k];
        uint4 snd = lo;
        if (k < 7 && lane == 0) snd = q[k < 7 ? k + 1 : k];
        uint4 hi;
        hi.x = __shfl_sync(kFull, snd.x, src);
        hi.y = __shfl_sync(kFull, snd.y, src);
        hi.z = __shfl_sync(kFull, snd.z, src);
        hi.w = __shfl_sync(kFull, snd.w, src);
        if (k == 7 && lane == 31) hi = qt;
        const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        // (for binary32 hs is 0 and the funnel shifts are moves; written as
        // shifts they keep the compiler from hoisting the moves across the
        // group, which made the binary32 instances spill)
        q[k] = make_uint4(__funnelshift_r(w[P], w[P + 1], hs), __funnelshift_r(w[P + 1], w[P + 2], hs),
                          __funnelshift_r(w[P + 2], w[P + 3], hs), __funnelshift_r(w[P + 3], w[P + 4], hs));
    }
}

// The raw granules of a group (q, qt) into its 8 vectors, in place; inputs
// past len read as the fill.
template <int DT, bool NEGZERO>
__device__ __forceinline__ void realign_group(uint4 (&q)[8], const uint4 &qt,
                                              const typename Elem<DT>::T *seg, size_t len, size_t gbase,
                                              int lane)
{
    constexpr int V = Elem<DT>::kPerVec;
    constexpr int EB = (int)sizeof(typename Elem<DT>::T);
    const uint32_t sb = (uint32_t)((uintptr_t)seg & 15);
    const uint32_t hs = (sb & 3u) * 8u;
    switch (sb >> 2) {                                   // the same in every lane
    case 0:
        if (sb != 0) shift_group<DT, 0>(q, qt, hs, lane);
        break;
    case 1: shift_group<DT, 1>(q, qt, hs, lane); break;
    case 2: shift_group<DT, 2>(q, qt, hs, lane); break;
    default: shift_group<DT, 3>(q, qt, hs, lane); break;
    }
    if (gbase + group_len<DT>() > len) {
        // the segment's last group: inputs past len become the fill
        const uint32_t f = fill_word<DT, NEGZERO>();
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const long long left = (long long)len - (long long)(gbase + (size_t)V * (32 * k + lane));
            const int cnt = left <= 0 ? 0 : (left >= V ? V : (int)left);
            uint32_t o[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int kb = cnt * 8 * EB - 32 * i;
                const uint32_t m = __funnelshift_lc(0xffffffffu, 0u, (uint32_t)(kb < 0 ? 0 : kb));
                o[i] = (o[i] & m) | (f & ~m);
            }
            q[k] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// The group of loads in flight: for 16-byte aligned segments its 8
// vectors; for the others the raw granules, made into vectors by ready()
// just before the group is reduced -- or, when REALIGN is off (a reducer
// already bound by its own arithmetic, for which input-sized loads cost
// less than the shifts), the vectors loaded input by input.
template <int DT, bool ALIGNED, bool NEGZERO, bool REALIGN = true>
struct GroupIn {
    using T = typename Elem<DT>::T;
    static constexpr bool kRaw = !ALIGNED && REALIGN;
    uint4 q[8];
    uint4 qt;

    __device__ __forceinline__ void load(const T *seg, size_t len, size_t gbase, int lane)
    {
        if constexpr (kRaw) load_group_raw<DT, NEGZERO>(q, qt, seg, len, gbase, lane);
        else load_group<DT, ALIGNED, NEGZERO>(q, seg, len, gbase, lane);
    }
    __device__ __forceinline__ void ready(const T *seg, size_t len, size_t gbase, int lane)
    {
        if constexpr (kRaw) realign_group<DT, NEGZERO>(q, qt, seg, len, gbase, lane);
    }
};

// Whether a reducer's unaligned segments are read as granules (its
// kRealign, true when it has none).
template <class Red, class = void>
struct realigns : std::true_type {};
template <class Red>
struct realigns<Red, std::void_t<decltype(Red::kRealign)>> : std::bool_constant<Red::kRealign> {};

// ---------------------------------------------------------------- trees

// t[k]: the lane's vector subtree of warp load k (k = 0..7) of a group.
// Returns the aligned subtree of the whole group (256 vectors) in every
// lane.  The first three levels above the vectors are a reduce-scatter
// butterfly that halves the values each lane carries (12 shuffles per
// group instead of 43).  Level names below count 16-bit inputs (a binary32
// vector holds 4 inputs, so every span there is half as long).  Additions
// are commutative bit for bit, so which lane of a pair forms a node does
// not matter; which two children it adds is fixed.
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
//
// VRUN > 0 (sums only): the blocked order with runs of 2^VRUN inputs inside a
// vector -- each vector's value is vec_runs instead of its balanced tree;
// the tree above the vectors is the same.
template <int DT, int OP, int LEVELS, int VRUN = 0>
struct FixedReducer {
    static constexpr int kDT = DT;
    static constexpr bool kNegZeroPad = true;
    TreeCounter<LEVELS> tc;
    float t[8];

    __device__ __forceinline__ void take(const uint4 (&q)[8])
    {
        if constexpr (VRUN > 0) {
#pragma unroll
            for (int k = 0; k < 8; k++) t[k] = vec_runs<DT, VRUN>(q[k]);
        } else {
#pragma unroll
            for (int k = 0; k < 8; k++) t[k] = vec_tree<DT, OP>(q[k]);
        }
    }
    __device__ __forceinline__ void reduce(int lane) { tc.push(group_tree(t, lane)); }
    __device__ __forceinline__ float value(int) const { return tc.finish(); }
};

// SHUFFLE_TREE, one-warp team: lane j adds the vector trees of vectors
// j, j+32, j+64, ... in that order (group after group, load k after load
// k-1), starting from -0.0; the warp value is the butterfly with offsets
// 16, 8, 4, 2, 1.  Vectors past the segment are -0.0, the identity.
template <int DT, int OP>
struct ShuffleReducer {
    static constexpr int kDT = DT;
    static constexpr bool kNegZeroPad = true;
    float acc = -0.0f;
    float t[8];

    __device__ __forceinline__ void take(const uint4 (&q)[8])
    {
#pragma unroll
        for (int k = 0; k < 8; k++) t[k] = vec_tree<DT, OP>(q[k]);
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
    static constexpr int kDT = DT;
    static constexpr bool kNegZeroPad = false;
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
    static constexpr int kDT = DT;
    static constexpr bool kNegZeroPad = false;
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

// MMA_CHAIN for binary32 inputs.  Every binary32 x is split exactly into
// three bfloat16 parts, x = hi + mid + lo: hi is x rounded toward zero to
// bfloat16 (its top 8 significant bits), r = x - hi is exact (the low 16
// bits of the significand), mid is r's top 8 significant bits and
// lo = r - mid holds at most 8, so lo is a bfloat16 too.  The split is
// exact whenever lo is a normal number or zero; below 2^-126 lo loses the
// bits under 2^-133, less than 2^-133 per input.  A non-finite x has its
// whole value in hi (cvt keeps infinities and NaNs) and a zero residual.
// Per two warp loads (256 inputs) three m16n8k16 MMAs against ones run:
// the hi parts of both loads as one A tile into D_hi, and each load's mid
// and lo parts (128 + 128 bfloat16) as one A tile into D_ml.  Chains of R
// tiles (R MMAs into D_hi, 2R into D_ml) flush into the lane's fp32
// accumulators as MmaReducer does.  For sums of squares the leaf
// fl32(x * x) is split instead of x.
template <int OP>
__device__ __forceinline__ void split_bf16x3(uint32_t ua, uint32_t ub, uint32_t &hi,
                                             uint32_t &mid, uint32_t &lo)
{
    const float a = leaf32<OP>(ua), b = leaf32<OP>(ub);
    // packed {a in the low half, b in the high half}, rounded toward zero
    asm("cvt.rz.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(b), "f"(a));
    float ra = __fsub_rn(a, __uint_as_float(__float_as_uint(a) & 0xffff0000u));
    float rb = __fsub_rn(b, __uint_as_float(__float_as_uint(b) & 0xffff0000u));
    // a NaN residual comes only from a non-finite leaf: drop it (min and max
    // return the non-NaN operand), leaving the leaf's value to hi
    ra = fminf(fmaxf(ra, 0.0f), ra);
    rb = fminf(fmaxf(rb, 0.0f), rb);
    const uint32_t ma = __float_as_uint(ra) & 0xffff0000u, mb = __float_as_uint(rb) & 0xffff0000u;
    mid = __byte_perm(ma, mb, 0x7632);
    const float la = __fsub_rn(ra, __uint_as_float(ma)), lb = __fsub_rn(rb, __uint_as_float(mb));
    lo = __byte_perm(__float_as_uint(la), __float_as_uint(lb), 0x7632);
}

template <int R, int OP>
struct MmaSplitReducer {
    static constexpr int kDT = kF32;
    static constexpr bool kNegZeroPad = false;
    // the split issues about 7 instructions per input: unaligned inputs are
    // loaded input by input (4-byte loads) rather than shifted out of granules
    static constexpr bool kRealign = false;
    float h0 = 0.f, h1 = 0.f, h2 = 0.f, h3 = 0.f;    // D_hi
    float m0 = 0.f, m1 = 0.f, m2 = 0.f, m3 = 0.f;    // D_ml
    float acc_lo = 0.f, acc_hi = 0.f;
    int cnt = 0;

    __device__ __forceinline__ void flush()
    {
        acc_lo = __fadd_rn(acc_lo, h0);
        acc_hi = __fadd_rn(acc_hi, h2);
        acc_lo = __fadd_rn(acc_lo, m0);
        acc_hi = __fadd_rn(acc_hi, m2);
        h0 = h1 = h2 = h3 = m0 = m1 = m2 = m3 = 0.f;
        cnt = 0;
    }
    __device__ __forceinline__ void take(const uint4 (&q)[8])
    {
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            uint32_t ha0, ma0, la0, ha1, ma1, la1, hb0, mb0, lb0, hb1, mb1, lb1;
            split_bf16x3<OP>(q[k].x, q[k].y, ha0, ma0, la0);
            split_bf16x3<OP>(q[k].z, q[k].w, ha1, ma1, la1);
            split_bf16x3<OP>(q[k + 1].x, q[k + 1].y, hb0, mb0, lb0);
            split_bf16x3<OP>(q[k + 1].z, q[k + 1].w, hb1, mb1, lb1);
            mma_ones<kBF16>(h0, h1, h2, h3, ha0, ha1, hb0, hb1);
            mma_ones<kBF16>(m0, m1, m2, m3, ma0, ma1, la0, la1);
            mma_ones<kBF16>(m0, m1, m2, m3, mb0, mb1, lb0, lb1);
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

// FIXED_ORDER, sum and sum of squares side by side (each leaf unpacked
// once): the values of FixedReducer<DT, kOpSum> and <DT, kOpSquares>.
template <int DT, int LEVELS>
struct FixedPairReducer {
    static constexpr int kDT = DT;
    static constexpr bool kNegZeroPad = true;
    TreeCounter<LEVELS> ca, cb;
    float ta[8], tb[8];

    __device__ __forceinline__ void take(const uint4 (&q)[8])
    {
#pragma unroll
        for (int k = 0; k < 8; k++) vec_tree_pair<DT>(q[k], ta[k], tb[k]);
    }
    __device__ __forceinline__ void reduce(int lane)
    {
        ca.push(group_tree(ta, lane));
        cb.push(group_tree(tb, lane));
    }
    __device__ __forceinline__ void value2(int, float &va, float &vb) const
    {
        va = ca.finish();
        vb = cb.finish();
    }
};

// SHUFFLE_TREE one-warp team, sum and sum of squares side by side.
template <int DT>
struct ShufflePairReducer {
    static constexpr int kDT = DT;
    static constexpr bool kNegZeroPad = true;
    float acc_a = -0.0f, acc_b = -0.0f;
    float ta[8], tb[8];

    __device__ __forceinline__ void take(const uint4 (&q)[8])
    {
#pragma unroll
        for (int k = 0; k < 8; k++) vec_tree_pair<DT>(q[k], ta[k], tb[k]);
    }
    __device__ __forceinline__ void reduce(int)
    {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            acc_a = __fadd_rn(acc_a, ta[k]);
            acc_b = __fadd_rn(acc_b, tb[k]);
        }
    }
    __device__ __forceinline__ void value2(int, float &va, float &vb) const
    {
        float a = acc_a, b = acc_b;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            a = __fadd_rn(a, __shfl_xor_sync(kFull, a, off));
            b = __fadd_rn(b, __shfl_xor_sync(kFull, b, off));
        }
        va = a;
        vb = b;
    }
};

// The MMA_CHAIN policy of an input type and leaf operation.
template <int DT, int R, int OP>
using MmaRed = typename std::conditional<
    DT == kF32, MmaSplitReducer<R, OP>,
    typename std::conditional<OP == kOpSquares, MmaSqReducer<DT, R>, MmaReducer<DT, R>>::type>::type;

// Two reductions of the same inputs in one pass -- a sum and a sum of
// squares: both policies take every group, and their values come out
// together.  Each value is the one its policy gives alone, bit for bit.
template <class A, class B>
struct PairReducer {
    static_assert(A::kDT == B::kDT && A::kNegZeroPad == B::kNegZeroPad, "pair of unlike streams");
    static constexpr int kDT = A::kDT;
    static constexpr bool kNegZeroPad = A::kNegZeroPad;
    static constexpr bool kRealign = realigns<A>::value && realigns<B>::value;
    A a;
    B b;

    __device__ __forceinline__ void take(const uint4 (&q)[8])
    {
        a.take(q);
        b.take(q);
    }
    __device__ __forceinline__ void reduce(int lane)
    {
        a.reduce(lane);
        b.reduce(lane);
    }
    __device__ __forceinline__ void value2(int lane, float &va, float &vb)
    {
        va = a.value(lane);
        vb = b.value(lane);
    }
};

// ---------------------------------------------------------------- kernels

// Chunked: CTA work unit u = (segment u / cps, chunk u % cps); the chunk of
// 2^chunk_log2 inputs is split into one aligned span per warp; dst[u] is
// the balanced tree over the CTA's warp values (warp order, -0.0 pad).
// CTA b takes units b, b + grid, b + 2*grid, ... (launched with one CTA
// per unit, so a CTA normally takes one).
template <class Red, bool ALIGNED>
__device__ __forceinline__ void chunk_body(const void *__restrict__ xv, size_t seg_len,
                                           size_t units, size_t cps, int chunk_log2,
                                           float *__restrict__ dst)
{
    pdl_launch_dependents();   // the combine may launch now; it waits for this grid to finish
    pdl_wait_primary();        // the stream's previous kernel has finished
    constexpr int DT = Red::kDT;
    constexpr bool NZ = Red::kNegZeroPad;
    using T = typename Elem<DT>::T;
    const T *__restrict__ x = static_cast<const T *>(xv);
    __shared__ float warp_val[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    // the chunk is one span per warp: chunk_log2 = log2 of the span's inputs
    // + log2 warps; a span is a whole number of groups (16 KiB, or 4-8 KiB
    // for small inputs, chosen by the host)
    const int span_log2 = chunk_log2 - (31 - __clz(nwarps));
    const size_t span = (size_t)1 << span_log2;
    const int ngroups = (int)(span / group_len<DT>());
    size_t u = blockIdx.x;
    if (u < units) {
        size_t s = u / cps;
        const T *seg = x + s * seg_len;
        size_t base = ((u - s * cps) << chunk_log2) + (size_t)warp * span;
        GroupIn<DT, ALIGNED, NZ, realigns<Red>::value> in;
        in.load(seg, seg_len, base, lane);
        for (;;) {
            const size_t nu = u + gridDim.x;
            const bool has_next = nu < units;
            const T *nseg = seg;
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
                in.ready(seg, seg_len, base + (size_t)g * group_len<DT>(), lane);
                red.take(in.q);
                if (g + 1 < ngroups)
                    in.load(seg, seg_len, base + (size_t)(g + 1) * group_len<DT>(), lane);
                else if (has_next)
                    in.load(nseg, seg_len, nbase, lane);
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
}

// One warp per row (rows of at most 2^LEVELS groups): out[r] is the row's
// value.  Warp w takes rows w, w + warps, w + 2*warps, ... (launched with
// one warp per row, so a warp normally takes one).
template <class Red, bool ALIGNED>
__device__ __forceinline__ void rows_body(const void *__restrict__ xv, size_t rows,
                                          size_t cols, float *__restrict__ out)
{
    pdl_launch_dependents();
    pdl_wait_primary();        // the stream's previous kernel has finished
    constexpr int DT = Red::kDT;
    constexpr bool NZ = Red::kNegZeroPad;
    using T = typename Elem<DT>::T;
    const T *__restrict__ x = static_cast<const T *>(xv);
    const int lane = threadIdx.x & 31;
    const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
    size_t r = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    constexpr size_t G = group_len<DT>();
    const size_t ngroups = (cols + G - 1) / G;
    if (r < rows && ngroups > 0) {
        GroupIn<DT, ALIGNED, NZ, realigns<Red>::value> in;
        in.load(x + r * cols, cols, 0, lane);
        for (;;) {
            const size_t nr = r + nw;
            const bool has_next = nr < rows;
            Red red;
#pragma unroll 1
            for (size_t g = 0; g < ngroups; g++) {
                in.ready(x + r * cols, cols, g * G, lane);
                red.take(in.q);
                if (g + 1 < ngroups)
                    in.load(x + r * cols, cols, (g + 1) * G, lane);
                else if (has_next)
                    in.load(x + nr * cols, cols, 0, lane);
                red.reduce(lane);
            }
            const float v = red.value(lane);
            if (lane == 0) out[r] = v;
            if (!has_next) break;
            r = nr;
        }
    }
}

// ---------------------------------------------------------------- pairs

// chunk_body for a PairReducer: dst_a[u], dst_b[u] are the chunk's two values.
template <class Red, bool ALIGNED>
__device__ __forceinline__ void chunk_pair_body(const void *__restrict__ xv, size_t seg_len,
                                                size_t units, size_t cps, int chunk_log2,
                                                float *__restrict__ dst_a,
                                                float *__restrict__ dst_b)
{
    pdl_launch_dependents();   // the combine may launch now; it waits for this grid to finish
    pdl_wait_primary();        // the stream's previous kernel has finished
    constexpr int DT = Red::kDT;
    constexpr bool NZ = Red::kNegZeroPad;
    using T = typename Elem<DT>::T;
    const T *__restrict__ x = static_cast<const T *>(xv);
    __shared__ float warp_val[2][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int span_log2 = chunk_log2 - (31 - __clz(nwarps));     // as in chunk_body
    const size_t span = (size_t)1 << span_log2;
    const int ngroups = (int)(span / group_len<DT>());
    for (size_t u = blockIdx.x; u < units; u += gridDim.x) {
        const size_t s = u / cps;
        const T *seg = x + s * seg_len;
        const size_t base = ((u - s * cps) << chunk_log2) + (size_t)warp * span;
        GroupIn<DT, ALIGNED, NZ, realigns<Red>::value> in;
        in.load(seg, seg_len, base, lane);
        Red red;
#pragma unroll 1
        for (int g = 0; g < ngroups; g++) {
            in.ready(seg, seg_len, base + (size_t)g * group_len<DT>(), lane);
            red.take(in.q);
            if (g + 1 < ngroups) in.load(seg, seg_len, base + (size_t)(g + 1) * group_len<DT>(), lane);
            red.reduce(lane);
        }
        float va, vb;
        red.value2(lane, va, vb);
        if (lane == 0) {
            warp_val[0][warp] = va;
            warp_val[1][warp] = vb;
        }
        __syncthreads();
        if (warp == 0) {
            const float a = warp_tree_lane_order(lane < nwarps ? warp_val[0][lane] : -0.0f);
            const float b = warp_tree_lane_order(lane < nwarps ? warp_val[1][lane] : -0.0f);
            if (lane == 0) {
                dst_a[u] = a;
                dst_b[u] = b;
            }
        }
        __syncthreads();
    }
}

// rows_body for a PairReducer: out_a[r], out_b[r] are the row's two values,
// or (mean_var) the row's mean and variance computed from them.  The next
// row's first group is loaded while the current row's last one is reduced.
template <class Red, bool ALIGNED>
__device__ __forceinline__ void rows_pair_body(const void *__restrict__ xv, size_t rows,
                                               size_t cols, float *__restrict__ out_a,
                                               float *__restrict__ out_b, int mean_var)
{
    pdl_launch_dependents();
    pdl_wait_primary();        // the stream's previous kernel has finished
    constexpr int DT = Red::kDT;
    constexpr bool NZ = Red::kNegZeroPad;
    using T = typename Elem<DT>::T;
    const T *__restrict__ x = static_cast<const T *>(xv);
    const int lane = threadIdx.x & 31;
    const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
    size_t r = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    constexpr size_t G = group_len<DT>();
    const size_t ngroups = (cols + G - 1) / G;
    if (r < rows && ngroups > 0) {
        GroupIn<DT, ALIGNED, NZ, realigns<Red>::value> in;
        in.load(x + r * cols, cols, 0, lane);
        for (;;) {
            const size_t nr = r + nw;
            const bool has_next = nr < rows;
            Red red;
#pragma unroll 1
            for (size_t g = 0; g < ngroups; g++) {
                in.ready(x + r * cols, cols, g * G, lane);
                red.take(in.q);
                if (g + 1 < ngroups)
                    in.load(x + r * cols, cols, (g + 1) * G, lane);
                else if (has_next)
                    in.load(x + nr * cols, cols, 0, lane);
                red.reduce(lane);
            }
            float va, vb;
            red.value2(lane, va, vb);
            if (lane == 0) {
                if (mean_var) mean_var_of(va, vb, cols, va, vb);
                out_a[r] = va;
                out_b[r] = vb;
            }
            if (!has_next) break;
            r = nr;
        }
    }
}

}  // namespace tcr
