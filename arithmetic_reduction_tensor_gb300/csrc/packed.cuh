// packed.cuh -- short rows, several to a warp group.
//
// The one-warp-per-row kernels walk a row in groups of 8 warp loads x 32
// lanes = 256 vectors (16 bytes each), so a row of a few hundred inputs
// leaves most of its group's loads empty and the warp holds too few bytes
// in flight.  Here a matrix whose rows hold at most 128 vectors is packed:
// a row gets W = 2^VLOG vector slots (the least power of two covering it;
// at least 4 for MMA_CHAIN), and a group's 256 slots hold 256 / W rows --
// lane j of load k holds slot 32 k + j, i.e. vector (32 k + j) mod W of
// group row (32 k + j) / W.  Slots past a row's vectors, or of rows past the
// matrix, read as the mode's pad (-0.0; zero bits for the tensor cores).
// The next group's loads are issued before the current group is reduced.
//
// Each mode keeps the order it declares for a row:
//
//   FIXED_ORDER   the vectors' trees, then the balanced tree over the row's
//                 vectors in lane order: lane pairs (j, j^1), then (j, j^2),
//                 ... within a sub-warp of W lanes (VLOG <= 5), or the whole
//                 load's tree followed by the tree over the row's loads
//                 (VLOG 6, 7) -- aligned subtrees of the row's balanced tree
//                 padded with -0.0;
//   SHUFFLE_TREE  the one-warp team: lane j of the row adds its vectors in
//                 load order from -0.0, then the butterfly with offsets 16,
//                 8, 4, 2, 1.  A row of W < 32 slots sits in a sub-warp whose
//                 missing lanes would hold -0.0, so the butterfly's steps
//                 with offsets >= W add -0.0 (no change) and the rest run
//                 inside the sub-warp;
//   MMA_CHAIN     one m16n8k16 tile against ones per load.  D row g of the
//                 MMA sums lane quad g's four vectors (d0 + d2), so a row of
//                 at least one quad is the sum over its quads; a row
//                 spanning L loads chains its L tiles, flushed every R.
//                 Squares: the tile's A * A^T diagonal.  Binary32: each
//                 input (or its square) split exactly into three bfloat16
//                 parts, a lane's hi and mid parts forming one tile and its
//                 lo parts a second one chained into the same accumulator
//                 (so a D row still holds one quad's inputs only).
//
// The lane-pair steps use a reduce-scatter: a lane carries one value per
// load (or row), and at each of the first steps the two lanes of a pair
// split the values -- the lane whose offset bit is set keeps the upper
// half -- so 8 values need 4 + 2 + 1 shuffles instead of 3 x 8.  Every sum
// is still the sum of the same two operands (addition commutes bit for
// bit), so the order is unchanged; only which lane forms it differs.
#pragma once

#include "common.cuh"
#include "kernels.cuh"
#include "stream.cuh"

namespace tcr {

constexpr int kPackedMaxVlog = 7;         // rows of at most 128 vectors

// One reduce-scatter step over H value pairs: v[i] (i < H) becomes the sum
// over lanes j, j^o of the item kept, item_base advancing by H in the lane
// that keeps the upper half.
template <int H>
__device__ __forceinline__ void rs_step(float (&v)[8], int lane, int o, int &item_base)
{
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < H; i++) {
        const float keep = up ? v[i + H] : v[i];
        const float send = up ? v[i] : v[i + H];
        v[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, o));
    }
    if (up) item_base += H;
}

// NS reduce-scatter steps over 8 items with offsets o1, o2, o3 (the first
// NS of them), leaving 8 >> NS values: v[i] = item item_base + i.
template <int NS>
__device__ __forceinline__ void rs_steps(float (&v)[8], int lane, int o1, int o2, int o3, int &item_base)
{
    if constexpr (NS >= 1) rs_step<4>(v, lane, o1, item_base);
    if constexpr (NS >= 2) rs_step<2>(v, lane, o2, item_base);
    if constexpr (NS >= 3) rs_step<1>(v, lane, o3, item_base);
}

// ---------------------------------------------------------------- loads
//
// Aligned rows (x 16-byte aligned, rows whole vectors): slot (k, lane) is
// one 16-byte load of its vector.
//
// Other rows: the group's rows are contiguous, so the vector of slot
// (k, lane) -- inputs e .. e + V - 1 of the group, e = row * cols + V * v --
// lies in 16-byte granule (hoff + e * EB) / 16 of the group (hoff: the
// group's byte offset in its first granule) and the next one.  Each slot
// loads its first granule whole (it holds an input of the matrix, so the
// load stays inside the data); the second one is the first granule of the
// next slot.  Inside a row that slot holds vector v + 1 (or, past the
// row's last vector, the granule after it).  After a row's last slot it is
// the next row's first slot, whose granule holds the row's end: when the
// last vector reaches into a second granule, the row ends inside that
// granule, so it is the one the next row starts in.  For the last row of
// the matrix the slot of the row past it loads that granule when it still
// holds data, and the group's own last slot takes the first granule of the
// rows after the group from one extra load (lane 31).  The vector is
// shifted out of the two granules when the group is reduced, while the
// next group's loads are in flight.

struct PackedGeom {
    const uint4 *gbase;   // the group's first granule
    uint32_t hoff;        // byte offset of the group's first input in it
    uint32_t glim;        // last granule index (from gbase) inside the data
};

template <int DT>
__device__ __forceinline__ PackedGeom packed_geom(const typename Elem<DT>::T *x, size_t rows, size_t cols,
                                                  size_t row0)
{
    const uintptr_t a = (uintptr_t)(x + row0 * cols);
    const uintptr_t last = (uintptr_t)(x + rows * cols) - 1;
    const uintptr_t gaddr = a & ~(uintptr_t)15;
    const size_t gl = (size_t)(last - gaddr) >> 4;
    PackedGeom g;
    g.gbase = reinterpret_cast<const uint4 *>(gaddr);
    g.hoff = (uint32_t)(a & 15);
    g.glim = gl > 0xffffffffu ? 0xffffffffu : (uint32_t)gl;
    return g;
}

// Vector v (v * V < len) of a row that starts on an 8-byte boundary and is
// a whole number of 8-byte words long: two 8-byte streaming loads, or for
// the row's last vector when it holds only one word, that word and the
// fill -- the same patterns a 16-byte load of an aligned row gives, with no
// realignment.  BRANCH (the trees on rows of 33 to 128 vectors): both words
// through L1 when the vector is whole, else the element-wise masked load --
// measured faster there, slower on every other kind of row.  `words`: the
// rows start on 4-byte boundaries only (and are whole 4-byte words): four
// 4-byte loads through L1 (the four of a warp share their lines), the words
// past the row the fill.
template <int DT, bool NEGZERO, bool BRANCH = false>
__device__ __forceinline__ uint4 ld_vec_half(const typename Elem<DT>::T *seg, size_t len, size_t v,
                                             bool words)
{
    constexpr int V = Elem<DT>::kPerVec;
    constexpr uint32_t EB = sizeof(typename Elem<DT>::T);
    if (words) {
        const uint32_t *p4 = reinterpret_cast<const uint32_t *>(seg + V * v);
        const size_t left = len - V * v;
        const uint32_t nb = left >= (size_t)V ? 16u : (uint32_t)left * EB;     // bytes of the row here
        const uint32_t f = fill_word<DT, NEGZERO>();
        uint4 r = make_uint4(0u, f, f, f);
        asm("ld.global.nc.u32 %0, [%1];" : "=r"(r.x) : "l"(p4));
        asm("{\n\t.reg .pred q;\n\tsetp.gt.u32 q, %3, 4;\n\t@q ld.global.nc.u32 %0, [%4];\n\t"
            "setp.gt.u32 q, %3, 8;\n\t@q ld.global.nc.u32 %1, [%5];\n\t"
            "setp.gt.u32 q, %3, 12;\n\t@q ld.global.nc.u32 %2, [%6];\n\t}"
            : "+r"(r.y), "+r"(r.z), "+r"(r.w)
            : "r"(nb), "l"(p4 + 1), "l"(p4 + 2), "l"(p4 + 3));
        return r;
    }
    const uint2 *p = reinterpret_cast<const uint2 *>(seg + V * v);
    if constexpr (BRANCH) {
        if (V * v + V <= len) {
            uint4 w;
            asm("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(w.x), "=r"(w.y) : "l"(p));
            asm("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(w.z), "=r"(w.w) : "l"(p + 1));
            return w;
        }
        return ld_vec_masked<DT, NEGZERO>(seg, len, v);
    }
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    // the second word as a predicated load (no branch, so the loads of a
    // group still issue together); it keeps the fill when not taken
    r.z = r.w = fill_word<DT, NEGZERO>();
    const uint32_t whole = V * v + V <= len ? 1u : 0u;
    asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t@q ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];\n\t}"
        : "+r"(r.z), "+r"(r.w)
        : "l"(p + 1), "r"(whole));
    return r;
}

// Load k (0..7) of the group whose first row is row0.  HALF (with ALIGNED):
// every row starts on a 4-byte boundary and is a whole number of 4-byte
// words long (on 8-byte boundaries and of 8-byte words unless `words`); x
// may not be 16-byte aligned.
template <int DT, bool ALIGNED, bool NEGZERO, int VLOG, bool HALF = false, bool BR = false>
__device__ __forceinline__ uint4 load_slot(const typename Elem<DT>::T *x, size_t rows, size_t cols,
                                           size_t row0, const PackedGeom &gm, int k, int lane,
                                           bool words = false)
{
    constexpr int V = Elem<DT>::kPerVec;
    constexpr uint32_t EB = sizeof(typename Elem<DT>::T);
    const uint32_t f = fill_word<DT, NEGZERO>();
    const int slot = 32 * k + lane;
    const uint32_t rr = (uint32_t)(slot >> VLOG);
    const uint32_t v = (uint32_t)(slot & ((1 << VLOG) - 1));
    const uint32_t c = (uint32_t)cols;                   // at most 128 vectors
    if constexpr (ALIGNED) {
        if (!(row0 + rr < rows && V * v < c)) return make_uint4(f, f, f, f);
        if constexpr (HALF) return ld_vec_half<DT, NEGZERO, BR>(x + (row0 + rr) * cols, cols, v, words);
        else return ld_vec<DT, true, NEGZERO>(x + (row0 + rr) * cols, cols, v);
    } else {
        // slots up to the one after the row's last vector, and the first
        // slot of the row past the matrix
        if (!((row0 + rr < rows && V * v < c + V) || (row0 + rr == rows && v == 0)))
            return make_uint4(f, f, f, f);
        const uint32_t gi = (gm.hoff + (rr * c + V * v) * EB) >> 4;
        return gi <= gm.glim ? ld_stream(gm.gbase + gi) : make_uint4(f, f, f, f);
    }
}

// Unaligned rows: the first granule of the rows after the group (lane 31).
template <int DT, int VLOG>
__device__ __forceinline__ uint4 load_tail(size_t rows, size_t cols, size_t row0, const PackedGeom &gm,
                                           int lane)
{
    constexpr uint32_t EB = sizeof(typename Elem<DT>::T);
    constexpr uint32_t RPG = 256u >> VLOG;
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 31 && row0 + RPG <= rows) {
        const uint32_t gi = (gm.hoff + RPG * (uint32_t)cols * EB) >> 4;
        if (gi <= gm.glim) r = ld_stream(gm.gbase + gi);
    }
    return r;
}

template <int DT, bool ALIGNED, bool NEGZERO, int VLOG, bool HALF = false, bool BR = false>
__device__ __forceinline__ void load_packed(uint4 (&q)[8], const typename Elem<DT>::T *x, size_t rows,
                                            size_t cols, size_t row0, const PackedGeom &gm, int lane,
                                            bool words = false)
{
#pragma unroll
    for (int k = 0; k < 8; k++)
        q[k] = load_slot<DT, ALIGNED, NEGZERO, VLOG, HALF, BR>(x, rows, cols, row0, gm, k, lane, words);
}

// The vector of slot (k, lane) of an unaligned group from the granules in
// q: this lane's q[k] and the next slot's (lane + 1's; lane 0's q[k + 1]
// for lane 31; the tail granule qt for the group's last slot), shifted by
// the vector's byte offset; inputs past the row, and every input of a row
// past the matrix, read as the fill.  Every lane of the warp takes part
// (shuffles).
template <int DT, bool NEGZERO, int VLOG>
__device__ __forceinline__ uint4 unaligned_vec(const uint4 (&q)[8], const uint4 &qt, int k, int lane,
                                               uint32_t hoff, size_t rows, size_t cols, size_t row0)
{
    constexpr int V = Elem<DT>::kPerVec;
    constexpr int EB = (int)sizeof(typename Elem<DT>::T);
    const uint4 lo = q[k];
    // lane j reads lane j + 1's value; lane 0 sends the next load's
    // granule, for lane 31
    uint4 snd = lo;
    if (k < 7 && lane == 0) snd = q[k < 7 ? k + 1 : k];
    const int src = (lane + 1) & 31;
    uint4 hi;
    hi.x = __shfl_sync(kFull, snd.x, src);
    hi.y = __shfl_sync(kFull, snd.y, src);
    hi.z = __shfl_sync(kFull, snd.z, src);
    hi.w = __shfl_sync(kFull, snd.w, src);
    if (k == 7 && lane == 31) hi = qt;
    const int slot = 32 * k + lane;
    const uint32_t rr = (uint32_t)(slot >> VLOG);
    const int v = slot & ((1 << VLOG) - 1);
    const uint32_t sb = (hoff + (rr * (uint32_t)cols + (uint32_t)(V * v)) * EB) & 15u;
    int cnt = (int)cols - V * v;
    cnt = cnt < 0 ? 0 : (cnt > V ? V : cnt);
    if (!(row0 + rr < rows)) cnt = 0;
    // shift the 8 words by sb bytes: 2 words, 1 word, then half a word
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t p = sb >> 2;
    uint32_t t[5], o[4];
    if constexpr (VLOG >= 5) {
        // a load holds vectors of one row only, so sb is the same in every
        // lane: a warp-uniform branch picks the words (no per-lane selects)
        switch (p) {
        case 0:
#pragma unroll
            for (int i = 0; i < 5; i++) t[i] = w[i];
            break;
        case 1:
#pragma unroll
            for (int i = 0; i < 5; i++) t[i] = w[i + 1];
            break;
        case 2:
#pragma unroll
            for (int i = 0; i < 5; i++) t[i] = w[i + 2];
            break;
        default:
#pragma unroll
            for (int i = 0; i < 5; i++) t[i] = w[i + 3];
            break;
        }
    } else {
        uint32_t u[6];
#pragma unroll
        for (int i = 0; i < 6; i++) u[i] = (p & 2) ? w[i + 2] : w[i];
#pragma unroll
        for (int i = 0; i < 5; i++) t[i] = (p & 1) ? u[i + 1] : u[i];
    }
    const uint32_t hs = (sb & 2u) << 3;                  // 0 or 16 (0 for binary32)
    const uint32_t f = fill_word<DT, NEGZERO>();
#pragma unroll
    for (int i = 0; i < 4; i++) {
        o[i] = __funnelshift_r(t[i], t[i + 1], hs);
        // keep the low bits of the word that hold inputs below cnt
        const int kb = cnt * 8 * EB - 32 * i;
        const uint32_t m = __funnelshift_lc(0xffffffffu, 0u, (uint32_t)(kb < 0 ? 0 : kb));
        o[i] = (o[i] & m) | (f & ~m);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------- rows of a group
//
// packed_reduce turns a lane's per-load values t[k] (FIXED_ORDER and
// SHUFFLE_TREE: vector trees; MMA_CHAIN: lane-quad totals for VLOG <= 5,
// per-row quad totals t[r] for VLOG 6, 7) into row values: afterwards the
// lane holds packed_m() values t[0..M-1], t[i] being group row
// packed_row(base, i, lane) when `writer` is set.

template <int MODE, int VLOG>
__host__ __device__ constexpr int packed_m()
{
    if (VLOG > 5) return 1;
    if (MODE == kPackedMma) return 8 >> (VLOG - 2);
    return 8 >> (VLOG < 3 ? VLOG : 3);
}

template <int MODE, int VLOG>
__device__ __forceinline__ uint32_t packed_row(int base, int i, int lane)
{
    if constexpr (VLOG <= 5) return (uint32_t)((base + i) * (32 >> VLOG) + (lane >> VLOG));
    else if constexpr (MODE == kPackedFixed) return (uint32_t)(base >> (VLOG - 5));
    else return (uint32_t)base;
}

template <int MODE, int VLOG>
__device__ __forceinline__ int packed_reduce(float (&t)[8], int lane, bool &writer)
{
    constexpr int W = 1 << VLOG;
    int base = 0;
    if constexpr (MODE == kPackedMma) {
        // sums over the row's lane quads: ascending offsets 4, 8, 16
        if constexpr (VLOG <= 5) {
            rs_steps<VLOG - 2>(t, lane, 4, 8, 16, base);   // offsets 4 .. W/2
            writer = (lane & 3) == 0;
        } else {
            constexpr int NS = VLOG == 6 ? 2 : 1;          // log2 rows per group
            if constexpr (NS == 2) {
                rs_step<2>(t, lane, 4, base);
                rs_step<1>(t, lane, 8, base);
            } else {
                rs_step<1>(t, lane, 4, base);
            }
#pragma unroll
            for (int o = 4 << NS; o < 32; o <<= 1) t[0] = __fadd_rn(t[0], __shfl_xor_sync(kFull, t[0], o));
            writer = (lane & 3) == 0 && lane < (4 << NS);
        }
    } else if constexpr (VLOG <= 5) {
        constexpr int NS = VLOG < 3 ? VLOG : 3;
        if constexpr (MODE == kPackedFixed) {
            // ascending offsets 1, 2, 4 (scatter), then 8, 16 below W
            rs_steps<NS>(t, lane, 1, 2, 4, base);
#pragma unroll
            for (int o = 8; o < W; o <<= 1) t[0] = __fadd_rn(t[0], __shfl_xor_sync(kFull, t[0], o));
            writer = (lane & (W - 1)) < (1 << NS);
        } else {
            // the one-warp butterfly: offsets W/2, W/4, W/8 (scatter), then
            // the rest down to 1; the lane's start value -0.0 + t is t
            rs_steps<NS>(t, lane, W >> 1, W >> 2, W >> 3, base);
#pragma unroll
            for (int o = W >> 4; o >= 1; o >>= 1) t[0] = __fadd_rn(t[0], __shfl_xor_sync(kFull, t[0], o));
            writer = (lane & ((W >> NS) - 1)) == 0;
        }
    } else {
        constexpr int LL = VLOG - 5;                     // log2 loads per row
        constexpr int L = 1 << LL;
        constexpr int M = 8 >> LL;                       // rows per group
        if constexpr (MODE == kPackedFixed) {
            // each load's tree (scatter 1, 2, 4, then 8, 16); loads k, k^1
            // then sit in lanes j, j^4 and loads k, k^2 in lanes j, j^2
            rs_steps<3>(t, lane, 1, 2, 4, base);
            t[0] = __fadd_rn(t[0], __shfl_xor_sync(kFull, t[0], 8));
            t[0] = __fadd_rn(t[0], __shfl_xor_sync(kFull, t[0], 16));
            t[0] = __fadd_rn(t[0], __shfl_xor_sync(kFull, t[0], 4));
            if constexpr (LL >= 2) t[0] = __fadd_rn(t[0], __shfl_xor_sync(kFull, t[0], 2));
            writer = lane < M;
        } else {
            // lane j adds its vectors of each row in load order, then the
            // butterfly 16, 8, 4, 2, 1 over the M row values
#pragma unroll
            for (int r = 0; r < M; r++) {
                float a = -0.0f;
#pragma unroll
                for (int k = 0; k < L; k++) a = __fadd_rn(a, t[r * L + k]);
                t[r] = a;
            }
            constexpr int NS = LL == 1 ? 2 : 1;          // log2 M
            if constexpr (NS == 2) {
                rs_step<2>(t, lane, 16, base);
                rs_step<1>(t, lane, 8, base);
            } else {
                rs_step<1>(t, lane, 16, base);
            }
#pragma unroll
            for (int o = 16 >> NS; o >= 1; o >>= 1) t[0] = __fadd_rn(t[0], __shfl_xor_sync(kFull, t[0], o));
            writer = (lane & ((32 >> NS) - 1)) == 0;
        }
    }
    return base;
}

// A row's result: out_a[row] = a (single reductions, or a pair's first
// value), out_b[row] = b (pairs), or the mean and variance from the pair.
template <bool PAIR>
__device__ __forceinline__ void packed_store(float *__restrict__ out_a, float *__restrict__ out_b,
                                             size_t row, float a, float b, size_t cols, int mean_var)
{
    if constexpr (PAIR) {
        if (mean_var) mean_var_of(a, b, cols, a, b);
        out_b[row] = b;
    }
    out_a[row] = a;
}

// The diagonal of A * A^T of one m16n8k16 tile (two MMAs, see MmaSqReducer
// in stream.cuh): lane quad g's sum of squares, in every lane of the quad.
template <int DT>
__device__ __forceinline__ void mma_sq_quad(const uint4 &a, float &p0, float &p1, float &p2, float &p3,
                                            float &q0, float &q1, float &q2, float &q3)
{
    mma_ab<DT>(p0, p1, p2, p3, a.x, a.y, a.z, a.w, a.x, a.z);
    mma_ab<DT>(q0, q1, q2, q3, a.x, a.y, a.z, a.w, a.y, a.w);
}
__device__ __forceinline__ float sq_diag(int lane, float p0, float p1, float q2, float q3)
{
    // D[g][g] and D[g+8][g+8] sit in lane (g, g / 2): d0 / d2 for even g,
    // d1 / d3 for odd g
    const int g = lane >> 2;
    return (g & 1) ? __fadd_rn(p1, q3) : __fadd_rn(p0, q2);
}
__device__ __forceinline__ float quad_bcast(float v, int lane)
{
    const int g = lane >> 2;
    return __shfl_sync(kFull, v, 4 * g + (g >> 1));
}

// Binary32: D += the tiles of load a's leaves (inputs for kOpSum, their
// binary32 squares for kOpSquares) split into bfloat16 parts (split_bf16x3
// in stream.cuh): A rows g / g+8 take the hi and mid parts of the lane
// quad's inputs 0, 1 / 2, 3, then a second tile their lo parts, so d0 + d2
// is lane quad g's total.
template <int LOP>
__device__ __forceinline__ void mma_f32_tiles(const uint4 &a, float &d0, float &d1, float &d2, float &d3)
{
    uint32_t h0, m0, l0, h1, m1, l1;
    split_bf16x3<LOP>(a.x, a.y, h0, m0, l0);
    split_bf16x3<LOP>(a.z, a.w, h1, m1, l1);
    mma_ones<kBF16>(d0, d1, d2, d3, h0, h1, m0, m1);
    mma_ones<kBF16>(d0, d1, d2, d3, l0, l1, 0u, 0u);
}

// The packed kernel: one warp per group of 256 / W rows, grid-stride over
// the groups.  PAIR: the sum and the sum of squares of every row in one
// pass (out_a, out_b), or their mean and variance (mean_var != 0); else
// the reduction OP into out_a.  R is the chain length of MMA_CHAIN (rows of
// VLOG 6 or 7 only; 1 otherwise).
// The tensor-core squares and binary32 splits hold two or three tiles'
// accumulators (or the split parts) beside the loads in flight: they get
// the registers of 2 resident CTAs per SM instead of 3.
template <int DT, int MODE, int OP, bool PAIR>
__host__ __device__ constexpr int packed_min_ctas()
{
    return MODE == kPackedMma && (PAIR || OP == kOpSquares || DT == kF32) ? 2 : kRowsMinCtas;
}

template <int DT, int OP, int MODE, int VLOG, int R, bool ALIGNED, bool PAIR, bool HALF = false>
__global__ void __launch_bounds__(kRowsBlock, packed_min_ctas<DT, MODE, OP, PAIR>())
packed_rows_kernel(const void *__restrict__ xv, size_t rows, size_t cols, float *__restrict__ out_a,
                   float *__restrict__ out_b, int mean_var)
{
    static_assert(MODE != kPackedMma || VLOG >= 2, "a tensor-core row is at least one lane quad");
    pdl_launch_dependents();
    pdl_wait_primary();        // the stream's previous kernel has finished
    using T = typename Elem<DT>::T;
    constexpr bool NZ = MODE != kPackedMma;
    constexpr int M = packed_m<MODE, VLOG>();
    const T *__restrict__ x = static_cast<const T *>(xv);
    const int lane = threadIdx.x & 31;
    const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
    constexpr size_t RPG = (size_t)256 >> VLOG;          // rows per group
    const size_t groups = (rows + RPG - 1) / RPG;
    size_t gi = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (gi >= groups) return;
    uint4 q[8], qt = make_uint4(0u, 0u, 0u, 0u);
    PackedGeom gm{};
    if constexpr (!ALIGNED) {
        gm = packed_geom<DT>(x, rows, cols, gi * RPG);
        qt = load_tail<DT, VLOG>(rows, cols, gi * RPG, gm, lane);
    }
    constexpr bool BR = MODE != kPackedMma && VLOG >= 6;     // the form of ld_vec_half
    // rows on 4-byte but not 8-byte boundaries, or not whole 8-byte words
    const bool words = HALF && ((((uintptr_t)xv) & 7u) != 0 || ((cols * sizeof(T)) & 7u) != 0);
    load_packed<DT, ALIGNED, NZ, VLOG, HALF, BR>(q, x, rows, cols, gi * RPG, gm, lane, words);
    for (;;) {
        const size_t row0 = gi * RPG;
        const size_t ngi = gi + nw;
        const bool has_next = ngi < groups;
        const size_t nrow0 = ngi * RPG;
        const uint32_t hoff = gm.hoff;                   // this group's (unaligned rows)
        if constexpr (!ALIGNED)
            if (has_next) gm = packed_geom<DT>(x, rows, cols, nrow0);
        // the vector of load k of this group
        auto vec = [&](int k) -> uint4 {
            if constexpr (ALIGNED) return q[k];
            else return unaligned_vec<DT, NZ, VLOG>(q, qt, k, lane, hoff, rows, cols, row0);
        };
        // once load k of this group is consumed: the next group's load k
        // (and after the last one its tail), so few registers are live
        // beside the loads in flight.  An unaligned vector is a copy made
        // from the granules, so the next load may replace them before the
        // vector is reduced; an aligned one is the loaded register itself.
        auto next = [&](int k) {
            if (has_next)
                q[k] = load_slot<DT, ALIGNED, NZ, VLOG, HALF, BR>(x, rows, cols, nrow0, gm, k, lane, words);
            if constexpr (!ALIGNED)
                if (k == 7 && has_next) qt = load_tail<DT, VLOG>(rows, cols, nrow0, gm, lane);
        };
        float ta[8], tb[8];
        // a load past the end of every row of the group (rows spanning 2 or
        // 4 loads with fewer vectors than slots, e.g. 96 of 128): every
        // vector of it is the pad, so the trees skip it -- the pad tree is
        // -0.0 (+0.0 for squares).  Aligned rows only: around the realigning
        // shuffles of other rows the branch left the trees waiting on their
        // loads (rows of 1001: 2.9 against 5.0 TB/s without it), and the
        // realigned pad vectors give the same -0.0 trees.  The MMA path keeps
        // its straight-line chain (a branch there cost more than the zero
        // tiles it saves)
        auto pad_load = [&](int k) -> bool {
            if constexpr (VLOG >= 6 && ALIGNED)
                return (size_t)(32 * Elem<DT>::kPerVec) * (size_t)(k & ((1 << (VLOG - 5)) - 1)) >= cols;
            else
                return false;
        };
        if constexpr (MODE == kPackedMma) {
            // sums: tiles against ones; squares: the tiles' A * A^T diagonals
            // (pairs: sums into ta, squares into tb)
            constexpr bool SUM = PAIR || OP == kOpSum;
            constexpr bool SQ = PAIR || OP == kOpSquares;
            float(&tq)[8] = PAIR ? tb : ta;
            if constexpr (VLOG <= 5) {
                // one tile per load: lane quad g's total is d0 + d2, its sum
                // of squares the tile's diagonal
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const uint4 a = vec(k);
                    if constexpr (!ALIGNED) next(k);
                    float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
                    if constexpr (DT == kF32) {
                        if constexpr (SUM) mma_f32_tiles<kOpSum>(a, d0, d1, d2, d3);
                        if constexpr (SQ) {
                            float e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
                            mma_f32_tiles<kOpSquares>(a, e0, e1, e2, e3);
                            tq[k] = __fadd_rn(e0, e2);
                        }
                    } else {
                        if constexpr (SUM) mma_ones<DT>(d0, d1, d2, d3, a.x, a.y, a.z, a.w);
                        if constexpr (SQ) {
                            float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f, r0 = 0.f, r1 = 0.f, r2 = 0.f,
                                  r3 = 0.f;
                            mma_sq_quad<DT>(a, p0, p1, p2, p3, r0, r1, r2, r3);
                            tq[k] = quad_bcast(sq_diag(lane, p0, p1, r2, r3), lane);
                        }
                    }
                    if constexpr (ALIGNED) next(k);
                    if constexpr (SUM) ta[k] = __fadd_rn(d0, d2);
                }
            } else {
                // a row's L loads: chains of R tiles, each chain's d0 and d2
                // (its diagonal) added into the row's accumulators
                constexpr int L = 1 << (VLOG - 5), MR = 8 / L;
#pragma unroll
                for (int r = 0; r < MR; r++) {
                    float lo = 0.f, hi = 0.f, d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
                    float sq = 0.f, p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f, r0 = 0.f, r1 = 0.f, r2 = 0.f,
                          r3 = 0.f;
#pragma unroll
                    for (int k = 0; k < L; k++) {
                        const int j = r * L + k;
                        const uint4 a = vec(j);
                        if constexpr (!ALIGNED) next(j);
                        const bool fl = (k + 1) % R == 0 || k == L - 1;     // chain ends
                        if constexpr (SUM) {
                            if constexpr (DT == kF32) mma_f32_tiles<kOpSum>(a, d0, d1, d2, d3);
                            else mma_ones<DT>(d0, d1, d2, d3, a.x, a.y, a.z, a.w);
                            if (fl) {
                                lo = __fadd_rn(lo, d0);
                                hi = __fadd_rn(hi, d2);
                                d0 = d1 = d2 = d3 = 0.f;
                            }
                        }
                        if constexpr (SQ && DT == kF32) {
                            // the squares' tiles: p0 / p2 as the sums' d0 / d2
                            mma_f32_tiles<kOpSquares>(a, p0, p1, p2, p3);
                            if (fl) {
                                sq = __fadd_rn(sq, __fadd_rn(p0, p2));
                                p0 = p1 = p2 = p3 = 0.f;
                            }
                        } else if constexpr (SQ) {
                            mma_sq_quad<DT>(a, p0, p1, p2, p3, r0, r1, r2, r3);
                            if (fl) {
                                sq = __fadd_rn(sq, sq_diag(lane, p0, p1, r2, r3));
                                p0 = p1 = p2 = p3 = r0 = r1 = r2 = r3 = 0.f;
                            }
                        }
                        if constexpr (ALIGNED) next(j);
                    }
                    if constexpr (SUM) ta[r] = __fadd_rn(lo, hi);
                    if constexpr (SQ) tq[r] = DT == kF32 ? sq : quad_bcast(sq, lane);
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; k++) {
                if (pad_load(k)) {
                    ta[k] = (!PAIR && OP == kOpSquares) ? 0.0f : -0.0f;
                    tb[k] = 0.0f;
                    next(k);
                    continue;
                }
                const uint4 a = vec(k);
                if constexpr (!ALIGNED) next(k);
                if constexpr (PAIR) vec_tree_pair<DT>(a, ta[k], tb[k]);
                else ta[k] = vec_tree<DT, OP>(a);
                if constexpr (ALIGNED) next(k);
                if constexpr (VLOG == 0) {
                    // a row is one vector: its value is the vector's tree
                    // (SHUFFLE_TREE: -0.0 + tree, the same bits)
                    const size_t row = row0 + (size_t)(32 * k + lane);
                    if (row < rows) packed_store<PAIR>(out_a, out_b, row, ta[k], tb[k], cols, mean_var);
                }
            }
        }
        if constexpr (MODE == kPackedMma || VLOG > 0) {
            bool writer;
            const int base = packed_reduce<MODE, VLOG>(ta, lane, writer);
            if constexpr (PAIR) packed_reduce<MODE, VLOG>(tb, lane, writer);
            if (writer) {
#pragma unroll
                for (int i = 0; i < M; i++) {
                    const size_t row = row0 + packed_row<MODE, VLOG>(base, i, lane);
                    if (row < rows) packed_store<PAIR>(out_a, out_b, row, ta[i], tb[i], cols, mean_var);
                }
            }
        }
        if (!has_next) break;
        gi = ngi;
    }
}

// Kernel pointers of each mode (k_packed_*.cu); nullptr where the mode has
// no packed kernel for the arguments.
// pair: the sum-and-squares kernel (op ignored).
// align: 0 rows read as whole granules and realigned, 1 16-byte aligned
// rows, 2 rows that all start on an 8-byte boundary (loads of 8 bytes)
const void *packed_pick_fixed(int dtype, int op, int vlog, int align, bool pair);
const void *packed_pick_shuffle(int dtype, int op, int vlog, int align, bool pair);
const void *packed_pick_mma(int dtype, int op, int vlog, int R, int align, bool pair);

}  // namespace tcr
