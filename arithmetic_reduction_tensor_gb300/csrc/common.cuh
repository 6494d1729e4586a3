// common.cuh -- device helpers shared by the reduction kernels.
//
// Inputs are 16-bit patterns (binary16 or bfloat16) or binary32 values.  A
// "vector" is 16 bytes = one 128-bit load per lane: 8 inputs of 16 bits or
// 4 of binary32.  A warp load of 32 vectors is 512 bytes: 256 16-bit inputs
// (exactly one 16x16 tensor-core A tile) or 128 binary32 inputs.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>

#include "config.cuh"

namespace tcr {

constexpr int kF16 = 0;
constexpr int kBF16 = 1;
constexpr int kF32 = 2;
constexpr unsigned kFull = 0xffffffffu;

// The storage of an input type: its pattern type T, the inputs per 16-byte
// vector, and the 32-bit word of -0.0 patterns -- the padding of the
// ordered modes (the identity of round-to-nearest addition for every x).
template <int DT>
struct Elem {
    using T = uint16_t;
    static constexpr int kPerVec = 8;
    static constexpr uint32_t kNegZeroWord = 0x80008000u;
};
template <>
struct Elem<kF32> {
    using T = uint32_t;
    static constexpr int kPerVec = 4;
    static constexpr uint32_t kNegZeroWord = 0x80000000u;
};

// Inputs per warp group (8 warp loads of 32 vectors) of an input type.
template <int DT>
__host__ __device__ constexpr size_t group_len()
{
    return (size_t)256 * Elem<DT>::kPerVec;
}

// ---------------------------------------------------------------- loads

// 16-byte streaming load through the read-only path.  Every input byte is
// read exactly once, so the line is not kept in L1.
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t pack2(uint16_t lo, uint16_t hi)
{
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// The fill word of a vector: -0.0 patterns (NEGZERO) or zero bits.
template <int DT, bool NEGZERO>
__device__ __forceinline__ uint32_t fill_word()
{
    return NEGZERO ? Elem<DT>::kNegZeroWord : 0u;
}

// Vector v of a segment of `len` inputs at `seg` (any alignment of the
// pattern type): the inputs past `len` read as the fill (-0.0 when
// NEGZERO, else zero bits).
template <int DT, bool NEGZERO>
__device__ __forceinline__ uint4 ld_vec_masked(const typename Elem<DT>::T *seg, size_t len,
                                               size_t v)
{
    if constexpr (DT == kF32) {
        const uint32_t f = fill_word<DT, NEGZERO>();
        uint32_t e[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const size_t i = 4 * v + (size_t)k;
            e[k] = i < len ? __ldg(seg + i) : f;
        }
        return make_uint4(e[0], e[1], e[2], e[3]);
    } else {
        const uint16_t f = NEGZERO ? (uint16_t)0x8000u : (uint16_t)0u;
        uint16_t e[8];
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const size_t i = 8 * v + (size_t)k;
            e[k] = i < len ? __ldg(seg + i) : f;
        }
        return make_uint4(pack2(e[0], e[1]), pack2(e[2], e[3]), pack2(e[4], e[5]),
                          pack2(e[6], e[7]));
    }
}

// Vector v: a single 16-byte load when the segment start is 16-byte
// aligned (ALIGNED) and the vector lies wholly inside the segment, the
// element-wise masked load otherwise.  Both give the same patterns.
template <int DT, bool ALIGNED, bool NEGZERO>
__device__ __forceinline__ uint4 ld_vec(const typename Elem<DT>::T *seg, size_t len, size_t v)
{
    constexpr int V = Elem<DT>::kPerVec;
    if (ALIGNED && V * v + V <= len) return ld_stream(seg + V * v);
    return ld_vec_masked<DT, NEGZERO>(seg, len, v);
}

// ---------------------------------------------------------------- leaves

// Exact binary32 value of the low / high 16-bit input of a 32-bit word
// (little-endian: the low half is the lower index).
template <int DT>
__device__ __forceinline__ float leaf_lo(uint32_t w)
{
    if constexpr (DT == kF16) {
        return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
    } else {
        return __uint_as_float(w << 16);
    }
}

template <int DT>
__device__ __forceinline__ float leaf_hi(uint32_t w)
{
    if constexpr (DT == kF16) {
        return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    } else {
        return __uint_as_float(w & 0xffff0000u);
    }
}

// The two leaves of a 32-bit word combined, low + high, binary32 round to
// nearest; for kOpSquares the leaves are the squares of the two inputs.
// For bfloat16 the unpacking (word << 16, word & 0xffff0000) and the
// arithmetic are one asm statement, which keeps the compiler from hoisting
// the unpacking of many words at once: the kernels that hold a group of
// loads in flight fit their register budget.
template <int DT, int OP>
__device__ __forceinline__ float pair_val(uint32_t w)
{
    if constexpr (DT == kF16) {
        const float lo = leaf_lo<DT>(w), hi = leaf_hi<DT>(w);
        if constexpr (OP == kOpSquares) return __fadd_rn(__fmul_rn(lo, lo), __fmul_rn(hi, hi));
        return __fadd_rn(lo, hi);
    } else {
        float r;
        if constexpr (OP == kOpSquares) {
            asm("{\n\t.reg .b32 lo, hi;\n\t"
                "shl.b32 lo, %1, 16;\n\t"
                "and.b32 hi, %1, 0xffff0000;\n\t"
                "mul.rn.f32 lo, lo, lo;\n\t"
                "mul.rn.f32 hi, hi, hi;\n\t"
                "add.rn.f32 %0, lo, hi;\n\t}"
                : "=f"(r)
                : "r"(w));
        } else {
            asm("{\n\t.reg .b32 lo, hi;\n\t"
                "shl.b32 lo, %1, 16;\n\t"
                "and.b32 hi, %1, 0xffff0000;\n\t"
                "add.rn.f32 %0, lo, hi;\n\t}"
                : "=f"(r)
                : "r"(w));
        }
        return r;
    }
}

// The leaf of one binary32 input: the value, or its square (one binary32
// multiplication, round to nearest).
template <int OP>
__device__ __forceinline__ float leaf32(uint32_t w)
{
    const float v = __uint_as_float(w);
    if constexpr (OP == kOpSquares) return __fmul_rn(v, v);
    return v;
}

// Balanced tree over the leaves of a vector: for 16-bit inputs
// ((e0 + e1) + (e2 + e3)) + ((e4 + e5) + (e6 + e7)), for binary32
// (e0 + e1) + (e2 + e3).
template <int DT, int OP = kOpSum>
__device__ __forceinline__ float vec_tree(uint4 q)
{
    if constexpr (DT == kF32) {
        // one asm statement, like pair_val for bfloat16: the additions stay
        // where the vector is consumed, so its registers free early
        float r;
        if constexpr (OP == kOpSquares) {
            asm("{\n\t.reg .f32 a, b, c, d;\n\t"
                "mul.rn.f32 a, %1, %1;\n\t"
                "mul.rn.f32 b, %2, %2;\n\t"
                "mul.rn.f32 c, %3, %3;\n\t"
                "mul.rn.f32 d, %4, %4;\n\t"
                "add.rn.f32 a, a, b;\n\t"
                "add.rn.f32 c, c, d;\n\t"
                "add.rn.f32 %0, a, c;\n\t}"
                : "=f"(r)
                : "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w));
        } else {
            asm("{\n\t.reg .f32 a, c;\n\t"
                "add.rn.f32 a, %1, %2;\n\t"
                "add.rn.f32 c, %3, %4;\n\t"
                "add.rn.f32 %0, a, c;\n\t}"
                : "=f"(r)
                : "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w));
        }
        return r;
    } else {
        const float p0 = pair_val<DT, OP>(q.x);
        const float p1 = pair_val<DT, OP>(q.y);
        const float p2 = pair_val<DT, OP>(q.z);
        const float p3 = pair_val<DT, OP>(q.w);
        return __fadd_rn(__fadd_rn(p0, p1), __fadd_rn(p2, p3));
    }
}

// (run + low leaf) + high leaf of a 32-bit word of two 16-bit inputs, one
// asm statement (as pair_val): the leaves are unpacked where they are added.
template <int DT>
__device__ __forceinline__ float seq_pair(float run, uint32_t w)
{
    float r;
    if constexpr (DT == kF16) {
        asm("{\n\t.reg .b16 l, h;\n\t.reg .f32 a;\n\t"
            "mov.b32 {l, h}, %2;\n\t"
            "cvt.f32.f16 a, l;\n\t"
            "add.rn.f32 %0, %1, a;\n\t"
            "cvt.f32.f16 a, h;\n\t"
            "add.rn.f32 %0, %0, a;\n\t}"
            : "=&f"(r)
            : "f"(run), "r"(w));
    } else {
        asm("{\n\t.reg .b32 a;\n\t"
            "shl.b32 a, %2, 16;\n\t"
            "add.rn.f32 %0, %1, a;\n\t"
            "and.b32 a, %2, 0xffff0000;\n\t"
            "add.rn.f32 %0, %0, a;\n\t}"
            : "=&f"(r)
            : "f"(run), "r"(w));
    }
    return r;
}

// ((x + y) + z) + w of four binary32 inputs, one asm statement.
__device__ __forceinline__ float seq_quad32(uint32_t x, uint32_t y, uint32_t z, uint32_t w)
{
    float r;
    asm("{\n\t.reg .f32 a;\n\t"
        "add.rn.f32 a, %1, %2;\n\t"
        "add.rn.f32 a, a, %3;\n\t"
        "add.rn.f32 %0, a, %4;\n\t}"
        : "=f"(r)
        : "r"(x), "r"(y), "r"(z), "r"(w));
    return r;
}

// Blocked order inside one vector: runs of 2^CLOG leaves added left to
// right, then the balanced tree over the runs (2 <= CLOG <= log2 V; runs of
// two leaves are the tree's own pairs).  A run starts from its first leaf,
// which equals starting from -0.0.
template <int DT, int CLOG>
__device__ __forceinline__ float vec_runs(uint4 q)
{
    static_assert(CLOG >= 2 && (1 << CLOG) <= Elem<DT>::kPerVec, "run outside 4..V");
    if constexpr (DT == kF32) {
        return seq_quad32(q.x, q.y, q.z, q.w);
    } else if constexpr (CLOG == 2) {
        const float r0 = seq_pair<DT>(seq_pair<DT>(-0.0f, q.x), q.y);
        const float r1 = seq_pair<DT>(seq_pair<DT>(-0.0f, q.z), q.w);
        return __fadd_rn(r0, r1);
    } else {
        return seq_pair<DT>(seq_pair<DT>(seq_pair<DT>(seq_pair<DT>(-0.0f, q.x), q.y), q.z), q.w);
    }
}

// run + (the leaves of a vector, left to right).
template <int DT>
__device__ __forceinline__ float vec_seq_add(float run, uint4 q)
{
    if constexpr (DT == kF32) {
        run = __fadd_rn(run, __uint_as_float(q.x));
        run = __fadd_rn(run, __uint_as_float(q.y));
        run = __fadd_rn(run, __uint_as_float(q.z));
        return __fadd_rn(run, __uint_as_float(q.w));
    } else {
        return seq_pair<DT>(seq_pair<DT>(seq_pair<DT>(seq_pair<DT>(run, q.x), q.y), q.z), q.w);
    }
}

// Both vector trees at once -- of the leaves and of their squares -- each
// leaf unpacked once, in one asm statement per vector (the values are those
// of vec_tree<DT, kOpSum> and vec_tree<DT, kOpSquares>, operation for
// operation).
template <int DT>
__device__ __forceinline__ void vec_tree_pair(uint4 q, float &ts, float &tq)
{
    if constexpr (DT == kF32) {
        asm("{\n\t.reg .f32 a, b, c, d;\n\t"
            "add.rn.f32 a, %2, %3;\n\t"
            "add.rn.f32 b, %4, %5;\n\t"
            "add.rn.f32 %0, a, b;\n\t"
            "mul.rn.f32 a, %2, %2;\n\t"
            "mul.rn.f32 b, %3, %3;\n\t"
            "add.rn.f32 c, a, b;\n\t"
            "mul.rn.f32 a, %4, %4;\n\t"
            "mul.rn.f32 b, %5, %5;\n\t"
            "add.rn.f32 d, a, b;\n\t"
            "add.rn.f32 %1, c, d;\n\t}"
            : "=&f"(ts), "=&f"(tq)
            : "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w));
    } else {
        // per word i: s_i = lo + hi, r_i = lo*lo + hi*hi; then
        // ts = (s0 + s1) + (s2 + s3), tq = (r0 + r1) + (r2 + r3)
#define TCR_UNPACK_F16(W) "mov.b32 {l, h}, " W ";\n\tcvt.f32.f16 lo, l;\n\tcvt.f32.f16 hi, h;\n\t"
#define TCR_UNPACK_BF16(W) "shl.b32 lo, " W ", 16;\n\tand.b32 hi, " W ", 0xffff0000;\n\t"
#define TCR_PAIR_STEP(S, R) \
    "add.rn.f32 " S ", lo, hi;\n\tmul.rn.f32 lo, lo, lo;\n\tmul.rn.f32 hi, hi, hi;\n\t" \
    "add.rn.f32 " R ", lo, hi;\n\t"
        if constexpr (DT == kF16) {
            asm("{\n\t.reg .b16 l, h;\n\t.reg .f32 lo, hi, s0, s1, s2, s3, r0, r1, r2, r3;\n\t"
                TCR_UNPACK_F16("%2") TCR_PAIR_STEP("s0", "r0")
                TCR_UNPACK_F16("%3") TCR_PAIR_STEP("s1", "r1")
                TCR_UNPACK_F16("%4") TCR_PAIR_STEP("s2", "r2")
                TCR_UNPACK_F16("%5") TCR_PAIR_STEP("s3", "r3")
                "add.rn.f32 s0, s0, s1;\n\tadd.rn.f32 s2, s2, s3;\n\tadd.rn.f32 %0, s0, s2;\n\t"
                "add.rn.f32 r0, r0, r1;\n\tadd.rn.f32 r2, r2, r3;\n\tadd.rn.f32 %1, r0, r2;\n\t}"
                : "=&f"(ts), "=&f"(tq)
                : "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w));
        } else {
            asm("{\n\t.reg .f32 lo, hi, s0, s1, s2, s3, r0, r1, r2, r3;\n\t"
                TCR_UNPACK_BF16("%2") TCR_PAIR_STEP("s0", "r0")
                TCR_UNPACK_BF16("%3") TCR_PAIR_STEP("s1", "r1")
                TCR_UNPACK_BF16("%4") TCR_PAIR_STEP("s2", "r2")
                TCR_UNPACK_BF16("%5") TCR_PAIR_STEP("s3", "r3")
                "add.rn.f32 s0, s0, s1;\n\tadd.rn.f32 s2, s2, s3;\n\tadd.rn.f32 %0, s0, s2;\n\t"
                "add.rn.f32 r0, r0, r1;\n\tadd.rn.f32 r2, r2, r3;\n\tadd.rn.f32 %1, r0, r2;\n\t}"
                : "=&f"(ts), "=&f"(tq)
                : "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w));
        }
#undef TCR_UNPACK_F16
#undef TCR_UNPACK_BF16
#undef TCR_PAIR_STEP
    }
}

// ---------------------------------------------------------------- trees

// Binary counter over a sequence of equal-height subtree values pushed in
// index order: after pushing c values it holds the aligned subtrees of the
// binary decomposition of c, and finish() returns the balanced tree over
// the c values padded with -0.0 to a power of two.  Indices into s[] are
// compile-time constants after unrolling, so s[] stays in registers.
template <int LEVELS>
struct TreeCounter {
    float s[LEVELS];
    uint32_t count;

    __device__ __forceinline__ TreeCounter() : count(0u) {}

    __device__ __forceinline__ void push(float v)
    {
        // carry up through the levels whose bit of count is set: the new
        // value is the right sibling of the subtree stored there
        bool carry = true;
#pragma unroll
        for (int l = 0; l < LEVELS; l++) {
            if (carry) {
                if ((count >> l) & 1u) {
                    v = __fadd_rn(s[l], v);        // left sibling + right sibling
                } else {
                    s[l] = v;
                    carry = false;
                }
            }
        }
        count++;
    }

    // Right-most partial subtree first: each higher stored subtree is the
    // left sibling of everything pushed after it; a missing right sibling
    // is -0.0, which passes its left sibling up unchanged.
    __device__ __forceinline__ float finish() const
    {
        float v = -0.0f;
#pragma unroll
        for (int l = 0; l < LEVELS; l++)
            if ((count >> l) & 1u) v = __fadd_rn(s[l], v);
        return v;
    }
};

// Balanced tree over the values of lanes 0..31 in lane order (offsets
// 1, 2, 4, 8, 16): every lane ends with the root.
__device__ __forceinline__ float warp_tree_lane_order(float v)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, off));
    return v;
}

// ---------------------------------------------------------------- MMA

// D += A * ones for one m16n8k16 tile: A is 16x16 inputs held 8 per lane
// (a0..a7 in the four 32-bit registers of q), B is the 16x8 all-ones
// matrix, D the 16x8 fp32 accumulator (d0, d1: row lane/4; d2, d3: row
// lane/4 + 8; every column of D holds the same row sums).
template <int DT>
__device__ __forceinline__ void mma_ones(float &d0, float &d1, float &d2, float &d3,
                                         uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3)
{
    if constexpr (DT == kF16) {
        const uint32_t one2 = 0x3c003c00u;    // binary16 1.0, twice
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
            : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(one2), "r"(one2));
    } else {
        const uint32_t one2 = 0x3f803f80u;    // bfloat16 1.0, twice
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
            : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(one2), "r"(one2));
    }
}

// D += A * B for one m16n8k16 tile with B given by registers: b0 holds
// B[2t][g], B[2t+1][g] and b1 holds B[2t+8][g], B[2t+9][g] (g = lane/4,
// t = lane%4).
template <int DT>
__device__ __forceinline__ void mma_ab(float &d0, float &d1, float &d2, float &d3, uint32_t a0,
                                       uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1)
{
    if constexpr (DT == kF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
            : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
            : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// ---------------------------------------------------------------- moments

// Mean and variance of n inputs from their sum s1 and sum of squares s2, in
// binary32 with one rounding to nearest per operation:
// m = s1 / n, v = s2 / n - m * m, a negative v (rounding only) becomes +0.
__device__ __forceinline__ void mean_var_of(float s1, float s2, size_t n, float &m, float &v)
{
    const float nf = __ull2float_rn((unsigned long long)n);
    m = __fdiv_rn(s1, nf);
    const float q = __fdiv_rn(s2, nf);
    v = __fsub_rn(q, __fmul_rn(m, m));
    if (v < 0.0f) v = 0.0f;
}

// ---------------------------------------------------------------- PDL

// Programmatic dependent launch: a producing kernel lets the next kernel
// on the stream start launching; the consumer waits until the producer has
// completed and its writes are visible.  Both are no-ops for a kernel
// launched without the attribute.  Every kernel of the library triggers its
// dependents as it starts, and every kernel launched with the attribute
// (a call's first kernel, its combines) waits before its first global
// memory access -- the wait covers the kernel before it on the stream,
// whichever it is.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_primary()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__host__ __device__ __forceinline__ int ceil_log2_sz(size_t n)
{
    int h = 0;
    while (((size_t)1 << h) < n) h++;
    return h;
}

}  // namespace tcr
