/*
 * tcr_oracle.c -- CPU oracle for the sum-reduction library.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously correct
 * restatement of what the reductions compute.  Only the test-suite, the
 * smoke check and the benchmark's CPU-baseline leg load it; the library
 * (the CUDA path) never does, and the two share no code, header or table.
 *
 * What the reduction is, and where each function comes from:
 *
 *  - "GPU Tensor Cores for fast Arithmetic Reductions" (arXiv 2001.05585),
 *    Abstract: the problem is the arithmetic reduction (sum) of n numbers;
 *    chain sub-results are kept as 32-bit floats and all of them are then
 *    reduced into a final 32-bit result.  The tensor-core method's exact
 *    rounding is not fixed by the page, so its oracle is the plain
 *    definition: the exact sum (oracle_exact_sum), against which the
 *    tensor-core result is held to an error bound.
 *
 *  - "Taming Bitwise Behavior in GPU Kernels with Tensor Core" (arXiv
 *    2609.11356), Abstract: reduction order is the primary cause of bitwise
 *    differences (with partial-sum precision, FMA and rounding placement);
 *    a fixed balanced-tree order makes results reproducible, and an order is
 *    pinned down by a descriptor.  oracle_fixed_order_f32 is the balanced
 *    binary32 tree over index order; oracle_shuffle_tree_f32 is the declared
 *    order of the conventional (grid-stride + butterfly) reduction.
 *
 * Readings taken where the pages are silent (each one is also listed in the
 * design notes):
 *  - Leaves are the exact binary32 values of the binary16 / bfloat16 /
 *    binary32 inputs (binary32 inputs are their own leaves).
 *  - The balanced tree is over index order with power-of-two aligned
 *    subtrees; the input is padded to the next power of two with -0.0,
 *    which is the identity of IEEE round-to-nearest addition for every x
 *    (including +0 and -0), so the pad equals "an absent child passes its
 *    sibling up".
 *  - Every addition is one binary32 add, round to nearest even, no fused
 *    multiply-add, no flush of subnormals.  The file is compiled with
 *    -ffp-contract=off and without fast-math, and only additions occur.
 *  - The empty sum is +0.0.
 *
 * Parity pins (the tests under tests/ check every function here against
 * brute-force rational sums, invariants, an independent vectorised
 * emulation and hand-worked trees).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define DT_F16 0
#define DT_BF16 1
#define DT_F32 2

/* ------------------------------------------------------------------ */
/* Decoding one input (IEEE 754 binary16, bfloat16 = the upper half of
 * binary32, or binary32 itself).  A finite value is (-1)^neg * m * 2^e with
 * an integer m.  Inputs are arrays of 16-bit patterns, or of 32-bit
 * patterns for binary32; raw_at() reads pattern i of either. */

typedef struct {
    int neg;      /* sign bit */
    int special;  /* 0 finite, 1 infinity, 2 NaN */
    uint32_t m;   /* integer significand (implicit bit included if normal) */
    int e;        /* exponent of the significand's unit bit */
} decoded_t;

static uint32_t raw_at(const void *x, size_t i, int dtype)
{
    if (dtype == DT_F32) return ((const uint32_t *)x)[i];
    return ((const uint16_t *)x)[i];
}

/* The address of pattern i (the start of row i / cols, for row calls). */
static const void *raw_ptr(const void *x, size_t i, int dtype)
{
    if (dtype == DT_F32) return (const uint32_t *)x + i;
    return (const uint16_t *)x + i;
}

static decoded_t decode(uint32_t h, int dtype)
{
    decoded_t d;
    d.special = 0;
    if (dtype == DT_F32) {
        /* binary32: 8 exponent bits (bias 127), 23 fraction bits */
        uint32_t ex = (h >> 23) & 0xff, fr = h & 0x7fffff;
        d.neg = (int)(h >> 31);
        if (ex == 0xff) {
            d.special = fr ? 2 : 1; d.m = 0; d.e = 0;
        } else if (ex == 0) {            /* subnormal: fr * 2^-149 */
            d.m = fr; d.e = -149;
        } else {                         /* (2^23 + fr) * 2^(ex - 127 - 23) */
            d.m = (1u << 23) + fr; d.e = (int)ex - 150;
        }
        return d;
    }
    d.neg = (h >> 15) & 1;
    if (dtype == DT_F16) {
        /* binary16: 5 exponent bits (bias 15), 10 fraction bits */
        uint32_t ex = (h >> 10) & 0x1f, fr = h & 0x3ff;
        if (ex == 0x1f) {
            d.special = fr ? 2 : 1; d.m = 0; d.e = 0;
        } else if (ex == 0) {            /* subnormal: fr * 2^-24 */
            d.m = fr; d.e = -24;
        } else {                         /* (1024 + fr) * 2^(ex - 15 - 10) */
            d.m = 1024 + fr; d.e = (int)ex - 25;
        }
    } else {
        /* bfloat16: 8 exponent bits (bias 127), 7 fraction bits */
        uint32_t ex = (h >> 7) & 0xff, fr = h & 0x7f;
        if (ex == 0xff) {
            d.special = fr ? 2 : 1; d.m = 0; d.e = 0;
        } else if (ex == 0) {            /* subnormal: fr * 2^-133 */
            d.m = fr; d.e = -133;
        } else {                         /* (128 + fr) * 2^(ex - 127 - 7) */
            d.m = 128 + fr; d.e = (int)ex - 134;
        }
    }
    return d;
}

/* The exact binary32 value of one input (every binary16 and bfloat16 value
 * is a binary32 value, so the conversion through double is exact). */
static float leaf_f32(uint32_t h, int dtype)
{
    decoded_t d = decode(h, dtype);
    if (d.special == 2) return NAN;
    if (d.special == 1) return d.neg ? -INFINITY : INFINITY;
    double v = ldexp((double)d.m, d.e);
    float f = (float)v;
    return d.neg ? -f : f;
}

/* ------------------------------------------------------------------ */
/* Exact sums: a two's-complement fixed-point accumulator of 10 x 64 bits
 * whose bit 0 weighs 2^-298 -- the square of the smallest binary32
 * subnormal 2^-149, so that every input (a multiple of 2^-149) and every
 * square of an input (a multiple of 2^-298) is an integer multiple of it.
 * The largest square of a binary32 or bfloat16 is below 2^256, so 2^40
 * terms stay below 2^296, far inside 639 bits. */

#define ACC_LIMBS 10
#define ACC_LSB_EXP (-298)

typedef struct { uint64_t w[ACC_LIMBS]; } acc_t;

static void acc_add(acc_t *a, const acc_t *b)
{
    uint64_t carry = 0;
    for (int i = 0; i < ACC_LIMBS; i++) {
        uint64_t s = a->w[i] + carry;
        uint64_t c1 = s < carry;
        uint64_t t = s + b->w[i];
        uint64_t c2 = t < s;
        a->w[i] = t;
        carry = c1 + c2;
    }
}

static void acc_negate(acc_t *a)
{
    for (int i = 0; i < ACC_LIMBS; i++) a->w[i] = ~a->w[i];
    acc_t one;
    memset(&one, 0, sizeof one);
    one.w[0] = 1;
    acc_add(a, &one);
}

/* acc += (neg ? -1 : 1) * m * 2^pos, m < 2^128, 0 <= pos < 64 * (ACC_LIMBS - 2) */
static void acc_add_term(acc_t *a, unsigned __int128 m, int pos, int neg)
{
    acc_t t;
    memset(&t, 0, sizeof t);
    int limb = pos / 64, sh = pos % 64;
    const uint64_t lo = (uint64_t)m, hi = (uint64_t)(m >> 64);
    t.w[limb] = lo << sh;
    t.w[limb + 1] = (sh ? lo >> (64 - sh) : 0) | (hi << sh);
    if (sh != 0) t.w[limb + 2] = hi >> (64 - sh);
    if (neg) acc_negate(&t);
    acc_add(a, &t);
}

static int acc_bit(const acc_t *a, int i) { return (int)((a->w[i / 64] >> (i % 64)) & 1u); }

/* Round the exact value held in the accumulator to the nearest binary64
 * (ties to even).  The accumulator's quantum 2^-298 is far above binary64's
 * subnormal range, so only the 53-bit significand limit applies. */
static double acc_to_double(const acc_t *a)
{
    acc_t mag = *a;
    int neg = (int)((mag.w[ACC_LIMBS - 1] >> 63) & 1u);
    if (neg) acc_negate(&mag);
    int top = -1;
    for (int i = ACC_LIMBS * 64 - 1; i >= 0; i--)
        if (acc_bit(&mag, i)) { top = i; break; }
    if (top < 0) return 0.0;
    uint64_t sig = 0;
    int low = top - 52;             /* lowest kept bit position */
    if (low < 0) low = 0;
    for (int i = top; i >= low; i--) sig = (sig << 1) | (uint64_t)acc_bit(&mag, i);
    if (low > 0) {
        int round = acc_bit(&mag, low - 1), sticky = 0;
        for (int i = low - 2; i >= 0; i--)
            if (acc_bit(&mag, i)) { sticky = 1; break; }
        if (round && (sticky || (sig & 1u))) sig += 1;   /* may carry to 2^53: still exact in double */
    }
    double v = ldexp((double)sig, low + ACC_LSB_EXP);
    return neg ? -v : v;
}

/* Exact summation by exponent buckets: every finite input is +-m * 2^e with
 * an integer m < 2^24 and e >= -149, and its square is m^2 * 2^(2e) with
 * m^2 < 2^48 and 2e >= -298.  Integer sums of m (or m^2) per exponent are
 * exact in 128 bits (below 2^48 * n < 2^88 for n < 2^40), and the buckets
 * are then added into the long accumulator, m_e * 2^e each.  Bucket index =
 * exponent + 298. */
#define N_EXP 560

typedef struct {
    __int128 signed_m[N_EXP];            /* sum of +-m (or m^2) per exponent */
    unsigned __int128 abs_m[N_EXP];      /* sum of m (or m^2) per exponent */
    size_t pos_inf, neg_inf, nan;
} exact_state_t;

/* squares != 0: accumulate x^2 (always >= 0) instead of x.  Inputs
 * lo .. lo+n-1 of x. */
static void exact_accumulate(exact_state_t *st, const void *x, size_t lo, size_t n, int dtype,
                             int squares)
{
    for (size_t i = lo; i < lo + n; i++) {
        decoded_t d = decode(raw_at(x, i, dtype), dtype);
        if (d.special == 2) { st->nan++; continue; }
        if (d.special == 1) {
            if (d.neg && !squares) st->neg_inf++; else st->pos_inf++;
            continue;
        }
        if (squares) {
            int pos = 2 * d.e - ACC_LSB_EXP;
            uint64_t m2 = (uint64_t)d.m * (uint64_t)d.m;
            st->signed_m[pos] += (__int128)m2;
            st->abs_m[pos] += m2;
        } else {
            int pos = d.e - ACC_LSB_EXP;
            st->signed_m[pos] += d.neg ? -(__int128)d.m : (__int128)d.m;
            st->abs_m[pos] += d.m;
        }
    }
}

/*
 * oracle_exact_sum: the exact sum of the n inputs, rounded once to binary64
 * (round to nearest even), and the exact sum of their magnitudes, rounded
 * the same way.  Non-finite inputs follow IEEE: any NaN, or +Inf together
 * with -Inf, gives NaN; otherwise an infinity gives that infinity.
 * Threads only split the index range; integer addition is exact, so the
 * result does not depend on the thread count.
 */
static void exact_sum_any(const void *x, size_t n, int dtype, int squares, int threads,
                          double *sum_out, double *abs_out)
{
    int nt = threads > 0 ? threads : 1;
#ifndef _OPENMP
    nt = 1;
#endif
    exact_state_t *parts = (exact_state_t *)calloc((size_t)nt, sizeof(exact_state_t));
    size_t per = (n + (size_t)nt - 1) / (size_t)nt;
#pragma omp parallel for num_threads(nt) schedule(static, 1)
    for (int t = 0; t < nt; t++) {
        size_t lo = (size_t)t * per, hi = lo + per;
        if (lo > n) lo = n;
        if (hi > n) hi = n;
        exact_accumulate(&parts[t], x, lo, hi - lo, dtype, squares);
    }
    exact_state_t tot;
    memset(&tot, 0, sizeof tot);
    for (int t = 0; t < nt; t++) {
        for (int e = 0; e < N_EXP; e++) {
            tot.signed_m[e] += parts[t].signed_m[e];
            tot.abs_m[e] += parts[t].abs_m[e];
        }
        tot.pos_inf += parts[t].pos_inf;
        tot.neg_inf += parts[t].neg_inf;
        tot.nan += parts[t].nan;
    }
    free(parts);
    if (tot.nan || (tot.pos_inf && tot.neg_inf)) {
        *sum_out = NAN;
        *abs_out = tot.nan ? NAN : INFINITY;
        return;
    }
    if (tot.pos_inf || tot.neg_inf) {
        *sum_out = tot.pos_inf ? INFINITY : -INFINITY;
        *abs_out = INFINITY;
        return;
    }
    acc_t sum, abs_sum;
    memset(&sum, 0, sizeof sum);
    memset(&abs_sum, 0, sizeof abs_sum);
    for (int e = 0; e < N_EXP; e++) {
        __int128 sm = tot.signed_m[e];
        unsigned __int128 mag = sm < 0 ? (unsigned __int128)0 - (unsigned __int128)sm
                                       : (unsigned __int128)sm;
        if (mag) acc_add_term(&sum, mag, e, sm < 0);
        if (tot.abs_m[e]) acc_add_term(&abs_sum, tot.abs_m[e], e, 0);
    }
    *sum_out = acc_to_double(&sum);
    *abs_out = acc_to_double(&abs_sum);
}

void oracle_exact_sum(const void *x, size_t n, int dtype, int threads, double *sum_out,
                      double *abs_out)
{
    exact_sum_any(x, n, dtype, 0, threads, sum_out, abs_out);
}

/* The exact sum of x_i^2, rounded once to binary64 (abs_out receives the
 * same value: every term is non-negative). */
void oracle_exact_sum_squares(const void *x, size_t n, int dtype, int threads,
                              double *sum_out, double *abs_out)
{
    exact_sum_any(x, n, dtype, 1, threads, sum_out, abs_out);
}

void oracle_exact_sum_rows(const void *x, size_t rows, size_t cols, int dtype,
                           int threads, double *sum_out, double *abs_out)
{
    int nt = threads > 0 ? threads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 64)
    for (size_t r = 0; r < rows; r++)
        exact_sum_any(raw_ptr(x, r * cols, dtype), cols, dtype, 0, 1, &sum_out[r], &abs_out[r]);
}

void oracle_exact_sum_squares_rows(const void *x, size_t rows, size_t cols, int dtype,
                                   int threads, double *sum_out, double *abs_out)
{
    int nt = threads > 0 ? threads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 64)
    for (size_t r = 0; r < rows; r++)
        exact_sum_any(raw_ptr(x, r * cols, dtype), cols, dtype, 1, 1, &sum_out[r], &abs_out[r]);
}

/* ------------------------------------------------------------------ */
/* Balanced binary32 trees. */

static int ceil_log2(size_t n)
{
    int h = 0;
    while (((size_t)1 << h) < n) h++;
    return h;
}

/* The leaf of input h: its binary32 value, or for sums of squares the
 * binary32 product of that value with itself (one rounding to nearest even;
 * the product of two binary32 values -- 24-bit significands, exponents
 * within binary64's normal range -- is exact in binary64). */
static float leaf_op(uint32_t h, int dtype, int squares)
{
    float f = leaf_f32(h, dtype);
    if (!squares) return f;
    return (float)((double)f * (double)f);
}

/* Node of height h whose leftmost leaf is input lo: the sum of its two
 * children, left + right, in binary32.  Leaves past n are the -0.0 pad.
 * A subtree that lies wholly in the pad has the value -0.0 (every leaf is
 * -0.0 and -0.0 + -0.0 = -0.0), so it is returned without descending. */
static float tree_node_in(const void *x, size_t n, int dtype, int squares, size_t lo, int h)
{
    if (lo >= n) return -0.0f;
    if (h == 0) return leaf_op(raw_at(x, lo, dtype), dtype, squares);
    size_t half = (size_t)1 << (h - 1);
    float left = tree_node_in(x, n, dtype, squares, lo, h - 1);
    float right = tree_node_in(x, n, dtype, squares, lo + half, h - 1);
    return left + right;
}

/* Same tree over binary32 values a[0..m), padded with -0.0. */
static float tree_node32(const float *a, size_t m, size_t lo, int h)
{
    if (lo >= m) return -0.0f;
    if (h == 0) return a[lo];
    size_t half = (size_t)1 << (h - 1);
    float left = tree_node32(a, m, lo, h - 1);
    float right = tree_node32(a, m, lo + half, h - 1);
    return left + right;
}

static float tree_f32(const float *a, size_t m)
{
    if (m == 0) return -0.0f;
    return tree_node32(a, m, 0, ceil_log2(m));
}

/*
 * oracle_fixed_order_f32: the balanced binary32 tree over the n inputs in
 * index order.  Threads evaluate disjoint subtrees of the same tree; the
 * top levels are then formed from those subtree values in the same shape,
 * so the result is that of the single recursive definition.
 */
static float fixed_order_any(const void *x, size_t n, int dtype, int squares, int threads)
{
    if (n == 0) return 0.0f;
    int H = ceil_log2(n);
    int k = H < 10 ? H : 10;                 /* 2^k subtrees of height H - k */
    size_t parts = (size_t)1 << k;
    float *node = (float *)malloc(parts * sizeof(float));
    int nt = threads > 0 ? threads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (size_t i = 0; i < parts; i++)
        node[i] = tree_node_in(x, n, dtype, squares, i << (H - k), H - k);
    float r = tree_node32(node, parts, 0, k);
    free(node);
    return r;
}

float oracle_fixed_order_f32(const void *x, size_t n, int dtype, int threads)
{
    return fixed_order_any(x, n, dtype, 0, threads);
}

/* The same tree over the leaves x_i^2 (sum of squares). */
float oracle_fixed_order_sq_f32(const void *x, size_t n, int dtype, int threads)
{
    return fixed_order_any(x, n, dtype, 1, threads);
}

void oracle_fixed_order_rows_f32(const void *x, size_t rows, size_t cols, int dtype,
                                 int squares, int threads, float *out)
{
    int nt = threads > 0 ? threads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 64)
    for (size_t r = 0; r < rows; r++)
        out[r] = fixed_order_any(raw_ptr(x, r * cols, dtype), cols, dtype, squares, 1);
}

/* ------------------------------------------------------------------ */
/* Blocked-sequential-then-tree order ("Taming Bitwise Behavior in GPU
 * Kernels with Tensor Core", Abstract: an order is pinned by a descriptor;
 * this is a second declared order for the fixed-order mode, with a run
 * length chosen by the caller).
 *
 * The segment of n inputs is cut into runs of C = 2^run_log2 consecutive
 * inputs (the last one shorter).  A run's value is its leaves added left to
 * right in binary32, starting from -0.0 (so a run of one input is that
 * input).  The result is the balanced binary32 tree over the run values in
 * run order, padded with -0.0 -- for C = 1 the plain fixed-order tree, for
 * C >= n the plain left-to-right sum. */

static float run_value(const void *x, size_t n, int dtype, size_t lo, size_t C)
{
    float s = -0.0f;
    size_t hi = lo + C < n ? lo + C : n;
    for (size_t i = lo; i < hi; i++) s = s + leaf_f32(raw_at(x, i, dtype), dtype);
    return s;
}

static float blocked_order_any(const void *x, size_t n, int dtype, int run_log2, int threads)
{
    if (n == 0) return 0.0f;
    if (run_log2 < 0 || run_log2 > 40) return NAN;
    const size_t C = (size_t)1 << run_log2;
    const size_t m = (n + C - 1) / C;       /* runs */
    float *runs = (float *)malloc(m * sizeof(float));
    int nt = threads > 0 ? threads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 64)
    for (size_t r = 0; r < m; r++) runs[r] = run_value(x, n, dtype, r * C, C);
    float v = tree_f32(runs, m);
    free(runs);
    return v;
}

float oracle_blocked_order_f32(const void *x, size_t n, int dtype, int run_log2, int threads)
{
    return blocked_order_any(x, n, dtype, run_log2, threads);
}

void oracle_blocked_order_rows_f32(const void *x, size_t rows, size_t cols, int dtype,
                                   int run_log2, int threads, float *out)
{
    int nt = threads > 0 ? threads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 16)
    for (size_t r = 0; r < rows; r++)
        out[r] = blocked_order_any(raw_ptr(x, r * cols, dtype), cols, dtype, run_log2, 1);
}

/* ------------------------------------------------------------------ */
/* Declared order of the conventional reduction (SHUFFLE_TREE).
 *
 * A segment of L inputs is split into vectors of V consecutive inputs, the
 * inputs of 16 bytes: V = 8 for binary16 and bfloat16, V = 4 for binary32
 * (v = inputs V*v .. V*v+V-1, the last one padded with -0.0).  It is
 * reduced by a team of G blocks of Bt threads (T = G*Bt threads, thread
 * g = b*Bt + t):
 *   1. vector value   = balanced tree over its V leaves;
 *   2. thread value   = acc, acc starts at -0.0 and for v = g, g+T, g+2T, ...
 *                       acc = acc + vector value (in that order);
 *   3. warp value     = butterfly over the 32 lanes of the warp: for the
 *                       offsets 16, 8, 4, 2, 1 in turn, every lane i replaces
 *                       its value by value[i] + value[i xor offset];
 *                       the warp value is what lane 0 holds at the end;
 *   4. block value    = balanced tree over the block's Bt/32 warp values,
 *                       in warp-index order;
 *   5. segment value  = balanced tree over the G block values in block
 *                       order, padded with -0.0.
 */
static size_t vector_len(int dtype) { return dtype == DT_F32 ? 4 : 8; }

static float vector_tree(const void *x, size_t L, int dtype, int squares, size_t v)
{
    const size_t V = vector_len(dtype);
    float e[8];
    for (size_t k = 0; k < V; k++) {
        size_t i = V * v + k;
        e[k] = i < L ? leaf_op(raw_at(x, i, dtype), dtype, squares) : -0.0f;
    }
    if (V == 4) return (e[0] + e[1]) + (e[2] + e[3]);
    return ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
}

static float shuffle_block_value(const void *x, size_t L, int dtype, int squares, int Bt, int G,
                                 int b)
{
    size_t T = (size_t)G * (size_t)Bt;
    size_t V = vector_len(dtype);
    size_t nvec = (L + V - 1) / V;
    int W = Bt / 32;
    float warp_value[32];
    for (int w = 0; w < W; w++) {
        float lane[32], next[32];
        for (int j = 0; j < 32; j++) {
            size_t g = (size_t)b * (size_t)Bt + (size_t)w * 32 + (size_t)j;
            float acc = -0.0f;
            for (size_t v = g; v < nvec; v += T) acc = acc + vector_tree(x, L, dtype, squares, v);
            lane[j] = acc;
        }
        for (int off = 16; off >= 1; off /= 2) {
            for (int j = 0; j < 32; j++) next[j] = lane[j] + lane[j ^ off];
            memcpy(lane, next, sizeof lane);
        }
        warp_value[w] = lane[0];
    }
    return tree_f32(warp_value, (size_t)W);
}

static float shuffle_tree_any(const void *x, size_t L, int dtype, int squares, int Bt, int G,
                              int threads)
{
    if (L == 0) return 0.0f;
    if (Bt < 32 || Bt > 1024 || (Bt & (Bt - 1)) != 0 || G < 1) return NAN;
    float *block = (float *)malloc((size_t)G * sizeof(float));
    int nt = threads > 0 ? threads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (int b = 0; b < G; b++) block[b] = shuffle_block_value(x, L, dtype, squares, Bt, G, b);
    float r = tree_f32(block, (size_t)G);
    free(block);
    return r;
}

float oracle_shuffle_tree_f32(const void *x, size_t L, int dtype, int Bt, int G, int threads)
{
    return shuffle_tree_any(x, L, dtype, 0, Bt, G, threads);
}

/* The same declared order over the leaves x_i^2 (sum of squares). */
float oracle_shuffle_tree_sq_f32(const void *x, size_t L, int dtype, int Bt, int G,
                                 int threads)
{
    return shuffle_tree_any(x, L, dtype, 1, Bt, G, threads);
}

void oracle_shuffle_tree_rows_f32(const void *x, size_t rows, size_t cols, int dtype,
                                  int squares, int Bt, int G, int threads, float *out)
{
    int nt = threads > 0 ? threads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 64)
    for (size_t r = 0; r < rows; r++)
        out[r] = shuffle_tree_any(raw_ptr(x, r * cols, dtype), cols, dtype, squares, Bt, G, 1);
}

/* ------------------------------------------------------------------ */
/* Mean and variance of rows from their sum S1 and sum of squares S2 (the
 * cascaded reductions named by the "RedFuser" title in the first page's list
 * of work built on the method: two reductions of one row in one pass).  The
 * formula, in binary32 with one rounding to nearest per operation:
 *   m = S1 / n,  q = S2 / n,  v = q - m * m,  var = v < 0 ? +0 : v
 * (n = cols as a binary32; a negative v can only come from rounding). */
void oracle_mean_var_f32(const float *s1, const float *s2, size_t rows, size_t cols, float *mean,
                         float *var)
{
    const float n = (float)cols;
    for (size_t r = 0; r < rows; r++) {
        const float m = s1[r] / n;
        const float q = s2[r] / n;
        const float mm = m * m;
        const float v = q - mm;
        mean[r] = m;
        var[r] = v < 0.0f ? 0.0f : v;
    }
}

/* ------------------------------------------------------------------ */
/* Split-K GEMM ("Taming Bitwise Behavior in GPU Kernels with Tensor Core",
 * Abstract: the descriptor of reduction order covers GEMM, including the
 * split-K partitioning of K).  C = A * W^T with A (M x K) and W (N x K)
 * row-major 16-bit inputs.
 *
 * oracle_gemm_f64: every element as a binary64 sum of the exact products
 * a_ik * w_jk (each exact in binary64) in k order, and the same sum of
 * |a_ik * w_jk| -- the reference for the error bound.
 *
 * oracle_gemm_splitk_f32: the declared order with each split's partial
 * taken exactly (as far as binary64 holds it) and rounded once to
 * binary32: P_s = fl32(sum over k in [s * k_split, (s + 1) * k_split)),
 * C = the balanced binary32 tree over P_0 .. P_{S-1} (-0.0 pad).  Where
 * every partial is exact in binary32 and the tensor core adds it without
 * rounding (small integers, one scale per split), this is the GPU's result
 * bit for bit; elsewhere the two differ by the tensor core's rounding. */

void oracle_gemm_f64(const void *A, const void *W, size_t M, size_t N, size_t K, int dtype,
                     int threads, double *out, double *abs_out)
{
    int nt = threads > 0 ? threads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (size_t i = 0; i < M; i++) {
        for (size_t j = 0; j < N; j++) {
            double acc = 0.0, aacc = 0.0;
            for (size_t k = 0; k < K; k++) {
                const double p = (double)leaf_f32(raw_at(A, i * K + k, dtype), dtype) *
                                 (double)leaf_f32(raw_at(W, j * K + k, dtype), dtype);
                acc += p;
                aacc += fabs(p);
            }
            out[i * N + j] = acc;
            abs_out[i * N + j] = aacc;
        }
    }
}

void oracle_gemm_splitk_f32(const void *A, const void *W, size_t M, size_t N, size_t K, int dtype,
                            int splits, size_t k_split, int threads, float *out)
{
    int nt = threads > 0 ? threads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (size_t i = 0; i < M; i++) {
        float *part = (float *)malloc((size_t)(splits > 0 ? splits : 1) * sizeof(float));
        for (size_t j = 0; j < N; j++) {
            for (int s = 0; s < splits; s++) {
                const size_t k0 = (size_t)s * k_split;
                const size_t k1 = k0 + k_split < K ? k0 + k_split : K;
                double acc = 0.0;
                for (size_t k = k0; k < k1; k++)
                    acc += (double)leaf_f32(raw_at(A, i * K + k, dtype), dtype) *
                           (double)leaf_f32(raw_at(W, j * K + k, dtype), dtype);
                part[s] = (float)acc;
            }
            out[i * N + j] = tree_f32(part, (size_t)splits);
        }
        free(part);
    }
}

/* Exact binary32 value of each input (used by the tests to compare the
 * decoder with independent conversions). */
void oracle_leaves_f32(const void *x, size_t n, int dtype, float *out)
{
    for (size_t i = 0; i < n; i++) out[i] = leaf_f32(raw_at(x, i, dtype), dtype);
}
