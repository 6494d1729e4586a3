"""Pins for the CPU oracle, checked against things other than itself.

Each test ties an oracle function to brute force, an invariant of the
mathematics, an independent implementation written differently, or a value
worked out by hand (``tests/golden``).  A plausible slip in the oracle -- a
dropped term, a wrong index or shift, a wrong rounding rule, a transposed
tree -- fails at least one of them.
"""
from fractions import Fraction
import math
import os

import numpy as np
import pytest

import oracle
from arithmetic_reduction_tensor_gb300 import synth

F16, BF16, F32 = oracle.F16, oracle.BF16, oracle.F32


# ---------------------------------------------------------------- helpers

def np_leaves(bits, dtype):
    """binary32 values decoded by numpy (independent of the oracle's decoder)."""
    if dtype == F32:
        return np.asarray(bits, np.uint32).view(np.float32)
    bits = np.asarray(bits, np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def frac_sum(bits, dtype):
    """Exact rational sum and sum of magnitudes of finite inputs."""
    vals = np_leaves(bits, dtype).astype(np.float64)
    s = sum((Fraction(float(v)) for v in vals), Fraction(0))
    a = sum((Fraction(abs(float(v))) for v in vals), Fraction(0))
    return s, a


@np.errstate(over="ignore", invalid="ignore")
def np_tree(values_f32):
    """Balanced binary32 tree, level by level with numpy, -0.0 pad."""
    v = np.asarray(values_f32, np.float32)
    n = v.size
    if n == 0:
        return np.float32(0.0)
    size = 1
    while size < n:
        size *= 2
    a = np.full(size, -0.0, np.float32)
    a[:n] = v
    while a.size > 1:
        a = a[0::2] + a[1::2]
    return a[0]


@np.errstate(over="ignore", invalid="ignore")
def np_shuffle(bits, dtype, bt, g, leaf_values=None):
    """Vectorised emulation of the declared SHUFFLE_TREE order (vectors of
    16 bytes: 8 inputs of 16 bits, 4 of binary32)."""
    v = np_leaves(bits, dtype) if leaf_values is None else leaf_values
    L = v.size
    if L == 0:
        return np.float32(0.0)
    V = 4 if dtype == F32 else 8
    nvec = (L + V - 1) // V
    e = np.full(nvec * V, -0.0, np.float32)
    e[:L] = v
    e = e.reshape(nvec, V)
    while e.shape[1] > 1:
        e = e[:, 0::2] + e[:, 1::2]
    vec = e[:, 0]
    T = bt * g
    acc = np.full(T, -0.0, np.float32)
    for start in range(0, nvec, T):
        m = min(T, nvec - start)
        acc[:m] = acc[:m] + vec[start:start + m]
    lanes = acc.reshape(-1, 32)
    idx = np.arange(32)
    for off in (16, 8, 4, 2, 1):
        lanes = lanes + lanes[:, idx ^ off]
    warp = lanes[:, 0].reshape(g, bt // 32)
    while warp.shape[1] > 1:
        warp = warp[:, 0::2] + warp[:, 1::2]
    return np_tree(warp[:, 0])


def same_f32(a, b):
    a, b = np.float32(a), np.float32(b)
    if np.isnan(a) or np.isnan(b):
        return bool(np.isnan(a) and np.isnan(b))
    return a.tobytes() == b.tobytes()


def special_patterns(dtype):
    """Bit patterns at the edges of each format: zeros, subnormals, extremes."""
    if dtype == F32:
        return [0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x007FFFFF, 0x807FFFFF,
                0x00800000, 0x80800000, 0x3F800000, 0xBF800000, 0x7F7FFFFF, 0xFF7FFFFF,
                0x3F7FFFFF, 0x3F800001]
    if dtype == F16:
        return [0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x83FF, 0x0400, 0x8400,
                0x3C00, 0xBC00, 0x7BFF, 0xFBFF, 0x3BFF, 0x3C01]
    return [0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x807F, 0x0080, 0x8080,
            0x3F80, 0xBF80, 0x7F7F, 0xFF7F, 0x3F7F, 0x3F81]


def random_finite(rng, n, dtype):
    """Random finite bit patterns (any exponent, both signs, subnormals)."""
    if dtype == F32:
        b = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
        bad = (b & np.uint32(0x7F800000)) == np.uint32(0x7F800000)
        b[bad] &= np.uint32(0xBFFFFFFF)
        return b
    b = rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16)
    exp_mask = 0x7C00 if dtype == F16 else 0x7F80
    bad = (b & exp_mask) == exp_mask
    b[bad] &= np.uint16(0xBFFF)      # clear the top exponent bit: finite again
    return b


# ---------------------------------------------------------------- decoder

@pytest.mark.parametrize("dtype", [F16, BF16])
def test_leaves_match_numpy_for_every_pattern(dtype):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.leaves(bits, dtype)
    ref = np_leaves(bits, dtype)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ---------------------------------------------------------------- exact sum

@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("seed", range(6))
def test_exact_sum_brute_force(dtype, seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 65))
    bits = np.concatenate([random_finite(rng, n, dtype),
                           np.array(special_patterns(dtype), np.uint16)])
    rng.shuffle(bits)
    s, a = oracle.exact_sum(bits, dtype, threads=3)
    fs, fa = frac_sum(bits, dtype)
    assert s == float(fs)      # float(Fraction) rounds to nearest even
    assert a == float(fa)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_exact_sum_permutation_invariant(dtype):
    bits = synth.generate(200_003, "normal", dtype, seed=11)
    rng = np.random.default_rng(5)
    perm = bits[rng.permutation(bits.size)]
    assert oracle.exact_sum(bits, dtype) == oracle.exact_sum(perm, dtype, threads=7)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_exact_sum_all_ones_is_n(dtype):
    one = 0x3C00 if dtype == F16 else 0x3F80
    n = 3_000_017
    s, a = oracle.exact_sum(np.full(n, one, np.uint16), dtype)
    assert s == float(n) and a == float(n)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_exact_sum_x_and_minus_x_cancel(dtype):
    bits = synth.generate(500_000, "uniform_pm1", dtype, seed=12)
    both = np.concatenate([bits, bits ^ np.uint16(0x8000)])
    s, a = oracle.exact_sum(both, dtype)
    s1, a1 = oracle.exact_sum(bits, dtype)
    assert s == 0.0
    assert a == 2 * a1


def test_exact_sum_rounding_needs_sticky_and_ties_to_even():
    # bfloat16 can hold 2^-52, 2^-53 and 2^-133 exactly.
    def bf(x):
        return int(np.float32(x).view(np.uint32) >> 16)
    tie_to_even_down = np.array([bf(1.0), bf(2.0 ** -53)], np.uint16)
    assert oracle.exact_sum(tie_to_even_down, BF16)[0] == 1.0
    tie_to_even_up = np.array([bf(1.0), bf(2.0 ** -52), bf(2.0 ** -53)], np.uint16)
    assert oracle.exact_sum(tie_to_even_up, BF16)[0] == 1.0 + 2.0 ** -51
    sticky = np.array([bf(1.0), bf(2.0 ** -53), 0x0001], np.uint16)   # + 2^-133
    assert oracle.exact_sum(sticky, BF16)[0] == 1.0 + 2.0 ** -52


def test_exact_sum_extremes():
    big = np.full(1 << 20, 0x7F7F, np.uint16)          # largest bfloat16
    s, _ = oracle.exact_sum(big, BF16)
    assert s == float(Fraction(float(np_leaves([0x7F7F], BF16)[0])) * (1 << 20))
    f16max = np.full(1 << 20, 0x7BFF, np.uint16)       # 65504
    assert oracle.exact_sum(f16max, F16)[0] == 65504.0 * (1 << 20)
    tiny = np.full(1000, 0x0001, np.uint16)             # 2^-24 each
    assert oracle.exact_sum(tiny, F16)[0] == 1000 * 2.0 ** -24


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_exact_sum_non_finite(dtype):
    inf = 0x7C00 if dtype == F16 else 0x7F80
    nan = 0x7E00 if dtype == F16 else 0x7FC0
    one = 0x3C00 if dtype == F16 else 0x3F80
    assert oracle.exact_sum(np.array([one, inf], np.uint16), dtype)[0] == math.inf
    assert oracle.exact_sum(np.array([one, inf | 0x8000], np.uint16), dtype)[0] == -math.inf
    assert math.isnan(oracle.exact_sum(np.array([inf, inf | 0x8000], np.uint16), dtype)[0])
    assert math.isnan(oracle.exact_sum(np.array([one, nan], np.uint16), dtype)[0])


def test_exact_sum_rows_match_whole_rows():
    x = synth.generate(37 * 301, "normal", F16, seed=13).reshape(37, 301)
    s, a = oracle.exact_sum_rows(x, F16)
    for r in range(37):
        assert (s[r], a[r]) == oracle.exact_sum(x[r], F16, threads=1)


def test_exact_sum_empty():
    assert oracle.exact_sum(np.zeros(0, np.uint16), F16) == (0.0, 0.0)


# ---------------------------------------------------------------- fixed order

def _read_tree16(golden_dir):
    vals = {}
    with open(os.path.join(golden_dir, "fixed_order_tree16.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(None, 1)
            vals[key] = rest
    bits = np.array([int(b, 16) for b in vals["bits"].split()], np.uint16)
    return bits, vals


def test_fixed_order_hand_worked_tree(golden_dir):
    bits, vals = _read_tree16(golden_dir)
    got = oracle.fixed_order(bits, F16, threads=1)
    assert got == np.float32(float(Fraction(vals["fixed_order"])))
    # the same inputs in other orders give the other two printed values
    seq = np.float32(0.0)
    for v in np_leaves(bits, F16):
        seq = np.float32(seq + v)
    assert seq == np.float32(float(Fraction(vals["sequential"])))
    exact = Fraction(oracle.exact_sum(bits, F16)[0])
    assert np.float32(float(exact)) == np.float32(float(Fraction(vals["exact_f32"])))
    assert got != seq and got != np.float32(float(exact))


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("n", [1, 2, 3, 7, 8, 9, 15, 16, 17, 255, 256, 257, 1000, 4095, 4097,
                               65536, 65537, 100_003])
def test_fixed_order_matches_levelwise_numpy(dtype, n):
    rng = np.random.default_rng(n)
    bits = random_finite(rng, n, dtype) if n < 5000 else synth.generate(n, "normal", dtype, seed=n)
    got = oracle.fixed_order(bits, dtype, threads=4)
    ref = np_tree(np_leaves(bits, dtype))
    assert same_f32(got, ref)


def test_fixed_order_thread_count_does_not_change_result():
    bits = synth.generate(1_000_003, "uniform_pm1", F16, seed=14)
    r = [oracle.fixed_order(bits, F16, threads=t) for t in (1, 2, 5, 8)]
    assert all(x.tobytes() == r[0].tobytes() for x in r)


def test_fixed_order_negative_zero_pad_is_identity():
    bits = synth.generate(1000, "uniform_pm1", F16, seed=15)
    padded = np.concatenate([bits, np.full(24, 0x8000, np.uint16)])   # 1024 = next power of two
    assert same_f32(oracle.fixed_order(bits, F16), oracle.fixed_order(padded, F16))


def test_fixed_order_integer_inputs_are_exact():
    # small integers: every partial sum is an integer below 2^24, so every
    # order gives the exact sum
    rng = np.random.default_rng(16)
    v = rng.integers(-64, 65, 300_001).astype(np.float16)
    bits = v.view(np.uint16)
    assert float(oracle.fixed_order(bits, F16)) == oracle.exact_sum(bits, F16)[0]


def test_fixed_order_degenerate_cases():
    assert oracle.fixed_order(np.zeros(0, np.uint16), F16).tobytes() == np.float32(0.0).tobytes()
    assert oracle.fixed_order(np.array([0x3555], np.uint16), F16) == np.float16(0.333251953125)
    negz = oracle.fixed_order(np.full(5, 0x8000, np.uint16), F16)
    assert negz.tobytes() == np.float32(-0.0).tobytes()
    assert np.isnan(oracle.fixed_order(np.array([0x3C00, 0x7E00, 0x3C00], np.uint16), F16))


def test_fixed_order_rows_match_whole_rows():
    x = synth.generate(29 * 1031, "uniform_pm1", BF16, seed=17).reshape(29, 1031)
    got = oracle.fixed_order_rows(x, BF16)
    for r in range(29):
        assert same_f32(got[r], oracle.fixed_order(x[r], BF16, threads=1))


# ---------------------------------------------------------------- shuffle tree

def _read_shuffle_cases(golden_dir):
    cases = []
    with open(os.path.join(golden_dir, "shuffle_tree_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, bt, g, L, items, result = [p.strip() for p in line.split("|")]
            bits = np.zeros(int(L), np.uint16)
            for it in items.split(","):
                i, b = it.split("=")
                bits[int(i)] = int(b, 16)
            cases.append((name, int(bt), int(g), bits, Fraction(result)))
    return cases


def test_shuffle_tree_hand_worked_cases(golden_dir):
    cases = _read_shuffle_cases(golden_dir)
    assert len(cases) == 4
    for name, bt, g, bits, expect in cases:
        got = oracle.shuffle_tree(bits, F16, bt, g, threads=1)
        assert got == np.float32(float(expect)), name


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("L,bt,g", [(1, 32, 1), (8, 32, 1), (9, 32, 1), (255, 32, 1), (256, 32, 1),
                                    (1000, 32, 1), (4097, 32, 1), (8192, 32, 1), (10_000, 64, 1),
                                    (10_000, 128, 3), (33_333, 256, 2), (65_536, 1024, 1),
                                    (70_001, 32, 7), (100_000, 512, 5)])
def test_shuffle_tree_matches_vectorised_emulation(dtype, L, bt, g):
    rng = np.random.default_rng(L + bt + g)
    bits = random_finite(rng, L, dtype) if L < 5000 else synth.generate(L, "normal", dtype, seed=L)
    got = oracle.shuffle_tree(bits, dtype, bt, g, threads=3)
    assert same_f32(got, np_shuffle(bits, dtype, bt, g))


@pytest.mark.parametrize("bt,g", [(32, 1), (64, 2), (256, 5), (1024, 3)])
def test_shuffle_tree_integer_inputs_are_exact(bt, g):
    rng = np.random.default_rng(bt * g)
    bits = rng.integers(-64, 65, 123_457).astype(np.float16).view(np.uint16)
    assert float(oracle.shuffle_tree(bits, F16, bt, g)) == oracle.exact_sum(bits, F16)[0]


def test_shuffle_tree_single_vector_is_the_eight_leaf_tree():
    # with at most one vector, only lane 0 holds data: the result is the
    # 8-leaf balanced tree, i.e. the fixed-order tree of those inputs
    rng = np.random.default_rng(18)
    for L in range(1, 9):
        bits = random_finite(rng, L, F16)
        assert same_f32(oracle.shuffle_tree(bits, F16, 32, 1), oracle.fixed_order(bits, F16))


def test_shuffle_tree_rows_match_whole_rows():
    x = synth.generate(23 * 9001, "normal", F16, seed=19).reshape(23, 9001)
    got = oracle.shuffle_tree_rows(x, F16, 64, 2)
    for r in range(23):
        assert same_f32(got[r], oracle.shuffle_tree(x[r], F16, 64, 2, threads=1))


def test_shuffle_tree_empty_is_positive_zero():
    assert oracle.shuffle_tree(np.zeros(0, np.uint16), F16, 32, 1).tobytes() == \
        np.float32(0.0).tobytes()


# ---------------------------------------------------------------- sum of squares

def np_square_leaves(bits, dtype):
    """binary32 squares by numpy (one rounding of the exact product)."""
    v = np_leaves(bits, dtype).astype(np.float32)
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        return v * v


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("seed", range(6))
def test_exact_sum_squares_brute_force(dtype, seed):
    rng = np.random.default_rng(200 + seed)
    n = int(rng.integers(1, 65))
    bits = np.concatenate([random_finite(rng, n, dtype),
                           np.array(special_patterns(dtype), np.uint16)])
    s, a = oracle.exact_sum_squares(bits, dtype, threads=3)
    vals = np_leaves(bits, dtype).astype(np.float64)
    exact = sum((Fraction(float(v)) ** 2 for v in vals), Fraction(0))
    assert s == float(exact) and a == s


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_exact_sum_squares_invariants(dtype):
    bits = synth.generate(300_001, "normal", dtype, seed=31)
    s1, _ = oracle.exact_sum_squares(bits, dtype)
    s2, _ = oracle.exact_sum_squares(bits ^ np.uint16(0x8000), dtype)    # x -> -x
    assert s1 == s2 > 0
    three = int(np.float16(3.0).view(np.uint16)) if dtype == F16 else 0x4040
    assert oracle.exact_sum_squares(np.full(1_000_003, three, np.uint16), dtype)[0] == 9.0 * 1_000_003
    # the extremes of the formats: bfloat16 squares reach 2^-266 and 2^255
    if dtype == BF16:
        tiny = np.full(7, 0x0001, np.uint16)
        assert oracle.exact_sum_squares(tiny, BF16)[0] == 7 * 2.0 ** -266
        big = np.array([0x7F7F], np.uint16)
        b = float(np_leaves(big, BF16)[0])
        assert oracle.exact_sum_squares(big, BF16)[0] == float(Fraction(b) ** 2)
    inf = 0x7C00 if dtype == F16 else 0x7F80
    assert oracle.exact_sum_squares(np.array([inf | 0x8000, inf], np.uint16), dtype)[0] == math.inf


def test_fixed_order_sq_hand_worked_tree(golden_dir):
    # squares of [2^-12 x8, 1.0, 2^-12 x7] are the leaves of the hand-worked
    # 16-leaf tree: 2^-24 x8, 1.0, 2^-24 x7 -> 1 + 7 * 2^-23
    _, vals = _read_tree16(golden_dir)
    bits = np.array([0x0C00] * 8 + [0x3C00] + [0x0C00] * 7, np.uint16)
    assert oracle.fixed_order_sq(bits, F16, threads=1) == np.float32(float(Fraction(vals["fixed_order"])))


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 255, 256, 1000, 4097, 65537, 100_003])
def test_fixed_order_sq_matches_levelwise_numpy(dtype, n):
    rng = np.random.default_rng(n + 7)
    bits = random_finite(rng, n, dtype) if n < 5000 else synth.generate(n, "normal", dtype, seed=n)
    got = oracle.fixed_order_sq(bits, dtype, threads=4)
    assert same_f32(got, np_tree(np_square_leaves(bits, dtype)))


def np_shuffle_sq(bits, dtype, bt, g):
    """Vectorised emulation of the declared order over squared leaves."""
    return np_shuffle(bits, dtype, bt, g, leaf_values=np_square_leaves(bits, dtype))


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("L,bt,g", [(9, 32, 1), (1000, 32, 1), (8192, 32, 1), (10_000, 128, 3),
                                    (70_001, 32, 7), (100_000, 512, 5)])
def test_shuffle_tree_sq_matches_vectorised_emulation(dtype, L, bt, g):
    rng = np.random.default_rng(L + 11)
    bits = random_finite(rng, L, dtype) if L < 5000 else synth.generate(L, "normal", dtype, seed=L)
    assert same_f32(oracle.shuffle_tree_sq(bits, dtype, bt, g, threads=3),
                    np_shuffle_sq(bits, dtype, bt, g))


def test_sum_squares_rows_match_whole_rows():
    x = synth.generate(19 * 9001, "normal", F16, seed=33).reshape(19, 9001)
    s, _ = oracle.exact_sum_rows(x, F16, squares=True)
    f = oracle.fixed_order_rows(x, F16, squares=True)
    t = oracle.shuffle_tree_rows(x, F16, 128, 2, squares=True)
    for r in range(19):
        assert s[r] == oracle.exact_sum_squares(x[r], F16, threads=1)[0]
        assert same_f32(f[r], oracle.fixed_order_sq(x[r], F16, threads=1))
        assert same_f32(t[r], oracle.shuffle_tree_sq(x[r], F16, 128, 2, threads=1))


# ---------------------------------------------------------------- binary32 inputs

def test_leaves_f32_are_the_patterns_themselves():
    rng = np.random.default_rng(40)
    bits = np.concatenate([random_finite(rng, 200_000, F32),
                           np.array(special_patterns(F32), np.uint32),
                           np.array([0x7F800000, 0xFF800000, 0x7FC00000, 0xFF812345], np.uint32)])
    got = oracle.leaves(bits, F32)
    nan = np.isnan(bits.view(np.float32))
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got.view(np.uint32)[~nan], bits[~nan])


@pytest.mark.parametrize("seed", range(8))
def test_exact_sum_f32_brute_force(seed):
    rng = np.random.default_rng(300 + seed)
    n = int(rng.integers(1, 65))
    bits = np.concatenate([random_finite(rng, n, F32), np.array(special_patterns(F32), np.uint32)])
    rng.shuffle(bits)
    s, a = oracle.exact_sum(bits, F32, threads=3)
    fs, fa = frac_sum(bits, F32)
    assert s == float(fs) and a == float(fa)
    s2, _ = oracle.exact_sum_squares(bits, F32, threads=2)
    exact = sum((Fraction(float(v)) ** 2 for v in np_leaves(bits, F32).astype(np.float64)),
                Fraction(0))
    assert s2 == float(exact)


def test_exact_sum_f32_rounding_and_extremes():
    def f(x):
        return int(np.float32(x).view(np.uint32))
    # ties to even and sticky, with the smallest binary32 subnormal 2^-149
    assert oracle.exact_sum(np.array([f(1.0), f(2.0 ** -53)], np.uint32), F32)[0] == 1.0
    sticky = np.array([f(1.0), f(2.0 ** -53), 0x00000001], np.uint32)
    assert oracle.exact_sum(sticky, F32)[0] == 1.0 + 2.0 ** -52
    # 2^20 copies of the largest binary32: the per-exponent integer sum and,
    # for the squares, m^2 sums beyond 2^64 must stay exact
    big = np.full(1 << 20, 0x7F7FFFFF, np.uint32)
    fmax = Fraction(float(np.float32(np.finfo(np.float32).max)))
    assert oracle.exact_sum(big, F32)[0] == float(fmax * (1 << 20))
    assert oracle.exact_sum_squares(big, F32)[0] == float(fmax ** 2 * (1 << 20))
    m = np.full(3_000_001, 0x3F7FFFFF, np.uint32)    # 1 - 2^-24: m^2 near 2^48
    one_less = Fraction(float(np.float32(1.0) - np.float32(2.0 ** -24)))
    assert oracle.exact_sum_squares(m, F32)[0] == float(one_less ** 2 * 3_000_001)
    tiny = np.full(7, 0x00000001, np.uint32)          # squares 2^-298 each
    assert oracle.exact_sum_squares(tiny, F32)[0] == 7 * 2.0 ** -298
    both = np.concatenate([big, big ^ np.uint32(0x80000000)])
    assert oracle.exact_sum(both, F32)[0] == 0.0


def test_exact_sum_f32_non_finite():
    one, inf, nan = 0x3F800000, 0x7F800000, 0x7FC00000
    assert oracle.exact_sum(np.array([one, inf], np.uint32), F32)[0] == math.inf
    assert oracle.exact_sum(np.array([one, inf | 0x80000000], np.uint32), F32)[0] == -math.inf
    assert math.isnan(oracle.exact_sum(np.array([inf, inf | 0x80000000], np.uint32), F32)[0])
    assert math.isnan(oracle.exact_sum(np.array([one, nan], np.uint32), F32)[0])
    assert oracle.exact_sum_squares(np.array([inf | 0x80000000], np.uint32), F32)[0] == math.inf


@pytest.mark.parametrize("n", [1, 3, 4, 5, 8, 1000, 4097, 65537, 100_003])
def test_fixed_order_f32_matches_levelwise_numpy(n):
    rng = np.random.default_rng(n + 41)
    bits = random_finite(rng, n, F32) if n < 5000 else synth.generate(n, "normal", F32, seed=n)
    assert same_f32(oracle.fixed_order(bits, F32, threads=4), np_tree(np_leaves(bits, F32)))
    assert same_f32(oracle.fixed_order_sq(bits, F32, threads=3),
                    np_tree(np_square_leaves(bits, F32)))


@pytest.mark.parametrize("L,bt,g", [(1, 32, 1), (4, 32, 1), (5, 32, 1), (128, 32, 1), (129, 32, 1),
                                    (4096, 32, 1), (4097, 32, 1), (10_000, 64, 1),
                                    (10_000, 128, 3), (70_001, 32, 7), (100_000, 512, 5)])
def test_shuffle_tree_f32_matches_vectorised_emulation(L, bt, g):
    rng = np.random.default_rng(L + bt + g + 42)
    bits = random_finite(rng, L, F32) if L < 5000 else synth.generate(L, "normal", F32, seed=L)
    assert same_f32(oracle.shuffle_tree(bits, F32, bt, g, threads=3),
                    np_shuffle(bits, F32, bt, g))
    assert same_f32(oracle.shuffle_tree_sq(bits, F32, bt, g, threads=2),
                    np_shuffle_sq(bits, F32, bt, g))


def test_shuffle_tree_f32_vector_is_four_inputs():
    # one binary32 vector holds 4 inputs: up to 4 inputs, the declared order
    # is their 4-leaf tree (the fixed-order tree); a fifth input starts
    # lane 1's vector, joined by the butterfly rather than inside the tree
    rng = np.random.default_rng(43)
    for L in range(1, 5):
        bits = random_finite(rng, L, F32)
        assert same_f32(oracle.shuffle_tree(bits, F32, 32, 1), oracle.fixed_order(bits, F32))
    # nine inputs make three vectors of 4 (lanes 0, 1, 2); the butterfly
    # adds lane 2 to lane 0 (offset 2) before lane 1 (offset 1).  With
    # x0 = 1, x4 = 2^-24, x8 = 3 * 2^-25 and zeros elsewhere:
    #   (1 + 3*2^-25) + 2^-24 = (1 + 2^-23) + 2^-24 -> tie, even: 1 + 2^-22
    # whereas vectors of 8 would give (1 + 2^-24) + 3*2^-25 = 1 + 2^-23.
    bits = np.zeros(9, np.uint32)
    bits[0], bits[4] = 0x3F800000, 0x33800000
    bits[8] = int(np.float32(3 * 2.0 ** -25).view(np.uint32))
    assert oracle.shuffle_tree(bits, F32, 32, 1) == np.float32(1 + 2.0 ** -22)
    assert oracle.fixed_order(bits, F32) == np.float32(1 + 2.0 ** -23)
    assert same_f32(oracle.shuffle_tree(bits, F32, 32, 1), np_shuffle(bits, F32, 32, 1))


def test_f32_rows_match_whole_rows():
    x = synth.generate(17 * 3001, "normal", F32, seed=44).reshape(17, 3001)
    s, a = oracle.exact_sum_rows(x, F32)
    f = oracle.fixed_order_rows(x, F32)
    t = oracle.shuffle_tree_rows(x, F32, 64, 2, squares=True)
    for r in range(17):
        assert (s[r], a[r]) == oracle.exact_sum(x[r], F32, threads=1)
        assert same_f32(f[r], oracle.fixed_order(x[r], F32, threads=1))
        assert same_f32(t[r], oracle.shuffle_tree_sq(x[r], F32, 64, 2, threads=1))


def test_f32_inputs_holding_16_bit_values_sum_like_them():
    # a binary32 array holding binary16 values has the same exact sum and the
    # same fixed-order result (the order is over index, not over bytes)
    h = synth.generate(50_001, "normal", F16, seed=45)
    w = synth.as_float(h, F16).view(np.uint32)
    assert oracle.exact_sum(w, F32) == oracle.exact_sum(h, F16)
    assert same_f32(oracle.fixed_order(w, F32), oracle.fixed_order(h, F16))
    assert oracle.exact_sum_squares(w, F32) == oracle.exact_sum_squares(h, F16)


# ---------------------------------------------------------------- blocked order

def np_blocked(bits, dtype, run_log2):
    """Runs summed left to right by numpy's accumulate (a plain sequential
    loop in float32), then the level-wise numpy tree over the runs."""
    v = np_leaves(bits, dtype).astype(np.float32)
    if v.size == 0:
        return np.float32(0.0)
    C = 1 << run_log2
    m = -(-v.size // C)
    e = np.full(m * C, -0.0, np.float32)
    e[:v.size] = v
    with np.errstate(over="ignore", invalid="ignore"):
        runs = np.add.accumulate(e.reshape(m, C), axis=1, dtype=np.float32)[:, -1]
    return np_tree(runs)


def test_blocked_order_hand_worked_cases(golden_dir):
    n_cases = 0
    with open(os.path.join(golden_dir, "blocked_order_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, bits, expect = [p.strip() for p in line.split("|")]
            b = np.array([int(h, 16) for h in bits.split()], np.uint16)
            got = oracle.blocked_order(b, F16, int(c), threads=1)
            assert got == np.float32(float(Fraction(expect))), line
            n_cases += 1
    assert n_cases == 5


@pytest.mark.parametrize("dtype", [F16, BF16, F32])
@pytest.mark.parametrize("n", [1, 5, 8, 63, 64, 65, 1000, 4097, 100_003])
@pytest.mark.parametrize("c", [0, 1, 2, 3, 5, 7, 12])
def test_blocked_order_matches_numpy(dtype, n, c):
    rng = np.random.default_rng(n * 16 + c)
    bits = random_finite(rng, n, dtype) if n < 5000 else synth.generate(n, "normal", dtype, seed=n)
    assert same_f32(oracle.blocked_order(bits, dtype, c, threads=3), np_blocked(bits, dtype, c))


def test_blocked_order_limits_are_the_tree_and_the_sequential_sum():
    bits = synth.generate(30_001, "uniform_pm1", F16, seed=46)
    tree = oracle.fixed_order(bits, F16)
    assert same_f32(oracle.blocked_order(bits, F16, 0), tree)
    assert same_f32(oracle.blocked_order(bits, F16, 1), tree)       # runs of two = pairs
    seq = np.float32(0.0)
    for v in np_leaves(bits, F16):
        seq = np.float32(seq + v)
    for c in (15, 16, 20):                                           # one run
        assert same_f32(oracle.blocked_order(bits, F16, c), seq)
    # the orders differ in between: C = 4 is neither the tree nor the run of all
    c4 = oracle.blocked_order(bits, F16, 2)
    assert not same_f32(c4, seq) or not same_f32(c4, tree)


def test_blocked_order_rows_and_degenerate():
    x = synth.generate(21 * 3001, "normal", BF16, seed=47).reshape(21, 3001)
    got = oracle.blocked_order_rows(x, BF16, 6)
    for r in range(21):
        assert same_f32(got[r], oracle.blocked_order(x[r], BF16, 6, threads=1))
    assert oracle.blocked_order(np.zeros(0, np.uint16), F16, 4).tobytes() == \
        np.float32(0.0).tobytes()
    negz = oracle.blocked_order(np.full(9, 0x8000, np.uint16), F16, 2)
    assert negz.tobytes() == np.float32(-0.0).tobytes()
    assert np.isnan(oracle.blocked_order(np.array([0x3C00, 0x7E00], np.uint16), F16, 1))


# ---------------------------------------------------------------- mean / variance

def test_mean_var_formula_against_float64():
    # normal rows: the binary32 formula is within a few ulps of the float64
    # mean and variance of the same sums
    x = synth.generate(300 * 4096, "normal", F16, seed=53).reshape(300, 4096)
    s1 = oracle.fixed_order_rows(x, F16)
    s2 = oracle.fixed_order_rows(x, F16, squares=True)
    m, v = oracle.mean_var(s1, s2, 4096)
    m64 = s1.astype(np.float64) / 4096
    v64 = s2.astype(np.float64) / 4096 - m64 * m64
    assert np.all(np.abs(m - m64) <= 2.0 ** -23 * np.abs(m64) + 1e-30)
    assert np.all(np.abs(v - v64) <= 2.0 ** -22 * (s2 / 4096) + 1e-30)
    # and the float64 statistics of the data themselves, within the sums' rounding
    xf = np.asarray(np_leaves(x.reshape(-1), F16), np.float64).reshape(300, 4096)
    assert np.allclose(m, xf.mean(axis=1), rtol=0, atol=1e-5)
    assert np.allclose(v, xf.var(axis=1), rtol=1e-5, atol=1e-6)


def test_mean_var_special_cases():
    # constant rows: variance exactly 0; [a, b]: ((a + b)/2, ((a - b)/2)^2)
    s1 = np.array([7 * 5.0, 3.0 + 5.0, 0.0], np.float32)
    s2 = np.array([7 * 25.0, 9.0 + 25.0, 0.0], np.float32)
    m, v = oracle.mean_var(s1[:1], s2[:1], 7)
    assert m[0] == 5.0 and v[0] == 0.0
    m, v = oracle.mean_var(s1[1:2], s2[1:2], 2)
    assert m[0] == 4.0 and v[0] == 1.0
    # cancellation that would go negative is clamped to +0
    m, v = oracle.mean_var(np.array([3.0000002], np.float32), np.array([3.0], np.float32), 3)
    assert v[0] == 0.0 and np.signbit(v[0]) == False
    # no inputs: 0 / 0
    m, v = oracle.mean_var(np.zeros(1, np.float32), np.zeros(1, np.float32), 0)
    assert np.isnan(m[0]) and np.isnan(v[0])


# ---------------------------------------------------------------- split-K GEMM

def test_gemm_f64_matches_numpy_and_brute_force():
    rng = np.random.default_rng(70)
    for dtype, (M, N, K) in ((F16, (5, 7, 33)), (BF16, (9, 4, 130)), (F16, (1, 1, 1))):
        A = synth.generate(M * K, "normal", dtype, seed=M).reshape(M, K)
        W = synth.generate(N * K, "normal", dtype, seed=N + 100).reshape(N, K)
        c, a = oracle.gemm_f64(A, W, dtype, threads=2)
        fa = np_leaves(A.reshape(-1), dtype).astype(np.float64).reshape(M, K)
        fw = np_leaves(W.reshape(-1), dtype).astype(np.float64).reshape(N, K)
        assert np.allclose(c, fa @ fw.T, rtol=1e-12, atol=1e-12)
        assert np.allclose(a, np.abs(fa) @ np.abs(fw).T, rtol=1e-12, atol=1e-12)
    # exact on a tiny case (every product and partial sum exact in binary64)
    A = random_finite(rng, 12, F16).reshape(3, 4)
    W = random_finite(rng, 20, F16).reshape(5, 4)
    c, _ = oracle.gemm_f64(A, W, F16)
    fa = np_leaves(A.reshape(-1), F16).reshape(3, 4)
    fw = np_leaves(W.reshape(-1), F16).reshape(5, 4)
    for i in range(3):
        for j in range(5):
            exact = sum((Fraction(float(fa[i, k])) * Fraction(float(fw[j, k])) for k in range(4)),
                        Fraction(0))
            assert abs(Fraction(c[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)


def exact_partials_operands(M, N, K, k_split, scales, dtype, seed):
    """Small integers in A; in W, integers times 2^-scales[s] on split s: every
    split's partial is an exact binary32 value that any order of addition
    reaches without rounding, so only the combine of the splits rounds."""
    rng = np.random.default_rng(seed)
    a = rng.integers(-8, 9, (M, K)).astype(np.float64)
    w = rng.integers(-8, 9, (N, K)).astype(np.float64)
    for s, e in enumerate(scales):
        w[:, s * k_split:(s + 1) * k_split] *= 2.0 ** -e
    if dtype == F16:
        return a.astype(np.float16).view(np.uint16), w.astype(np.float16).view(np.uint16)
    def bf(x):
        return (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return bf(a), bf(w)


def test_gemm_splitk_declared_combine_hand_worked():
    # K = 256 in 4 splits of 64: row 0 of A all ones; column 0 of W has 1.0
    # in split 0 and 2^-24 once in each other split -> P = (1, t, t, t);
    # the tree (1 + t) + (t + t): 1 + t ties to 1, + 2^-23 -> 1 + 2^-23.
    # One split rounds the exact 1 + 3 * 2^-24 once: halfway between 1 + 2^-23
    # and 1 + 2^-22, to even -> 1 + 2^-22.
    A = np.full((1, 256), 0x3C00, np.uint16)
    W = np.zeros((1, 256), np.uint16)
    W[0, 0] = 0x3C00
    W[0, 64] = W[0, 128] = W[0, 192] = 0x0001
    assert oracle.gemm_splitk(A, W, F16, 4, 64)[0, 0] == np.float32(1 + 2.0 ** -23)
    assert oracle.gemm_splitk(A, W, F16, 1, 256)[0, 0] == np.float32(1 + 2.0 ** -22)
    c, _ = oracle.gemm_f64(A, W, F16)
    assert c[0, 0] == 1 + 3 * 2.0 ** -24


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_gemm_splitk_exact_partials_and_bound(dtype):
    M, N, K, ks = 7, 9, 320, 64
    scales = (0, 13, 24, 7, 20)
    A, W = exact_partials_operands(M, N, K, ks, scales, dtype, seed=71)
    got = oracle.gemm_splitk(A, W, dtype, 5, ks)
    # each partial exactly, then the tree in numpy
    fa = np_leaves(A.reshape(-1), dtype).astype(np.float64).reshape(M, K)
    fw = np_leaves(W.reshape(-1), dtype).astype(np.float64).reshape(N, K)
    parts = np.stack([(fa[:, s * ks:(s + 1) * ks] @ fw[:, s * ks:(s + 1) * ks].T).astype(np.float32)
                      for s in range(5)])
    for i in range(M):
        for j in range(N):
            assert same_f32(got[i, j], np_tree(parts[:, i, j]))
    # general inputs: within the rounding of the partials and of the tree
    A = synth.generate(6 * 500, "normal", dtype, seed=72).reshape(6, 500)
    W = synth.generate(5 * 500, "normal", dtype, seed=73).reshape(5, 500)
    c, a = oracle.gemm_f64(A, W, dtype)
    for S, ks in ((1, 512), (4, 128), (8, 64)):
        g = oracle.gemm_splitk(A, W, dtype, S, ks).astype(np.float64)
        assert np.all(np.abs(g - c) <= 2.0 ** -24 * (1 + int(np.ceil(np.log2(S))) * 2) * a + 1e-30)
