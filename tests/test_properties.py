"""Property-based checks (hypothesis; skipped where it is not installed) of
the oracle and of the declared rules, over generated shapes and patterns."""
import math

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
import arithmetic_reduction_tensor_gb300 as tcr  # noqa: E402
from arithmetic_reduction_tensor_gb300.build import build_library  # noqa: E402
from tests import spec  # noqa: E402
from tests.test_oracle import (F16, BF16, F32, np_blocked, np_leaves, np_shuffle, np_tree,  # noqa: E402
                               random_finite, same_f32)

SETTINGS = settings(max_examples=60, deadline=None)


@SETTINGS
@given(n=st.integers(0, 3000), dtype=st.sampled_from([F16, BF16, F32]), seed=st.integers(0, 2**31))
def test_fixed_order_is_the_levelwise_tree(n, dtype, seed):
    bits = random_finite(np.random.default_rng(seed), n, dtype)
    got = oracle.fixed_order(bits, dtype, threads=2)
    ref = np_tree(np_leaves(bits, dtype)) if n else np.float32(0.0)
    assert same_f32(got, ref)


@SETTINGS
@given(n=st.integers(1, 5000), dtype=st.sampled_from([F16, BF16, F32]), c=st.integers(0, 14),
       seed=st.integers(0, 2**31))
def test_blocked_order_is_accumulate_then_tree(n, dtype, c, seed):
    bits = random_finite(np.random.default_rng(seed), n, dtype)
    assert same_f32(oracle.blocked_order(bits, dtype, c, threads=2), np_blocked(bits, dtype, c))


@SETTINGS
@given(L=st.integers(1, 20000), bt=st.sampled_from([32, 64, 128, 256]), g=st.integers(1, 6),
       dtype=st.sampled_from([F16, F32]), seed=st.integers(0, 2**31))
def test_shuffle_tree_is_its_vectorised_emulation(L, bt, g, dtype, seed):
    bits = random_finite(np.random.default_rng(seed), L, dtype)
    assert same_f32(oracle.shuffle_tree(bits, dtype, bt, g, threads=2), np_shuffle(bits, dtype, bt, g))


@SETTINGS
@given(n=st.integers(0, 400), dtype=st.sampled_from([F16, BF16, F32]), seed=st.integers(0, 2**31))
def test_exact_sum_is_the_rational_sum(n, dtype, seed):
    from fractions import Fraction
    bits = random_finite(np.random.default_rng(seed), n, dtype)
    s, a = oracle.exact_sum(bits, dtype)
    vals = np_leaves(bits, dtype).astype(np.float64)
    assert s == float(sum((Fraction(float(v)) for v in vals), Fraction(0)))
    assert a == float(sum((Fraction(abs(float(v))) for v in vals), Fraction(0)))


@pytest.fixture(scope="module")
def lib():
    build_library()
    return tcr.c_api()


@SETTINGS
@given(L=st.integers(1, 1 << 34), block=st.sampled_from([0, 32, 64, 128, 256, 512, 1024]),
       dtype=st.sampled_from([F16, BF16, F32]))
def test_shuffle_descriptor_follows_the_rule(lib, L, block, dtype):
    d = tcr.tcr_order_descriptor(n=L, mode=tcr.Mode(tcr.SHUFFLE_TREE, block_threads=block, dtype=dtype))
    assert (d["team_threads"], d["team_blocks"]) == spec.shuffle_team(L, block, dtype)


@SETTINGS
@given(M=st.integers(1, 70000), N=st.integers(1, 70000), K=st.integers(0, 1 << 20).map(lambda k: 8 * k),
       S=st.integers(0, 64))
def test_gemm_descriptor_follows_the_rule(lib, M, N, K, S):
    d = tcr.tcr_gemm_descriptor(M, N, K, S, F16)
    assert (d["splits"], d["k_split"]) == spec.gemm_splits(M, N, K, S)
    # whole 64-column boxes, every split non-empty, together covering K
    assert d["k_split"] % 64 == 0
    assert (d["splits"] - 1) * d["k_split"] < max(K, 1) <= d["splits"] * d["k_split"] or K == 0


@SETTINGS
@given(n=st.integers(1, 1 << 20), c1=st.integers(0, 16), c2=st.integers(0, 16))
def test_blocked_equivalence_is_the_effective_run(lib, n, c1, c2):
    h = max(0, math.ceil(math.log2(n)))

    def eff(c):
        c = min(c, h)
        return 0 if c <= 1 else c
    a = {"n": n, "mode": tcr.Mode(tcr.FIXED_ORDER, run_log2=c1)}
    b = {"n": n, "mode": tcr.Mode(tcr.FIXED_ORDER, run_log2=c2)}
    assert tcr.tcr_order_equivalent(a, b) == (eff(c1) == eff(c2))
