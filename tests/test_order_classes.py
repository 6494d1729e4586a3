"""Bit-equivalence classes decided from order descriptors
(tcr_order_equivalent), checked against the CPU oracle: calls the checker
puts in one class must agree bit for bit on every input tried, and calls it
separates must be told apart by some input."""
import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library
from tests.test_oracle import same_f32

M = tcr.Mode
BLOCKS = (32, 64, 128, 256, 512, 1024)


@pytest.fixture(scope="module", autouse=True)
def lib():
    build_library()
    return tcr.c_api()


def team(L, block):
    d = tcr.tcr_order_descriptor(n=L, mode=M(tcr.SHUFFLE_TREE, block_threads=block))
    return d["team_threads"], d["team_blocks"]


def samples(L):
    out = [synth.generate(L, dist, tcr.F16, seed=L + i)
           for i, dist in enumerate(("normal", "uniform01", "uniform_pm1"))]
    # order-sensitive: one large value among many tiny ones at scattered places
    crafted = np.full(L, 0x0001, np.uint16)
    crafted[L // 3] = 0x3C00
    out.append(crafted)
    return out


@pytest.mark.parametrize("L", [5, 8, 100, 250, 2048, 8192, 8193, 10_000, 33_333, 262_144, 1_000_003])
def test_shuffle_tree_classes_agree_with_the_oracle(L):
    xs = samples(L)
    results = {b: [oracle.shuffle_tree(x, tcr.F16, *team(L, b)) for x in xs] for b in BLOCKS}
    for i, a in enumerate(BLOCKS):
        for b in BLOCKS[i + 1:]:
            eq = tcr.tcr_order_equivalent(dict(n=L, mode=M(tcr.SHUFFLE_TREE, block_threads=a)),
                                          dict(n=L, mode=M(tcr.SHUFFLE_TREE, block_threads=b)))
            same = all(same_f32(p, q) for p, q in zip(results[a], results[b]))
            if eq:
                assert same, (L, a, b)
            else:
                # separated classes really are different orders: some input shows it
                extra = [synth.generate(L, "normal", tcr.F16, seed=7 * L + s) for s in range(6)]
                differ = not same or any(
                    not same_f32(oracle.shuffle_tree(x, tcr.F16, *team(L, a)),
                                 oracle.shuffle_tree(x, tcr.F16, *team(L, b))) for x in extra)
                assert differ, (L, a, b)


def test_whole_team_rule_is_one_class_on_large_sums():
    for L in (1 << 20, 1 << 28, 1 << 30):
        for b in BLOCKS:
            assert tcr.tcr_order_equivalent(dict(n=L, mode=M(tcr.SHUFFLE_TREE)),
                                            dict(n=L, mode=M(tcr.SHUFFLE_TREE, block_threads=b)))


def test_fixed_order_is_one_class_per_length():
    for b in BLOCKS:
        assert tcr.tcr_order_equivalent(dict(n=12345, mode=M(tcr.FIXED_ORDER)),
                                        dict(n=12345, mode=M(tcr.FIXED_ORDER, block_threads=b)))
        assert tcr.tcr_order_equivalent(dict(n=12345, mode=M(tcr.FIXED_ORDER)),
                                        dict(rows=7, cols=12345, mode=M(tcr.FIXED_ORDER, block_threads=b)))
    assert not tcr.tcr_order_equivalent(dict(n=12345, mode=M(tcr.FIXED_ORDER)),
                                        dict(n=12346, mode=M(tcr.FIXED_ORDER)))
    assert not tcr.tcr_order_equivalent(dict(n=12345, mode=M(tcr.FIXED_ORDER)),
                                        dict(n=12345, mode=M(tcr.SHUFFLE_TREE)))


def test_mma_chain_classes():
    base = dict(n=1 << 24, mode=M(tcr.MMA_CHAIN, R=4))
    assert tcr.tcr_order_equivalent(base, dict(n=1 << 24, mode=M(tcr.MMA_CHAIN, R=4)))
    assert not tcr.tcr_order_equivalent(base, dict(n=1 << 24, mode=M(tcr.MMA_CHAIN, R=5)))
    assert not tcr.tcr_order_equivalent(base, dict(n=1 << 24, mode=M(tcr.MMA_CHAIN, R=4, block_threads=512)))


def test_equivalence_rejects_null(lib):
    d = tcr.tcr_order_desc()
    assert lib.tcr_order_equivalent(None, None, None) == tcr.ERR_INVALID_ARG
    import ctypes
    assert lib.tcr_order_equivalent(ctypes.byref(d), ctypes.byref(d), None) == tcr.ERR_INVALID_ARG
