"""GPU parity for the sum of squares (tcr_reduce_sum_squares,
tcr_reduce_rows_sum_squares), through the C ABI.

FIXED_ORDER and SHUFFLE_TREE must equal the oracle's emulation of their
declared orders over the leaves fl32(x_i * x_i) bit for bit; MMA_CHAIN (the
A * A^T contraction on the tensor cores) must be within
2^-20 * sum x_i^2 + 1e-6 of the exact sum of squares.
"""
import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library
from tests import spec
from tests.test_gpu_parity import assert_within_mma_tolerance, same_bits, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F16, BF16 = tcr.F16, tcr.BF16
SIZES = [1, 7, 8, 9, 255, 256, 257, 2048, 2049, 8193, 65537, 1 << 20, (1 << 22) + 13]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


def sq_sum(bits, mode):
    return np.float32(tcr.tcr_reduce_sum_squares(dev(bits), mode).cpu().numpy()[0])


def sq_rows(bits2d, mode):
    return tcr.tcr_reduce_rows_sum_squares(dev(bits2d), mode).cpu().numpy()


def inputs(n, dtype, dist="normal", seed=None):
    return synth.generate(n, dist, dtype, seed=n + 1000 if seed is None else seed)


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("n", SIZES)
def test_fixed_order_sum_squares_bit_exact(dtype, n):
    x = inputs(n, dtype)
    assert same_bits(sq_sum(x, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)), oracle.fixed_order_sq(x, dtype))


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("block", [0, 32, 1024])
def test_shuffle_tree_sum_squares_bit_exact(dtype, n, block):
    x = inputs(n, dtype)
    got = sq_sum(x, tcr.Mode(tcr.SHUFFLE_TREE, block_threads=block, dtype=dtype))
    assert same_bits(got, oracle.shuffle_tree_sq(x, dtype, *spec.shuffle_team(n, block)))


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("kind,R", [(tcr.MMA_CHAIN, 0), (tcr.MMA_CHAIN, 1), (tcr.MMA_CHAIN, 5),
                                    (tcr.MMA_CHAIN, 8), (tcr.MMA_CHAIN_TMEM, 0)])
def test_mma_chain_sum_squares_within_tolerance(dtype, n, kind, R):
    x = inputs(n, dtype, "uniform_pm1")
    got = sq_sum(x, tcr.Mode(kind, R=R, dtype=dtype))
    assert_within_mma_tolerance(got, *oracle.exact_sum_squares(x, dtype))


def test_fixed_order_sum_squares_one_equivalence_class():
    n = (1 << 21) + 3
    x = inputs(n, F16, "uniform_pm1")
    ref = oracle.fixed_order_sq(x, F16)
    for b in (32, 64, 128, 256, 512, 1024):
        assert same_bits(sq_sum(x, tcr.Mode(tcr.FIXED_ORDER, block_threads=b)), ref)
    assert same_bits(sq_rows(x.reshape(1, n), tcr.Mode(tcr.FIXED_ORDER))[0], ref)


ROW_SHAPES = [(1, 1), (17, 100), (64, 4096), (1000, 4096), (40, 16384), (9, 16385), (3, 1 << 20)]


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("shape", ROW_SHAPES)
def test_rows_sum_squares_all_modes(dtype, shape):
    rows, cols = shape
    x = inputs(rows * cols, dtype, seed=rows * 3 + cols).reshape(rows, cols)
    assert same_bits(sq_rows(x, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)),
                     oracle.fixed_order_rows(x, dtype, squares=True))
    bt, g = spec.shuffle_team(cols)
    assert same_bits(sq_rows(x, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype)),
                     oracle.shuffle_tree_rows(x, dtype, bt, g, squares=True))
    s, a = oracle.exact_sum_rows(x, dtype, squares=True)
    for kind in (tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM):
        assert_within_mma_tolerance(sq_rows(x, tcr.Mode(kind, dtype=dtype)), s, a)


def test_sum_squares_rows_65536x4096():
    rows, cols = 65536, 4096
    x = synth.generate(rows * cols, "normal", F16, seed=2).reshape(rows, cols)
    t = dev(x.reshape(-1)).view(rows, cols)
    got = tcr.tcr_reduce_rows_sum_squares(t, tcr.Mode(tcr.FIXED_ORDER)).cpu().numpy()
    assert same_bits(got, oracle.fixed_order_rows(x, F16, squares=True))
    s, a = oracle.exact_sum_rows(x, F16, squares=True)
    got = tcr.tcr_reduce_rows_sum_squares(t, tcr.Mode(tcr.MMA_CHAIN)).cpu().numpy()
    assert_within_mma_tolerance(got, s, a)


def test_sum_squares_misaligned_and_special():
    x = inputs(100_003, F16)
    t = dev(x)[5:]
    got = np.float32(tcr.tcr_reduce_sum_squares(t, tcr.Mode(tcr.FIXED_ORDER)).cpu().numpy()[0])
    assert same_bits(got, oracle.fixed_order_sq(x[5:], F16))
    got = np.float32(tcr.tcr_reduce_sum_squares(t, tcr.Mode(tcr.MMA_CHAIN)).cpu().numpy()[0])
    assert_within_mma_tolerance(got, *oracle.exact_sum_squares(x[5:], F16))
    for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN):
        y = x.copy()
        y[17] = 0xFC00                      # -inf: its square is +inf
        assert sq_sum(y, tcr.Mode(kind)) == np.inf
        y[18] = 0x7E00
        assert np.isnan(sq_sum(y, tcr.Mode(kind)))
        z = np.full(1000, 0x8000, np.uint16)
        assert same_bits(sq_sum(z, tcr.Mode(kind)), np.float32(0.0))
