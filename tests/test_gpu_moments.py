"""GPU parity for the fused row moments: tcr_reduce_rows_moments (sum and sum
of squares of every row in one pass) and tcr_reduce_rows_mean_var.

FIXED_ORDER and SHUFFLE_TREE: both sums bit-exact to the oracle's emulation
of the declared orders (and to the single-reduction calls), and the mean and
variance bit-exact to the oracle's binary32 formula applied to them.
MMA_CHAIN (and the tcgen05 kind, which runs it): each sum within
2^-20 * sum|leaf| + 1e-6 of the exact one, the mean and variance within the
bound that follows from those two errors and the formula's four roundings.
"""
import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library
from tests import spec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F16, BF16, F32 = tcr.F16, tcr.BF16, tcr.F32


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


def dev2(bits, rows, cols):
    a = np.ascontiguousarray(bits)
    t = torch.from_numpy(a.view(np.float32) if a.dtype == np.uint32 else a.view(np.int16))
    return t.to("cuda").view(rows, cols)


def same_bits(a, b):
    a = np.asarray(a, np.float32).reshape(-1)
    b = np.asarray(b, np.float32).reshape(-1)
    nan = np.isnan(a) & np.isnan(b)
    return np.array_equal(a.view(np.uint32)[~nan], b.view(np.uint32)[~nan]) and \
        np.array_equal(np.isnan(a), np.isnan(b))


def moments(x, m):
    s1, s2 = tcr.tcr_reduce_rows_moments(x, m)
    return s1.cpu().numpy(), s2.cpu().numpy()


def mean_var(x, m):
    a, b = tcr.tcr_reduce_rows_mean_var(x, m)
    return a.cpu().numpy(), b.cpu().numpy()


SHAPES = [(3, 5), (1000, 4096), (333, 4095), (64, 16384), (50, 16385), (4, 1_000_003)]


@pytest.mark.parametrize("dtype", [F16, BF16, F32])
@pytest.mark.parametrize("shape", SHAPES)
def test_ordered_moments_bit_exact(dtype, shape):
    rows, cols = shape
    x = synth.generate(rows * cols, "normal", dtype, seed=rows + cols).reshape(rows, cols)
    t = dev2(x, rows, cols)
    f1 = oracle.fixed_order_rows(x, dtype)
    f2 = oracle.fixed_order_rows(x, dtype, squares=True)
    s1, s2 = moments(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype))
    assert same_bits(s1, f1) and same_bits(s2, f2)
    m, v = mean_var(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype))
    om, ov = oracle.mean_var(f1, f2, cols)
    assert same_bits(m, om) and same_bits(v, ov)
    bt, g = spec.shuffle_team(cols, 0, dtype)
    g1 = oracle.shuffle_tree_rows(x, dtype, bt, g)
    g2 = oracle.shuffle_tree_rows(x, dtype, bt, g, squares=True)
    s1, s2 = moments(t, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype))
    assert same_bits(s1, g1) and same_bits(s2, g2)
    m, v = mean_var(t, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype))
    om, ov = oracle.mean_var(g1, g2, cols)
    assert same_bits(m, om) and same_bits(v, ov)


def test_fused_equals_the_two_single_calls():
    rows, cols = 700, 5000
    x = synth.generate(rows * cols, "uniform_pm1", BF16, seed=60).reshape(rows, cols)
    t = dev2(x, rows, cols)
    for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN):
        m = tcr.Mode(kind, dtype=BF16)
        s1, s2 = moments(t, m)
        assert same_bits(s1, tcr.tcr_reduce_rows(t, m).cpu().numpy())
        assert same_bits(s2, tcr.tcr_reduce_rows_sum_squares(t, m).cpu().numpy())


@pytest.mark.parametrize("dtype", [F16, BF16, F32])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("kind", [tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM])
def test_mma_moments_within_tolerance(dtype, shape, kind):
    rows, cols = shape
    x = synth.generate(rows * cols, "normal", dtype, seed=rows * 3 + cols).reshape(rows, cols)
    t = dev2(x, rows, cols)
    e1, a1 = oracle.exact_sum_rows(x, dtype)
    e2, _ = oracle.exact_sum_rows(x, dtype, squares=True)
    s1, s2 = moments(t, tcr.Mode(kind, dtype=dtype))
    t1, t2 = spec.mma_tolerance(a1), spec.mma_tolerance(e2)
    assert np.all(np.abs(s1 - e1) <= t1) and np.all(np.abs(s2 - e2) <= t2)
    m, v = mean_var(t, tcr.Mode(kind, dtype=dtype))
    n = float(cols)
    mu = e1 / n
    ex2 = e2 / n
    var_exact = ex2 - mu * mu
    u = 2.0 ** -24
    dm = t1 / n + u * np.abs(s1 / n)
    # |dv| <= dq + 2|mu| dm + dm^2 + the formula's roundings of q, m*m and q - m*m
    dv = t2 / n + 2 * np.abs(mu) * dm + dm * dm + 3 * u * (ex2 + mu * mu) + 1e-12
    assert np.all(np.abs(m - mu) <= dm)
    assert np.all(np.abs(v - np.maximum(var_exact, 0)) <= dv)


@pytest.mark.parametrize("block", [32, 128, 1024])
def test_long_rows_do_not_depend_on_the_block_size(block):
    rows, cols = 9, 300_001
    x = synth.generate(rows * cols, "normal", F16, seed=61).reshape(rows, cols)
    t = dev2(x, rows, cols)
    s1, s2 = moments(t, tcr.Mode(tcr.FIXED_ORDER, block_threads=block))
    assert same_bits(s1, oracle.fixed_order_rows(x, F16))
    assert same_bits(s2, oracle.fixed_order_rows(x, F16, squares=True))


def test_misaligned_rows_and_base():
    rows, cols = 257, 1001
    x = synth.generate(rows * cols + 1, "normal", F16, seed=62)
    t = torch.from_numpy(x.view(np.int16)).cuda()[1:].view(rows, cols)
    xs = x[1:].reshape(rows, cols)
    s1, s2 = moments(t, tcr.Mode(tcr.FIXED_ORDER))
    assert same_bits(s1, oracle.fixed_order_rows(xs, F16))
    assert same_bits(s2, oracle.fixed_order_rows(xs, F16, squares=True))


def test_degenerate_shapes_and_non_finite():
    out_a = torch.full((4,), 7.0, device="cuda")
    out_b = torch.full((4,), 7.0, device="cuda")
    empty = torch.empty(4, 0, dtype=torch.float16, device="cuda")
    tcr.tcr_reduce_rows_moments(empty, tcr.Mode(tcr.FIXED_ORDER), sums=out_a, sums_of_squares=out_b)
    assert same_bits(out_a.cpu().numpy(), np.zeros(4, np.float32))
    assert same_bits(out_b.cpu().numpy(), np.zeros(4, np.float32))
    tcr.tcr_reduce_rows_mean_var(empty, tcr.Mode(tcr.FIXED_ORDER), mean=out_a, var=out_b)
    assert np.all(np.isnan(out_a.cpu().numpy())) and np.all(np.isnan(out_b.cpu().numpy()))
    a, b = tcr.tcr_reduce_rows_moments(torch.empty(0, 9, dtype=torch.float16, device="cuda"),
                                       tcr.Mode(tcr.FIXED_ORDER))
    assert a.numel() == 0 and b.numel() == 0
    # constant rows: variance exactly 0
    x = np.full(16 * 3000, np.float16(0.75).view(np.uint16), np.uint16)
    m, v = mean_var(dev2(x, 16, 3000), tcr.Mode(tcr.FIXED_ORDER))
    assert np.all(m == 0.75) and np.all(v == 0.0)
    # an infinity in a row: both sums infinite, the formula's NaN variance
    rows, cols = 8, 2000
    x = synth.generate(rows * cols, "normal", F16, seed=63).reshape(rows, cols)
    x[3, 17] = 0x7C00
    t = dev2(x, rows, cols)
    for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN):
        s1, s2 = moments(t, tcr.Mode(kind))
        assert s1[3] == np.inf and s2[3] == np.inf and np.all(np.isfinite(np.delete(s1, 3)))
        m, v = mean_var(t, tcr.Mode(kind))
        assert m[3] == np.inf and np.isnan(v[3])


def test_blocked_order_is_refused():
    x = torch.zeros(4, 100, dtype=torch.float16, device="cuda")
    with pytest.raises(tcr.TcrError) as e:
        tcr.tcr_reduce_rows_moments(x, tcr.Mode(tcr.FIXED_ORDER, run_log2=3))
    assert e.value.status == tcr.ERR_UNSUPPORTED
