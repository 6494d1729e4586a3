"""GPU parity for inputs that do not start on a 16-byte boundary: a base
pointer a few inputs past one, and rows whose stride is not whole vectors.
The kernels read such segments as whole aligned granules and shift each
vector out of two of them; every result must still be the declared order's
(bit-exact to the oracle for FIXED_ORDER and SHUFFLE_TREE, within the
MMA_CHAIN bound), at every offset in the granule, over group boundaries and
ragged ends, in every kernel family (warp per row, chunked, block team).
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


def dev(bits):
    a = np.ascontiguousarray(bits).reshape(-1)
    return torch.from_numpy(a.view(np.float32) if a.dtype == np.uint32 else a.view(np.int16)).to("cuda")


def same_bits(a, b):
    a = np.asarray(a, np.float32).reshape(-1)
    b = np.asarray(b, np.float32).reshape(-1)
    nan = np.isnan(a) & np.isnan(b)
    return np.array_equal(a.view(np.uint32)[~nan], b.view(np.uint32)[~nan]) and \
        np.array_equal(np.isnan(a), np.isnan(b))


def within(got, exact, abs_sum):
    err = np.abs(np.asarray(got, np.float64) - np.asarray(exact))
    return bool(np.all(err <= spec.mma_tolerance(np.asarray(abs_sum))))


SIZES = [1, 7, 9, 2047, 2049, 4097, 300_001, (1 << 22) + 5]


@pytest.mark.parametrize("dtype", [F16, BF16, F32])
@pytest.mark.parametrize("offset", [1, 2, 3, 5, 7])
def test_sums_from_a_misaligned_base(dtype, offset):
    V = spec.vector_len(dtype)
    if offset % V == 0:
        pytest.skip("aligned")
    for n in SIZES:
        x = synth.generate(n + offset, "normal", dtype, seed=n + 7 * offset)
        t = dev(x)[offset:]
        xs = x[offset:]
        got = tcr.tcr_reduce_sum(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)).cpu().numpy()
        assert same_bits(got, oracle.fixed_order(xs, dtype)), n
        for block in (32, 256, 1024):
            got = tcr.tcr_reduce_sum(t, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype, block_threads=block))
            assert same_bits(got.cpu().numpy(), oracle.shuffle_tree(xs, dtype, *spec.shuffle_team(n, block, dtype))), \
                (n, block)
        e, a = oracle.exact_sum(xs, dtype)
        for kind in (tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM):
            assert within(tcr.tcr_reduce_sum(t, tcr.Mode(kind, dtype=dtype)).cpu().numpy(), e, a), (n, kind)
        got = tcr.tcr_reduce_sum_squares(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)).cpu().numpy()
        assert same_bits(got, oracle.fixed_order_sq(xs, dtype)), n


# long rows: one warp per row up to 32 KiB, chunked (FIXED, MMA) or a block
# team (SHUFFLE) beyond
ROWS = [(300, 4095), (64, 16383), (9, 100_003), (3, 1_000_001)]


@pytest.mark.parametrize("dtype", [F16, F32])
@pytest.mark.parametrize("shape", ROWS)
def test_rows_whose_stride_is_not_whole_vectors(dtype, shape):
    rows, cols = shape
    x = synth.generate(rows * cols, "normal", dtype, seed=rows + cols).reshape(rows, cols)
    t = dev(x).view(rows, cols)
    got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)).cpu().numpy()
    assert same_bits(got, oracle.fixed_order_rows(x, dtype))
    for block in (64, 1024):
        bt, g = spec.shuffle_team(cols, block, dtype)
        got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype, block_threads=block)).cpu().numpy()
        assert same_bits(got, oracle.shuffle_tree_rows(x, dtype, bt, g)), block
    e, a = oracle.exact_sum_rows(x, dtype)
    for R in (1, 4):
        got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.MMA_CHAIN, R=R, dtype=dtype)).cpu().numpy()
        assert within(got, e, a), R
    # both sums in one pass
    s1, s2 = tcr.tcr_reduce_rows_moments(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype))
    assert same_bits(s1.cpu().numpy(), oracle.fixed_order_rows(x, dtype))
    assert same_bits(s2.cpu().numpy(), oracle.fixed_order_rows(x, dtype, squares=True))
    s1, s2 = tcr.tcr_reduce_rows_moments(t, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype))
    bt, g = spec.shuffle_team(cols, 0, dtype)
    assert same_bits(s1.cpu().numpy(), oracle.shuffle_tree_rows(x, dtype, bt, g))
    assert same_bits(s2.cpu().numpy(), oracle.shuffle_tree_rows(x, dtype, bt, g, squares=True))
    s1, s2 = tcr.tcr_reduce_rows_moments(t, tcr.Mode(tcr.MMA_CHAIN, dtype=dtype))
    e2, _ = oracle.exact_sum_rows(x, dtype, squares=True)
    assert within(s1.cpu().numpy(), e, a) and within(s2.cpu().numpy(), e2, e2)


@pytest.mark.parametrize("offset", [1, 3, 6])
def test_rows_from_a_misaligned_base(offset):
    # whole-vector rows, every one starting `offset` inputs past a boundary
    rows, cols = 40, 8192
    x = synth.generate(rows * cols + offset, "normal", BF16, seed=offset)
    t = dev(x)[offset:].view(rows, cols)
    xs = x[offset:].reshape(rows, cols)
    for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        got = tcr.tcr_reduce_rows(t, tcr.Mode(kind, dtype=BF16)).cpu().numpy()
        ref = oracle.fixed_order_rows(xs, BF16) if kind == tcr.FIXED_ORDER else \
            oracle.shuffle_tree_rows(xs, BF16, *spec.shuffle_team(cols, 0, BF16))
        assert same_bits(got, ref), kind
    e, a = oracle.exact_sum_rows(xs, BF16)
    for kind in (tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM):
        assert within(tcr.tcr_reduce_rows(t, tcr.Mode(kind, dtype=BF16)).cpu().numpy(), e, a), kind


def test_segment_ending_at_the_end_of_its_buffer():
    # the last granule holds the data's last bytes and nothing after them is
    # read: the input ends exactly at the end of its allocation
    for n in (2049, 40_000, 300_001):
        for tail in range(1, 8):
            x = synth.generate(n, "normal", F16, seed=n + tail)
            buf = torch.empty(n + tail, dtype=torch.int16, device="cuda")
            buf[tail:] = torch.from_numpy(x.view(np.int16)).cuda()
            t = buf[tail:]
            got = tcr.tcr_reduce_sum(t, tcr.Mode(tcr.FIXED_ORDER)).cpu().numpy()
            assert same_bits(got, oracle.fixed_order(x, F16)), (n, tail)
            got = tcr.tcr_reduce_sum(t, tcr.Mode(tcr.SHUFFLE_TREE, block_threads=128)).cpu().numpy()
            assert same_bits(got, oracle.shuffle_tree(x, F16, *spec.shuffle_team(n, 128))), (n, tail)
