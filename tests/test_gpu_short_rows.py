"""GPU parity for short rows -- rows of at most 128 vectors (1024 16-bit or 512
binary32 inputs), which the library packs several to a warp group.

FIXED_ORDER and SHUFFLE_TREE: every row bit-exact to the oracle's emulation
of the declared order (the same as a single reduction of that row), for
every row width around each packing width, ragged row counts, both input
alignments, sums and sums of squares.  MMA_CHAIN: every row within
2^-20 * sum|x| + 1e-6 of the exact sum, at every chain length.
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


def within_mma_tolerance(got, exact, abs_sum):
    err = np.abs(np.asarray(got, np.float64) - np.asarray(exact))
    return bool(np.all(err <= spec.mma_tolerance(np.asarray(abs_sum))))


# row widths around every packing width (2^v vectors, v = 0..7) and past the last;
# widths of an odd number of 8-byte words (12, 36, ... for 16-bit inputs, 6, 50, ...
# for binary32) make every other row start 8 bytes into a granule: 8-byte loads;
# an odd number of 4-byte words (10, 50, ... 16-bit, every odd binary32 width):
# 4-byte loads
COLS16 = [1, 5, 8, 9, 10, 12, 16, 17, 31, 32, 33, 36, 50, 63, 64, 65, 100, 127, 128, 129, 130,
          132, 255, 256, 257, 383, 511, 512, 513, 514, 516, 777, 1000, 1020, 1022, 1023, 1024,
          1025]
COLS32 = [1, 3, 4, 5, 6, 8, 13, 16, 31, 32, 33, 50, 64, 100, 102, 128, 129, 255, 256, 257, 258,
          400, 510, 511, 512, 513]


def rows_for(cols, dtype):
    # several groups of packed rows and a ragged tail
    V = spec.vector_len(dtype)
    nvec = -(-cols // V)
    per_group = 256 // (1 << max(0, (nvec - 1).bit_length()))
    return 3 * per_group + 5


def rows_call(x, mode, squares=False):
    rows, cols = x.shape
    t = dev(x).view(rows, cols)
    f = tcr.tcr_reduce_rows_sum_squares if squares else tcr.tcr_reduce_rows
    return f(t, mode).cpu().numpy()


@pytest.mark.parametrize("dtype", [F16, BF16, F32])
def test_fixed_and_shuffle_bit_exact(dtype):
    for cols in (COLS32 if dtype == F32 else COLS16):
        rows = rows_for(cols, dtype)
        x = synth.generate(rows * cols, "normal", dtype, seed=cols).reshape(rows, cols)
        for squares in (False, True):
            got = rows_call(x, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype), squares)
            assert same_bits(got, oracle.fixed_order_rows(x, dtype, squares=squares)), (cols, squares)
            bt, g = spec.shuffle_team(cols, 0, dtype)
            got = rows_call(x, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype), squares)
            assert same_bits(got, oracle.shuffle_tree_rows(x, dtype, bt, g, squares=squares)), \
                (cols, squares)


@pytest.mark.parametrize("dtype", [F16, BF16, F32])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
def test_mma_chain_within_tolerance(dtype, R):
    for cols in (COLS32 if dtype == F32 else COLS16):
        rows = rows_for(cols, dtype)
        x = synth.generate(rows * cols, "uniform_pm1", dtype, seed=cols + R).reshape(rows, cols)
        e, a = oracle.exact_sum_rows(x, dtype)
        assert within_mma_tolerance(rows_call(x, tcr.Mode(tcr.MMA_CHAIN, R=R, dtype=dtype)), e, a), cols
        e2, _ = oracle.exact_sum_rows(x, dtype, squares=True)
        got = rows_call(x, tcr.Mode(tcr.MMA_CHAIN, R=R, dtype=dtype), squares=True)
        assert within_mma_tolerance(got, e2, e2), cols


@pytest.mark.parametrize("dtype", [F16, F32])
@pytest.mark.parametrize("offset", [1, 2, 3, 4, 7])
def test_misaligned_base_and_rows(dtype, offset):
    # a base `offset` inputs past a 16-byte boundary: rows start at every
    # offset in their granule; widths around each packing width, whole
    # vectors or not (a row gets one slot more than vectors); a base 8 bytes
    # past the boundary with rows of whole 8-byte words takes 8-byte loads
    for cols in ((7, 8, 12, 15, 31, 36, 63, 64, 100, 127, 249, 255, 256, 333, 516, 1001, 1017)
                 if dtype == F16 else (3, 4, 6, 7, 31, 32, 50, 100, 127, 255, 256, 258, 509)):
        rows = 777
        x = synth.generate(rows * cols + offset, "normal", dtype, seed=cols + offset)
        t = dev(x)[offset:].view(rows, cols)
        xs = x[offset:].reshape(rows, cols)
        got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)).cpu().numpy()
        assert same_bits(got, oracle.fixed_order_rows(xs, dtype)), cols
        got = tcr.tcr_reduce_rows_sum_squares(t, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype)).cpu().numpy()
        bt, g = spec.shuffle_team(cols, 0, dtype)
        assert same_bits(got, oracle.shuffle_tree_rows(xs, dtype, bt, g, squares=True)), cols
        e, a = oracle.exact_sum_rows(xs, dtype)
        for R in (1, 4):
            got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.MMA_CHAIN, R=R, dtype=dtype)).cpu().numpy()
            assert within_mma_tolerance(got, e, a), (cols, R)


def test_last_row_ends_the_allocation():
    # the matrix ends exactly at the end of its buffer, at every offset in
    # the last granule: the loads stay inside the data
    for cols in (5, 9, 100, 255):
        for tail in range(8):
            rows = 64 + tail
            x = synth.generate(rows * cols, "normal", F16, seed=cols * 8 + tail)
            buf = torch.empty(rows * cols + 8 - tail, dtype=torch.int16, device="cuda")
            buf[8 - tail:] = torch.from_numpy(x.view(np.int16)).cuda()
            t = buf[8 - tail:].view(rows, cols)
            got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.FIXED_ORDER)).cpu().numpy()
            assert same_bits(got, oracle.fixed_order_rows(x.reshape(rows, cols), F16)), (cols, tail)


@pytest.mark.parametrize("kind", [tcr.FIXED_ORDER, tcr.SHUFFLE_TREE])
@pytest.mark.parametrize("cols", [3, 40, 200, 700])
def test_rows_equal_single_reductions(kind, cols):
    # batch invariance: a row's bits do not depend on its neighbours or on
    # where it falls in a warp group
    rows = 301
    x = synth.generate(rows * cols, "normal", F16, seed=7 * cols).reshape(rows, cols)
    whole = rows_call(x, tcr.Mode(kind))
    for r in (0, 1, 37, 150, 300):
        single = tcr.tcr_reduce_sum(dev(x[r]), tcr.Mode(kind)).cpu().numpy()
        assert same_bits(whole[r], single), r
    part = rows_call(np.ascontiguousarray(x[37:44]), tcr.Mode(kind))
    assert same_bits(part, whole[37:44])


@pytest.mark.parametrize("cols", [8, 64, 300])
def test_non_finite_and_signed_zero_rows(cols):
    rows = 100
    x = synth.generate(rows * cols, "normal", F16, seed=cols).reshape(rows, cols)
    x[3, cols // 2] = 0x7C00                  # +inf
    x[4, 0] = 0xFC00                          # -inf
    x[5, 0], x[5, cols - 1] = 0x7C00, 0xFC00  # inf - inf
    x[6, cols - 1] = 0x7E00                   # NaN
    x[7, :] = 0x8000                          # every input -0.0
    for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN):
        got = rows_call(x, tcr.Mode(kind))
        assert got[3] == np.inf and got[4] == -np.inf
        assert np.isnan(got[5]) and np.isnan(got[6])
        fin = np.delete(got, [3, 4, 5, 6])
        assert np.all(np.isfinite(fin))
        if kind != tcr.MMA_CHAIN:
            # the ordered modes pad with -0.0, so a row of -0.0 sums to -0.0
            assert same_bits(got[7], np.float32(-0.0))
            assert same_bits(got, oracle.fixed_order_rows(x, F16) if kind == tcr.FIXED_ORDER else
                             oracle.shuffle_tree_rows(x, F16, *spec.shuffle_team(cols)))
        else:
            assert got[7] == 0.0


def test_descriptor_reports_one_launch_and_no_scratch():
    for cols, dtype in ((64, F16), (1024, F16), (512, F32)):
        for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN):
            d = tcr.tcr_order_descriptor(rows=1 << 20, cols=cols, mode=tcr.Mode(kind, dtype=dtype))
            assert d["launches"] == 1 and d["partials"] == 0 and d["launch_block"] == 256


# ---------------------------------------------------------------- row moments

def moments_call(t, mode, mean_var=False):
    f = tcr.tcr_reduce_rows_mean_var if mean_var else tcr.tcr_reduce_rows_moments
    a, b = f(t, mode)
    return a.cpu().numpy(), b.cpu().numpy()


@pytest.mark.parametrize("dtype", [F16, BF16, F32])
def test_moments_of_short_rows(dtype):
    # both sums bit-exact to the single-reduction orders, the mean and
    # variance to the oracle's binary32 formula on them; MMA_CHAIN within
    # the bound of each sum
    for cols in (COLS32 if dtype == F32 else COLS16):
        rows = rows_for(cols, dtype)
        x = synth.generate(rows * cols, "normal", dtype, seed=3 * cols).reshape(rows, cols)
        t = dev(x).view(rows, cols)
        f1, f2 = oracle.fixed_order_rows(x, dtype), oracle.fixed_order_rows(x, dtype, squares=True)
        s1, s2 = moments_call(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype))
        assert same_bits(s1, f1) and same_bits(s2, f2), cols
        m, v = moments_call(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype), mean_var=True)
        om, ov = oracle.mean_var(f1, f2, cols)
        assert same_bits(m, om) and same_bits(v, ov), cols
        bt, g = spec.shuffle_team(cols, 0, dtype)
        g1 = oracle.shuffle_tree_rows(x, dtype, bt, g)
        g2 = oracle.shuffle_tree_rows(x, dtype, bt, g, squares=True)
        s1, s2 = moments_call(t, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype))
        assert same_bits(s1, g1) and same_bits(s2, g2), cols
        e1, a1 = oracle.exact_sum_rows(x, dtype)
        e2, _ = oracle.exact_sum_rows(x, dtype, squares=True)
        for R in (1, 2, 4):
            s1, s2 = moments_call(t, tcr.Mode(tcr.MMA_CHAIN, R=R, dtype=dtype))
            assert within_mma_tolerance(s1, e1, a1) and within_mma_tolerance(s2, e2, e2), (cols, R)


@pytest.mark.parametrize("offset", [1, 4, 5])
def test_moments_of_misaligned_short_rows(offset):
    for cols in (7, 31, 36, 64, 100, 255, 516, 777):
        rows = 513
        x = synth.generate(rows * cols + offset, "normal", BF16, seed=cols + offset)
        t = dev(x)[offset:].view(rows, cols)
        xs = x[offset:].reshape(rows, cols)
        f1, f2 = oracle.fixed_order_rows(xs, BF16), oracle.fixed_order_rows(xs, BF16, squares=True)
        m, v = moments_call(t, tcr.Mode(tcr.FIXED_ORDER, dtype=BF16), mean_var=True)
        om, ov = oracle.mean_var(f1, f2, cols)
        assert same_bits(m, om) and same_bits(v, ov), cols
        e1, a1 = oracle.exact_sum_rows(xs, BF16)
        e2, _ = oracle.exact_sum_rows(xs, BF16, squares=True)
        s1, s2 = moments_call(t, tcr.Mode(tcr.MMA_CHAIN, dtype=BF16))
        assert within_mma_tolerance(s1, e1, a1) and within_mma_tolerance(s2, e2, e2), cols
        # the fused pass gives the single calls' bits
        for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN):
            s1, s2 = moments_call(t, tcr.Mode(kind, dtype=BF16))
            assert same_bits(s1, tcr.tcr_reduce_rows(t, tcr.Mode(kind, dtype=BF16)).cpu().numpy())
            assert same_bits(s2, tcr.tcr_reduce_rows_sum_squares(t, tcr.Mode(kind, dtype=BF16)).cpu().numpy())


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_every_16_bit_pattern_converts_exactly(dtype):
    # rows of one input: each row's value is that input's binary32 leaf, so
    # the GPU's conversion of all 65536 patterns is compared with the
    # oracle's decoder (itself pinned to numpy); squares give fl32(x * x)
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(-1, 1)
    leaves = oracle.leaves(bits.reshape(-1), dtype)
    for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        assert same_bits(rows_call(bits, tcr.Mode(kind, dtype=dtype)), leaves)
        with np.errstate(over="ignore", invalid="ignore"):
            sq = (leaves * leaves).astype(np.float32)
        assert same_bits(rows_call(bits, tcr.Mode(kind, dtype=dtype), squares=True), sq)
