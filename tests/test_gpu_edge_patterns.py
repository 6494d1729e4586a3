"""The ordered modes on bit patterns from the whole range of the 16-bit formats.

FIXED_ORDER, SHUFFLE_TREE and the blocked order must equal the oracle's
emulation of their declared order bit for bit ("Taming Bitwise Behavior in
GPU Kernels with Tensor Core", Abstract: partial-sum precision and where
rounding happens decide the bits).  The synthetic workloads keep every
partial well inside binary32's range; these inputs do not: random finite
patterns of any exponent (binary16 and bfloat16 subnormals, down to
bfloat16's 2^-133), binary16's largest values +-65504, and bfloat16
magnitudes near 2^127 whose partial sums overflow binary32 to +-inf (and
+inf + -inf to NaN) part way up the tree.  Every path of the kernels is
covered: chunked sums with a combine, one CTA, packed short rows, one warp
per row, long rows through the chunked kernels, and misaligned bases.
NaN results are compared as a class (payloads are not claimed).
"""
import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300.build import build_library
from tests import spec
from tests.test_oracle import random_finite, special_patterns

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F16, BF16 = tcr.F16, tcr.BF16


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


def same_bits(a, b):
    a = np.asarray(a, np.float32).reshape(-1)
    b = np.asarray(b, np.float32).reshape(-1)
    nan = np.isnan(a) & np.isnan(b)
    return np.array_equal(a.view(np.uint32)[~nan], b.view(np.uint32)[~nan]) and \
        np.array_equal(np.isnan(a), np.isnan(b))


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def edge_inputs(n, dtype, seed, kind):
    """kind 'random': random finite patterns with the format's edge patterns
    sprinkled in; 'wide': the same with bfloat16 exponents capped at 2^100, so
    that sums of up to 2^22 inputs stay finite while spanning 2^-133 to 2^100
    (binary16 sums are always finite: 'wide' is 'random' there); 'huge': the
    largest finite magnitudes of both signs (sums overflow binary32 for
    bfloat16; for binary16 they stay finite);
    'tiny': subnormals and the smallest normals of both signs."""
    rng = np.random.default_rng(seed)
    if kind in ("random", "wide"):
        x = random_finite(rng, n, dtype)
        sp = np.array(special_patterns(dtype), np.uint16)
        pos = rng.integers(0, n, max(1, n // 64))
        x[pos] = sp[rng.integers(0, sp.size, pos.size)]
        if kind == "wide" and dtype == BF16:
            e = (x >> np.uint16(7)) & np.uint16(0xFF)
            x = (x & np.uint16(0x807F)) | ((e % np.uint16(228)) << np.uint16(7))
        return x
    if kind == "huge":
        top = 0x7BFF if dtype == F16 else 0x7F7F
        mags = np.arange(top - 15, top + 1, dtype=np.uint16)
    else:
        top = 0x03FF if dtype == F16 else 0x007F
        mags = np.concatenate([np.arange(1, top + 1, dtype=np.uint16),
                               np.array([top + 1, top + 2], np.uint16)])
    x = mags[rng.integers(0, mags.size, n)]
    # mostly positive, so that the bfloat16 sums run into +inf before a -inf meets them
    neg = rng.random(n) < 0.3
    return (x | (neg.astype(np.uint16) << np.uint16(15))).astype(np.uint16)


SUM_SIZES = [9, 2049, 65537, (1 << 20) + 13, (1 << 22) + 5]
KINDS = ["random", "wide", "huge", "tiny"]


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", SUM_SIZES)
def test_sums(dtype, kind, n):
    x = edge_inputs(n, dtype, seed=n + 7 * dtype, kind=kind)
    t = to_dev(x)
    for lo in (0, 1):                    # aligned, and a base 2 bytes past a boundary
        xs, ts = x[lo:], t[lo:]
        m = tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)
        assert same_bits(tcr.tcr_reduce_sum(ts, m).cpu().numpy(), oracle.fixed_order(xs, dtype)), lo
        m = tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype)
        ref = oracle.shuffle_tree(xs, dtype, *spec.shuffle_team(xs.size))
        assert same_bits(tcr.tcr_reduce_sum(ts, m).cpu().numpy(), ref), lo
    for c in (2, 3, 5, 8):
        m = tcr.Mode(tcr.FIXED_ORDER, dtype=dtype, run_log2=c)
        assert same_bits(tcr.tcr_reduce_sum(t, m).cpu().numpy(), oracle.blocked_order(x, dtype, c)), c


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("kind", KINDS)
def test_sums_of_squares(dtype, kind):
    n = (1 << 20) + 13
    x = edge_inputs(n, dtype, seed=99 + dtype, kind=kind)
    t = to_dev(x)
    got = tcr.tcr_reduce_sum_squares(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)).cpu().numpy()
    assert same_bits(got, oracle.fixed_order_sq(x, dtype))
    got = tcr.tcr_reduce_sum_squares(t, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype)).cpu().numpy()
    assert same_bits(got, oracle.shuffle_tree_sq(x, dtype, *spec.shuffle_team(n)))


# packed short rows (aligned 64, unaligned 100, 8-byte rows of 36), one warp
# per row (4096), long rows through the chunked kernels (40000)
@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("cols", [36, 64, 100, 4096, 40000])
def test_rows(dtype, kind, cols):
    rows = max(5, (1 << 22) // cols)
    x = edge_inputs(rows * cols, dtype, seed=cols + 3 * dtype, kind=kind).reshape(rows, cols)
    t = to_dev(x.reshape(-1)).view(rows, cols)
    got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)).cpu().numpy()
    assert same_bits(got, oracle.fixed_order_rows(x, dtype))
    got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype)).cpu().numpy()
    assert same_bits(got, oracle.shuffle_tree_rows(x, dtype, *spec.shuffle_team(cols)))
    got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype, run_log2=5)).cpu().numpy()
    assert same_bits(got, oracle.blocked_order_rows(x, dtype, 5))
    # every row misaligned: a base one input past the matrix's start
    xm = x.reshape(-1)[1:1 + (rows - 1) * cols].reshape(rows - 1, cols)
    tm = t.view(-1)[1:1 + (rows - 1) * cols].view(rows - 1, cols)
    got = tcr.tcr_reduce_rows(tm, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)).cpu().numpy()
    assert same_bits(got, oracle.fixed_order_rows(xm, dtype))
    got = tcr.tcr_reduce_rows(tm, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype)).cpu().numpy()
    assert same_bits(got, oracle.shuffle_tree_rows(xm, dtype, *spec.shuffle_team(cols)))


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_overflow_shapes(dtype):
    # binary16: 2^22 + 5 inputs of +65504 sum to about 2.7e11, finite in
    # binary32.  bfloat16: +max in the first half and -max in the second
    # overflow to +inf and -inf in the two halves of the tree, which meet at
    # the root as NaN; +max alone overflows to +inf.
    n = (1 << 22) + 5
    top = 0x7BFF if dtype == F16 else 0x7F7F
    cases = [np.full(n, top, np.uint16)]
    half = np.full(n, top, np.uint16)
    half[n // 2:] |= np.uint16(0x8000)
    cases.append(half)
    for x in cases:
        t = to_dev(x)
        got = tcr.tcr_reduce_sum(t, tcr.Mode(tcr.FIXED_ORDER, dtype=dtype)).cpu().numpy()
        ref = oracle.fixed_order(x, dtype)
        assert same_bits(got, ref)
        got = tcr.tcr_reduce_sum(t, tcr.Mode(tcr.SHUFFLE_TREE, dtype=dtype)).cpu().numpy()
        assert same_bits(got, oracle.shuffle_tree(x, dtype, *spec.shuffle_team(n)))
    if dtype == BF16:
        assert np.isposinf(oracle.fixed_order(cases[0], dtype))
        assert np.isnan(oracle.fixed_order(cases[1], dtype))
