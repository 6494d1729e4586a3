"""Tensor-core accumulation probe: what the MMA does with small addends.

The pages state only that chain sub-results are kept in fp32; how the
tensor core aligns and rounds the 16 products of a row plus the
accumulator is the hardware's.  These crafted single-tile inputs, run
through the public MMA_CHAIN call, put one 1.0 and fifteen 2^-24 in the
same A row (lane t of the first four holds inputs 8t, 8t+1, 8t+4, 8t+5 in
row 0), so the observed sum tells the behaviours apart:

  1.0                  each small addend truncated away after alignment
  1 + 7 * 2^-23        exact row sum, then rounded toward zero
  1 + 2^-20            exact row sum, then rounded to nearest even

The tests assert the stated error bound only; the observed values are
printed (pytest -s) and recorded in the design notes.
"""
import numpy as np
import pytest

import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300.build import build_library

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROW0 = [8 * t + k for t in range(4) for k in (0, 1, 4, 5)]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


def bits_of(value, dtype):
    if dtype == tcr.F16:
        return int(np.float16(value).view(np.uint16))
    return int(np.float32(value).view(np.uint32) >> 16)


def run(x_bits, kind, R, dtype):
    t = torch.from_numpy(np.asarray(x_bits, np.uint16).view(np.int16)).cuda()
    return float(tcr.tcr_reduce_sum(t, tcr.Mode(kind, R=R, dtype=dtype)).item())


@pytest.mark.parametrize("dtype", [tcr.F16, tcr.BF16])
@pytest.mark.parametrize("kind", [tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM])
def test_small_addends_in_one_row(dtype, kind):
    n = 256 if kind == tcr.MMA_CHAIN else 2048
    x = np.zeros(n, np.uint16)
    x[ROW0[0]] = bits_of(1.0, dtype)
    for i in ROW0[1:]:
        x[i] = bits_of(2.0 ** -24, dtype)
    got = run(x, kind, 1, dtype)
    exact = 1.0 + 15 * 2.0 ** -24
    labels = {1.0: "addends truncated after alignment", 1 + 7 * 2.0 ** -23: "exact, then toward zero",
              1 + 2.0 ** -20: "exact, then nearest even"}
    print(f"\n{tcr.KIND_NAMES[kind]} {'f16' if dtype == tcr.F16 else 'bf16'}: "
          f"1 + 15*2^-24 -> {got!r} ({labels.get(got, 'other')})")
    assert abs(got - exact) <= 2.0 ** -20 * exact + 1e-6


@pytest.mark.parametrize("dtype", [tcr.F16, tcr.BF16])
def test_chain_accumulator_keeps_small_sums(dtype):
    # two MMAs in one chain: the first leaves D = 1.0 in row 0, the second
    # adds fifteen 2^-24 to it through the accumulator input
    x = np.zeros(512, np.uint16)
    x[ROW0[0]] = bits_of(1.0, dtype)
    for i in ROW0[1:]:
        x[256 + i] = bits_of(2.0 ** -24, dtype)
    got = run(x, tcr.MMA_CHAIN, 2, dtype)
    print(f"\nMMA_CHAIN R=2 {'f16' if dtype == tcr.F16 else 'bf16'}: "
          f"1.0 then + 15*2^-24 in the chain -> {got!r}")
    exact = 1.0 + 15 * 2.0 ** -24
    assert abs(got - exact) <= 2.0 ** -20 * exact + 1e-6
