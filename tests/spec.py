"""The declared orders, restated for the tests from their specification.

The SHUFFLE_TREE order of a segment of L inputs at block size B is fixed by
its team (Bt threads per block, G blocks).  With V inputs per 16-byte vector
(8 for 16-bit inputs, 4 for binary32) and nvec = ceil(L / V) vectors: one
warp (Bt = 32, G = 1) when nvec <= 1024, otherwise Bt = B and
G = ceil(nvec / (B * 16)).  Written here from
that statement, not taken from the library, so that a test can check the
library's descriptor against it and feed the oracle with it.
"""
import math

DEFAULT_BLOCK = 256
F32 = 2


def vector_len(dtype: int = 0) -> int:
    return 4 if dtype == F32 else 8


def span_log2(dtype: int = 0) -> int:
    """log2 inputs of a 16 KiB warp span (the tree kernels' work per warp)."""
    return 12 if dtype == F32 else 13


def shuffle_team(L: int, block: int = 0, dtype: int = 0) -> tuple[int, int]:
    B = block or DEFAULT_BLOCK
    nvec = math.ceil(L / vector_len(dtype))
    if nvec <= 1024:
        return 32, 1
    g = math.ceil(nvec / (B * 16))
    return B, max(1, g)


def default_R(block: int = 0) -> int:
    """Default MMA chain length: 4 at every block size."""
    return 4


def mma_tolerance(abs_sum: float) -> float:
    """|gpu - exact| <= 2^-20 * sum|x_i| + 1e-6."""
    return 2.0 ** -20 * abs_sum + 1e-6


def gemm_splits(M: int, N: int, K: int, splits: int = 0) -> tuple[int, int]:
    """(effective S, k_split) of a split-K GEMM, from the rule stated in
    include/tcr.h: with T the 128 x 256 output tiles, S = 1 when T >= 152,
    else min(32, floor(152 / T)); a requested S is taken as given; either is
    limited to ceil(K / 64) boxes, split evenly in whole boxes."""
    tiles = math.ceil(M / 128) * math.ceil(N / 256)
    kboxes = math.ceil(K / 64)
    s = splits or (1 if tiles >= 152 else min(32, 152 // max(tiles, 1)))
    s = max(1, min(s, kboxes))
    kbps = math.ceil(kboxes / s) if kboxes else 1
    return (math.ceil(kboxes / kbps) if kboxes else 1), kbps * 64


def gemm_bound(k_split: int, S: int, abs_sum):
    """|C - exact| <= (2^-22 * k_split / 16 + 2^-24 * ceil(log2 S)) * sum|a w| + 1e-30."""
    return (2.0 ** -22 * k_split / 16 + 2.0 ** -24 * math.ceil(math.log2(S))) * abs_sum + 1e-30
