"""The declared orders, restated for the tests from their specification.

The SHUFFLE_TREE order of a segment of L inputs at block size B is fixed by
its team (Bt threads per block, G blocks).  With V inputs per 16-byte vector
(8 for 16-bit inputs, 4 for binary32) and nvec = ceil(L / V) vectors: one
warp (Bt = 32, G = 1) when nvec <= 1024, otherwise Bt = B and
G = ceil(nvec / (B * 16)) clamped to [1, 152 * 1024 / B].  Written here from
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
    return B, max(1, min(g, 152 * 1024 // B))


def default_R(block: int = 0) -> int:
    """Default MMA chain length: 4 at every block size."""
    return 4


def mma_tolerance(abs_sum: float) -> float:
    """|gpu - exact| <= 2^-20 * sum|x_i| + 1e-6."""
    return 2.0 ** -20 * abs_sum + 1e-6
