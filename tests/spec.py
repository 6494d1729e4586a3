"""The declared orders, restated for the tests from their specification.

The SHUFFLE_TREE order of a segment of L inputs at block size B is fixed by
its team (Bt threads per block, G blocks): one warp (Bt = 32, G = 1) when
L <= 8192, otherwise Bt = B and G = ceil(L / (8 * B * 16)) clamped to
[1, 152 * 1024 / B].  Written here from that statement, not taken from the
library, so that a test can check the library's descriptor against it and
feed the oracle with it.
"""
import math

DEFAULT_BLOCK = 256


def shuffle_team(L: int, block: int = 0) -> tuple[int, int]:
    B = block or DEFAULT_BLOCK
    if L <= 8192:
        return 32, 1
    g = math.ceil(L / (8 * B * 16))
    return B, max(1, min(g, 152 * 1024 // B))


def default_R(block: int = 0) -> int:
    """Default MMA chain length: 4 at every block size."""
    return 4


def mma_tolerance(abs_sum: float) -> float:
    """|gpu - exact| <= 2^-20 * sum|x_i| + 1e-6."""
    return 2.0 ** -20 * abs_sum + 1e-6
