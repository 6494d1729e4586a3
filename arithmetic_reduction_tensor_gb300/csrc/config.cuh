// config.cuh -- the work-split constants the kernels are compiled with.
//
// Kept apart from the launcher declarations (kernels.cuh): a change here
// changes kernel code, a change there does not.
#pragma once

#include <cstddef>

namespace tcr {

// Operations on the leaves: the sum of the inputs, or the sum of their
// squares (each square one binary32 multiplication, round to nearest, of an
// exact binary32 value -- exact for binary16 inputs).
constexpr int kOpSum = 0;
constexpr int kOpSquares = 1;

// Inputs per warp group of the tree kernels: 8 warp loads of 256 inputs.
constexpr size_t kGroup = 2048;
// Inputs per warp of one CTA work unit (chunk) of the chunked kernels.
constexpr int kWarpSpanLog2 = 13;
// Longest row served by one warp; longer rows go through the chunked
// kernels (FIXED_ORDER, MMA_CHAIN) or the block team (SHUFFLE_TREE).
constexpr size_t kRowsWarpMaxCols = 16384;
// CTA size of the one-warp-per-row kernels, and the CTAs per SM their
// register budget is set for (65536 / (256 * 3) -> up to 80 registers).
constexpr int kRowsBlock = 256;
constexpr int kRowsMinCtas = 3;

}  // namespace tcr
