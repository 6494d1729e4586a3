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

// Bytes per warp group of the stream kernels (log2): 8 warp loads of 512
// bytes (2048 16-bit inputs, 1024 binary32 inputs).
constexpr int kGroupBytesLog2 = 12;
// Bytes per warp of one CTA work unit (chunk) of the chunked kernels (log2):
// 2^14 = 4 groups (2^13 16-bit inputs, 2^12 binary32 inputs); inputs too
// small to give every SM two work units get shorter spans, down to one
// group.
constexpr int kWarpSpanBytesLog2 = 14;
// Longest row served by one warp, in bytes (8 groups: 16384 16-bit or 8192
// binary32 inputs); longer rows go through the chunked kernels
// (FIXED_ORDER, MMA_CHAIN) or the block team (SHUFFLE_TREE).
constexpr size_t kRowsWarpMaxBytes = 32768;
// CTA size of the one-warp-per-row kernels, and the CTAs per SM their
// register budget is set for (65536 / (256 * 3) -> up to 80 registers).
constexpr int kRowsBlock = 256;
constexpr int kRowsMinCtas = 3;

}  // namespace tcr
