// plan.h -- host-side planning shared by the entry points of tcr_api.cu and
// tcr_noalloc.cu: argument checks, device queries and the work split of the
// chunked sum kernels.  One definition of each, in tcr_api.cu, so that the
// two entry points of the 1-D sum cut the same input into the same chunks
// (and so return the same bits).
#pragma once

#include <cstddef>

#include "../../include/tcr.h"
#include "config.cuh"

namespace tcr {
namespace plan {

// Largest input count of a call (exclusive).
constexpr size_t kMaxInputs = (size_t)1 << 40;
// Longest run of the blocked order (log2 inputs).
constexpr int kMaxRunLog2 = 16;
constexpr int kDefaultBlock = 256;
// GB300: 152 SMs.  Used only by the declared SHUFFLE_TREE team rule and the
// small-input split rule (so both are the same on every device), and as the
// launch-plan SM count when no device can be queried.
constexpr int kRuleSMs = 152;

// Kernel families of the occupancy cache.
enum Family { kPackedF };

// The current device, or -1 (the CUDA error is cleared).
int current_device();
// SMs of `dev` (kRuleSMs when it cannot be queried); cached per device.
int sm_count(int dev);
// Resident CTAs per SM of a kernel variant at a block size; cached per
// (device, variant, block size), so only a variant's first use queries the
// runtime.  At least 1.
int occupancy(int dev, Family fam, bool rows, int dtype, int op, bool aligned, int R, int block);

int log2_exact(int v);
size_t elem_bytes(int dtype);
int vector_len(int dtype);

// Mode fields: kind, dtype, run_log2 (FIXED_ORDER only), block size (0:
// the default 256; else a power of two in 32..1024), R (chain kinds: 0 the
// default 4, else 1..8).  TCR_ERR_INVALID_ARG on any bad field.
tcr_status check_mode(const tcr_mode &m, int *block, int *R);
// check_mode plus out (non-null, 4-byte aligned), the input count (below
// kMaxInputs) and x (non-null and aligned to its element when total > 0).
tcr_status check_common(const void *x, size_t total, const float *out, const tcr_mode &mode,
                        int *block, int *R);

// The work split of the chunked kernels (FIXED_ORDER and MMA_CHAIN) over
// `segments` segments of seg_len inputs at a requested block size.
struct ChunkSplit {
    int block;        // CTA size used
    int chunk_log2;   // log2 inputs per CTA work unit
    size_t cps;       // chunks per segment
};
ChunkSplit chunk_split(size_t segments, size_t seg_len, int dtype, int block, bool may_shrink);

// The grid of a warp-stream kernel launched with one CTA per work unit
// (CTAs walk the units grid-stride, so a grid clamped to the launch limit
// still covers them all).
inline int unit_grid(size_t units)
{
    return (int)(units < (size_t)0x7fffffff ? units : (size_t)0x7fffffff);
}

}  // namespace plan
}  // namespace tcr
