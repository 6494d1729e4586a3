// tcr_noalloc.cu -- tcr_reduce_sum_noalloc: the chunked sum without any
// device allocation.
//
// Who needs it: callers that must not allocate device memory while they
// run -- for instance code that works inside a fixed, pre-reserved memory
// budget (a long-running service that sized all of its device memory at
// start-up and treats any later cudaMalloc as a fault), code that runs while
// another component owns the device allocator, or a host thread with a
// hard deadline that cannot afford the allocator's occasional trip to the
// driver.  tcr_reduce_sum takes its partials from a stream-ordered pool;
// this entry point instead keeps them in one fixed array in device memory,
// reserved when the library's device code is loaded on a GPU.
//
// There is no counterpart on the pages: this is an interface choice of the
// library, not part of the reduction method.
//
// Behaviour a caller must know:
//  * The array holds kNoAllocMaxPartials floats (256 KiB) on every GPU that
//    loads the library, for as long as the process runs.
//  * The first call on each device, with that device current, looks up the
//    array's device address (cudaGetSymbolAddress) and makes the driver
//    load every kernel this entry point can launch (the runtime otherwise
//    loads each kernel at its first launch, and loading code reserves
//    device memory): after that first call no call loads anything.  Make
//    the first call before any stream capture.
//  * Every call on a device uses the same array, and it keeps whatever the
//    last call left there.  Nothing in it needs clearing: the reduction
//    kernel writes every partial slot the combine kernel then reads, in the
//    same call and on the same stream.  Calls whose work overlaps on the GPU
//    (two streams, or two host threads without ordering between them) race
//    on the array and give wrong results: order them on one stream or with
//    events.
//  * Only the chunked kernels are served (TCR_FIXED_ORDER with the plain
//    tree, TCR_MMA_CHAIN), with the work split of tcr_reduce_sum (one plan
//    function serves both), so the results are tcr_reduce_sum's bit for bit.
//    TCR_SHUFFLE_TREE, TCR_MMA_CHAIN_TMEM and a blocked order return
//    TCR_ERR_UNSUPPORTED; an n whose chunk count exceeds the array returns
//    TCR_ERR_UNSUPPORTED before any GPU work; malformed arguments return
//    TCR_ERR_INVALID_ARG exactly as for tcr_reduce_sum.
//  * No cudaMalloc, cudaFree or allocating library routine is called.
#include <cstdint>
#include <mutex>

#include "../../include/tcr.h"
#include "kernels.cuh"
#include "plan.h"

namespace {

using namespace tcr;
using namespace tcr::plan;

constexpr size_t kNoAllocMaxPartials = 65536;
constexpr int kMaxDevices = 64;

// the partials of a call; one copy per device that loads this module
static __device__ __align__(256) float g_noalloc_partials[kNoAllocMaxPartials];

struct NoAllocDevice {
    bool ready = false;
    float *partials = nullptr;   // device address of g_noalloc_partials
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kMaxDevices];

// Set-up, once per device, with that device current: the array's address,
// and every kernel variant this entry point launches loaded.
tcr_status noalloc_setup(int dev, float **partials)
{
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || p == nullptr ||
            preload_fixed_chunk_sums() != cudaSuccess || preload_mma_chunk_sums() != cudaSuccess ||
            preload_combine() != cudaSuccess) {
            (void)cudaGetLastError();
            return TCR_ERR_CUDA;
        }
        d.partials = (float *)p;
        d.ready = true;
    }
    *partials = d.partials;
    return TCR_OK;
}

}  // namespace

extern "C" tcr_status tcr_reduce_sum_noalloc(const void *x, size_t n, float *out, tcr_mode mode,
                                             void *stream)
{
    int block = 0, R = 0;
    tcr_status st = check_common(x, n, out, mode, &block, &R);
    if (st != TCR_OK) return st;
    if (mode.kind != TCR_FIXED_ORDER && mode.kind != TCR_MMA_CHAIN) return TCR_ERR_UNSUPPORTED;
    if (mode.run_log2 != 0) return TCR_ERR_UNSUPPORTED;     // the plain tree only

    // the split of tcr_reduce_sum for this mode (the CTA size is free for
    // FIXED_ORDER and for a default block size)
    const ChunkSplit c = chunk_split(1, n, mode.dtype, block,
                                     mode.kind == TCR_FIXED_ORDER || mode.block_threads == 0);
    if (c.cps > kNoAllocMaxPartials) return TCR_ERR_UNSUPPORTED;

    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return TCR_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (n == 0) return cudaMemsetAsync(out, 0, sizeof(float), s) == cudaSuccess ? TCR_OK : TCR_ERR_CUDA;

    float *partials = nullptr;
    st = noalloc_setup(dev, &partials);
    if (st != TCR_OK) return st;

    const bool aligned = ((uintptr_t)x & 15u) == 0;
    const bool fixed = mode.kind == TCR_FIXED_ORDER;
    const int grid = unit_grid(c.cps);      // one CTA per chunk, as tcr_reduce_sum launches
    float *dst = c.cps > 1 ? partials : out;
    cudaError_t e = fixed ? launch_fixed_chunk(mode.dtype, kOpSum, aligned, x, n, c.cps, c.cps,
                                               c.chunk_log2, dst, grid, c.block, s)
                          : launch_mma_chunk(mode.dtype, kOpSum, aligned, R, x, n, c.cps, c.cps,
                                             c.chunk_log2, dst, grid, c.block, s);
    if (e == cudaSuccess && c.cps > 1) e = launch_combine(partials, 1, c.cps, out, s);
    return e == cudaSuccess ? TCR_OK : TCR_ERR_CUDA;
}
