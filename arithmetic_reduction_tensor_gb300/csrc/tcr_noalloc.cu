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
//  * The first call on each device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.
//  * Every call on a device uses the same array, and it keeps whatever the
//    last call left there.  Nothing in it needs clearing: the reduction
//    kernel writes every partial slot the combine kernel then reads, in the
//    same call and on the same stream.  Calls whose work overlaps on the GPU
//    (two streams, or two host threads without ordering between them) race
//    on the array and give wrong results: order them on one stream or with
//    events.
//  * Only the chunked kernels are served (TCR_FIXED_ORDER and TCR_MMA_CHAIN);
//    TCR_SHUFFLE_TREE returns TCR_ERR_UNSUPPORTED.  An n whose chunk count
//    exceeds the array returns TCR_ERR_UNSUPPORTED before any GPU work.
//  * No cudaMalloc, cudaFree or allocating library routine is called.
#include <cstdint>
#include <mutex>

#include "../../include/tcr.h"
#include "kernels.cuh"

namespace {

using namespace tcr;

constexpr size_t kNoAllocMaxPartials = 65536;
constexpr int kMaxDevices = 64;

// the partials of a call; one copy per device that loads this module
static __device__ __align__(256) float g_noalloc_partials[kNoAllocMaxPartials];

struct NoAllocDevice {
    bool ready = false;
    float *partials = nullptr;   // device address of g_noalloc_partials
    int sms = 0;
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kMaxDevices];

// Set-up, once per device, with that device current.
tcr_status noalloc_setup(int dev, NoAllocDevice *out)
{
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return TCR_ERR_CUDA;
        }
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0) {
            (void)cudaGetLastError();
            return TCR_ERR_CUDA;
        }
        d.partials = (float *)p;
        d.sms = sms;
        d.ready = true;
    }
    *out = d;
    return TCR_OK;
}

}  // namespace

extern "C" tcr_status tcr_reduce_sum_noalloc(const void *x, size_t n, float *out, tcr_mode mode,
                                             void *stream)
{
    if (!out || ((uintptr_t)out & 3u) != 0) return TCR_ERR_INVALID_ARG;
    if (n >= ((size_t)1 << 40)) return TCR_ERR_INVALID_ARG;
    if (mode.dtype != TCR_F16 && mode.dtype != TCR_BF16 && mode.dtype != TCR_F32)
        return TCR_ERR_INVALID_ARG;
    const int elem_log2 = mode.dtype == TCR_F32 ? 2 : 1;
    if (n > 0 && (!x || ((uintptr_t)x & ((1u << elem_log2) - 1u)) != 0)) return TCR_ERR_INVALID_ARG;
    if (mode.run_log2 < 0 || mode.run_log2 > 16) return TCR_ERR_INVALID_ARG;
    if (mode.run_log2 != 0) return TCR_ERR_UNSUPPORTED;     // the plain tree only
    const int block = mode.block_threads == 0 ? 256 : mode.block_threads;
    if (block < 32 || block > 1024 || (block & (block - 1)) != 0) return TCR_ERR_INVALID_ARG;
    int R = 0;
    if (mode.kind == TCR_MMA_CHAIN) {
        if (mode.R < 0 || mode.R > 8) return TCR_ERR_INVALID_ARG;
        R = mode.R != 0 ? mode.R : 4;    // the same default as tcr_reduce_sum
    } else if (mode.kind == TCR_SHUFFLE_TREE) {
        return TCR_ERR_UNSUPPORTED;
    } else if (mode.kind != TCR_FIXED_ORDER) {
        return TCR_ERR_INVALID_ARG;
    }

    // 2^kWarpSpanBytesLog2 bytes per warp, and the same choice of CTA size
    // and span for small inputs, as in the allocating entry point
    int block_used = block;
    int warps_log2 = 0;
    while ((32 << warps_log2) < block_used) warps_log2++;
    int span_log2 = kWarpSpanBytesLog2 - elem_log2;
    const int group_log2 = kGroupBytesLog2 - elem_log2;
    int chunk_log2 = span_log2 + warps_log2;
    size_t cps = (n + ((size_t)1 << chunk_log2) - 1) >> chunk_log2;
    const bool may_shrink = mode.kind == TCR_FIXED_ORDER || mode.block_threads == 0;
    const bool one_cta = may_shrink && n <= ((size_t)1 << (group_log2 + 1 + 5));
    if (one_cta) {
        // one CTA, as in the allocating entry point
        span_log2 = n > ((size_t)1 << (group_log2 + 5)) ? group_log2 + 1 : group_log2;
        block_used = 32;
        warps_log2 = 0;
        while (((size_t)block_used << (span_log2 - 5)) < n) {
            block_used *= 2;
            warps_log2++;
        }
        chunk_log2 = span_log2 + warps_log2;
        cps = 1;
    }
    while (may_shrink && !one_cta && cps < (size_t)2 * 152 && (block_used > 32 || span_log2 > group_log2)) {
        if (block_used > 32) {
            block_used /= 2;
            warps_log2--;
        } else {
            span_log2--;
        }
        chunk_log2 = span_log2 + warps_log2;
        cps = (n + ((size_t)1 << chunk_log2) - 1) >> chunk_log2;
    }
    if (cps > kNoAllocMaxPartials) return TCR_ERR_UNSUPPORTED;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return TCR_ERR_CUDA;
    }
    cudaStream_t s = (cudaStream_t)stream;
    if (n == 0) return cudaMemsetAsync(out, 0, sizeof(float), s) == cudaSuccess ? TCR_OK : TCR_ERR_CUDA;

    NoAllocDevice d;
    tcr_status st = noalloc_setup(dev, &d);
    if (st != TCR_OK) return st;

    const bool aligned = ((uintptr_t)x & 15u) == 0;
    int occ = mode.kind == TCR_FIXED_ORDER ? occupancy_fixed(false, mode.dtype, kOpSum, aligned, block_used)
                                           : occupancy_mma(false, mode.dtype, kOpSum, aligned, R, block_used);
    if (occ <= 0) occ = 1;
    const size_t resident = (size_t)d.sms * (size_t)occ;
    const int grid = (int)(cps < resident ? cps : resident);
    float *dst = cps > 1 ? d.partials : out;
    cudaError_t e = mode.kind == TCR_FIXED_ORDER
                        ? launch_fixed_chunk(mode.dtype, kOpSum, aligned, x, n, cps, cps,
                                             chunk_log2, dst, grid, block_used, s)
                        : launch_mma_chunk(mode.dtype, kOpSum, aligned, R, x, n, cps, cps,
                                           chunk_log2, dst, grid, block_used, s);
    if (e == cudaSuccess && cps > 1) e = launch_combine(d.partials, 1, cps, out, s);
    return e == cudaSuccess ? TCR_OK : TCR_ERR_CUDA;
}
