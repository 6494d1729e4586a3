// k_probe.cu -- the read ceiling of this GPU: a kernel that only streams its
// input in, with the same 16-byte streaming loads as the reduction kernels
// and no arithmetic beyond an XOR per word (so the loads cannot be dropped).
//
// Not part of the reduction method: a measurement of what any read-only
// kernel can reach, beside the copy bandwidth (read + write) that is the
// usual HBM figure.  A reduction reads every byte once and writes almost
// nothing, so this is the ceiling it is held against.
#include "../../include/tcr.h"
#include "common.cuh"

namespace tcr {
namespace {

// Thread t of the grid reads vectors t, t + T, t + 2T, ... (T = all
// threads), eight in flight before any is used, and XORs their words.
__global__ void __launch_bounds__(1024)
read_probe_kernel(const uint4 *__restrict__ x, size_t nvec, unsigned int *__restrict__ out)
{
    const size_t T = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 7 * T < nvec; i += 8 * T) {
        uint4 v[8];
#pragma unroll
        for (int k = 0; k < 8; k++) v[k] = ld_stream(x + i + k * T);
#pragma unroll
        for (int k = 0; k < 8; k++) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
    }
    for (; i < nvec; i += T) {
        const uint4 v = ld_stream(x + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc ^= __shfl_xor_sync(kFull, acc, off);
    if ((threadIdx.x & 31) == 0 && acc != 0) atomicXor(out, acc);
}

// One CTA per chunk of 8 x blockDim.x vectors: thread t reads vectors
// chunk + t + k * blockDim.x (k = 0..7), all eight in flight, then the CTA
// exits and the block scheduler starts the next chunk on whichever SM has
// room -- the launch shape of the reduction kernels.
__global__ void __launch_bounds__(1024)
read_probe_chunk_kernel(const uint4 *__restrict__ x, size_t nvec, unsigned int *__restrict__ out)
{
    const size_t base = (size_t)blockIdx.x * 8 * blockDim.x + threadIdx.x;
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const size_t i = base + (size_t)k * blockDim.x;
        v[k] = i < nvec ? ld_stream(x + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t acc = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc ^= __shfl_xor_sync(kFull, acc, off);
    if ((threadIdx.x & 31) == 0 && acc != 0) atomicXor(out, acc);
}

}  // namespace
}  // namespace tcr

extern "C" tcr_status tcr_read_probe(const void *x, size_t bytes, unsigned int *out, int ctas_per_sm,
                                     int block_threads, void *stream)
{
    if (!out || ((uintptr_t)out & 3u) != 0) return TCR_ERR_INVALID_ARG;
    if ((bytes & 15u) != 0 || (bytes > 0 && (!x || ((uintptr_t)x & 15u) != 0)))
        return TCR_ERR_INVALID_ARG;
    const int block = block_threads == 0 ? 512 : block_threads;
    if (block < 32 || block > 1024 || (block & (block - 1)) != 0) return TCR_ERR_INVALID_ARG;
    if (ctas_per_sm < -1 || ctas_per_sm > 64) return TCR_ERR_INVALID_ARG;
    int dev = -1, sms = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, tcr::read_probe_kernel, block, 0) !=
            cudaSuccess) {
        (void)cudaGetLastError();
        return TCR_ERR_CUDA;
    }
    int per_sm = ctas_per_sm == 0 ? occ : ctas_per_sm;
    if (per_sm > occ) per_sm = occ;
    if (per_sm < 1) per_sm = 1;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(out, 0, sizeof(unsigned int), s) != cudaSuccess) return TCR_ERR_CUDA;
    if (bytes == 0) return TCR_OK;
    const uint4 *xv = (const uint4 *)x;
    size_t nvec = bytes / 16;
    void *args[] = {(void *)&xv, (void *)&nvec, (void *)&out};
    if (ctas_per_sm == -1) {
        const size_t chunk = (size_t)8 * (size_t)block;
        const size_t ctas = (nvec + chunk - 1) / chunk;
        if (ctas > 0x7fffffffu) return TCR_ERR_INVALID_ARG;
        return cudaLaunchKernel((const void *)tcr::read_probe_chunk_kernel, dim3((unsigned)ctas), dim3(block),
                                args, 0, s) == cudaSuccess
                   ? TCR_OK
                   : TCR_ERR_CUDA;
    }
    return cudaLaunchKernel((const void *)tcr::read_probe_kernel, dim3(sms * per_sm), dim3(block), args, 0,
                            s) == cudaSuccess
               ? TCR_OK
               : TCR_ERR_CUDA;
}
