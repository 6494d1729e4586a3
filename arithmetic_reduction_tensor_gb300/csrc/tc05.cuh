// tc05.cuh -- fifth-generation tensor-core helpers shared by the tcgen05
// kernels: mbarrier waits with a time limit, bulk and tensor-map copies,
// shared-memory matrix descriptors, tcgen05 MMA / commit / load wrappers, and
// the host-side shared-memory opt-in and tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"

namespace tcr {

constexpr uint64_t kWaitLimitNs = 1000000000ull;    // about one second

// ---------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of parity `parity` of `bar` to complete, giving up
// after about a second (or soon after another role gave up); giving up sets
// `abort` for the CTA's other roles and bit 0 of the device fault word.
__device__ __forceinline__ bool mbar_wait_f(uint32_t bar, uint32_t parity, volatile uint32_t *abort,
                                            unsigned int *fault)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; i++) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0u) {
            if (*abort) return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                *abort = 1u;
                atomicOr(fault, 1u);
                return false;
            }
        }
    }
}

// One bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global memory into this CTA's shared memory, completing on
// mbarrier `bar`.  The inputs are read once, so the copy carries an L2
// evict-first policy: L2 drops its lines ahead of lines that other data
// (partials, outputs) may still need.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar)
{
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, no swizzle, K-major: 8-row x 16-byte
// core matrices; lbo = byte step between core matrices along K, sbo = byte
// step between 8-row groups; bits 46..48 hold the fixed value 0b001.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3fffu) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16, M = 128: D fp32 (bits 4-5 = 1), A
// and B binary16 (0) or bfloat16 (1) in bits 7-9 and 10-12, both K-major,
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
template <int DT, uint32_t N>
__device__ __forceinline__ uint32_t instr_desc_n()
{
    constexpr uint32_t ab = DT == kF16 ? 0u : 1u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((N >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar)
                 : "memory");
}

// Column 0 of the n D buffers b0, b0 + 1, ... (mod 8; buffer b at columns
// `base + stride * b`) for the calling thread's TMEM lane, n <= 8, the loads
// issued together and waited for once; v[i] for i >= n is left unchanged.
// Warp-collective: b0 and n must be the same in every lane.
__device__ __forceinline__ void tc_ld_chain_cols(uint32_t base, uint32_t stride, int b0, int n,
                                                 uint32_t (&v)[8])
{
#pragma unroll
    for (int i = 0; i < 8; i++)
        if (i < n)
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                         : "=r"(v[i])
                         : "r"(base + stride * (uint32_t)((b0 + i) & 7))
                         : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                   "+r"(v[7])
                 :
                 : "memory");
}

__device__ __forceinline__ float tc_ld_lane(uint32_t taddr)
{
    uint32_t v;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr) : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    return __uint_as_float(v);
}

// Cluster launch control (sm_100 and later): ask the hardware to cancel the
// launch of a CTA of this grid that has not started yet, so that the asking
// CTA runs that CTA's work instead.  The 16-byte response lands in shared
// memory at `resp` (16-byte aligned) and completes 16 transaction bytes on
// `bar`.  Once a response has said that nothing was cancelled, the CTA must
// not ask again.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar)
{
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];"
        ::"r"(resp), "r"(bar)
        : "memory");
}

// Read a completed response: true and the cancelled CTA's x index, or false
// when no CTA was left to cancel.
__device__ __forceinline__ bool clc_query(uint32_t resp, uint32_t *ctaid_x)
{
    uint32_t ok, x;
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b128 c;\n\t"
        "ld.shared.b128 c, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, c;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "mov.u32 %1, 0;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, c;\n\t"
        "}"
        : "=r"(ok), "=r"(x)
        : "r"(resp)
        : "memory");
    *ctaid_x = x;
    return ok != 0;
}

// Wait for a phase with a time limit and no abort flag (drain paths).
__device__ __forceinline__ bool mbar_wait_limited(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// SWIZZLE_128B K-major descriptor: 8-row groups 1024 bytes apart (the
// leading-dimension field is not used by this layout), swizzle code 2 in
// bits 61..63; the atom base is 1024-byte aligned, so the base offset is 0.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr)
{
    return (uint64_t)((addr >> 4) & 0x3fffu) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------- host

// The shared-memory opt-in (and, where given, the preferred shared-memory
// carveout, in percent of the maximum) are per-kernel attributes: set them
// once per device and kernel instance.
inline cudaError_t set_smem_once(void *k, int bytes, int carveout_percent = -1)
{
    static std::mutex mu;
    static std::vector<std::pair<int, void *>> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
    std::lock_guard<std::mutex> lk(mu);
    for (auto &d : done)
        if (d.first == dev && d.second == k) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && carveout_percent >= 0)
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, carveout_percent);
    if (e == cudaSuccess) done.emplace_back(dev, k);
    return e;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library does not link the driver library itself.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
        else
            (void)cudaGetLastError();
    });
    return fn;
}

}  // namespace tcr
