// k_gemm.cu -- split-K GEMM with a declared, bit-reproducible K-partition
// combine.
//
// "Taming Bitwise Behavior in GPU Kernels with Tensor Core" (arXiv
// 2609.11356), Abstract: reduction order is the primary cause of bitwise
// differences, and a descriptor of reduction order -- for GEMM including the
// split-K partitioning of K -- pins it down.  Here C = A * W^T (A: M x K, W:
// N x K, both row-major 16-bit, C: M x N binary32) with K cut into S splits
// of k_split columns (a multiple of 64; the last split shorter):
//
//   P_s = the tensor core's sum over split s (one chain of tcgen05 MMAs,
//         K = 16 each, accumulating in one fp32 TMEM tile), s = 0 .. S-1;
//   C   = the balanced binary32 tree over P_0 .. P_{S-1} in split order
//         (-0.0 pad), formed by a second kernel -- never by atomics, so C
//         does not depend on which CTA finished first.
//
// A work unit is one 128 x 256 output tile of one split; units are ordered
// in groups of 8 tile rows (tile column outermost within a group) so that
// the CTAs in flight share A and W tiles through L2 -- the order of units
// never changes a result.  CTA roles (192 threads, one persistent CTA per
// SM), as in the tcgen05 reduction kernels:
//   warp 0, lane 0   producer: per stage a 64-column x 128-row box of A and
//                    a 64-column x 256-row box of W (2-D tensor maps,
//                    128-byte swizzle: the SWIZZLE_128B K-major operand
//                    layout) into a 4-stage shared-memory ring, completion
//                    by transaction count;
//   warp 1           owns the TMEM allocation (two 256-column fp32 tiles, all
//                    512 columns); lane 0 issues
//                    tcgen05.mma.cta_group::1.kind::f16 with M = 128,
//                    N = 256 -- four per stage, the k-th slice 32 bytes
//                    further in both operands -- and commits a stage when
//                    its MMAs are done and a tile when the split is;
//   warps 2..5       epilogue: thread m reads row m of the tile from TMEM
//                    (tcgen05.ld 32x32b, 32 columns at a time) and stores it
//                    to P_s (or straight to C when S = 1).
// Every mbarrier wait gives up after about a second, raises g_gemm_fault,
// drains its own copies and MMAs, frees TMEM and writes NaN to its tiles.
#include <cstdlib>
#include <cstring>

#include "kernels.cuh"
#include "tc05.cuh"

namespace tcr {

constexpr int kGmBM = 128;                       // tile rows (TMEM lanes)
constexpr int kGmBN = 256;                       // tile columns (MMA N, the most for M = 128)
constexpr int kGmBK = 64;                        // K per box: one 128-byte swizzle row
constexpr int kGmABoxBytes = kGmBM * kGmBK * 2;  // 16 KiB
constexpr int kGmWBoxBytes = kGmBN * kGmBK * 2;  // 32 KiB
constexpr int kGmStageBytes = kGmABoxBytes + kGmWBoxBytes;   // 48 KiB
constexpr int kGmStages = 4;                     // 192 KiB ring
constexpr int kGmDBuffers = 2;
constexpr uint32_t kGmTmemCols = kGmDBuffers * kGmBN;     // 512: all of TMEM
constexpr int kGmGroupM = 8;                     // tile rows per raster group (L2 reuse)
constexpr int kGmThreads = 192;
constexpr int kGmEpilogueThreads = 128;
constexpr int kGmOffBars = kGmStages * kGmStageBytes;
// barriers: full[S], empty[S], dfull[D], dempty[D], drain
constexpr int kGmNumBars = 2 * kGmStages + 2 * kGmDBuffers + 1;
constexpr int kGmOffMisc = kGmOffBars + 8 * kGmNumBars;
constexpr int kGmSmemBytes = kGmOffMisc + 64 + 1024;   // + alignment slack

__device__ unsigned int g_gemm_fault;

__device__ __forceinline__ bool gm_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort)
{
    return mbar_wait_f(bar, parity, abort, &g_gemm_fault);
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_ld_row32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
}

struct GemmArgs {
    size_t M, N;
    int kboxes;            // 64-column boxes of K
    int kbps;              // boxes per split
    int splits;            // S
    int tiles_m, tiles_n;
    size_t units;          // tiles_m * tiles_n * splits
    float *out;            // C when splits == 1, else P (splits x M x N)
    uint32_t inject_stall; // withhold the first tile's publication (tests of the failure path)
};

template <int DT>
__global__ void __launch_bounds__(kGmThreads, 1)
gemm_splitk_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmw,
                   const GemmArgs g)
{
    pdl_launch_dependents();   // the combine may launch now; it waits for this grid to finish
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t ring = sbase;
    const uint32_t bars = sbase + kGmOffBars;
    auto full_bar = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bars + 8u * (uint32_t)(kGmStages + s); };
    auto dfull_bar = [&](int b) { return bars + 8u * (uint32_t)(2 * kGmStages + b); };
    auto dempty_bar = [&](int b) { return bars + 8u * (uint32_t)(2 * kGmStages + kGmDBuffers + b); };
    const uint32_t drain_bar = bars + 8u * (uint32_t)(2 * kGmStages + 2 * kGmDBuffers);
    uint32_t *misc = (uint32_t *)(smem + kGmOffMisc);
    volatile uint32_t *tmem_holder = misc;
    volatile uint32_t *abort = misc + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // unit u = (split s, tile t); tiles in groups of kGmGroupM tile rows,
    // the tile row fastest within a group
    auto decode = [&](size_t u, int &s, int &tm, int &tn) {
        const size_t tiles = (size_t)g.tiles_m * (size_t)g.tiles_n;
        s = (int)(u / tiles);
        const size_t t = u - (size_t)s * tiles;
        const size_t group = (size_t)kGmGroupM * (size_t)g.tiles_n;
        const size_t first = (t / group) * kGmGroupM;
        const size_t in_group = (size_t)g.tiles_m - first < (size_t)kGmGroupM ? (size_t)g.tiles_m - first
                                                                             : (size_t)kGmGroupM;
        const size_t r = t % group;
        tm = (int)(first + r % in_group);
        tn = (int)(r / in_group);
    };
    auto split_boxes = [&](int s) {
        const int b0 = s * g.kbps;
        return min(g.kbps, g.kboxes - b0);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGmStages; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < kGmDBuffers; b++) {
            mbar_init(dfull_bar(b), 1);
            mbar_init(dempty_bar(b), kGmEpilogueThreads);
        }
        mbar_init(drain_bar, 1);
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tma) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmw) : "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr((const void *)tmem_holder)), "r"(kGmTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // the set-up above ran beside the stream's previous kernel; global
    // memory is touched only after it has finished
    pdl_wait_primary();

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            int st = 0;
            uint32_t phase = 0;
            bool armed[kGmStages];
            uint32_t armed_phase[kGmStages];
            for (int i = 0; i < kGmStages; i++) {
                armed[i] = false;
                armed_phase[i] = 0;
            }
            for (size_t u = blockIdx.x; u < g.units && !*abort; u += gridDim.x) {
                int s, tm, tn;
                decode(u, s, tm, tn);
                const int nb = split_boxes(s);
                bool ok = true;
                for (int j = 0; j < nb; j++) {
                    if (!gm_wait(empty_bar(st), phase ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = ring + (uint32_t)st * kGmStageBytes;
                    const int kc = (s * g.kbps + j) * kGmBK;      // a multiple of 64 columns
                    mbar_arrive_expect_tx(full_bar(st), (uint32_t)kGmStageBytes);
                    tma_load_2d(dst, &tma, kc, tm * kGmBM, full_bar(st));
                    tma_load_2d(dst + kGmABoxBytes, &tmw, kc, tn * kGmBN, full_bar(st));
                    armed[st] = true;
                    armed_phase[st] = phase;
                    if (++st == kGmStages) {
                        st = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            if (*abort) {
                for (int i = 0; i < kGmStages; i++) {
                    if (!armed[i]) continue;
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(full_bar(i), armed_phase[i]) &&
                           global_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = instr_desc_n<DT, (uint32_t)kGmBN>();
            const uint64_t ring_desc = smem_desc_sw128(ring);
            constexpr uint64_t kKStep = 32u >> 4;                       // 16 columns = 32 bytes
            constexpr uint64_t kBoxStep = (uint64_t)kGmABoxBytes >> 4;
            constexpr uint64_t kStageStep = (uint64_t)kGmStageBytes >> 4;
            int st = 0, b = 0;
            uint32_t phase = 0, dphase = 0;
            bool withhold = g.inject_stall != 0u;
            for (size_t u = blockIdx.x; u < g.units && !*abort; u += gridDim.x) {
                int s, tm, tn;
                decode(u, s, tm, tn);
                const int nb = split_boxes(s);
                if (!gm_wait(dempty_bar(b), ((dphase >> b) & 1u) ^ 1u, abort)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)b * kGmBN;
                bool ok = true;
                for (int j = 0; j < nb; j++) {
                    if (!gm_wait(full_bar(st), phase, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = ring_desc + (uint64_t)st * kStageStep;
                    const uint64_t w_desc = a_desc + kBoxStep;
#pragma unroll
                    for (int k = 0; k < 4; k++)
                        tc_mma(d, a_desc + (uint64_t)k * kKStep, w_desc + (uint64_t)k * kKStep, idesc,
                               (j > 0 || k > 0) ? 1u : 0u);
                    tc_commit(empty_bar(st));
                    if (++st == kGmStages) {
                        st = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (withhold)
                    withhold = false;
                else
                    tc_commit(dfull_bar(b));
                dphase ^= 1u << b;
                b ^= 1;
            }
            tc_commit(drain_bar);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(drain_bar, 0u) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: thread m stores row m of the tile
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int m = 32 * (warp & 3) + lane;
        int b = 0;
        uint32_t dphase = 0;
        const size_t mn = g.M * g.N;
        for (size_t u = blockIdx.x; u < g.units; u += gridDim.x) {
            int s, tm, tn;
            decode(u, s, tm, tn);
            float *out = g.out + (size_t)s * mn;
            const size_t row = (size_t)tm * kGmBM + (size_t)m;
            const size_t col0 = (size_t)tn * kGmBN;
            // tcgen05.ld is warp-collective: a warp reads the tile only if
            // every lane's wait succeeded
            const bool ready = !*abort && gm_wait(dfull_bar(b), (dphase >> b) & 1u, abort);
            const bool live = __all_sync(kFull, ready);
            if (live) tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < kGmBN / 32; c++) {
                float v[32];
                if (live) {
                    tc_ld_row32(tmem + lane_base + (uint32_t)b * kGmBN + (uint32_t)(32 * c), v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j++) v[j] = __int_as_float(0x7fc00000);
                }
                if (row < g.M) {
                    float *dst = out + row * g.N + col0 + (size_t)(32 * c);
                    const size_t left = g.N - (col0 + (size_t)(32 * c));
                    if (col0 + (size_t)(32 * c) >= g.N) continue;
                    if (left >= 32 && (((uintptr_t)dst) & 15u) == 0) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4 *>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j++)
                            if ((size_t)j < left) dst[j] = v[j];
                    }
                }
            }
            if (live) {
                tc_fence_before();
                mbar_arrive(dempty_bar(b));
            }
            dphase ^= 1u << b;
            b ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kGmTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- CTA pairs
//
// The same units and order, on a pair of CTAs (a cluster of two on two SMs)
// that issues tcgen05.mma.cta_group::2 with M = 256, N = 256: a unit is a
// 256 x 256 output tile of one split; CTA r of the pair loads rows
// 128 r .. 128 r + 127 of the A box and of the W box (64 K-columns each,
// 16 KiB + 16 KiB a stage) into its own shared memory, and the leader
// (rank 0) issues every MMA, which reads both CTAs' halves at the same
// shared-memory offsets and writes rows 128 r .. of D into CTA r's tensor
// memory.  Per 2 x 128 x 256 x 64 multiply-adds an SM thus takes in 32 KiB
// of operands instead of the 48 KiB of a 128 x 256 tile on one SM -- the
// one-SM kernel is bound by that intake (with the W box left out it ran
// 8192^3 at the cuBLAS rate).  Both CTAs allocate the tensor memory
// together (one warp each; two 256-column accumulators); the peer's copies
// complete on the leader's full barrier, the leader's commits arrive on
// both CTAs' barriers (multicast), and both epilogues report the
// accumulator read on the leader's barrier.  Cluster barriers order the
// set-up and the teardown.  Waits give up after about a second as in the
// one-SM kernel.
constexpr int kG2BM = 256;                       // tile rows of the pair (128 per CTA)
constexpr int kG2BN = 256;                       // tile columns (128 W rows per CTA)
constexpr int kG2HalfBytes = 128 * kGmBK * 2;    // 16 KiB: a CTA's half of a box
constexpr int kG2StageBytes = 2 * kG2HalfBytes;  // its A half + its W half
constexpr int kG2Stages = 7;                     // 224 KiB ring (230.6 KB of shared memory in all)
constexpr int kG2DBuffers = 2;                   // accumulators: a tile's epilogue beside the next's MMAs
constexpr uint32_t kG2TmemCols = kG2DBuffers * kG2BN;    // 512: all of TMEM
constexpr int kG2OffBars = kG2Stages * kG2StageBytes;
// barriers: full[S] (leader's: both CTAs' copies), empty[S], dfull[D], dempty[D] (leader's), drain
constexpr int kG2NumBars = 2 * kG2Stages + 2 * kG2DBuffers + 1;
constexpr int kG2OffMisc = kG2OffBars + 8 * kG2NumBars;
constexpr int kG2SmemBytes = kG2OffMisc + 64 + 1024;
static_assert(kG2SmemBytes <= 232448, "the pair kernel's shared memory fits one SM's 227 KiB");

// Instruction descriptor of kind::f16 for the pair: M = 256, N = 256.
template <int DT>
__device__ __forceinline__ uint32_t instr_desc_pair()
{
    constexpr uint32_t ab = DT == kF16 ? 0u : 1u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(kG2BN >> 3) << 17) | ((uint32_t)(kG2BM >> 4) << 24);
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of `addr` (this CTA's shared memory) in CTA
// `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A tensor-map box into this CTA's shared memory whose completion counts on
// an mbarrier of either CTA of the pair (bar: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                                 uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at `bar` in both CTAs of the pair when every
// tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(bar), "h"((uint16_t)3)
        : "memory");
}

// The same, on this CTA's barrier only.
__device__ __forceinline__ void tc_commit_pair_local(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

template <int DT>
__global__ void __launch_bounds__(kGmThreads, 1)
gemm_splitk_pair_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmw,
                        const GemmArgs g)
{
    pdl_launch_dependents();   // the combine may launch now; it waits for this grid to finish
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t ring = sbase;
    const uint32_t bars = sbase + kG2OffBars;
    auto full_bar = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bars + 8u * (uint32_t)(kG2Stages + s); };
    auto dfull_bar = [&](int b) { return bars + 8u * (uint32_t)(2 * kG2Stages + b); };
    auto dempty_bar = [&](int b) { return bars + 8u * (uint32_t)(2 * kG2Stages + kG2DBuffers + b); };
    const uint32_t drain_bar = bars + 8u * (uint32_t)(2 * kG2Stages + 2 * kG2DBuffers);
    uint32_t *misc = (uint32_t *)(smem + kG2OffMisc);
    volatile uint32_t *tmem_holder = misc;
    volatile uint32_t *abort = misc + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const size_t pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;

    auto decode = [&](size_t u, int &s, int &tm, int &tn) {
        const size_t tiles = (size_t)g.tiles_m * (size_t)g.tiles_n;
        s = (int)(u / tiles);
        const size_t t = u - (size_t)s * tiles;
        const size_t group = (size_t)kGmGroupM * (size_t)g.tiles_n;
        const size_t first = (t / group) * kGmGroupM;
        const size_t in_group = (size_t)g.tiles_m - first < (size_t)kGmGroupM ? (size_t)g.tiles_m - first
                                                                             : (size_t)kGmGroupM;
        const size_t r = t % group;
        tm = (int)(first + r % in_group);
        tn = (int)(r / in_group);
    };
    auto split_boxes = [&](int s) {
        const int b0 = s * g.kbps;
        return min(g.kbps, g.kboxes - b0);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kG2Stages; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < kG2DBuffers; b++) {
            mbar_init(dfull_bar(b), 1);
            mbar_init(dempty_bar(b), 2 * kGmEpilogueThreads);     // both CTAs' epilogues
        }
        mbar_init(drain_bar, 1);
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tma) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmw) : "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 1) {
        // together with the peer CTA's warp 1
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr((const void *)tmem_holder)), "r"(kG2TmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync_all();        // both CTAs' barriers and allocation are in place
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    pdl_wait_primary();

    if (warp == 0) {
        // ---------------- producer: this CTA's halves; completion on the leader's full barrier
        if (lane == 0) {
            int st = 0;
            uint32_t phase = 0;
            bool armed[kG2Stages];
            uint32_t armed_phase[kG2Stages];
            for (int i = 0; i < kG2Stages; i++) {
                armed[i] = false;
                armed_phase[i] = 0;
            }
            for (size_t u = pair; u < g.units && !*abort; u += pairs) {
                int s, tm, tn;
                decode(u, s, tm, tn);
                const int nb = split_boxes(s);
                bool ok = true;
                for (int j = 0; j < nb; j++) {
                    if (!gm_wait(empty_bar(st), phase ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = ring + (uint32_t)st * kG2StageBytes;
                    const int kc = (s * g.kbps + j) * kGmBK;
                    const uint32_t fb = map_to_rank(full_bar(st), 0u);
                    if (leader) mbar_arrive_expect_tx(full_bar(st), (uint32_t)(2 * kG2StageBytes));
                    tma_load_2d_pair(dst, &tma, kc, tm * kG2BM + 128 * (int)rank, fb);
                    tma_load_2d_pair(dst + kG2HalfBytes, &tmw, kc, tn * kG2BN + 128 * (int)rank, fb);
                    armed[st] = true;
                    armed_phase[st] = phase;
                    if (++st == kG2Stages) {
                        st = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            if (*abort && leader) {
                // the full barriers count both CTAs' copies: let them land
                for (int i = 0; i < kG2Stages; i++)
                    if (armed[i]) (void)mbar_wait_limited(full_bar(i), armed_phase[i]);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (the leader's lane 0)
        if (leader && lane == 0) {
            const uint32_t idesc = instr_desc_pair<DT>();
            const uint64_t ring_desc = smem_desc_sw128(ring);
            constexpr uint64_t kKStep = 32u >> 4;
            constexpr uint64_t kHalfStep = (uint64_t)kG2HalfBytes >> 4;
            constexpr uint64_t kStageStep = (uint64_t)kG2StageBytes >> 4;
            int st = 0, b = 0;
            uint32_t phase = 0, dphase = 0;       // bit b: uses of accumulator b so far, mod 2
            bool withhold = g.inject_stall != 0u;
            for (size_t u = pair; u < g.units && !*abort; u += pairs) {
                int s, tm, tn;
                decode(u, s, tm, tn);
                const int nb = split_boxes(s);
                // both epilogues have read accumulator b
                if (!gm_wait(dempty_bar(b), ((dphase >> b) & 1u) ^ 1u, abort)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)b * kG2BN;
                bool ok = true;
                for (int j = 0; j < nb; j++) {
                    if (!gm_wait(full_bar(st), phase, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = ring_desc + (uint64_t)st * kStageStep;
                    const uint64_t w_desc = a_desc + kHalfStep;
#pragma unroll
                    for (int k = 0; k < 4; k++)
                        tc_mma_pair(d, a_desc + (uint64_t)k * kKStep, w_desc + (uint64_t)k * kKStep, idesc,
                                    (j > 0 || k > 0) ? 1u : 0u);
                    tc_commit_pair(empty_bar(st));               // both CTAs' stage is free
                    if (++st == kG2Stages) {
                        st = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (withhold)
                    withhold = false;
                else
                    tc_commit_pair(dfull_bar(b));                // the tile is in both CTAs' TMEM
                dphase ^= 1u << b;
                b ^= 1;
            }
            tc_commit_pair_local(drain_bar);
            (void)mbar_wait_limited(drain_bar, 0u);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: thread m stores row 128 rank + m of the tile
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int m = 32 * (warp & 3) + lane;
        int b = 0;
        uint32_t dphase = 0;
        const size_t mn = g.M * g.N;
        for (size_t u = pair; u < g.units; u += pairs) {
            int s, tm, tn;
            decode(u, s, tm, tn);
            float *out = g.out + (size_t)s * mn;
            const size_t row = (size_t)tm * kG2BM + 128u * rank + (size_t)m;
            const size_t col0 = (size_t)tn * kG2BN;
            const bool ready = !*abort && gm_wait(dfull_bar(b), (dphase >> b) & 1u, abort);
            const bool live = __all_sync(kFull, ready);
            if (live) tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < kG2BN / 32; c++) {
                float v[32];
                if (live) {
                    tc_ld_row32(tmem + lane_base + (uint32_t)b * kG2BN + (uint32_t)(32 * c), v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j++) v[j] = __int_as_float(0x7fc00000);
                }
                if (row < g.M) {
                    float *dst = out + row * g.N + col0 + (size_t)(32 * c);
                    const size_t left = g.N - (col0 + (size_t)(32 * c));
                    if (col0 + (size_t)(32 * c) >= g.N) continue;
                    if (left >= 32 && (((uintptr_t)dst) & 15u) == 0) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4 *>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j++)
                            if ((size_t)j < left) dst[j] = v[j];
                    }
                }
            }
            if (live) {
                tc_fence_before();
                mbar_arrive_cluster(map_to_rank(dempty_bar(b), 0u));
            }
            dphase ^= 1u << b;
            b ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    // the leader's MMAs read the peer's shared memory and write its tensor
    // memory: neither CTA leaves or frees before both are done
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kG2TmemCols)
                     : "memory");
    }
}

// C[i] = balanced binary32 tree over P[s * mn + i], s = 0 .. splits-1, in
// split order, -0.0 pad (a binary counter over the splits), one element per
// thread.  (Four elements per thread with 16-byte loads, and eight loads
// issued ahead of their additions, both measured slower: fewer threads in
// flight.)
__global__ void splitk_combine_kernel(const float *__restrict__ P, size_t mn, int splits,
                                      float *__restrict__ C)
{
    pdl_launch_dependents();
    pdl_wait_primary();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < mn;
         i += (size_t)gridDim.x * blockDim.x) {
        TreeCounter<7> tc;
        for (int s = 0; s < splits; s++) tc.push(__ldg(P + (size_t)s * mn + i));
        C[i] = tc.finish();
    }
}

// ---------------------------------------------------------------- host

int gemm_tile_m() { return kGmBM; }
int gemm_tile_n() { return kGmBN; }
int gemm_tile_k() { return kGmBK; }
int gemm_block_threads() { return kGmThreads; }

// The CTA pairs of the pair kernel that can be resident at once on the
// current device (a pair needs two SMs of one GPC), cached per device; 0
// when a pair cannot be scheduled (the one-SM kernel runs instead), or when
// TCR_GEMM_ONE_SM is set in the environment (the one-SM kernel on request,
// e.g. to test it on a device that does schedule pairs).
int gemm_resident_pairs()
{
    const char *one = std::getenv("TCR_GEMM_ONE_SM");
    if (one && one[0] != '\0' && one[0] != '0') return 0;
    static std::mutex mu;
    static std::vector<std::pair<int, int>> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    {
        std::lock_guard<std::mutex> lk(mu);
        for (auto &c : cache)
            if (c.first == dev) return c.second;
    }
    void *kp = (void *)gemm_splitk_pair_kernel<kBF16>;
    int sms = 0, n = 0;
    if (set_smem_once(kp, kG2SmemBytes) == cudaSuccess &&
        set_smem_once((void *)gemm_splitk_pair_kernel<kF16>, kG2SmemBytes) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)sms & ~1u);
        cfg.blockDim = dim3(kGmThreads);
        cfg.dynamicSmemBytes = kG2SmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kp, &cfg) != cudaSuccess) n = 0;
    }
    (void)cudaGetLastError();
    std::lock_guard<std::mutex> lk(mu);
    cache.emplace_back(dev, n);
    return n;
}

int gemm_tile_m_run() { return gemm_resident_pairs() > 0 ? kG2BM : kGmBM; }
int gemm_tile_n_run() { return gemm_resident_pairs() > 0 ? kG2BN : kGmBN; }

int gemm_launch_grid(size_t M, size_t N, int splits)
{
    const int pairs = gemm_resident_pairs();
    const size_t tm = pairs > 0 ? kG2BM : kGmBM, tn = pairs > 0 ? kG2BN : kGmBN;
    const size_t units = ((M + tm - 1) / tm) * ((N + tn - 1) / tn) * (size_t)splits;
    if (pairs > 0) return 2 * (int)(units < (size_t)pairs ? units : (size_t)pairs);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        sms = 152;
    }
    return (int)(units < (size_t)sms ? units : (size_t)sms);
}

cudaError_t launch_gemm_splitk(int dtype, const void *A, const void *W, size_t M, size_t N, size_t K,
                               int splits, int kbps, float *out, bool inject_stall, cudaStream_t stream)
{
    if (dtype != kF16 && dtype != kBF16) return cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const bool pair = gemm_resident_pairs() > 0;
    const int bm = pair ? kG2BM : kGmBM, bn = pair ? kG2BN : kGmBN;
    // boxes of 64 K-columns: 128 rows of A and W per CTA of a pair, else 128
    // rows of A and 256 of W
    alignas(64) CUtensorMap ma, mw;
    const cuuint32_t abox[2] = {kGmBK, 128};
    const cuuint32_t wbox[2] = {kGmBK, (cuuint32_t)(pair ? 128 : kGmBN)};
    const cuuint32_t estride[2] = {1, 1};
    const cuuint64_t gstride[1] = {(cuuint64_t)K * 2};
    const cuuint64_t da[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t dw[2] = {(cuuint64_t)K, (cuuint64_t)N};
    if (encode(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (void *)A, da, gstride, abox, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (void *)W, dw, gstride, wbox, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    GemmArgs g;
    g.M = M;
    g.N = N;
    g.kboxes = (int)((K + kGmBK - 1) / kGmBK);
    g.kbps = kbps;
    g.splits = splits;
    g.tiles_m = (int)((M + bm - 1) / bm);
    g.tiles_n = (int)((N + bn - 1) / bn);
    g.units = (size_t)g.tiles_m * (size_t)g.tiles_n * (size_t)splits;
    g.out = out;
    g.inject_stall = inject_stall ? 1u : 0u;
    void *args[] = {(void *)&ma, (void *)&mw, (void *)&g};
    const int grid = gemm_launch_grid(M, N, splits);
    if (!pair) {
        void *k = dtype == kF16 ? (void *)gemm_splitk_kernel<kF16> : (void *)gemm_splitk_kernel<kBF16>;
        cudaError_t e = set_smem_once(k, kGmSmemBytes);
        if (e != cudaSuccess) return e;
        return launch_first(k, dim3(grid), dim3(kGmThreads), args, kGmSmemBytes, stream);
    }
    // CTA pairs (clusters of two), launched as programmatic dependents too
    void *kp = dtype == kF16 ? (void *)gemm_splitk_pair_kernel<kF16> : (void *)gemm_splitk_pair_kernel<kBF16>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kGmThreads);
    cfg.dynamicSmemBytes = kG2SmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelExC(&cfg, kp, args);
}

cudaError_t launch_splitk_combine(const float *P, size_t mn, int splits, float *C, cudaStream_t stream)
{
    if (mn == 0) return cudaSuccess;
    const size_t blocks = (mn + 255) / 256;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)(blocks < 152 * 8 ? blocks : 152 * 8));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, splitk_combine_kernel, P, mn, splits, C);
}

cudaError_t read_gemm_faults(unsigned int *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_gemm_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0u;
    return cudaMemcpyToSymbol(g_gemm_fault, &zero, sizeof(unsigned int));
}

}  // namespace tcr
