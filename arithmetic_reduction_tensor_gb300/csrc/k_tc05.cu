// k_tc05.cu -- MMA_CHAIN on the fifth-generation tensor cores (tcgen05):
// inputs staged into shared memory by bulk asynchronous copies, tensor-core
// MMAs against an all-ones matrix issued by one thread, the accumulator in
// tensor memory (TMEM).
//
// The method is that of "GPU Tensor Cores for fast Arithmetic Reductions"
// (arXiv 2001.05585), Abstract: the sum of n numbers as chains of m x m
// MMAs; each chain of R MMAs keeps its sub-result in 32-bit floating point
// and the sub-results are then reduced into one 32-bit result.  Here one
// MMA is tcgen05.mma.cta_group::1.kind::f16 with M = 128, N = 16, K = 16:
// A is a 4 KiB tile of 2048 inputs (128 rows x 16), B is 16 x 16 ones, so
// every column of the 128 x 16 fp32 D holds the 128 row sums.  Since B is
// all ones the sum of column 0 is the sum of the tile whatever element sits
// in whatever slot, so a contiguous 4 KiB of input is a valid A tile as it
// lies in memory: no layout transform, no swizzle.
//
// CTA roles (192 threads, one persistent CTA per SM):
//   warp 0, lane 0   producer: 32 KiB bulk copies (8 tiles) global -> a
//                    6-stage shared-memory ring, completion by mbarrier
//                    transaction count;
//   warp 1           owns the TMEM allocation; lane 0 issues the MMAs:
//                    R per chain into one of 8 D buffers, the first of a
//                    chain without accumulate, tcgen05.commit after a chain
//                    (D full) and after a stage (stage free);
//   warps 2..5       epilogue: each thread reads its TMEM lane of column 0
//                    of a full D buffer, adds it to its fp32 accumulator and
//                    frees the buffer; at the end of a work unit (2^16
//                    inputs) the 128 accumulators and any tail inputs past
//                    the last whole tile are reduced into the unit's partial.
//
// Every wait on an mbarrier gives up after about one second: the CTA then
// raises a device-wide fault flag, drains its own copies and MMAs (again
// with a limit), frees its TMEM and writes NaN as its partials, so a broken
// pipeline shows up as a NaN result, never as a hang.
#include "kernels.cuh"
#include "tc05.cuh"

namespace tcr {

constexpr int kTcTileInputs = 2048;                 // one MMA: 128 x 16 inputs
constexpr int kTcTileBytes = kTcTileInputs * 2;     // 4 KiB
constexpr int kTcTilesPerStage = 8;                 // 32 KiB bulk copies
constexpr int kTcStageBytes = kTcTileBytes * kTcTilesPerStage;
constexpr int kTcStages = 6;                        // 192 KiB in flight per SM
constexpr int kTcUnitLog2 = 16;                     // work unit: 2^16 inputs ...
constexpr int kTcMinUnitLog2 = 11;                  // ... down to one tile for small inputs
constexpr size_t kTcMinUnits = 2 * 152;             // the units small inputs are cut into
constexpr int kTcThreads = 192;
constexpr int kTcEpilogueThreads = 128;
constexpr int kTcDBuffers = 8;                      // chains the MMA may run ahead
constexpr uint32_t kTcDBufferStride = 32;           // columns per D buffer (N = 16 used)
constexpr uint32_t kTcTmemCols = kTcDBuffers * kTcDBufferStride;    // 256

// Dynamic shared memory layout (offsets from a 1024-byte aligned base).
constexpr int kTcOffRing = 0;
constexpr int kTcOffOnes = kTcOffRing + kTcStages * kTcStageBytes;     // 512 B of ones
constexpr int kTcOffBars = kTcOffOnes + 1024;
// barriers: full[S], empty[S], dfull[B], dempty[B], drain
constexpr int kTcNumBars = 2 * kTcStages + 2 * kTcDBuffers + 1;
constexpr int kTcOffMisc = kTcOffBars + 8 * kTcNumBars;                 // tmem addr, abort, red[4]
constexpr int kTcSmemBytes = kTcOffMisc + 64 + 1024;                    // + alignment slack

__device__ unsigned int g_tc05_fault;               // non-zero once any wait gave up

// Waits of these kernels give up into g_tc05_fault.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort)
{
    return mbar_wait_f(bar, parity, abort, &g_tc05_fault);
}

template <int DT>
__device__ __forceinline__ uint32_t instr_desc()
{
    return instr_desc_n<DT, 16>();
}

// ---------------------------------------------------------------- kernel

// Work unit u covers inputs [u * 2^L, min(n, (u+1) * 2^L)), L = unit_log2
// (16, or less for small inputs: tmem_unit_log2); its whole 2048-input
// tiles go through the tensor cores, the inputs past the last whole tile of
// the array (fewer than 2048) are added by the epilogue.
__device__ __forceinline__ int unit_tiles(size_t n, size_t u, int unit_log2)
{
    const size_t base = u << unit_log2;
    const size_t left = n - base;
    const size_t t = left / kTcTileInputs;
    const size_t per_unit = (size_t)1 << (unit_log2 - kTcMinUnitLog2);
    return (int)(t < per_unit ? t : per_unit);
}

template <int DT, int R>
__global__ void __launch_bounds__(kTcThreads, 1)
mma_tmem_kernel(const uint16_t *__restrict__ x, size_t n, size_t units, int unit_log2,
                float *__restrict__ dst, uint32_t inject_stall)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t ring = sbase + kTcOffRing;
    const uint32_t ones = sbase + kTcOffOnes;
    const uint32_t bars = sbase + kTcOffBars;
    auto full_bar = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bars + 8u * (uint32_t)(kTcStages + s); };
    auto dfull_bar = [&](int b) { return bars + 8u * (uint32_t)(2 * kTcStages + b); };
    auto dempty_bar = [&](int b) { return bars + 8u * (uint32_t)(2 * kTcStages + kTcDBuffers + b); };
    const uint32_t drain_bar = bars + 8u * (uint32_t)(2 * kTcStages + 2 * kTcDBuffers);
    uint32_t *misc = (uint32_t *)(smem + kTcOffMisc);
    volatile uint32_t *tmem_holder = misc;
    volatile uint32_t *abort = misc + 1;
    float *red = (float *)(misc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ones matrix B (16 x 16 inputs, 512 bytes), barriers, flags
    {
        const uint32_t one2 = DT == kF16 ? 0x3c003c00u : 0x3f803f80u;
        uint32_t *o = (uint32_t *)(smem + kTcOffOnes);
        for (int i = threadIdx.x; i < 128; i += blockDim.x) o[i] = one2;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < kTcDBuffers; b++) {
            mbar_init(dfull_bar(b), 1);
            mbar_init(dempty_bar(b), kTcEpilogueThreads);
        }
        mbar_init(drain_bar, 1);
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // make the generic-proxy writes (ones, barriers) visible to the async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr((const void *)tmem_holder)), "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            int s = 0;
            uint32_t phase = 0;
            bool armed[kTcStages];
            uint32_t armed_phase[kTcStages];
#pragma unroll
            for (int i = 0; i < kTcStages; i++) {
                armed[i] = false;
                armed_phase[i] = 0;
            }
            for (size_t u = blockIdx.x; u < units && !*abort; u += gridDim.x) {
                const int tiles = unit_tiles(n, u, unit_log2);
                const uint16_t *src = x + (u << unit_log2);
                for (int t0 = 0; t0 < tiles; t0 += kTcTilesPerStage) {
                    const int nt = min(kTcTilesPerStage, tiles - t0);
                    if (!mbar_wait(empty_bar(s), phase ^ 1u, abort)) break;
                    const uint32_t bytes = (uint32_t)nt * kTcTileBytes;
                    mbar_arrive_expect_tx(full_bar(s), bytes);
                    bulk_copy_g2s(ring + (uint32_t)s * kTcStageBytes, src + (size_t)t0 * kTcTileInputs,
                                  bytes, full_bar(s));
                    armed[s] = true;
                    armed_phase[s] = phase;
                    if (++s == kTcStages) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort) {
                // let the copies already issued land before the CTA exits
#pragma unroll
                for (int i = 0; i < kTcStages; i++) {
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
            const uint32_t idesc = instr_desc<DT>();
            const uint64_t b_desc = smem_desc(ones, 128, 256);
            // descriptor of tile 0 of stage 0; a tile is 4096 bytes further
            // (256 in the descriptor's 16-byte units), a stage 8 tiles
            const uint64_t ring_desc = smem_desc(ring, 128, 256);
            constexpr uint64_t kTileStep = kTcTileBytes >> 4;
            constexpr uint64_t kStageStep = kTcStageBytes >> 4;
            int s = 0, b = 0;
            uint32_t phase = 0, dphase = 0u;     // bit b: uses of D buffer b so far, mod 2
            auto begin_chain = [&]() -> bool {
                // the chain's D buffer must have been read out
                if (!mbar_wait(dempty_bar(b), ((dphase >> b) & 1u) ^ 1u, abort)) return false;
                tc_fence_after();
                return true;
            };
            // A host-requested stall leaves the first chain unpublished, so
            // the epilogue's wait runs out its limit (failure-path test).
            bool withhold = inject_stall != 0u;
            auto end_chain = [&]() {
                if (withhold)
                    withhold = false;
                else
                    tc_commit(dfull_bar(b));      // chain sub-result ready
                dphase ^= 1u << b;
                if (++b == kTcDBuffers) b = 0;
            };
            for (size_t u = blockIdx.x; u < units && !*abort; u += gridDim.x) {
                const int tiles = unit_tiles(n, u, unit_log2);
                int in_chain = 0;
                for (int t0 = 0; t0 < tiles && !*abort; t0 += kTcTilesPerStage) {
                    const int nt = min(kTcTilesPerStage, tiles - t0);
                    if (!mbar_wait(full_bar(s), phase, abort)) break;
                    tc_fence_after();
                    const uint64_t sdesc = ring_desc + (uint64_t)s * kStageStep;
                    bool ok = true;
                    if (kTcTilesPerStage % R == 0 && nt == kTcTilesPerStage) {
                        // whole stage, chains aligned to it: static boundaries
#pragma unroll
                        for (int t = 0; t < kTcTilesPerStage; t++) {
                            if (t % R == 0 && !(ok = begin_chain())) break;
                            tc_mma(tmem + (uint32_t)b * kTcDBufferStride, sdesc + (uint64_t)t * kTileStep,
                                   b_desc, idesc, t % R != 0 ? 1u : 0u);
                            if (t % R == R - 1) end_chain();
                        }
                    } else {
                        for (int t = 0; t < nt; t++) {
                            if (in_chain == 0 && !(ok = begin_chain())) break;
                            tc_mma(tmem + (uint32_t)b * kTcDBufferStride, sdesc + (uint64_t)t * kTileStep,
                                   b_desc, idesc, in_chain > 0 ? 1u : 0u);
                            if (++in_chain == R || t0 + t + 1 == tiles) {
                                end_chain();
                                in_chain = 0;
                            }
                        }
                    }
                    tc_commit(empty_bar(s));                  // stage may be refilled
                    if (++s == kTcStages) {
                        s = 0;
                        phase ^= 1u;
                    }
                    if (!ok) break;
                }
            }
            // every MMA issued has completed once the drain barrier flips
            tc_commit(drain_bar);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(drain_bar, 0u) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warps 2..5, TMEM lanes 32*(warp%4) ..
        const int et = threadIdx.x - 64;                   // 0..127
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        int b = 0;
        uint32_t dphase = 0u;
        for (size_t u = blockIdx.x; u < units; u += gridDim.x) {
            const int tiles = unit_tiles(n, u, unit_log2);
            const int chains = (tiles + R - 1) / R;
            float acc = 0.f;
            for (int c = 0; c < chains && !*abort; c++) {
                if (!mbar_wait(dfull_bar(b), (dphase >> b) & 1u, abort)) break;
                tc_fence_after();
                const float v = tc_ld_lane(tmem + lane_base + (uint32_t)b * kTcDBufferStride);
                acc = __fadd_rn(acc, v);
                tc_fence_before();
                mbar_arrive(dempty_bar(b));
                dphase ^= 1u << b;
                if (++b == kTcDBuffers) b = 0;
            }
            // inputs of this unit past its whole tiles (only in the last unit)
            const size_t base = u << unit_log2;
            const size_t tail_lo = base + (size_t)tiles * kTcTileInputs;
            size_t tail_hi = base + ((size_t)1 << unit_log2);
            if (tail_hi > n) tail_hi = n;
            for (size_t i = tail_lo + (size_t)et; i < tail_hi; i += kTcEpilogueThreads)
                acc = __fadd_rn(acc, DT == kF16 ? leaf_lo<kF16>(__ldg(x + i)) : leaf_lo<kBF16>(__ldg(x + i)));
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, off));
            if (lane == 0) red[warp - 2] = acc;
            named_sync(1, kTcEpilogueThreads);
            if (et == 0) {
                float v = __fadd_rn(__fadd_rn(red[0], red[1]), __fadd_rn(red[2], red[3]));
                dst[u] = *abort ? __int_as_float(0x7fc00000) : v;
            }
            named_sync(1, kTcEpilogueThreads);
        }
    }

    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTcTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- rows

// Rows: D's 128 lanes are 128 consecutive data rows.  A 2-D tensor map over
// the row-major matrix (dims: cols, rows) with a 64-column x 128-row box and
// the 128-byte swizzle lands a row block as 128 rows of 128 bytes (8-row
// atoms of 1024 bytes, the 16-byte chunks of row r permuted by r mod 8) --
// the SWIZZLE_128B K-major layout the MMA descriptor names, so one box is
// four MMAs of K = 16, the k-th starting 32 bytes further.  The swizzle only
// permutes chunks within a row, so each MMA row still holds one data row.
// The column of D read out after a chain holds the 128 rows' sums over that
// chain's columns.  Work unit: 128 rows x kTcRowsChunkCols columns, one
// partial per row and unit; the tensor map zero-fills rows and columns past
// the matrix.
constexpr int kTcRowsChunkCols = 1024;                // columns per work unit
constexpr int kTcRowsBoxCols = 64;                    // columns per tensor-map box
constexpr int kTcRowsBoxBytes = 128 * kTcRowsBoxCols * 2;     // 16 KiB
constexpr int kTcRowsBoxesPerStage = 4;               // 64 KiB, 16 MMAs per stage
constexpr int kTcRowsStageBytes = kTcRowsBoxBytes * kTcRowsBoxesPerStage;
constexpr int kTcRowsStages = 3;                      // 192 KiB ring
constexpr int kTcRowsOffOnes = kTcRowsStages * kTcRowsStageBytes;
constexpr int kTcRowsOffBars = kTcRowsOffOnes + 1024;
constexpr int kTcRowsNumBars = 2 * kTcRowsStages + 2 * kTcDBuffers + 1;
constexpr int kTcRowsOffMisc = kTcRowsOffBars + 8 * kTcRowsNumBars;
constexpr int kTcRowsSmemBytes = kTcRowsOffMisc + 64 + 1024;

template <int DT, int R>
__global__ void __launch_bounds__(kTcThreads, 1)
mma_tmem_rows_kernel(const __grid_constant__ CUtensorMap tmap, size_t rows, size_t cols,
                     size_t cpr, size_t units, float *__restrict__ dst, uint32_t inject_stall)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t ring = sbase;
    const uint32_t ones = sbase + kTcRowsOffOnes;
    const uint32_t bars = sbase + kTcRowsOffBars;
    auto full_bar = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bars + 8u * (uint32_t)(kTcRowsStages + s); };
    auto dfull_bar = [&](int b) { return bars + 8u * (uint32_t)(2 * kTcRowsStages + b); };
    auto dempty_bar = [&](int b) { return bars + 8u * (uint32_t)(2 * kTcRowsStages + kTcDBuffers + b); };
    const uint32_t drain_bar = bars + 8u * (uint32_t)(2 * kTcRowsStages + 2 * kTcDBuffers);
    uint32_t *misc = (uint32_t *)(smem + kTcRowsOffMisc);
    volatile uint32_t *tmem_holder = misc;
    volatile uint32_t *abort = misc + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // boxes (64 columns) of work unit u
    auto unit_boxes = [&](size_t u) -> int {
        const size_t c0 = (u % cpr) * kTcRowsChunkCols;
        const size_t nc = cols - c0 < (size_t)kTcRowsChunkCols ? cols - c0 : (size_t)kTcRowsChunkCols;
        return (int)((nc + kTcRowsBoxCols - 1) / kTcRowsBoxCols);
    };

    {
        const uint32_t one2 = DT == kF16 ? 0x3c003c00u : 0x3f803f80u;
        uint32_t *o = (uint32_t *)(smem + kTcRowsOffOnes);
        for (int i = threadIdx.x; i < 128; i += blockDim.x) o[i] = one2;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcRowsStages; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < kTcDBuffers; b++) {
            mbar_init(dfull_bar(b), 1);
            mbar_init(dempty_bar(b), kTcEpilogueThreads);
        }
        mbar_init(drain_bar, 1);
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmap) : "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr((const void *)tmem_holder)), "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ---------------- producer: one 64-column x 128-row box per stage
        if (lane == 0) {
            int s = 0;
            uint32_t phase = 0;
            bool armed[kTcRowsStages];
            uint32_t armed_phase[kTcRowsStages];
            for (int i = 0; i < kTcRowsStages; i++) {
                armed[i] = false;
                armed_phase[i] = 0;
            }
            for (size_t u = blockIdx.x; u < units && !*abort; u += gridDim.x) {
                const int row0 = (int)((u / cpr) * 128);
                const int col0 = (int)((u % cpr) * kTcRowsChunkCols);
                const int boxes = unit_boxes(u);
                for (int j = 0; j < boxes; j += kTcRowsBoxesPerStage) {
                    const int nb = min(kTcRowsBoxesPerStage, boxes - j);
                    if (!mbar_wait(empty_bar(s), phase ^ 1u, abort)) break;
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)nb * kTcRowsBoxBytes);
                    for (int q = 0; q < nb; q++)
                        tma_load_2d(ring + (uint32_t)s * kTcRowsStageBytes + (uint32_t)q * kTcRowsBoxBytes,
                                    &tmap, col0 + (j + q) * kTcRowsBoxCols, row0, full_bar(s));
                    armed[s] = true;
                    armed_phase[s] = phase;
                    if (++s == kTcRowsStages) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort) {
                for (int i = 0; i < kTcRowsStages; i++) {
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
        // ---------------- MMA issuer: four MMAs (K = 16) per stage
        if (lane == 0) {
            const uint32_t idesc = instr_desc<DT>();
            const uint64_t b_desc = smem_desc(ones, 128, 256);
            const uint64_t ring_desc = smem_desc_sw128(ring);
            constexpr uint64_t kKStep = 32u >> 4;                    // 16 columns = 32 bytes
            constexpr uint64_t kBoxStep = (uint64_t)kTcRowsBoxBytes >> 4;
            constexpr uint64_t kStageStep = (uint64_t)kTcRowsStageBytes >> 4;
            constexpr int kMmasPerStage = 4 * kTcRowsBoxesPerStage;
            int s = 0, b = 0;
            uint32_t phase = 0, dphase = 0u;
            auto begin_chain = [&]() -> bool {
                if (!mbar_wait(dempty_bar(b), ((dphase >> b) & 1u) ^ 1u, abort)) return false;
                tc_fence_after();
                return true;
            };
            bool withhold = inject_stall != 0u;
            auto end_chain = [&]() {
                if (withhold)
                    withhold = false;
                else
                    tc_commit(dfull_bar(b));
                dphase ^= 1u << b;
                if (++b == kTcDBuffers) b = 0;
            };
            for (size_t u = blockIdx.x; u < units && !*abort; u += gridDim.x) {
                const int boxes = unit_boxes(u);
                const int mmas = 4 * boxes;
                int in_chain = 0;
                bool ok = true;
                for (int j = 0; j < boxes && ok; j += kTcRowsBoxesPerStage) {
                    const int nm = 4 * min(kTcRowsBoxesPerStage, boxes - j);
                    if (!mbar_wait(full_bar(s), phase, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t sdesc = ring_desc + (uint64_t)s * kStageStep;
                    // MMA k of the stage: box k / 4, 32-byte slice k % 4
                    if (kMmasPerStage % R == 0 && nm == kMmasPerStage) {
#pragma unroll
                        for (int k = 0; k < kMmasPerStage; k++) {
                            if (k % R == 0 && !(ok = begin_chain())) break;
                            tc_mma(tmem + (uint32_t)b * kTcDBufferStride,
                                   sdesc + (uint64_t)(k / 4) * kBoxStep + (uint64_t)(k % 4) * kKStep,
                                   b_desc, idesc, k % R != 0 ? 1u : 0u);
                            if (k % R == R - 1) end_chain();
                        }
                    } else {
                        for (int k = 0; k < nm; k++) {
                            if (in_chain == 0 && !(ok = begin_chain())) break;
                            tc_mma(tmem + (uint32_t)b * kTcDBufferStride,
                                   sdesc + (uint64_t)(k / 4) * kBoxStep + (uint64_t)(k % 4) * kKStep,
                                   b_desc, idesc, in_chain > 0 ? 1u : 0u);
                            if (++in_chain == R || 4 * j + k + 1 == mmas) {
                                end_chain();
                                in_chain = 0;
                            }
                        }
                    }
                    tc_commit(empty_bar(s));
                    if (++s == kTcRowsStages) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            tc_commit(drain_bar);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(drain_bar, 0u) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: thread m holds row row0 + m of the unit
        const int et = threadIdx.x - 64;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int m = 32 * (warp & 3) + lane;              // TMEM lane = row in the block
        (void)et;
        int b = 0;
        uint32_t dphase = 0u;
        for (size_t u = blockIdx.x; u < units; u += gridDim.x) {
            const int chains = (4 * unit_boxes(u) + R - 1) / R;
            float acc = 0.f;
            for (int c = 0; c < chains && !*abort; c++) {
                if (!mbar_wait(dfull_bar(b), (dphase >> b) & 1u, abort)) break;
                tc_fence_after();
                acc = __fadd_rn(acc, tc_ld_lane(tmem + lane_base + (uint32_t)b * kTcDBufferStride));
                tc_fence_before();
                mbar_arrive(dempty_bar(b));
                dphase ^= 1u << b;
                if (++b == kTcDBuffers) b = 0;
            }
            const size_t row = (u / cpr) * 128 + (size_t)m;
            if (row < rows) dst[row * cpr + (u % cpr)] = *abort ? __int_as_float(0x7fc00000) : acc;
        }
    }

    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTcTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host

template <int DT>
static void *pick_dt(int R)
{
    switch (R) {
    case 1: return (void *)mma_tmem_kernel<DT, 1>;
    case 2: return (void *)mma_tmem_kernel<DT, 2>;
    case 3: return (void *)mma_tmem_kernel<DT, 3>;
    case 4: return (void *)mma_tmem_kernel<DT, 4>;
    case 5: return (void *)mma_tmem_kernel<DT, 5>;
    case 6: return (void *)mma_tmem_kernel<DT, 6>;
    case 7: return (void *)mma_tmem_kernel<DT, 7>;
    case 8: return (void *)mma_tmem_kernel<DT, 8>;
    default: return nullptr;
    }
}

// 2^16 inputs per unit (one unit -- one launch, no partials -- up to 2^16
// inputs); above that halved while it leaves fewer than two units per SM of
// the 152 the rules assume, down to one tile.  A function of n only, so the
// chunking (and MMA_CHAIN's bits) is the same on every device.
int tmem_unit_log2(size_t n)
{
    int l = kTcUnitLog2;
    if (n <= ((size_t)1 << kTcUnitLog2)) return l;
    while (l > kTcMinUnitLog2 && ((n + ((size_t)1 << l) - 1) >> l) < kTcMinUnits) l--;
    return l;
}

size_t tmem_units(size_t n)
{
    const int l = tmem_unit_log2(n);
    return (n + ((size_t)1 << l) - 1) >> l;
}

int tmem_block_threads() { return kTcThreads; }

cudaError_t launch_mma_tmem(int dtype, int R, const uint16_t *x, size_t n, float *dst, int grid,
                            bool inject_stall, cudaStream_t stream)
{
    void *k = dtype == kF16 ? pick_dt<kF16>(R) : pick_dt<kBF16>(R);
    if (!k) return cudaErrorInvalidValue;
    cudaError_t e = set_smem_once(k, kTcSmemBytes);
    if (e != cudaSuccess) return e;
    size_t units = tmem_units(n);
    int unit_log2 = tmem_unit_log2(n);
    uint32_t stall = inject_stall ? 1u : 0u;
    void *args[] = {(void *)&x, (void *)&n, (void *)&units, (void *)&unit_log2, (void *)&dst,
                    (void *)&stall};
    return cudaLaunchKernel(k, dim3(grid), dim3(kTcThreads), args, kTcSmemBytes, stream);
}

template <int DT>
static void *pick_rows_dt(int R)
{
    switch (R) {
    case 1: return (void *)mma_tmem_rows_kernel<DT, 1>;
    case 2: return (void *)mma_tmem_rows_kernel<DT, 2>;
    case 3: return (void *)mma_tmem_rows_kernel<DT, 3>;
    case 4: return (void *)mma_tmem_rows_kernel<DT, 4>;
    case 5: return (void *)mma_tmem_rows_kernel<DT, 5>;
    case 6: return (void *)mma_tmem_rows_kernel<DT, 6>;
    case 7: return (void *)mma_tmem_rows_kernel<DT, 7>;
    case 8: return (void *)mma_tmem_rows_kernel<DT, 8>;
    default: return nullptr;
    }
}

size_t tmem_rows_chunks(size_t cols)
{
    return (cols + kTcRowsChunkCols - 1) / kTcRowsChunkCols;
}

size_t tmem_rows_units(size_t rows, size_t cols)
{
    return ((rows + 127) / 128) * tmem_rows_chunks(cols);
}

cudaError_t launch_mma_tmem_rows(int dtype, int R, const uint16_t *x, size_t rows, size_t cols,
                                 float *dst, int grid, bool inject_stall, cudaStream_t stream)
{
    void *k = dtype == kF16 ? pick_rows_dt<kF16>(R) : pick_rows_dt<kBF16>(R);
    if (!k) return cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    alignas(64) CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {kTcRowsBoxCols, 128};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (void *)x, gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaError_t e = set_smem_once(k, kTcRowsSmemBytes);
    if (e != cudaSuccess) return e;
    size_t cpr = tmem_rows_chunks(cols);
    size_t units = tmem_rows_units(rows, cols);
    uint32_t stall = inject_stall ? 1u : 0u;
    void *args[] = {(void *)&map, (void *)&rows, (void *)&cols, (void *)&cpr, (void *)&units,
                    (void *)&dst, (void *)&stall};
    return cudaLaunchKernel(k, dim3(grid), dim3(kTcThreads), args, kTcRowsSmemBytes, stream);
}

cudaError_t read_device_faults(unsigned int *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_tc05_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0u;
    return cudaMemcpyToSymbol(g_tc05_fault, &zero, sizeof(unsigned int));
}

}  // namespace tcr
