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
// CTA roles (192 threads; one CTA per work unit, two resident per SM):
//   warp 0, lane 0   producer: 32 KiB bulk copies (8 tiles) global -> a
//                    2-stage shared-memory ring, completion by mbarrier
//                    transaction count; while a unit's last stage streams
//                    in it asks the hardware to cancel a CTA that has not
//                    launched yet (cluster launch control) and takes that
//                    CTA's unit next -- the other roles read the same
//                    answers, so fast SMs take more units;
//   warp 1           owns the TMEM allocation; lane 0 issues the MMAs:
//                    R per chain into one of 8 D buffers, the first of a
//                    chain without accumulate, tcgen05.commit after a chain
//                    (D full) and after a stage (stage free);
//   warps 2..5       epilogue: each thread reads its TMEM lane of column 0
//                    of a stage's full D buffers (one wait for the stage's
//                    last chain, the loads issued together), adds them to
//                    its fp32 accumulator and frees the buffers; at the end
//                    of a work unit (2^16 inputs) the 128 accumulators and
//                    any tail inputs past the last whole tile are reduced
//                    into the unit's partial.
// The set-up (barriers, ones, TMEM) runs before griddepcontrol.wait, beside
// the stream's previous kernel (programmatic dependent launch).
//
// Every wait on an mbarrier gives up after about one second: the CTA then
// raises a device-wide fault flag, drains its own copies and MMAs (again
// with a limit), frees its TMEM and writes NaN as its partials (and as the
// partials of every unit it still takes over), so a broken pipeline shows
// up as a NaN result, never as a hang.
#include <cstring>

#include "kernels.cuh"
#include "tc05.cuh"

namespace tcr {

constexpr int kTcTileInputs = 2048;                 // one MMA: 128 x 16 inputs
constexpr int kTcTileBytes = kTcTileInputs * 2;     // 4 KiB
constexpr int kTcTilesPerStage = 8;                 // 32 KiB bulk copies
constexpr int kTcStageBytes = kTcTileBytes * kTcTilesPerStage;
constexpr int kTcStages = 2;                        // 64 KiB a CTA, 128 KiB in flight per SM
// Resident CTAs of the sum and flat rows kernels, and the shared-memory
// carveout their launches ask for (percent of the 228 KiB maximum: the
// 164 KiB configuration).  Two CTAs per SM take over units faster than one
// with a deeper ring; three need the 228 KiB configuration, and an SM keeps
// its configuration while the stream's next kernel runs on it: with 28 KiB
// (or 60 KiB) of L1 left, the streaming kernels after a tcgen05 call ran
// about 14% slower.
constexpr int kTcCtasPerSm = 2;
constexpr int kTcCarveoutPercent = 72;
constexpr int kTcCarveoutBytes = 164 * 1024;
constexpr int kTcUnitLog2 = 16;                     // work unit: 2^16 inputs ...
constexpr int kTcMinUnitLog2 = 11;                  // ... down to one tile for small inputs
constexpr size_t kTcMinUnits = 152 / 2;            // the units small inputs are cut into
constexpr int kTcThreads = 192;
constexpr int kTcEpilogueThreads = 128;
constexpr int kTcDBuffers = 8;                      // chains the MMA may run ahead
constexpr uint32_t kTcDBufferStride = 16;           // columns per D buffer (N = 16)
constexpr uint32_t kTcTmemCols = kTcDBuffers * kTcDBufferStride;    // 128
static_assert(kTcCtasPerSm * kTcTmemCols <= 512, "the resident CTAs' TMEM fits an SM's 512 columns");

constexpr uint32_t kTcClcSlots = 16;                // cancellation responses in flight
constexpr uint32_t kTcRecent = 32;                  // units the producer remembers (abort path)

// Dynamic shared memory layout (offsets from a 1024-byte aligned base).
constexpr int kTcOffRing = 0;
constexpr int kTcOffOnes = kTcOffRing + kTcStages * kTcStageBytes;     // 512 B of ones
constexpr int kTcOffClc = kTcOffOnes + 512;                             // 16 B per response
constexpr int kTcOffBars = kTcOffOnes + 1024;
static_assert(512 + 16 * kTcClcSlots <= 1024, "responses fit beside the ones");
// barriers: full[S], empty[S], dfull[B], dempty[B], drain, clc_full[C], clc_empty[C]
constexpr int kTcNumBars = 2 * kTcStages + 2 * kTcDBuffers + 1 + 2 * kTcClcSlots;
constexpr int kTcOffMisc = kTcOffBars + 8 * kTcNumBars;     // tmem addr, abort, red[4], next unit
constexpr int kTcSmemBytes = kTcOffMisc + 64 + 1024;                    // + alignment slack
// an SM has 228 KiB of shared memory, of which each CTA reserves 1 KiB
static_assert(kTcCtasPerSm * (kTcSmemBytes + 1024) <= kTcCarveoutBytes,
              "the resident CTAs fit the carveout (each CTA reserves 1 KiB more)");

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

// Issue NM MMAs (k = 0 .. NM-1) in chains of R: a chain starts on a free D
// buffer (begin), its first MMA overwrites D, the rest accumulate, and its
// end publishes D (end).  The boundaries are compile-time constants: MMAs
// issued under run-time chain logic issued several times slower.  Returns
// false when a wait gave up.
template <int R, int NM, class Begin, class End, class Issue>
__device__ __forceinline__ bool issue_chains(Begin &begin, End &end, Issue &issue)
{
#pragma unroll
    for (int k = 0; k < NM; k++) {
        if (k % R == 0 && !begin()) return false;
        issue(k, k % R != 0 ? 1u : 0u);
        if (k % R == R - 1 || k == NM - 1) end();
    }
    return true;
}

// Chains of R over n MMAs that run through stages of P: a chain ends with
// its stage, so each whole stage holds ceil(P / R) chains.
template <int R, int P>
__device__ __forceinline__ int stage_chains(int n)
{
    return (n / P) * ((P + R - 1) / R) + (n % P + R - 1) / R;
}

// issue_chains for a run-time count 1 <= nm <= NM
template <int R, int NM, class Begin, class End, class Issue>
__device__ __forceinline__ bool issue_chains_upto(int nm, Begin &begin, End &end, Issue &issue)
{
    if constexpr (NM == 1) {
        return issue_chains<R, 1>(begin, end, issue);
    } else {
        if (nm >= NM) return issue_chains<R, NM>(begin, end, issue);
        return issue_chains_upto<R, NM - 1>(nm, begin, end, issue);
    }
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
__global__ void __launch_bounds__(kTcThreads, kTcCtasPerSm)
mma_tmem_kernel(const uint16_t *__restrict__ x, size_t n, int unit_log2, float *__restrict__ dst,
                uint32_t inject_stall)
{
    pdl_launch_dependents();   // the combine may launch now; it waits for this grid to finish
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
    auto clc_full_bar = [&](uint32_t k) { return drain_bar + 8u * (1u + k % kTcClcSlots); };
    auto clc_empty_bar = [&](uint32_t k) { return drain_bar + 8u * (1u + kTcClcSlots + k % kTcClcSlots); };
    auto clc_resp = [&](uint32_t k) { return sbase + kTcOffClc + 16u * (k % kTcClcSlots); };
    auto clc_parity = [](uint32_t k) { return (k / kTcClcSlots) & 1u; };
    uint32_t *misc = (uint32_t *)(smem + kTcOffMisc);
    volatile uint32_t *tmem_holder = misc;
    volatile uint32_t *abort = misc + 1;
    float *red = (float *)(misc + 4);
    volatile uint32_t *next_unit = misc + 8;       // the epilogue's next unit, or
    volatile uint32_t *more_units = misc + 9;      // none (more_units == 0)

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
        for (uint32_t k = 0; k < kTcClcSlots; k++) {
            mbar_init(clc_full_bar(k), 1);
            mbar_init(clc_empty_bar(k), 2);        // the MMA issuer and the epilogue
        }
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
    // the set-up above ran beside the stream's previous kernel; global
    // memory is touched only after it has finished
    pdl_wait_primary();

    // The CTA's k-th unit is blockIdx.x for k = 0, then the CTA the k-th
    // cancellation request took over (one CTA of the grid per unit): each
    // role walks the same sequence, reading response k - 1 from slot
    // (k - 1) mod kTcClcSlots once its unit k - 1 is done.
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
            uint32_t recent[kTcRecent];     // the last units started, for the abort path
            uint32_t u = blockIdx.x, k = 0;
            bool asked = false;             // request k is in flight
            // request k: asked while unit k's last stage streams in, so that
            // the unit taken over is claimed as late as the pipeline allows
            auto ask = [&]() -> bool {
                if (!mbar_wait(clc_empty_bar(k), clc_parity(k) ^ 1u, abort)) return false;
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive_expect_tx(clc_full_bar(k), 16);
                clc_try_cancel(clc_resp(k), clc_full_bar(k));
                asked = true;
                return true;
            };
            for (;;) {
                recent[k % kTcRecent] = u;
                const int tiles = unit_tiles(n, u, unit_log2);
                const int stages = (tiles + kTcTilesPerStage - 1) / kTcTilesPerStage;
                const uint16_t *src = x + ((size_t)u << unit_log2);
                bool ok = stages > 0 || ask();
                for (int st = 0; st < stages && ok; st++) {
                    if (st == stages - 1 && !(ok = ask())) break;
                    if (!(ok = mbar_wait(empty_bar(s), phase ^ 1u, abort))) break;
                    const int nt = min(kTcTilesPerStage, tiles - st * kTcTilesPerStage);
                    const uint32_t bytes = (uint32_t)nt * kTcTileBytes;
                    mbar_arrive_expect_tx(full_bar(s), bytes);
                    bulk_copy_g2s(ring + (uint32_t)s * kTcStageBytes,
                                  src + (size_t)st * kTcTilesPerStage * kTcTileInputs, bytes, full_bar(s));
                    armed[s] = true;
                    armed_phase[s] = phase;
                    if (++s == kTcStages) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok || !mbar_wait(clc_full_bar(k), clc_parity(k), abort)) break;
                asked = false;
                uint32_t next;
                if (!clc_query(clc_resp(k), &next)) break;
                u = next;
                k++;
            }
            if (*abort) {
                // let the copies already issued land before the CTA exits
#pragma unroll
                for (int i = 0; i < kTcStages; i++)
                    if (armed[i]) (void)mbar_wait_limited(full_bar(i), armed_phase[i]);
                // the units started may lack a partial (the epilogue stops at
                // the failed unit): mark them NaN -- a finished one among them
                // may lose its value, the sum is NaN either way
                const float nan = __int_as_float(0x7fc00000);
                for (uint32_t j = 0; j < kTcRecent && j <= k; j++) dst[recent[(k - j) % kTcRecent]] = nan;
                // take over every CTA still waiting to launch and mark its unit
                if (!asked) {
                    mbar_arrive_expect_tx(clc_full_bar(k), 16);
                    clc_try_cancel(clc_resp(k), clc_full_bar(k));
                }
                for (;;) {
                    uint32_t v;
                    if (!mbar_wait_limited(clc_full_bar(k), clc_parity(k)) || !clc_query(clc_resp(k), &v))
                        break;
                    dst[v] = nan;
                    k++;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive_expect_tx(clc_full_bar(k), 16);
                    clc_try_cancel(clc_resp(k), clc_full_bar(k));
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
            // A host-requested stall leaves the first stage's last chain
            // unpublished (the epilogue waits for a stage's last chain), so
            // the epilogue's wait runs out its limit (failure-path test).
            bool withhold = inject_stall != 0u;
            auto end_chain = [&](bool ends_stage) {
                if (withhold && ends_stage)
                    withhold = false;
                else
                    tc_commit(dfull_bar(b));      // chain sub-result ready
                dphase ^= 1u << b;
                if (++b == kTcDBuffers) b = 0;
            };
            // one unit's MMAs: chains of R, each ending with its stage
            // (when R divides a stage they fall on stage boundaries anyway);
            // a whole stage is issued with static chain boundaries -- MMAs
            // issued under run-time chain logic issue several times slower
            auto unit_mmas = [&](int tiles) -> bool {
                bool ok = true;
                for (int t0 = 0; t0 < tiles && ok; t0 += kTcTilesPerStage) {
                    const int nt = min(kTcTilesPerStage, tiles - t0);
                    if (!mbar_wait(full_bar(s), phase, abort)) return false;
                    tc_fence_after();
                    const uint64_t sdesc = ring_desc + (uint64_t)s * kStageStep;
                    if (nt == kTcTilesPerStage) {
#pragma unroll
                        for (int t = 0; t < kTcTilesPerStage; t++) {
                            if (t % R == 0 && !(ok = begin_chain())) break;
                            tc_mma(tmem + (uint32_t)b * kTcDBufferStride, sdesc + (uint64_t)t * kTileStep,
                                   b_desc, idesc, t % R != 0 ? 1u : 0u);
                            if (t % R == R - 1 || t == kTcTilesPerStage - 1)
                                end_chain(t == kTcTilesPerStage - 1);
                        }
                    } else {
                        // a unit's last, partial stage (the array's end; every stage
                        // of the units of fewer than 8 tiles that small inputs use)
                        for (int t = 0; t < nt; t++) {
                            if (t % R == 0 && !(ok = begin_chain())) break;
                            tc_mma(tmem + (uint32_t)b * kTcDBufferStride, sdesc + (uint64_t)t * kTileStep,
                                   b_desc, idesc, t % R != 0 ? 1u : 0u);
                            if (t % R == R - 1 || t == nt - 1) end_chain(t == nt - 1);
                        }
                    }
                    tc_commit(empty_bar(s));                  // stage may be refilled
                    if (++s == kTcStages) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
                return ok;
            };
            uint32_t u = blockIdx.x, k = 0;
            for (;;) {
                if (!unit_mmas(unit_tiles(n, u, unit_log2)) || *abort) break;
                if (!mbar_wait(clc_full_bar(k), clc_parity(k), abort)) break;
                uint32_t next;
                const bool more = clc_query(clc_resp(k), &next);
                mbar_arrive(clc_empty_bar(k));
                if (!more) break;
                u = next;
                k++;
            }
            // every MMA issued has completed once the drain barrier flips
            tc_commit(drain_bar);
            (void)mbar_wait_limited(drain_bar, 0u);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warps 2..5, TMEM lanes 32*(warp%4) ..
        const int et = threadIdx.x - 64;                   // 0..127
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        int b = 0;
        uint32_t dphase = 0u;
        uint32_t u = blockIdx.x, k = 0;
        for (;;) {
            const int tiles = unit_tiles(n, u, unit_log2);
            float acc = 0.f;
            for (int t0 = 0; t0 < tiles; t0 += kTcTilesPerStage) {
                // the stage's chains (a chain ends with its stage): wait for the
                // last one -- its commit covers every MMA issued before it --
                // then read them together and add them in chain order
                const int nc = (min(kTcTilesPerStage, tiles - t0) + R - 1) / R;
                const int bl = (b + nc - 1) % kTcDBuffers;
                // the warp takes the wait's outcome together: tcgen05.ld is warp-wide
                const bool ok = !*abort && mbar_wait(dfull_bar(bl), (dphase >> bl) & 1u, abort);
                if (!__all_sync(kFull, ok)) break;
                tc_fence_after();
                uint32_t v[8];
                tc_ld_chain_cols(tmem + lane_base, kTcDBufferStride, b, nc, v);
#pragma unroll
                for (int i = 0; i < 8; i++)
                    if (i < nc) acc = __fadd_rn(acc, __uint_as_float(v[i]));
                tc_fence_before();
                for (int i = 0; i < nc; i++) {
                    mbar_arrive(dempty_bar(b));
                    dphase ^= 1u << b;
                    if (++b == kTcDBuffers) b = 0;
                }
            }
            // inputs of this unit past its whole tiles (only in the last unit)
            const size_t base = (size_t)u << unit_log2;
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
                // the next unit, for all four warps (one decision: the named
                // barriers below need every epilogue thread)
                uint32_t next = 0, more = 0;
                if (!*abort && mbar_wait(clc_full_bar(k), clc_parity(k), abort)) {
                    more = clc_query(clc_resp(k), &next) ? 1u : 0u;
                    mbar_arrive(clc_empty_bar(k));
                }
                *next_unit = next;
                *more_units = more;
            }
            named_sync(1, kTcEpilogueThreads);
            if (!*more_units) break;
            u = *next_unit;
            k++;
        }
    }

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

// Rows: one MMA tile holds 16 data rows, 8 TMEM lanes to a row.  A 64 KiB
// stage of the ring holds 16 G rows x S columns, row-major with a pitch of
// 2S bytes (S = 2048 columns and G = 1 for rows of more than 1024 columns,
// S = 1024 and G = 2 for rows of 768 to 1024; the library sends shorter
// rows to the mma.sync kernels), brought in by one 3-D tensor-map box (rows
// of whole 128-column blocks) or one 1-D bulk copy per row: either reads
// each row's bytes contiguously, 4 KiB at a time on long rows.
// Read through a K-major descriptor with no swizzle whose 8-row groups are
// one stage row apart and whose two K halves are 128 bytes apart, lane
// 8g + i of an MMA takes 16 inputs of data row g of its group (bytes 16i and
// 128 + 16i of the MMA's 256-byte column slice), so D lanes 8g .. 8g+7 hold
// row g's partial sums; the next MMA of a chain takes the next 128 columns
// of the same rows.  The MMAs cover a row's whole 128-column slices; the
// last cols % 128 inputs of a row are added by the epilogue from global
// memory; rows past the matrix are zero-filled by the tensor map or not
// copied at all (their lanes then hold stale values), and never stored.
// Work unit: 16 G rows x the whole row, or chunks of kTcRowsMaxChunkCols
// columns of longer rows; a chain ends with its stage; per row group the
// epilogue adds the chain results per lane, then each row's 8 lanes by an
// xor butterfly.
constexpr int kTcRowsGroup = 16;                       // data rows per MMA tile
constexpr int kTcRowsMmaCols = 128;                    // columns per MMA and row
constexpr int kTcRowsStageCols = 2048;                 // S of long rows (4 KiB a row)
constexpr int kTcRowsMinStageCols = 1024;              // S of the shortest rows (G = 2)
constexpr int kTcRowsStageBytes = kTcRowsGroup * kTcRowsStageCols * 2;     // 64 KiB
constexpr int kTcRowsStages = 3;                       // 192 KiB ring
constexpr size_t kTcRowsMaxChunkCols = 8192;           // columns per work unit, at most
constexpr int kTcRowsOffOnes = kTcRowsStages * kTcRowsStageBytes;
constexpr int kTcRowsOffBars = kTcRowsOffOnes + 1024;
constexpr int kTcRowsNumBars = 2 * kTcRowsStages + 2 * kTcDBuffers + 1;
constexpr int kTcRowsOffMisc = kTcRowsOffBars + 8 * kTcRowsNumBars;
constexpr int kTcRowsSmemBytes = kTcRowsOffMisc + 64 + 1024;

template <int DT, int R, bool SHORT>
__global__ void __launch_bounds__(kTcThreads, 1)
mma_tmem_rows_kernel(const __grid_constant__ CUtensorMap tmap, int use_map, const uint16_t *__restrict__ x,
                     size_t rows, size_t cols, size_t chunk_cols, size_t cpr, size_t units, int stage_cols,
                     float *__restrict__ dst, uint32_t inject_stall)
{
    pdl_launch_dependents();   // the combine may launch now; it waits for this grid to finish
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
    // G: row groups per unit (SHORT: rows of at most 1024 columns, G >= 2)
    const int groups = SHORT ? kTcRowsStageCols / stage_cols : 1;
    const int unit_rows = kTcRowsGroup * groups;
    const uint32_t pitch = 2u * (uint32_t)stage_cols;               // bytes per stage row
    // columns of column chunk c of a row, and of them the whole 128-column slices
    auto unit_cols = [&](size_t c) -> int {
        const size_t c0 = c * chunk_cols;
        return (int)(cols - c0 < chunk_cols ? cols - c0 : chunk_cols);
    };
    auto mma_cols = [&](int nc) -> int { return nc - nc % kTcRowsMmaCols; };
    // work unit u = (row block u / cpr, column chunk u % cpr), walked
    // u = blockIdx.x, + gridDim.x, ... with the quotient and remainder
    // carried (no 64-bit division per unit)
    struct Unit {
        size_t u, blk, chunk;
    };
    const size_t step_blk = gridDim.x / cpr, step_chunk = gridDim.x % cpr;
    auto first_unit = [&]() -> Unit { return {blockIdx.x, blockIdx.x / cpr, blockIdx.x % cpr}; };
    auto next_unit = [&](Unit &w) {
        w.u += gridDim.x;
        w.blk += step_blk;
        w.chunk += step_chunk;
        if (w.chunk >= cpr) {
            w.chunk -= cpr;
            w.blk++;
        }
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
        if (use_map) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmap) : "memory");
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
    // the set-up above ran beside the stream's previous kernel; global
    // memory is touched only after it has finished
    pdl_wait_primary();

    if (warp == 0) {
        // ---------------- producer: a stage is one 3-D tensor-map box (whole
        // 128-column rows), else one bulk copy per row, rows spread over the lanes
        int s = 0;
        uint32_t phase = 0;
        bool armed[kTcRowsStages];
        uint32_t armed_phase[kTcRowsStages];
        for (int i = 0; i < kTcRowsStages; i++) {
            armed[i] = false;
            armed_phase[i] = 0;
        }
        bool ok = true;
        for (Unit w = first_unit(); w.u < units && ok; next_unit(w)) {
            const size_t row0 = w.blk * (size_t)unit_rows;
            const size_t col0 = w.chunk * chunk_cols;
            const int live = (int)(rows - row0 < (size_t)unit_rows ? rows - row0 : (size_t)unit_rows);
            const int mc = mma_cols(unit_cols(w.chunk));
            for (int c = 0; c < mc; c += stage_cols) {
                const int sc = min(stage_cols, mc - c);
                const uint32_t row_bytes = (uint32_t)sc * 2u;
                if (lane == 0) {
                    ok = !*abort && mbar_wait(empty_bar(s), phase ^ 1u, abort);
                    if (ok && use_map) {
                        // box: 128 columns x S / 128 column blocks x 16 G rows (64 KiB,
                        // blocks and rows past the matrix zero-filled)
                        mbar_arrive_expect_tx(full_bar(s), (uint32_t)kTcRowsStageBytes);
                        tma_load_3d(ring + (uint32_t)s * kTcRowsStageBytes, &tmap, 0,
                                    (int)((col0 + (size_t)c) / kTcRowsMmaCols), (int)row0, full_bar(s));
                    } else if (ok) {
                        mbar_arrive_expect_tx(full_bar(s), (uint32_t)live * row_bytes);
                    }
                }
                ok = __shfl_sync(kFull, ok, 0);
                if (!ok) break;
                if (!use_map)
                    for (int r = lane; r < live; r += 32)
                        bulk_copy_g2s(ring + (uint32_t)s * kTcRowsStageBytes + (uint32_t)r * pitch,
                                      x + (row0 + (size_t)r) * cols + col0 + (size_t)c, row_bytes, full_bar(s));
                armed[s] = true;
                armed_phase[s] = phase;
                if (++s == kTcRowsStages) {
                    s = 0;
                    phase ^= 1u;
                }
            }
        }
        if (lane == 0 && *abort) {
            for (int i = 0; i < kTcRowsStages; i++) {
                if (!armed[i]) continue;
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(full_bar(i), armed_phase[i]) && global_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = instr_desc<DT>();
            const uint64_t b_desc = smem_desc(ones, 128, 256);
            // 8-row groups one stage row apart, K halves 128 bytes apart
            const uint64_t ring_desc = smem_desc(ring, 128, pitch);
            constexpr uint64_t kMmaStep = (uint64_t)(kTcRowsMmaCols * 2) >> 4;      // 256 bytes
            constexpr uint64_t kStageStep = (uint64_t)kTcRowsStageBytes >> 4;
            constexpr int kMmasPerStage = kTcRowsStageCols / kTcRowsMmaCols;         // 16 (G = 1)
            const uint64_t group_step = (uint64_t)(kTcRowsGroup * pitch) >> 4;
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
            for (Unit w = first_unit(); w.u < units && !*abort; next_unit(w)) {
                const int mmas = mma_cols(unit_cols(w.chunk)) / kTcRowsMmaCols;    // per row group
                bool ok = true;
                if constexpr (!SHORT) {
                    // one row group; its chains run along the row, each ending with its stage
                    for (int done = 0; done < mmas && ok; done += kMmasPerStage) {
                        const int nm = min(kMmasPerStage, mmas - done);
                        if (!mbar_wait(full_bar(s), phase, abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t sdesc = ring_desc + (uint64_t)s * kStageStep;
                        if (nm == kMmasPerStage) {
                            // whole stage: static chain boundaries (the MMAs issue
                            // several times slower under run-time chain logic)
#pragma unroll
                            for (int k = 0; k < kMmasPerStage; k++) {
                                if (k % R == 0 && !(ok = begin_chain())) break;
                                tc_mma(tmem + (uint32_t)b * kTcDBufferStride, sdesc + (uint64_t)k * kMmaStep,
                                       b_desc, idesc, k % R != 0 ? 1u : 0u);
                                if (k % R == R - 1 || k == kMmasPerStage - 1) end_chain();
                            }
                        } else {
                            // the row's (or chunk's) last, partial stage
                            auto issue = [&](int k, uint32_t acc) {
                                tc_mma(tmem + (uint32_t)b * kTcDBufferStride, sdesc + (uint64_t)k * kMmaStep,
                                       b_desc, idesc, acc);
                            };
                            ok = issue_chains_upto<R, kMmasPerStage - 1>(nm, begin_chain, end_chain, issue);
                        }
                        tc_commit(empty_bar(s));
                        if (++s == kTcRowsStages) {
                            s = 0;
                            phase ^= 1u;
                        }
                    }
                } else {
                    // G row groups of short rows in one stage, each row group its own chains
                    if (!mbar_wait(full_bar(s), phase, abort)) break;
                    tc_fence_after();
                    const uint64_t sdesc = ring_desc + (uint64_t)s * kStageStep;
                    for (int j = 0; j < groups && ok; j++) {
                        const uint64_t gdesc = sdesc + (uint64_t)j * group_step;
                        auto issue = [&](int k, uint32_t acc) {
                            tc_mma(tmem + (uint32_t)b * kTcDBufferStride, gdesc + (uint64_t)k * kMmaStep, b_desc,
                                   idesc, acc);
                        };
                        // a row group of short rows has at most 8 MMAs (S = 1024 columns)
                        ok = issue_chains_upto<R, kMmasPerStage / 2>(mmas, begin_chain, end_chain, issue);
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
        // ---------------- epilogue: TMEM lane m = 8g + i holds part of row g of a row group
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int m = 32 * (warp & 3) + lane;
        int b = 0;
        uint32_t dphase = 0u;
        for (Unit w = first_unit(); w.u < units; next_unit(w)) {
            const int nc = unit_cols(w.chunk);
            const int mc = mma_cols(nc);
            const int chains = stage_chains<R, kTcRowsStageCols / kTcRowsMmaCols>(mc / kTcRowsMmaCols);
            for (int j = 0; j < groups; j++) {
                float acc = 0.f;
                for (int c = 0; c < chains; c++) {
                    // the warp takes the wait's outcome together: tcgen05.ld is warp-wide
                    const bool ok = !*abort && mbar_wait(dfull_bar(b), (dphase >> b) & 1u, abort);
                    if (!__all_sync(kFull, ok)) break;
                    tc_fence_after();
                    acc = __fadd_rn(acc, tc_ld_lane(tmem + lane_base + (uint32_t)b * kTcDBufferStride));
                    tc_fence_before();
                    mbar_arrive(dempty_bar(b));
                    dphase ^= 1u << b;
                    if (++b == kTcDBuffers) b = 0;
                }
                const size_t row = w.blk * (size_t)unit_rows + (size_t)(kTcRowsGroup * j + (m >> 3));
                if (row < rows) {
                    // the row's last nc - mc inputs of the unit (fewer than 128):
                    // lane i adds inputs i, i + 8, ...
                    const uint16_t *t = x + row * cols + w.chunk * chunk_cols;
                    for (int q = mc + (m & 7); q < nc; q += 8)
                        acc = __fadd_rn(acc, DT == kF16 ? leaf_lo<kF16>(__ldg(t + q)) : leaf_lo<kBF16>(__ldg(t + q)));
                }
                // the row's 8 lanes (aligned within the warp): every lane gets the same bits
                acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, 1));
                acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, 2));
                acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, 4));
                if ((m & 7) == 0 && row < rows)
                    dst[row * cpr + w.chunk] = *abort ? __int_as_float(0x7fc00000) : acc;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTcTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- rows, flat

// Rows of 1024 k columns, k a divisor or a multiple of 16, laid out one
// after the other (row stride = cols): the matrix is read as the flat array
// it is, in the sum kernel's 32 KiB bulk copies, and only the MMA's view of
// a stage follows the rows.  A K-major descriptor with no swizzle, K halves
// 128 bytes apart and 8-row groups 2048 bytes apart gives MMA m of a stage
// (m = 0 .. 7, 256 bytes further each) lanes 8g + i the 16-byte pieces at
// 2048 g + 256 m + 16 i and + 128: over the stage's 8 MMAs the 8 lanes of
// group g take its 2 KiB (1024 inputs) g, which lies inside one row.  Row j
// of a stage of whole rows (k <= 16: 16 / k rows a stage) is TMEM lanes
// 8 k j .. 8 k (j + 1) - 1, a row of 16 384 inputs or more fills all 128
// lanes of each of its stages.  The epilogue adds a lane's chain results
// over the row's stages, then the row's lanes: an xor butterfly inside a
// warp, then the warps' totals in lane-quarter order, the same for every
// row whatever its position -- a row's bits depend on its inputs and cols
// only.  Every stage is 8 MMAs with static chain boundaries; lanes of the
// groups past the matrix in a unit's last stage read stale shared memory
// and are never stored.  Work unit: 65 536 / cols whole rows (65 536
// inputs), or one chunk of 65 536 columns of a longer row (partials merged
// by the rows combine).  One CTA per unit; the resident CTAs take over the
// rest by cluster launch control, as in the sum kernel.
constexpr int kFlatGroupInputs = 1024;                      // inputs of a lane group per stage
constexpr size_t kFlatUnitInputs = (size_t)1 << 16;         // 4 stages
// an MMA takes 256 bytes of each of the 16 lane groups: 8 MMAs cover a group's 2 KiB
constexpr int kFlatMmasPerStage = 2 * kFlatGroupInputs / (kTcRowsMmaCols * 2);
static_assert(kFlatMmasPerStage == 8 && 16 * 2 * kFlatGroupInputs == kTcStageBytes,
              "16 lane groups of 2 KiB fill a stage, 8 MMAs of 4 KiB");

__host__ __device__ inline bool flat_rows_shape(size_t cols)
{
    if (cols == 0 || cols % kFlatGroupInputs != 0) return false;
    const size_t k = cols / kFlatGroupInputs;
    return 16 % k == 0 || k % 16 == 0;
}

template <int DT, int R>
__global__ void __launch_bounds__(kTcThreads, kTcCtasPerSm)
mma_tmem_rows_flat_kernel(const uint16_t *__restrict__ x, uint32_t rows, uint32_t cols, uint32_t unit_rows,
                          uint32_t chunk_cols, uint32_t cpr, float *__restrict__ dst, uint32_t inject_stall)
{
    pdl_launch_dependents();   // the combine may launch now; it waits for this grid to finish
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
    auto clc_full_bar = [&](uint32_t k) { return drain_bar + 8u * (1u + k % kTcClcSlots); };
    auto clc_empty_bar = [&](uint32_t k) { return drain_bar + 8u * (1u + kTcClcSlots + k % kTcClcSlots); };
    auto clc_resp = [&](uint32_t k) { return sbase + kTcOffClc + 16u * (k % kTcClcSlots); };
    auto clc_parity = [](uint32_t k) { return (k / kTcClcSlots) & 1u; };
    uint32_t *misc = (uint32_t *)(smem + kTcOffMisc);
    volatile uint32_t *tmem_holder = misc;
    volatile uint32_t *abort = misc + 1;
    volatile float *red = (volatile float *)(misc + 4);
    volatile uint32_t *next_unit = misc + 8;
    volatile uint32_t *more_units = misc + 9;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t k_groups = cols / kFlatGroupInputs;             // lane groups per row
    // unit u: row block u / cpr (unit_rows rows), column chunk u % cpr
    // (chunk_cols columns); its inputs are contiguous
    auto unit_row0 = [&](uint32_t u) { return (size_t)(u / cpr) * unit_rows; };
    auto unit_col0 = [&](uint32_t u) { return (size_t)(u % cpr) * chunk_cols; };
    auto unit_inputs = [&](uint32_t u) -> size_t {
        const size_t r0 = unit_row0(u), c0 = unit_col0(u);
        const size_t live = rows - r0 < unit_rows ? rows - r0 : unit_rows;
        const size_t nc = cols - c0 < chunk_cols ? cols - c0 : chunk_cols;
        return live * nc;
    };
    auto unit_stages = [&](uint32_t u) {
        return (int)((unit_inputs(u) + kTcStageBytes / 2 - 1) / (kTcStageBytes / 2));
    };

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
        for (uint32_t k = 0; k < kTcClcSlots; k++) {
            mbar_init(clc_full_bar(k), 1);
            mbar_init(clc_empty_bar(k), 2);
        }
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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
    // the set-up above ran beside the stream's previous kernel; global
    // memory is touched only after it has finished
    pdl_wait_primary();

    if (warp == 0) {
        // ---------------- producer: the unit's contiguous inputs, 32 KiB a stage
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
            uint32_t recent[kTcRecent];
            uint32_t u = blockIdx.x, k = 0;
            bool asked = false;
            auto ask = [&]() -> bool {
                if (!mbar_wait(clc_empty_bar(k), clc_parity(k) ^ 1u, abort)) return false;
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive_expect_tx(clc_full_bar(k), 16);
                clc_try_cancel(clc_resp(k), clc_full_bar(k));
                asked = true;
                return true;
            };
            for (;;) {
                recent[k % kTcRecent] = u;
                const size_t total = unit_inputs(u);
                const int stages = unit_stages(u);
                const uint16_t *src = x + unit_row0(u) * cols + unit_col0(u);
                bool ok = true;
                for (int st = 0; st < stages && ok; st++) {
                    if (st == stages - 1 && !(ok = ask())) break;
                    if (!(ok = mbar_wait(empty_bar(s), phase ^ 1u, abort))) break;
                    const size_t i0 = (size_t)st * (kTcStageBytes / 2);
                    const size_t left = total - i0;
                    const uint32_t bytes = (uint32_t)(left < (size_t)kTcStageBytes / 2 ? left * 2 : kTcStageBytes);
                    mbar_arrive_expect_tx(full_bar(s), bytes);
                    bulk_copy_g2s(ring + (uint32_t)s * kTcStageBytes, src + i0, bytes, full_bar(s));
                    armed[s] = true;
                    armed_phase[s] = phase;
                    if (++s == kTcStages) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok || !mbar_wait(clc_full_bar(k), clc_parity(k), abort)) break;
                asked = false;
                uint32_t next;
                if (!clc_query(clc_resp(k), &next)) break;
                u = next;
                k++;
            }
            if (*abort) {
#pragma unroll
                for (int i = 0; i < kTcStages; i++)
                    if (armed[i]) (void)mbar_wait_limited(full_bar(i), armed_phase[i]);
                // the rows of the units started, and of every unit taken over
                // from here, are marked NaN (see the sum kernel)
                const float nan = __int_as_float(0x7fc00000);
                auto mark = [&](uint32_t v) {
                    const size_t r0 = unit_row0(v);
                    for (size_t r = r0; r < r0 + unit_rows && r < rows; r++) dst[r * cpr + v % cpr] = nan;
                };
                for (uint32_t j = 0; j < kTcRecent && j <= k; j++) mark(recent[(k - j) % kTcRecent]);
                if (!asked) {
                    mbar_arrive_expect_tx(clc_full_bar(k), 16);
                    clc_try_cancel(clc_resp(k), clc_full_bar(k));
                }
                for (;;) {
                    uint32_t v;
                    if (!mbar_wait_limited(clc_full_bar(k), clc_parity(k)) || !clc_query(clc_resp(k), &v))
                        break;
                    mark(v);
                    k++;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive_expect_tx(clc_full_bar(k), 16);
                    clc_try_cancel(clc_resp(k), clc_full_bar(k));
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer: 8 MMAs a stage, chains of R ending with it
        if (lane == 0) {
            const uint32_t idesc = instr_desc<DT>();
            const uint64_t b_desc = smem_desc(ones, 128, 256);
            const uint64_t ring_desc = smem_desc(ring, 128, 2 * kFlatGroupInputs);
            constexpr uint64_t kMmaStep = (uint64_t)(kTcRowsMmaCols * 2) >> 4;    // 256 bytes
            constexpr uint64_t kStageStep = kTcStageBytes >> 4;
            int s = 0, b = 0;
            uint32_t phase = 0, dphase = 0u;
            auto begin_chain = [&]() -> bool {
                if (!mbar_wait(dempty_bar(b), ((dphase >> b) & 1u) ^ 1u, abort)) return false;
                tc_fence_after();
                return true;
            };
            // a host-requested stall withholds the first stage's last chain
            bool withhold = inject_stall != 0u;
            auto end_chain = [&](bool ends_stage) {
                if (withhold && ends_stage)
                    withhold = false;
                else
                    tc_commit(dfull_bar(b));
                dphase ^= 1u << b;
                if (++b == kTcDBuffers) b = 0;
            };
            uint32_t u = blockIdx.x, k = 0;
            bool ok = true;
            for (;;) {
                const int stages = unit_stages(u);
                for (int st = 0; st < stages && ok; st++) {
                    if (!(ok = mbar_wait(full_bar(s), phase, abort))) break;
                    tc_fence_after();
                    const uint64_t sdesc = ring_desc + (uint64_t)s * kStageStep;
#pragma unroll
                    for (int m = 0; m < kFlatMmasPerStage; m++) {
                        if (m % R == 0 && !(ok = begin_chain())) break;
                        tc_mma(tmem + (uint32_t)b * kTcDBufferStride, sdesc + (uint64_t)m * kMmaStep, b_desc,
                               idesc, m % R != 0 ? 1u : 0u);
                        if (m % R == R - 1 || m == kFlatMmasPerStage - 1) end_chain(m == kFlatMmasPerStage - 1);
                    }
                    tc_commit(empty_bar(s));
                    if (++s == kTcStages) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok || *abort) break;
                if (!mbar_wait(clc_full_bar(k), clc_parity(k), abort)) break;
                uint32_t next;
                const bool more = clc_query(clc_resp(k), &next);
                mbar_arrive(clc_empty_bar(k));
                if (!more) break;
                u = next;
                k++;
            }
            tc_commit(drain_bar);
            (void)mbar_wait_limited(drain_bar, 0u);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: TMEM lane L = 32 q + lane, group L / 8
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t L = 32u * (uint32_t)q + (uint32_t)lane;
        constexpr int kChains = (kFlatMmasPerStage + R - 1) / R;
        // rows of a stage (k <= 16) or stages of a row chunk (k >= 16)
        const uint32_t lanes_per_row = k_groups <= 16 ? 8u * k_groups : 128u;
        const uint32_t rows_per_stage = k_groups <= 16 ? 16u / k_groups : 1u;
        const uint32_t stages_per_row = k_groups <= 16 ? 1u : k_groups / 16u;
        int b = 0;
        uint32_t dphase = 0u;
        uint32_t u = blockIdx.x, k = 0;
        for (;;) {
            const int stages = unit_stages(u);
            const size_t r0 = unit_row0(u);
            const uint32_t chunk = u % cpr;
            float acc = 0.f;
            bool ok = true;
            for (int st = 0; st < stages; st++) {
                // the stage's chains: wait for the last (its commit covers the
                // MMAs before it), read them together, add them in chain order
                const int bl = (b + kChains - 1) % kTcDBuffers;
                const bool w_ok = ok && !*abort && mbar_wait(dfull_bar(bl), (dphase >> bl) & 1u, abort);
                ok = __all_sync(kFull, w_ok);
                if (ok) {
                    tc_fence_after();
                    uint32_t v[8];
                    tc_ld_chain_cols(tmem + lane_base, kTcDBufferStride, b, kChains, v);
#pragma unroll
                    for (int i = 0; i < kChains; i++) acc = __fadd_rn(acc, __uint_as_float(v[i]));
                    tc_fence_before();
#pragma unroll
                    for (int i = 0; i < kChains; i++) {
                        mbar_arrive(dempty_bar(b));
                        dphase ^= 1u << b;
                        if (++b == kTcDBuffers) b = 0;
                    }
                }
                if ((uint32_t)(st + 1) % stages_per_row != 0 && st + 1 != stages) continue;
                // the stage ends rows (or the row's chunk): add each row's lanes
                for (uint32_t off = 1; off < 32u && off < lanes_per_row; off <<= 1)
                    acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, (int)off));
                const size_t row = r0 + (size_t)st / stages_per_row * rows_per_stage + L / lanes_per_row;
                const float nan = __int_as_float(0x7fc00000);
                if (lanes_per_row <= 32u) {
                    if ((L & (lanes_per_row - 1u)) == 0 && row < rows)
                        dst[row * cpr + chunk] = (*abort || !ok) ? nan : acc;
                } else {
                    // two or four warps to a row: their totals in lane-quarter order
                    if (lane == 0) red[q] = acc;
                    named_sync(1, kTcEpilogueThreads);
                    if (lanes_per_row == 64u && lane == 0 && (q & 1) == 0 && row < rows) {
                        const float v = __fadd_rn(red[q], red[q + 1]);
                        dst[row * cpr + chunk] = (*abort || !ok) ? nan : v;
                    } else if (lanes_per_row == 128u && et == 0 && row < rows) {
                        const float v = __fadd_rn(__fadd_rn(red[0], red[1]), __fadd_rn(red[2], red[3]));
                        dst[row * cpr + chunk] = (*abort || !ok) ? nan : v;
                    }
                    named_sync(1, kTcEpilogueThreads);
                }
                acc = 0.f;
            }
            if (et == 0) {
                uint32_t next = 0, more = 0;
                if (!*abort && mbar_wait(clc_full_bar(k), clc_parity(k), abort)) {
                    more = clc_query(clc_resp(k), &next) ? 1u : 0u;
                    mbar_arrive(clc_empty_bar(k));
                }
                *next_unit = next;
                *more_units = more;
            }
            named_sync(1, kTcEpilogueThreads);
            if (!*more_units) break;
            u = *next_unit;
            k++;
            named_sync(1, kTcEpilogueThreads);
        }
    }

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
// inputs); above that halved while it leaves fewer than one unit per two
// SMs of the 152 the rules assume, down to one tile: every unit a CTA takes
// over costs it a cancellation round trip, which small inputs cannot hide.
// A function of n only, so the chunking (and MMA_CHAIN's bits) is the same
// on every device.
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
    cudaError_t e = set_smem_once(k, kTcSmemBytes, kTcCarveoutPercent);
    if (e != cudaSuccess) return e;
    // one CTA per unit: the CTAs running take over those still waiting to
    // launch (cluster launch control), so fast SMs take more units
    const size_t units = tmem_units(n);
    if (units != (size_t)grid) return cudaErrorInvalidValue;
    int unit_log2 = tmem_unit_log2(n);
    uint32_t stall = inject_stall ? 1u : 0u;
    void *args[] = {(void *)&x, (void *)&n, (void *)&unit_log2, (void *)&dst, (void *)&stall};
    return launch_first(k, dim3(grid), dim3(kTcThreads), args, kTcSmemBytes, stream);
}

template <int DT, bool SHORT>
static void *pick_rows_dt(int R)
{
    switch (R) {
    case 1: return (void *)mma_tmem_rows_kernel<DT, 1, SHORT>;
    case 2: return (void *)mma_tmem_rows_kernel<DT, 2, SHORT>;
    case 3: return (void *)mma_tmem_rows_kernel<DT, 3, SHORT>;
    case 4: return (void *)mma_tmem_rows_kernel<DT, 4, SHORT>;
    case 5: return (void *)mma_tmem_rows_kernel<DT, 5, SHORT>;
    case 6: return (void *)mma_tmem_rows_kernel<DT, 6, SHORT>;
    case 7: return (void *)mma_tmem_rows_kernel<DT, 7, SHORT>;
    case 8: return (void *)mma_tmem_rows_kernel<DT, 8, SHORT>;
    default: return nullptr;
    }
}

// Work units: 16 G rows (G = row groups per stage, tmem_rows_stage_cols)
// x the whole row up to kTcRowsMaxChunkCols columns, else chunks of that
// many.  A function of cols only, so a row's chains (and MMA_CHAIN's bits)
// do not depend on the number of rows or the device.
size_t tmem_rows_chunks(size_t cols)
{
    if (flat_rows_shape(cols)) return (cols + kFlatUnitInputs - 1) / kFlatUnitInputs;
    return (cols + kTcRowsMaxChunkCols - 1) / kTcRowsMaxChunkCols;
}

// Rows of the flat layout: 65 536 / cols whole rows a unit, or one row
// (its chunks of 65 536 columns being units of their own).
static size_t flat_unit_rows(size_t cols)
{
    return cols < kFlatUnitInputs ? kFlatUnitInputs / cols : 1;
}

// S: the columns of a row in one stage -- 2048, or 1024 for rows whose
// whole 128-column slices fit 1024 columns; G = 2048 / S row groups share a
// stage.
static int tmem_rows_stage_cols(size_t cols)
{
    const size_t mc = (cols < kTcRowsMaxChunkCols ? cols : kTcRowsMaxChunkCols) / kTcRowsMmaCols *
                      kTcRowsMmaCols;
    int s = kTcRowsMinStageCols;
    while (s < kTcRowsStageCols && (size_t)s < mc) s *= 2;
    return s;
}

size_t tmem_rows_units(size_t rows, size_t cols)
{
    if (flat_rows_shape(cols)) {
        const size_t ur = flat_unit_rows(cols);
        return ((rows + ur - 1) / ur) * tmem_rows_chunks(cols);
    }
    const size_t unit_rows = (size_t)kTcRowsGroup * (kTcRowsStageCols / tmem_rows_stage_cols(cols));
    return ((rows + unit_rows - 1) / unit_rows) * tmem_rows_chunks(cols);
}

cudaError_t launch_mma_tmem_rows(int dtype, int R, const uint16_t *x, size_t rows, size_t cols,
                                 float *dst, int grid, bool inject_stall, cudaStream_t stream)
{
    uint32_t stall = inject_stall ? 1u : 0u;
    if (flat_rows_shape(cols)) {
        // one CTA per unit, the resident ones taking over the rest
        void *k = nullptr;
        switch (R) {
#define TCR_FLAT_CASE(r)                                                                              \
    case r:                                                                                           \
        k = dtype == kF16 ? (void *)mma_tmem_rows_flat_kernel<kF16, r> : (void *)mma_tmem_rows_flat_kernel<kBF16, r>; \
        break;
            TCR_FLAT_CASE(1) TCR_FLAT_CASE(2) TCR_FLAT_CASE(3) TCR_FLAT_CASE(4)
            TCR_FLAT_CASE(5) TCR_FLAT_CASE(6) TCR_FLAT_CASE(7) TCR_FLAT_CASE(8)
#undef TCR_FLAT_CASE
        default: return cudaErrorInvalidValue;
        }
        const size_t units = tmem_rows_units(rows, cols);
        if (units != (size_t)grid || rows >= ((size_t)1 << 31) || cols >= ((size_t)1 << 31))
            return cudaErrorInvalidValue;
        cudaError_t e = set_smem_once(k, kTcSmemBytes, kTcCarveoutPercent);
        if (e != cudaSuccess) return e;
        uint32_t r32 = (uint32_t)rows, c32 = (uint32_t)cols, ur = (uint32_t)flat_unit_rows(cols);
        uint32_t cc = (uint32_t)(cols < kFlatUnitInputs ? cols : kFlatUnitInputs);
        uint32_t cpr = (uint32_t)tmem_rows_chunks(cols);
        void *args[] = {(void *)&x, (void *)&r32, (void *)&c32, (void *)&ur, (void *)&cc, (void *)&cpr,
                        (void *)&dst, (void *)&stall};
        return launch_first(k, dim3(grid), dim3(kTcThreads), args, kTcSmemBytes, stream);
    }
    int stage_cols = tmem_rows_stage_cols(cols);
    const bool short_rows = stage_cols < kTcRowsStageCols;
    void *k = dtype == kF16 ? (short_rows ? pick_rows_dt<kF16, true>(R) : pick_rows_dt<kF16, false>(R))
                            : (short_rows ? pick_rows_dt<kBF16, true>(R) : pick_rows_dt<kBF16, false>(R));
    if (!k) return cudaErrorInvalidValue;
    cudaError_t e = set_smem_once(k, kTcRowsSmemBytes);
    if (e != cudaSuccess) return e;
    size_t chunk_cols = kTcRowsMaxChunkCols;
    size_t cpr = tmem_rows_chunks(cols);
    size_t units = tmem_rows_units(rows, cols);
    // rows of whole 128-column blocks: a 3-D view (128 columns, cols / 128
    // blocks, rows) whose 64 KiB box is one stage as laid out above
    alignas(64) CUtensorMap map;
    std::memset(&map, 0, sizeof map);
    int use_map = 0;
    if (cols % kTcRowsMmaCols == 0) {
        PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
        if (!encode) return cudaErrorNotSupported;
        const cuuint64_t gdim[3] = {(cuuint64_t)kTcRowsMmaCols, (cuuint64_t)(cols / kTcRowsMmaCols),
                                    (cuuint64_t)rows};
        const cuuint64_t gstride[2] = {(cuuint64_t)kTcRowsMmaCols * 2, (cuuint64_t)cols * 2};
        const cuuint32_t box[3] = {(cuuint32_t)kTcRowsMmaCols, (cuuint32_t)(stage_cols / kTcRowsMmaCols),
                                   (cuuint32_t)(kTcRowsGroup * (kTcRowsStageCols / stage_cols))};
        const cuuint32_t estride[3] = {1, 1, 1};
        if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, (void *)x, gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        use_map = 1;
    }
    void *args[] = {(void *)&map, (void *)&use_map, (void *)&x, (void *)&rows, (void *)&cols,
                    (void *)&chunk_cols, (void *)&cpr, (void *)&units, (void *)&stage_cols,
                    (void *)&dst, (void *)&stall};
    return launch_first(k, dim3(grid), dim3(kTcThreads), args, kTcRowsSmemBytes, stream);
}

int tmem_rows_grid(size_t rows, size_t cols, size_t sms)
{
    const size_t units = tmem_rows_units(rows, cols);
    if (flat_rows_shape(cols)) return units < ((size_t)1 << 31) ? (int)units : 0;
    return (int)(units < sms ? units : sms);
}

cudaError_t read_device_faults(unsigned int *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_tc05_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0u;
    return cudaMemcpyToSymbol(g_tc05_fault, &zero, sizeof(unsigned int));
}

}  // namespace tcr
