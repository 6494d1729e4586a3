// k_blocked.cu -- FIXED_ORDER's second declared order, blocked-sequential-
// then-tree, for runs longer than a vector.
//
// "Taming Bitwise Behavior in GPU Kernels with Tensor Core" (arXiv
// 2609.11356), Abstract: an order pinned by a descriptor makes results
// reproducible.  Here the caller chooses a run length C = 2^run_log2: every
// run of C consecutive inputs is added left to right in binary32, and the
// balanced tree (over index order, -0.0 pad) runs over the run values.
//
// A run is a serial chain, so each lane owns whole runs: a round is 32
// consecutive pieces of P = max(C, 8V) inputs (V inputs per 16-byte
// vector), lane j's piece the j-th -- one run, or 8V / C short runs.  A pass
// moves the next 8 vectors of every piece of the round: warp load k has lane
// L fetch vector L mod 8 of piece 4k + L / 8, so each load instruction reads
// four whole 128-byte lines.  The vectors go through a per-warp shared-memory
// stage (rows padded by one vector so neither the writes nor the
// lane-per-row reads conflict), then lane j adds its row's leaves in order.
// The next pass's loads are issued before the current pass is added.  A
// lane's short runs end in a lane-local binary counter (the balanced tree
// over them); after P / 8V passes the lane holds its piece's value, the
// lane-order butterfly forms the round's subtree, a binary counter the warp
// span's, a shared-memory tree the CTA chunk's, and the combine kernel the
// segment's -- every one an aligned subtree of the declared tree.  Runs of
// at most one vector go through the warp stream instead (k_fixed.cu,
// vec_runs).
#include "stream.cuh"

namespace tcr {

constexpr int kBlockedMaxWarps = 8;
constexpr int kStageRow = 9;    // vectors per stage row: 8 + 1 of padding
constexpr size_t kStageBytesPerWarp = 32 * kStageRow * sizeof(uint4);

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(32 * kBlockedMaxWarps, 4)
blocked_chunk_kernel(const void *__restrict__ xv, size_t seg_len, size_t units, size_t cps,
                     int chunk_log2, int run_log2, float *__restrict__ dst)
{
    pdl_launch_dependents();   // the combine may launch now; it waits for this grid to finish
    pdl_wait_primary();        // the stream's previous kernel has finished
    using T = typename Elem<DT>::T;
    constexpr int V = Elem<DT>::kPerVec;
    constexpr int LV = V == 8 ? 3 : 2;
    extern __shared__ uint4 stage[];                  // kStageBytesPerWarp per warp
    __shared__ float warp_val[kBlockedMaxWarps];
    const T *__restrict__ x = static_cast<const T *>(xv);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    // piece of 2^piece_log2 inputs per lane and round; run_log2 > LV
    const int piece_log2 = run_log2 > LV + 3 ? run_log2 : LV + 3;
    const int lpasses = piece_log2 - LV - 3;                  // log2 passes per round
    const int vrun_log2 = run_log2 - LV;                       // vectors per run (log2)
    const bool short_runs = run_log2 < LV + 3;                 // several runs per piece
    const int span_log2 = chunk_log2 - ceil_log2_sz((size_t)nwarps);
    const size_t steps = (size_t)1 << (span_log2 - piece_log2 - 5 + lpasses);
    const size_t nvec = (seg_len + V - 1) / V;
    const uint32_t nz = Elem<DT>::kNegZeroWord;
    uint4 *buf = stage + warp * (32 * kStageRow);

    for (size_t u = blockIdx.x; u < units; u += gridDim.x) {
        const size_t s = u / cps;
        const T *seg = x + s * seg_len;
        const size_t wbase = ((u - s * cps) << chunk_log2) + ((size_t)warp << span_log2);
        // step t = round (t >> lpasses), pass (t & (passes - 1)); the vector
        // that slot k of this lane loads at step t
        auto vec_of = [&](size_t t, int k) -> size_t {
            const size_t r = t >> lpasses, p = t & (((size_t)1 << lpasses) - 1);
            const size_t off = wbase + (r << (piece_log2 + 5)) +
                               ((size_t)(4 * k + (lane >> 3)) << piece_log2) + (p << (LV + 3)) +
                               (size_t)(lane & 7) * V;
            return off / V;
        };
        uint4 q[8];
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const size_t v = vec_of(0, k);
            q[k] = v < nvec ? ld_vec<DT, ALIGNED, true>(seg, seg_len, v) : make_uint4(nz, nz, nz, nz);
        }
        TreeCounter<5> tc;            // rounds of the span
        TreeCounter<3> lane_tc;       // short runs of the lane's piece (at most 4)
        float run = -0.0f;
#pragma unroll 1
        for (size_t t = 0; t < steps; t++) {
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; k++) buf[(4 * k + (lane >> 3)) * kStageRow + (lane & 7)] = q[k];
            __syncwarp();
            if (t + 1 < steps) {
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const size_t v = vec_of(t + 1, k);
                    q[k] = v < nvec ? ld_vec<DT, ALIGNED, true>(seg, seg_len, v)
                                    : make_uint4(nz, nz, nz, nz);
                }
            }
#pragma unroll
            for (int k = 0; k < 8; k++) {
                run = vec_seq_add<DT>(run, buf[lane * kStageRow + k]);
                if (short_runs && ((k + 1) & ((1 << vrun_log2) - 1)) == 0) {
                    lane_tc.push(run);
                    run = -0.0f;
                }
            }
            if (((t + 1) & (((size_t)1 << lpasses) - 1)) == 0) {
                // the round: the lane-order tree over 32 pieces
                float piece = run;
                if (short_runs) {
                    piece = lane_tc.finish();
                    lane_tc = TreeCounter<3>();
                }
                tc.push(warp_tree_lane_order(piece));
                run = -0.0f;
            }
        }
        const float w = tc.finish();
        if (lane == 0) warp_val[warp] = w;
        __syncthreads();
        if (warp == 0) {
            const float c = warp_tree_lane_order(lane < nwarps ? warp_val[lane] : -0.0f);
            if (lane == 0) dst[u] = c;
        }
        __syncthreads();
    }
}

// Rows of at most 16 pieces (a row's pieces padded to 2^lpr, lpr <= 4): a
// round of 32 pieces holds 32 >> lpr whole rows, lane group i (2^lpr
// lanes) row i's pieces in order; the passes, the stage and the lanes' runs
// are those of blocked_chunk_kernel, and the round ends in each row's tree
// over its pieces -- the lane-order butterfly over its 2^lpr lanes.  With
// one row to a round, the pieces past the row are -0.0 and the butterfly's
// upper levels would add only -0.0 to the row's tree, so the bits are the
// same; the round is no longer half padding.  Each warp walks the rounds
// grid-stride; there are no partials.
template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(32 * kBlockedMaxWarps, 4)
blocked_rows_kernel(const void *__restrict__ xv, size_t rows, size_t cols, int run_log2, int lpr,
                    float *__restrict__ out)
{
    pdl_launch_dependents();
    pdl_wait_primary();        // the stream's previous kernel has finished
    using T = typename Elem<DT>::T;
    constexpr int V = Elem<DT>::kPerVec;
    constexpr int LV = V == 8 ? 3 : 2;
    extern __shared__ uint4 stage[];                  // kStageBytesPerWarp per warp
    const T *__restrict__ x = static_cast<const T *>(xv);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int piece_log2 = run_log2 > LV + 3 ? run_log2 : LV + 3;
    const int passes = 1 << (piece_log2 - LV - 3);
    const int vrun_log2 = run_log2 - LV;
    const bool short_runs = run_log2 < LV + 3;
    const size_t rpr = (size_t)32 >> lpr;                     // rows per round
    const size_t rounds = (rows + rpr - 1) / rpr;
    const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
    const uint32_t nz = Elem<DT>::kNegZeroWord;
    uint4 *buf = stage + warp * (32 * kStageRow);
    // slot k of this lane at pass p of round r: vector lane mod 8 of piece
    // 4k + lane / 8, i.e. of piece q of row i of the round
    auto load = [&](size_t r, int p, int k) -> uint4 {
        const int piece = 4 * k + (lane >> 3);
        const size_t row = r * rpr + (size_t)(piece >> lpr);
        const size_t e = ((size_t)(piece & ((1 << lpr) - 1)) << piece_log2) + ((size_t)p << (LV + 3)) +
                         (size_t)(lane & 7) * V;
        if (row >= rows || e >= cols) return make_uint4(nz, nz, nz, nz);
        return ld_vec<DT, ALIGNED, true>(x + row * cols, cols, e / V);
    };
    size_t r = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (r >= rounds) return;
    uint4 q[8];
#pragma unroll
    for (int k = 0; k < 8; k++) q[k] = load(r, 0, k);
    TreeCounter<3> lane_tc;       // short runs of the lane's piece (at most 4)
    float run = -0.0f;
    int p = 0;
#pragma unroll 1
    for (;;) {
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; k++) buf[(4 * k + (lane >> 3)) * kStageRow + (lane & 7)] = q[k];
        __syncwarp();
        size_t nr = r;
        int np = p + 1;
        if (np == passes) {
            np = 0;
            nr = r + nw;
        }
        const bool more = nr < rounds;
        if (more) {
#pragma unroll
            for (int k = 0; k < 8; k++) q[k] = load(nr, np, k);
        }
#pragma unroll
        for (int k = 0; k < 8; k++) {
            run = vec_seq_add<DT>(run, buf[lane * kStageRow + k]);
            if (short_runs && ((k + 1) & ((1 << vrun_log2) - 1)) == 0) {
                lane_tc.push(run);
                run = -0.0f;
            }
        }
        if (p == passes - 1) {
            float piece = run;
            if (short_runs) {
                piece = lane_tc.finish();
                lane_tc = TreeCounter<3>();
            }
            // the row's tree over its 2^lpr pieces, in lane order
            for (int off = 1; off < (1 << lpr); off <<= 1)
                piece = __fadd_rn(piece, __shfl_xor_sync(kFull, piece, off));
            const size_t row = r * rpr + (size_t)(lane >> lpr);
            if ((lane & ((1 << lpr) - 1)) == 0 && row < rows) out[row] = piece;
            run = -0.0f;
        }
        if (!more) break;
        r = nr;
        p = np;
    }
}

// ---------------------------------------------------------------- host

static const void *pick(int dtype, bool aligned)
{
    switch (dtype) {
    case kF16: return aligned ? (const void *)blocked_chunk_kernel<kF16, true>
                              : (const void *)blocked_chunk_kernel<kF16, false>;
    case kBF16: return aligned ? (const void *)blocked_chunk_kernel<kBF16, true>
                               : (const void *)blocked_chunk_kernel<kBF16, false>;
    case kF32: return aligned ? (const void *)blocked_chunk_kernel<kF32, true>
                              : (const void *)blocked_chunk_kernel<kF32, false>;
    default: return nullptr;
    }
}

cudaError_t launch_blocked_chunk(int dtype, bool aligned, const void *x, size_t seg_len,
                                 size_t units, size_t cps, int chunk_log2, int run_log2,
                                 float *dst, int grid, int block, cudaStream_t stream)
{
    const void *k = pick(dtype, aligned);
    if (!k || block < 32 || block > 32 * kBlockedMaxWarps) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&seg_len, (void *)&units, (void *)&cps,
                    (void *)&chunk_log2, (void *)&run_log2, (void *)&dst};
    return launch_first(k, dim3(grid), dim3(block), args, kStageBytesPerWarp * (block / 32), stream);
}

static const void *pick_rows(int dtype, bool aligned)
{
    switch (dtype) {
    case kF16: return aligned ? (const void *)blocked_rows_kernel<kF16, true>
                              : (const void *)blocked_rows_kernel<kF16, false>;
    case kBF16: return aligned ? (const void *)blocked_rows_kernel<kBF16, true>
                               : (const void *)blocked_rows_kernel<kBF16, false>;
    case kF32: return aligned ? (const void *)blocked_rows_kernel<kF32, true>
                              : (const void *)blocked_rows_kernel<kF32, false>;
    default: return nullptr;
    }
}

cudaError_t launch_blocked_rows(int dtype, bool aligned, const void *x, size_t rows, size_t cols,
                                int run_log2, int lpr, float *out, int grid, int block, cudaStream_t stream)
{
    const void *k = pick_rows(dtype, aligned);
    if (!k || block < 32 || block > 32 * kBlockedMaxWarps || lpr < 0 || lpr > 4) return cudaErrorInvalidValue;
    void *args[] = {(void *)&x, (void *)&rows, (void *)&cols, (void *)&run_log2, (void *)&lpr, (void *)&out};
    return launch_first(k, dim3(grid), dim3(block), args, kStageBytesPerWarp * (block / 32), stream);
}

}  // namespace tcr
