// tcr_api.cu -- the C ABI of libtcr: argument checks, launch planning,
// stream-ordered scratch and the launch sequence of every call.
//
// The calls follow "GPU Tensor Cores for fast Arithmetic Reductions"
// (arXiv 2001.05585), Abstract: the arithmetic reduction of n numbers into
// one 32-bit result (tcr_reduce_sum), and the same per row (tcr_reduce_rows).
// The order descriptor restates for sums the descriptor of reduction order
// of "Taming Bitwise Behavior in GPU Kernels with Tensor Core" (arXiv
// 2609.11356), Abstract.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/tcr.h"
#include "kernels.cuh"
#include "plan.h"

namespace tcr {
namespace plan {


// -------------------------------------------------------------- devices

struct DeviceState {
    bool init = false;
    int sms = kRuleSMs;
    cudaMemPool_t pool = nullptr;
};

std::mutex g_mu;
std::vector<DeviceState> g_dev;

struct OccKey {
    int dev, fam, rows, dtype, aligned, R, block;
    bool operator==(const OccKey &o) const { return std::memcmp(this, &o, sizeof *this) == 0; }
};
std::vector<std::pair<OccKey, int>> g_occ;

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    return dev;
}

int sm_count(int dev)
{
    if (dev < 0) return kRuleSMs;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
    DeviceState &d = g_dev[dev];
    if (!d.init) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
            d.sms = n;
        else
            (void)cudaGetLastError();
        d.init = true;
    }
    return d.sms;
}

// The library's stream-ordered pool on `dev`.  Its release threshold keeps
// freed blocks reserved, so a steady stream of calls does not go back to
// the driver for memory.
cudaMemPool_t pool_for(int dev)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
    DeviceState &d = g_dev[dev];
    if (!d.pool) {
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof props);
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        uint64_t keep = UINT64_MAX;
        (void)cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        d.pool = p;
    }
    return d.pool;
}


int occupancy(int dev, Family fam, bool rows, int dtype, int op, bool aligned, int R, int block)
{
    OccKey key{dev, (int)fam, (rows ? 1 : 0) | (op << 1), dtype, aligned ? 1 : 0, R, block};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (auto &e : g_occ)
            if (e.first == key) return e.second;
    }
    int n = 0;
    if (dev >= 0) {
        switch (fam) {
        case kPackedF:
            // R carries the pair flag, the packed family, the row width and
            // the chain length
            n = occupancy_packed((R / 100) % 10, dtype, op, R % 10, (R / 10) % 10, aligned, R >= 1000);
            break;
        }
    }
    if (n <= 0) n = 1;
    std::lock_guard<std::mutex> lk(g_mu);
    g_occ.emplace_back(key, n);
    return n;
}

int log2_exact(int v)
{
    int l = 0;
    while ((1 << l) < v) l++;
    return l;
}

int ceil_log2_sz(size_t n)
{
    int h = 0;
    while (((size_t)1 << h) < n) h++;
    return h;
}

// Default chain length.  The Abstract of arXiv 2001.05585 finds R = 4 or 5
// best for 32- and 128-thread blocks and R = 1 for large ones; on GB300 the
// sum of 2^28 values is fastest at R = 4 for every block size (R = 1 and 2
// flush more often and hold more live registers), so R = 4 is the default
// throughout.
int default_R(int)
{
    return 4;
}

size_t elem_bytes(int dtype)
{
    return dtype == TCR_F32 ? 4 : 2;
}

// Inputs per 16-byte vector: 8 of 16 bits, 4 of binary32.
int vector_len(int dtype)
{
    return (int)(16 / elem_bytes(dtype));
}

tcr_status check_mode(const tcr_mode &m, int *block, int *R)
{
    if (m.kind < TCR_MMA_CHAIN || m.kind > TCR_MMA_CHAIN_TMEM) return TCR_ERR_INVALID_ARG;
    if (m.dtype != TCR_F16 && m.dtype != TCR_BF16 && m.dtype != TCR_F32) return TCR_ERR_INVALID_ARG;
    if (m.run_log2 < 0 || m.run_log2 > kMaxRunLog2) return TCR_ERR_INVALID_ARG;
    if (m.run_log2 != 0 && m.kind != TCR_FIXED_ORDER) return TCR_ERR_INVALID_ARG;
    int b = m.block_threads == 0 ? kDefaultBlock : m.block_threads;
    if (b < 32 || b > 1024 || (b & (b - 1)) != 0) return TCR_ERR_INVALID_ARG;
    int r = 0;
    if (m.kind == TCR_MMA_CHAIN || m.kind == TCR_MMA_CHAIN_TMEM) {
        if (m.R < 0 || m.R > 8) return TCR_ERR_INVALID_ARG;
        r = m.R == 0 ? default_R(b) : m.R;
    }
    *block = b;
    *R = r;
    return TCR_OK;
}

tcr_status check_common(const void *x, size_t total, const float *out, const tcr_mode &mode,
                        int *block, int *R)
{
    if (!out || ((uintptr_t)out & 3u) != 0) return TCR_ERR_INVALID_ARG;
    if (total >= kMaxInputs) return TCR_ERR_INVALID_ARG;
    tcr_status st = check_mode(mode, block, R);
    if (st != TCR_OK) return st;
    // x is aligned to its pattern type: 2 bytes, or 4 for binary32
    if (total > 0 && (!x || ((uintptr_t)x & (elem_bytes(mode.dtype) - 1)) != 0))
        return TCR_ERR_INVALID_ARG;
    return TCR_OK;
}

// may_shrink: the CTA size is free to choose (FIXED_ORDER, whose bits never
// depend on it, or a default block size): a sum small enough for one CTA
// whose warps take at most two groups each (2^17 16-bit or 2^16 binary32
// inputs) is one work unit -- one launch, no partials, no scratch; larger
// small inputs get smaller CTAs, then shorter warp spans (16 KiB down to
// one 4 KiB group), until there are two work units per SM of the 152 the
// rules assume.  Both are fixed functions of the input length, so
// MMA_CHAIN's chunking (reported by the descriptor) is the same on every
// device.
ChunkSplit chunk_split(size_t segments, size_t seg_len, int dtype, int block, bool may_shrink)
{
    ChunkSplit c;
    int span_log2 = kWarpSpanBytesLog2 - log2_exact((int)elem_bytes(dtype));
    const int group_log2 = kGroupBytesLog2 - log2_exact((int)elem_bytes(dtype));
    if (may_shrink && segments == 1 && seg_len <= ((size_t)1 << (group_log2 + 1 + 5))) {
        // one CTA: spans of one group (two above 32 groups), as few warps as cover it
        span_log2 = seg_len > ((size_t)1 << (group_log2 + 5)) ? group_log2 + 1 : group_log2;
        int warps = 1;
        while (((size_t)warps << span_log2) < seg_len) warps *= 2;
        c.block = 32 * warps;
        c.chunk_log2 = span_log2 + log2_exact(warps);
        c.cps = 1;
        return c;
    }
    c.block = block;
    for (;;) {
        c.chunk_log2 = span_log2 + log2_exact(c.block / 32);
        c.cps = (seg_len + ((size_t)1 << c.chunk_log2) - 1) >> c.chunk_log2;
        if (!may_shrink || segments * c.cps >= (size_t)2 * kRuleSMs) break;
        if (c.block > 32)
            c.block /= 2;
        else if (span_log2 > group_log2)
            span_log2--;
        else
            break;
    }
    return c;
}

}  // namespace plan
}  // namespace tcr

namespace {

using namespace tcr;
using namespace tcr::plan;

// -------------------------------------------------------------- planning

enum Path {
    kPathEmpty,          // nothing to reduce: memset out to +0.0
    kPathChunk,          // FIXED / MMA chunked kernel (+ combine if cps > 1)
    kPathFixedRowsWarp,  // FIXED, one warp per row
    kPathMmaRows,        // MMA, one warp per row
    kPathShuffleBlock,   // SHUFFLE block team (+ combine if G > 1)
    kPathShuffleRowsWarp, // SHUFFLE warp team, one warp per row
    kPathTmem,           // MMA_CHAIN on tcgen05 (+ combine if units > 1)
    kPathTmemRows,       // MMA_CHAIN rows on tcgen05 (+ combine if chunks > 1)
    kPathBlocked,        // FIXED blocked order, runs longer than a vector (+ combine)
    kPathBlockedRows,    // FIXED blocked order, rows of at most 16 pieces: several to a round
    kPathPackedRows      // short rows, several to a warp group (FIXED, SHUFFLE, MMA)
};

struct Plan {
    int kind, dtype, op, R, block;
    int run_log2;            // blocked order: log2 run length (0: the plain tree)
    int vrun;                // runs inside a vector: the warp-stream kernels' variant
    int packed, vlog;        // packed rows: kernel family, log2 vector slots per row
    bool aligned;
    Path path;
    size_t segments, seg_len;
    int grid, chunk_log2;
    size_t cps, units;       // chunks per segment, CTA work units
    int team_threads, team_blocks;
    size_t partials;         // fp32 scratch entries (0: writes out directly)
    size_t combine_count;    // partials per segment for the combine
    int launches;
};


// The declared SHUFFLE_TREE team for a segment of L inputs, in vectors of
// V inputs, at block size B: one warp for segments of at most 1024
// vectors, else G blocks of B threads with about 16 vectors per thread.
// (G is not capped at one wave of resident blocks: the blocks of a large
// segment run in several waves, which the block scheduler balances over
// the SMs -- a 2^30-input sum took 298.6 us with the team capped at
// 152 * 1024 threads, 290.6 us without.)
void shuffle_team(size_t L, int V, int B, int *Bt, int *G)
{
    const size_t nvec = (L + (size_t)V - 1) / (size_t)V;
    if (nvec <= 1024) {
        *Bt = 32;
        *G = 1;
        return;
    }
    const size_t per_block = (size_t)B * 16;
    size_t g = (nvec + per_block - 1) / per_block;
    if (g < 1) g = 1;
    *Bt = B;
    *G = (int)g;
}


// Grids of the warp-stream kernels.  Their CTAs walk work units (chunks,
// rows) grid-stride, so any grid gives the same bits.  They are launched
// with one CTA per unit (per 8 rows): the hardware block scheduler hands
// the next CTA to whichever SM frees a slot, so the SMs end within a unit
// of each other, and the CTAs resident beside a starting one keep the SM's
// loads in flight.  One persistent wave with units dealt round-robin ran
// 7-12 us longer on 2^30-input sums and 2 us on 65536 x 4096 rows: the
// static split left SMs streaming alone at the end.  Packed short rows keep
// a warp's next group in flight while it reduces the current one, so they
// take a few waves rather than one group per warp.
constexpr size_t kPackedWaves = 8;

// The chunked kernels' plan: the work split of chunk_split, one CTA per
// unit, and a combine launch when a segment has several chunks.
void plan_chunked(Plan &p, bool may_shrink)
{
    p.path = kPathChunk;
    const ChunkSplit c = chunk_split(p.segments, p.seg_len, p.dtype, p.block, may_shrink);
    p.block = c.block;
    p.chunk_log2 = c.chunk_log2;
    p.cps = c.cps;
    p.units = p.segments * c.cps;
    p.grid = unit_grid(p.units);
    p.partials = p.cps > 1 ? p.units : 0;
    p.combine_count = p.cps;
    p.launches = p.cps > 1 ? 2 : 1;
}

// The blocked order with runs longer than a vector: a warp's span is a
// whole number of rounds (32 pieces of one or more runs) and at least 16 KiB (for rows: at least
// the row, when the row is shorter); CTAs of up to 8 warps, fewer when that
// leaves too few CTA work units to fill the GPU (the tree above the spans
// is the same whatever the CTA size).
void plan_blocked(Plan &p, bool rows_call, int dev)
{
    p.path = kPathBlocked;
    const int sms = sm_count(dev);
    if (rows_call) {
        // rows of at most 16 pieces (a piece: max(run, 8 vectors) inputs),
        // padded to 2^lpr: 32 >> lpr rows to a warp's round, one launch
        const int lv0 = log2_exact(vector_len(p.dtype));
        const int pl = p.run_log2 > lv0 + 3 ? p.run_log2 : lv0 + 3;
        const int h = ceil_log2_sz(p.seg_len);
        const int lpr = h > pl ? h - pl : 0;
        if (lpr <= 4) {
            p.path = kPathBlockedRows;
            p.vlog = lpr;
            p.block = 32 * 8;
            const size_t rounds = (p.segments + ((size_t)32 >> lpr) - 1) / ((size_t)32 >> lpr);
            p.grid = unit_grid((rounds + 7) / 8);
            p.units = rounds;
            p.cps = 1;
            p.chunk_log2 = 0;
            p.partials = 0;
            p.combine_count = 1;
            p.launches = 1;
            return;
        }
    }
    const int s0 = kWarpSpanBytesLog2 - log2_exact((int)elem_bytes(p.dtype));
    int span_log2 = s0;
    if (rows_call && ceil_log2_sz(p.seg_len) < span_log2) span_log2 = ceil_log2_sz(p.seg_len);
    // a round is 32 pieces of max(run, 8 vectors) inputs
    const int lv = log2_exact(vector_len(p.dtype));
    const int piece_log2 = p.run_log2 > lv + 3 ? p.run_log2 : lv + 3;
    if (span_log2 < piece_log2 + 5) span_log2 = piece_log2 + 5;
    int w = p.block / 32 < 8 ? p.block / 32 : 8;
    if (rows_call) {
        // no more warps than spans in a row
        const size_t spans = (p.seg_len + ((size_t)1 << span_log2) - 1) >> span_log2;
        while (w > 1 && (size_t)(w / 2) >= spans) w /= 2;
    }
    for (;;) {
        p.chunk_log2 = span_log2 + log2_exact(w);
        p.cps = (p.seg_len + ((size_t)1 << p.chunk_log2) - 1) >> p.chunk_log2;
        p.units = p.segments * p.cps;
        if (w == 1 || p.units >= (size_t)4 * (size_t)sms) break;
        w /= 2;
    }
    p.block = 32 * w;
    p.grid = unit_grid(p.units);
    p.partials = p.cps > 1 ? p.units : 0;
    p.combine_count = p.cps;
    p.launches = p.cps > 1 ? 2 : 1;
}

constexpr size_t kTmemRowsMinCols = 768;

// Short rows, several to a warp group: one launch of kRowsBlock threads,
// as many CTAs as there are groups of 8 warps' rows, at most kPackedWaves
// full waves.
void plan_packed(Plan &p, int family, bool pair, int dev)
{
    p.path = kPathPackedRows;
    p.packed = family;
    p.vlog = packed_rows_vlog(family, p.seg_len, vector_len(p.dtype));
    p.block = kRowsBlock;
    const size_t warps_per_cta = (size_t)p.block / 32;
    const size_t groups = packed_rows_groups(p.segments, p.vlog);
    const size_t need = (groups + warps_per_cta - 1) / warps_per_cta;
    const int key = (pair ? 1000 : 0) + family * 100 + p.vlog * 10 + (p.R > 0 ? p.R : 1);
    const size_t resident = (size_t)sm_count(dev) *
                            (size_t)occupancy(dev, kPackedF, true, p.dtype, p.op, p.aligned, key, p.block);
    p.grid = unit_grid(need < kPackedWaves * resident ? need : kPackedWaves * resident);
    p.launches = 1;
}

// Plans tcr_reduce_sum (rows == 0: one segment of n) or tcr_reduce_rows;
// pair: the sum and sum of squares of every row in one pass (planned as
// the sum of squares).  Rows short enough to share a warp group take the
// packed kernels.
Plan make_plan(size_t segments, size_t seg_len, bool rows_call, const tcr_mode &m, int op,
               int block, int R, bool aligned, int dev, bool pair = false)
{
    Plan p;
    std::memset(&p, 0, sizeof p);
    p.kind = m.kind;
    // the tcgen05 kernels reduce plain sums of 16-bit inputs; sums of
    // squares of that kind run the mma.sync contraction (MmaSqReducer), and
    // binary32 inputs the mma.sync three-way split (MmaSplitReducer)
    if (p.kind == TCR_MMA_CHAIN_TMEM && (op != kOpSum || m.dtype == TCR_F32)) p.kind = TCR_MMA_CHAIN;
    p.dtype = m.dtype;
    p.op = op;
    p.R = R;
    p.block = block;
    p.aligned = aligned;
    p.segments = segments;
    p.seg_len = seg_len;
    p.run_log2 = m.kind == TCR_FIXED_ORDER ? m.run_log2 : 0;
    if (segments == 0 || seg_len == 0) {
        p.path = kPathEmpty;
        return p;
    }
    const size_t sms = (size_t)sm_count(dev);
    if (m.kind == TCR_SHUFFLE_TREE) {
        shuffle_team(seg_len, vector_len(p.dtype), block, &p.team_threads, &p.team_blocks);
        if (p.team_threads == 32 && p.team_blocks == 1 && rows_call &&
            packed_rows_supported(kPackedShuffle, p.dtype, op, seg_len, vector_len(p.dtype), aligned,
                                  pair)) {
            plan_packed(p, kPackedShuffle, pair, dev);
        } else if (p.team_threads == 32 && p.team_blocks == 1) {
            // a team of one warp: pack one segment per warp, 8 per CTA
            p.path = kPathShuffleRowsWarp;
            p.block = kRowsBlock;
            const size_t warps_per_cta = (size_t)p.block / 32;
            const size_t need = (segments + warps_per_cta - 1) / warps_per_cta;
            p.grid = unit_grid(need);
            p.launches = 1;
        } else {
            p.path = kPathShuffleBlock;
            p.grid = (int)(segments * (size_t)p.team_blocks);
            p.partials = p.team_blocks > 1 ? segments * (size_t)p.team_blocks : 0;
            p.combine_count = (size_t)p.team_blocks;
            p.launches = p.team_blocks > 1 ? 2 : 1;
        }
        return p;
    }
    // rows of fewer than 768 inputs run the packed mma.sync kernel: the
    // tcgen05 kernel would put 4 or 8 row groups, each its own chains and
    // read-out, in a 64 KiB stage -- its epilogue then bounds it
    if (p.kind == TCR_MMA_CHAIN_TMEM && rows_call && seg_len < kTmemRowsMinCols) p.kind = TCR_MMA_CHAIN;
    if (p.kind == TCR_MMA_CHAIN_TMEM && rows_call && aligned && segments < ((size_t)1 << 31) &&
        seg_len < ((size_t)1 << 31) && tmem_rows_grid(segments, seg_len, sms) > 0) {
        // rows of 1024 k columns as one flat array of 32 KiB copies (one CTA
        // per unit), else 16 rows per MMA tile by tensor-map boxes (one CTA
        // per SM)
        p.path = kPathTmemRows;
        p.block = tmem_block_threads();
        p.cps = tmem_rows_chunks(seg_len);
        p.units = tmem_rows_units(segments, seg_len);
        p.grid = tmem_rows_grid(segments, seg_len, sms);
        p.partials = p.cps > 1 ? segments * p.cps : 0;
        p.combine_count = p.cps;
        p.launches = p.cps > 1 ? 2 : 1;
        return p;
    }
    if (p.kind == TCR_MMA_CHAIN_TMEM && !rows_call && aligned && tmem_units(seg_len) < ((size_t)1 << 31)) {
        // one CTA per unit, two resident per SM; the resident CTAs take
        // over the units of those waiting
        p.path = kPathTmem;
        p.block = tmem_block_threads();
        p.chunk_log2 = tmem_unit_log2(seg_len);
        p.units = tmem_units(seg_len);
        p.cps = p.units;
        p.grid = (int)p.units;
        p.partials = p.units > 1 ? p.units : 0;
        p.combine_count = p.units;
        p.launches = p.units > 1 ? 2 : 1;
        return p;
    }
    if (m.kind == TCR_FIXED_ORDER && m.run_log2 > 1) {
        // blocked order: runs of at most a vector are the warp stream's
        // vector leaves (vrun); longer runs have their own kernel
        if ((1 << m.run_log2) <= vector_len(p.dtype)) {
            p.vrun = m.run_log2;
        } else {
            plan_blocked(p, rows_call, dev);
            return p;
        }
    }
    if (rows_call && p.vrun == 0) {
        const int pf = m.kind == TCR_FIXED_ORDER ? kPackedFixed : kPackedMma;
        if (packed_rows_supported(pf, p.dtype, op, seg_len, vector_len(p.dtype), aligned, pair)) {
            plan_packed(p, pf, pair, dev);
            return p;
        }
    }
    if (rows_call && seg_len <= kRowsWarpMaxBytes / elem_bytes(p.dtype)) {
        // one warp per row: the CTA size is a launch detail (the result does
        // not depend on it), fixed at kRowsBlock threads
        p.block = block = kRowsBlock;
        const size_t warps_per_cta = (size_t)block / 32;
        const size_t need = (segments + warps_per_cta - 1) / warps_per_cta;
        p.path = m.kind == TCR_FIXED_ORDER ? kPathFixedRowsWarp : kPathMmaRows;
        p.grid = unit_grid(need);
        p.launches = 1;
        return p;
    }
    plan_chunked(p, m.kind == TCR_FIXED_ORDER || m.block_threads == 0);
    return p;
}

bool fault_injected(const char *what)
{
    const char *e = std::getenv("TCR_FAULT_INJECT");
    return e && std::strcmp(e, what) == 0;
}

tcr_status run_plan(const Plan &p, const void *x, float *out, cudaStream_t s, int dev)
{
    if (p.path == kPathEmpty) {
        if (fault_injected("launch")) return TCR_ERR_CUDA;
        if (cudaMemsetAsync(out, 0, p.segments * sizeof(float), s) != cudaSuccess) return TCR_ERR_CUDA;
        return TCR_OK;
    }
    float *partials = nullptr;
    if (p.partials) {
        if (fault_injected("alloc")) return TCR_ERR_CUDA;
        cudaMemPool_t pool = pool_for(dev);
        if (!pool) return TCR_ERR_CUDA;
        if (cudaMallocFromPoolAsync((void **)&partials, p.partials * sizeof(float), pool, s) !=
            cudaSuccess)
            return TCR_ERR_CUDA;
    }
    if (fault_injected("launch")) {
        if (partials) (void)cudaFreeAsync(partials, s);
        return TCR_ERR_CUDA;
    }
    float *dst = partials ? partials : out;
    cudaError_t e = cudaSuccess;
    switch (p.path) {
    case kPathTmem:
        e = launch_mma_tmem(p.dtype, p.R, (const uint16_t *)x, p.seg_len, dst, p.grid,
                            fault_injected("stall"), s);
        break;
    case kPathTmemRows:
        e = launch_mma_tmem_rows(p.dtype, p.R, (const uint16_t *)x, p.segments, p.seg_len, dst,
                                 p.grid, fault_injected("stall"), s);
        break;
    case kPathChunk:
        e = p.kind == TCR_FIXED_ORDER
                ? launch_fixed_chunk(p.dtype, p.op, p.aligned, x, p.seg_len, p.units, p.cps,
                                     p.chunk_log2, dst, p.grid, p.block, s, p.vrun)
                : launch_mma_chunk(p.dtype, p.op, p.aligned, p.R, x, p.seg_len, p.units, p.cps,
                                   p.chunk_log2, dst, p.grid, p.block, s);
        break;
    case kPathFixedRowsWarp:
        e = launch_fixed_rows_warp(p.dtype, p.op, p.aligned, x, p.segments, p.seg_len, dst,
                                   p.grid, p.block, s, p.vrun);
        break;
    case kPathBlocked:
        e = launch_blocked_chunk(p.dtype, p.aligned, x, p.seg_len, p.units, p.cps, p.chunk_log2,
                                 p.run_log2, dst, p.grid, p.block, s);
        break;
    case kPathBlockedRows:
        e = launch_blocked_rows(p.dtype, p.aligned, x, p.segments, p.seg_len, p.run_log2, p.vlog, dst,
                                p.grid, p.block, s);
        break;
    case kPathMmaRows:
        e = launch_mma_rows(p.dtype, p.op, p.aligned, p.R, x, p.segments, p.seg_len, dst,
                            p.grid, p.block, s);
        break;
    case kPathShuffleBlock:
        e = launch_shuffle_block(p.dtype, p.op, p.aligned, x, p.seg_len, p.segments,
                                 p.team_blocks, dst, p.team_threads, s);
        break;
    case kPathShuffleRowsWarp:
        e = launch_shuffle_rows_warp(p.dtype, p.op, p.aligned, x, p.segments, p.seg_len, dst,
                                     p.grid, p.block, s);
        break;
    case kPathPackedRows:
        e = launch_packed_rows(p.packed, p.dtype, p.op, p.R, p.aligned, x, p.segments, p.seg_len,
                               p.vlog, dst, p.grid, p.block, s);
        break;
    default:
        e = cudaErrorInvalidValue;
        break;
    }
    if (e == cudaSuccess && partials)
        e = launch_combine(partials, p.segments, p.combine_count, out, s);
    if (partials) {
        cudaError_t f = cudaFreeAsync(partials, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? TCR_OK : TCR_ERR_CUDA;
}


bool mul_overflows(size_t a, size_t b)
{
    return a != 0 && b > SIZE_MAX / a;
}

tcr_status reduce_sum_op(const void *x, size_t n, float *out, const tcr_mode &mode, int op,
                         void *stream)
{
    int block = 0, R = 0;
    tcr_status st = check_common(x, n, out, mode, &block, &R);
    if (st != TCR_OK) return st;
    if (op != kOpSum && mode.run_log2 != 0) return TCR_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return TCR_ERR_CUDA;
    const bool aligned = ((uintptr_t)x & 15u) == 0;
    Plan p = make_plan(1, n, false, mode, op, block, R, aligned, dev);
    return run_plan(p, x, out, (cudaStream_t)stream, dev);
}

tcr_status reduce_rows_op(const void *x, size_t rows, size_t cols, float *out,
                          const tcr_mode &mode, int op, void *stream)
{
    if (mul_overflows(rows, cols)) return TCR_ERR_INVALID_ARG;
    if (rows == 0) {
        int block = 0, R = 0;
        return check_mode(mode, &block, &R);
    }
    int block = 0, R = 0;
    tcr_status st = check_common(x, rows * cols, out, mode, &block, &R);
    if (st != TCR_OK) return st;
    if (op != kOpSum && mode.run_log2 != 0) return TCR_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return TCR_ERR_CUDA;
    // every row starts 16-byte aligned when x does and a row is whole vectors
    const bool aligned = ((uintptr_t)x & 15u) == 0 && (cols % (size_t)vector_len(mode.dtype)) == 0;
    Plan p = make_plan(rows, cols, true, mode, op, block, R, aligned, dev);
    return run_plan(p, x, out, (cudaStream_t)stream, dev);
}

// What a fixed-order descriptor's run length does: 0 for the plain tree
// (runs of one or two inputs), the segment's tree height for one run
// covering it (the left-to-right sum), else the run length itself.
int effective_run_log2(const tcr_order_desc *d)
{
    int c = d->order == TCR_ORDER_BLOCKED_TREE ? d->run_log2 : 0;
    const int h = ceil_log2_sz(d->segment_len);
    if (c > h) c = h;
    return c <= 1 ? 0 : c;
}

// The sum and sum of squares of every row in one pass (mean_var == 0:
// out_a = sums, out_b = sums of squares) or their mean and variance.
tcr_status run_pair_plan(const Plan &p, const void *x, float *out_a, float *out_b, int mean_var,
                         cudaStream_t s, int dev)
{
    if (p.path == kPathEmpty) {
        if (fault_injected("launch")) return TCR_ERR_CUDA;
        // no inputs: sums +0.0; mean and variance 0 / 0 (NaN)
        const int byte = mean_var ? 0xff : 0;
        if (cudaMemsetAsync(out_a, byte, p.segments * sizeof(float), s) != cudaSuccess ||
            cudaMemsetAsync(out_b, byte, p.segments * sizeof(float), s) != cudaSuccess)
            return TCR_ERR_CUDA;
        return TCR_OK;
    }
    const int family = p.kind == TCR_FIXED_ORDER ? kPairFixed
                       : p.kind == TCR_SHUFFLE_TREE ? kPairShuffle
                                                    : kPairMma;
    if (p.path == kPathPackedRows) {
        if (fault_injected("launch")) return TCR_ERR_CUDA;
        return launch_packed_rows_pair(p.packed, p.dtype, p.R, p.aligned, x, p.segments, p.seg_len,
                                       p.vlog, out_a, out_b, mean_var, p.grid, p.block, s) == cudaSuccess
                   ? TCR_OK
                   : TCR_ERR_CUDA;
    }
    if (p.path == kPathFixedRowsWarp || p.path == kPathMmaRows || p.path == kPathShuffleRowsWarp) {
        if (fault_injected("launch")) return TCR_ERR_CUDA;
        return launch_rows_pair(family, p.dtype, p.aligned, p.R, x, p.segments, p.seg_len, out_a,
                                out_b, mean_var, p.grid, p.block, s) == cudaSuccess
                   ? TCR_OK
                   : TCR_ERR_CUDA;
    }
    if (p.path != kPathChunk && p.path != kPathShuffleBlock) return TCR_ERR_UNSUPPORTED;
    // scratch: two partial arrays, and the two sums per row before the
    // mean/variance epilogue
    const size_t np = p.partials;
    const size_t nt = mean_var ? p.segments : 0;
    float *scratch = nullptr;
    if (np + nt > 0) {
        if (fault_injected("alloc")) return TCR_ERR_CUDA;
        cudaMemPool_t pool = pool_for(dev);
        if (!pool) return TCR_ERR_CUDA;
        if (cudaMallocFromPoolAsync((void **)&scratch, 2 * (np + nt) * sizeof(float), pool, s) !=
            cudaSuccess)
            return TCR_ERR_CUDA;
    }
    if (fault_injected("launch")) {
        if (scratch) (void)cudaFreeAsync(scratch, s);
        return TCR_ERR_CUDA;
    }
    float *sum_a = mean_var ? scratch + 2 * np : out_a;
    float *sum_b = mean_var ? scratch + 2 * np + nt : out_b;
    float *dst_a = np ? scratch : sum_a;
    float *dst_b = np ? scratch + np : sum_b;
    cudaError_t e = p.path == kPathChunk
                        ? launch_chunk_pair(family, p.dtype, p.aligned, p.R, x, p.seg_len, p.units,
                                            p.cps, p.chunk_log2, dst_a, dst_b, p.grid, p.block, s)
                        : launch_shuffle_block_pair(p.dtype, p.aligned, x, p.seg_len, p.segments,
                                                    p.team_blocks, dst_a, dst_b, p.team_threads, s);
    if (e == cudaSuccess && np) e = launch_combine(dst_a, p.segments, p.combine_count, sum_a, s);
    if (e == cudaSuccess && np) e = launch_combine(dst_b, p.segments, p.combine_count, sum_b, s);
    if (e == cudaSuccess && mean_var)
        e = launch_mean_var(sum_a, sum_b, p.segments, p.seg_len, out_a, out_b, s);
    if (scratch) {
        cudaError_t f = cudaFreeAsync(scratch, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? TCR_OK : TCR_ERR_CUDA;
}

tcr_status reduce_rows_pair(const void *x, size_t rows, size_t cols, float *out_a, float *out_b,
                            const tcr_mode &mode, int mean_var, void *stream)
{
    if (mul_overflows(rows, cols)) return TCR_ERR_INVALID_ARG;
    int block = 0, R = 0;
    if (rows == 0) return check_mode(mode, &block, &R);
    tcr_status st = check_common(x, rows * cols, out_a, mode, &block, &R);
    if (st != TCR_OK) return st;
    if (!out_b || ((uintptr_t)out_b & 3u) != 0) return TCR_ERR_INVALID_ARG;
    if (mode.run_log2 != 0) return TCR_ERR_UNSUPPORTED;     // squares have no blocked order
    const int dev = current_device();
    if (dev < 0) return TCR_ERR_CUDA;
    const bool aligned = ((uintptr_t)x & 15u) == 0 && (cols % (size_t)vector_len(mode.dtype)) == 0;
    // planned as the sum of squares (the tcgen05 kind runs the mma.sync pair)
    Plan p = make_plan(rows, cols, true, mode, kOpSquares, block, R, aligned, dev, true);
    return run_pair_plan(p, x, out_a, out_b, mean_var, (cudaStream_t)stream, dev);
}

// ---------------------------------------------------------------- GEMM

constexpr int kGemmMaxSplits = 64;

struct GemmPlan {
    int splits, kbps, grid;
    size_t k_split, workspace;
};

tcr_status gemm_check(size_t M, size_t N, size_t K, int splits, int dtype)
{
    if (dtype != TCR_F16 && dtype != TCR_BF16) return TCR_ERR_INVALID_ARG;
    if (M >= ((size_t)1 << 31) || N >= ((size_t)1 << 31) || K >= ((size_t)1 << 31))
        return TCR_ERR_INVALID_ARG;
    if (K % 8 != 0) return TCR_ERR_INVALID_ARG;
    if (splits < 0 || splits > kGemmMaxSplits) return TCR_ERR_INVALID_ARG;
    return TCR_OK;
}

// The K partition: a fixed function of (M, N, K, splits) -- never of the
// device -- so the declared order is the same on every GPU.
GemmPlan gemm_plan(size_t M, size_t N, size_t K, int splits, int dev)
{
    GemmPlan g;
    // the default: as many splits as fill one wave of 152 CTAs with tiles x S
    // units, at most 32
    const size_t tiles = ((M + gemm_tile_m() - 1) / gemm_tile_m()) *
                         ((N + gemm_tile_n() - 1) / gemm_tile_n());
    const size_t kboxes = (K + gemm_tile_k() - 1) / gemm_tile_k();
    size_t s = (size_t)splits;
    if (s == 0) {
        s = tiles >= (size_t)kRuleSMs ? 1 : (size_t)kRuleSMs / (tiles ? tiles : 1);
        if (s > 32) s = 32;
    }
    if (s > kboxes) s = kboxes;
    if (s < 1) s = 1;
    const size_t kbps = kboxes ? (kboxes + s - 1) / s : 1;
    g.kbps = (int)kbps;
    g.splits = kboxes ? (int)((kboxes + kbps - 1) / kbps) : 1;
    g.k_split = kbps * (size_t)gemm_tile_k();
    g.workspace = g.splits > 1 ? (size_t)g.splits * M * N * sizeof(float) : 0;
    const size_t units = tiles * (size_t)g.splits;
    const size_t sms = (size_t)sm_count(dev);
    g.grid = (int)(units < sms ? units : sms);
    return g;
}

}  // namespace

extern "C" {

tcr_status tcr_reduce_sum(const void *x, size_t n, float *out, tcr_mode mode, void *stream)
{
    return reduce_sum_op(x, n, out, mode, kOpSum, stream);
}

tcr_status tcr_reduce_rows(const void *x, size_t rows, size_t cols, float *out, tcr_mode mode,
                           void *stream)
{
    return reduce_rows_op(x, rows, cols, out, mode, kOpSum, stream);
}

tcr_status tcr_reduce_sum_squares(const void *x, size_t n, float *out, tcr_mode mode, void *stream)
{
    return reduce_sum_op(x, n, out, mode, kOpSquares, stream);
}

tcr_status tcr_reduce_rows_sum_squares(const void *x, size_t rows, size_t cols, float *out,
                                       tcr_mode mode, void *stream)
{
    return reduce_rows_op(x, rows, cols, out, mode, kOpSquares, stream);
}

tcr_status tcr_reduce_rows_moments(const void *x, size_t rows, size_t cols, float *sums,
                                   float *sums_of_squares, tcr_mode mode, void *stream)
{
    return reduce_rows_pair(x, rows, cols, sums, sums_of_squares, mode, 0, stream);
}

tcr_status tcr_reduce_rows_mean_var(const void *x, size_t rows, size_t cols, float *mean,
                                    float *var, tcr_mode mode, void *stream)
{
    return reduce_rows_pair(x, rows, cols, mean, var, mode, 1, stream);
}

tcr_status tcr_gemm_descriptor(size_t M, size_t N, size_t K, int splits, int dtype,
                               tcr_gemm_desc *desc)
{
    if (!desc) return TCR_ERR_INVALID_ARG;
    tcr_status st = gemm_check(M, N, K, splits, dtype);
    if (st != TCR_OK) return st;
    const GemmPlan g = gemm_plan(M, N, K, splits, current_device());
    std::memset(desc, 0, sizeof *desc);
    desc->M = M;
    desc->N = N;
    desc->K = K;
    desc->dtype = dtype;
    desc->splits = g.splits;
    desc->k_split = g.k_split;
    desc->tile_m = (current_device() >= 0) ? gemm_tile_m_run() : gemm_tile_m();
    desc->tile_n = (current_device() >= 0) ? gemm_tile_n_run() : gemm_tile_n();
    desc->tile_k = gemm_tile_k();
    desc->combine_order = TCR_ORDER_BALANCED_TREE;
    desc->workspace_bytes = g.workspace;
    desc->launch_grid = (current_device() >= 0) ? gemm_launch_grid(M, N, g.splits) : g.grid;
    desc->launch_block = gemm_block_threads();
    desc->launches = (M * N == 0) ? 0 : (K == 0 ? 0 : (g.splits > 1 ? 2 : 1));
    return TCR_OK;
}

tcr_status tcr_gemm_splitk(const void *A, const void *W, float *C, size_t M, size_t N, size_t K,
                           int splits, int dtype, void *stream)
{
    tcr_status st = gemm_check(M, N, K, splits, dtype);
    if (st != TCR_OK) return st;
    if (M == 0 || N == 0) return TCR_OK;
    if (!C || ((uintptr_t)C & 3u) != 0) return TCR_ERR_INVALID_ARG;
    if (K > 0 && (!A || !W || ((uintptr_t)A & 15u) != 0 || ((uintptr_t)W & 15u) != 0))
        return TCR_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0) return TCR_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (K == 0)
        return cudaMemsetAsync(C, 0, M * N * sizeof(float), s) == cudaSuccess ? TCR_OK : TCR_ERR_CUDA;
    const GemmPlan g = gemm_plan(M, N, K, splits, dev);
    float *P = nullptr;
    if (g.splits > 1) {
        if (fault_injected("alloc")) return TCR_ERR_CUDA;
        cudaMemPool_t pool = pool_for(dev);
        if (!pool) return TCR_ERR_CUDA;
        if (cudaMallocFromPoolAsync((void **)&P, g.workspace, pool, s) != cudaSuccess) return TCR_ERR_CUDA;
    }
    if (fault_injected("launch")) {
        if (P) (void)cudaFreeAsync(P, s);
        return TCR_ERR_CUDA;
    }
    cudaError_t e = launch_gemm_splitk(dtype, A, W, M, N, K, g.splits, g.kbps, P ? P : C,
                                       fault_injected("stall"), s);
    if (e == cudaSuccess && P) e = launch_splitk_combine(P, M * N, g.splits, C, s);
    if (P) {
        cudaError_t f = cudaFreeAsync(P, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? TCR_OK : TCR_ERR_CUDA;
}

tcr_status tcr_order_descriptor(size_t n, size_t rows, size_t cols, tcr_mode mode,
                                tcr_order_desc *desc)
{
    if (!desc) return TCR_ERR_INVALID_ARG;
    int block = 0, R = 0;
    tcr_status st = check_mode(mode, &block, &R);
    if (st != TCR_OK) return st;
    const bool rows_call = rows > 0;
    if (rows_call && mul_overflows(rows, cols)) return TCR_ERR_INVALID_ARG;
    const size_t segments = rows_call ? rows : 1;
    const size_t seg_len = rows_call ? cols : n;
    if (segments * seg_len >= kMaxInputs) return TCR_ERR_INVALID_ARG;
    const int dev = current_device();
    // the plan of a 16-byte aligned x (rows: aligned when they are whole
    // vectors); another alignment differs only in speed
    const bool aligned = !rows_call || cols % (size_t)vector_len(mode.dtype) == 0;
    Plan p = make_plan(segments, seg_len, rows_call, mode, kOpSum, block, R, aligned, dev);
    std::memset(desc, 0, sizeof *desc);
    desc->kind = mode.kind;
    desc->order = mode.kind == TCR_SHUFFLE_TREE ? TCR_ORDER_GRID_STRIDE
                  : mode.kind == TCR_FIXED_ORDER
                      ? (mode.run_log2 > 0 ? TCR_ORDER_BLOCKED_TREE : TCR_ORDER_BALANCED_TREE)
                      : TCR_ORDER_TENSOR_CORE;
    desc->run_log2 = mode.kind == TCR_FIXED_ORDER ? mode.run_log2 : 0;
    desc->segment_len = seg_len;
    desc->segments = segments;
    desc->vector_len = vector_len(mode.dtype);
    desc->dtype = mode.dtype;
    desc->chain_R = (mode.kind == TCR_MMA_CHAIN || mode.kind == TCR_MMA_CHAIN_TMEM) ? R : 0;
    desc->pad_negative_zero = 1;
    if (mode.kind == TCR_SHUFFLE_TREE) {
        shuffle_team(seg_len, desc->vector_len, block, &desc->team_threads, &desc->team_blocks);
    }
    desc->launch_grid = p.grid;
    desc->launch_block = p.path == kPathShuffleBlock ? p.team_threads : p.block;
    desc->chunk_log2 =
        (p.path == kPathChunk || p.path == kPathTmem || p.path == kPathBlocked) ? p.chunk_log2 : 0;
    desc->partials = p.partials;
    desc->launches = p.launches;
    return TCR_OK;
}

tcr_status tcr_order_equivalent(const tcr_order_desc *a, const tcr_order_desc *b,
                                int *equivalent)
{
    if (!a || !b || !equivalent) return TCR_ERR_INVALID_ARG;
    *equivalent = 0;
    const bool tree_a = a->order == TCR_ORDER_BALANCED_TREE || a->order == TCR_ORDER_BLOCKED_TREE;
    const bool tree_b = b->order == TCR_ORDER_BALANCED_TREE || b->order == TCR_ORDER_BLOCKED_TREE;
    if (a->kind != b->kind || (a->order != b->order && !(tree_a && tree_b)) ||
        a->segment_len != b->segment_len || a->dtype != b->dtype ||
        a->vector_len != b->vector_len || a->vector_len <= 0)
        return TCR_OK;
    if (tree_a) {
        *equivalent = effective_run_log2(a) == effective_run_log2(b);
        return TCR_OK;
    }
    switch (a->order) {
    case TCR_ORDER_GRID_STRIDE: {
        const size_t nvec = (a->segment_len + (size_t)a->vector_len - 1) / (size_t)a->vector_len;
        const size_t ta = (size_t)a->team_threads * (size_t)a->team_blocks;
        const size_t tb = (size_t)b->team_threads * (size_t)b->team_blocks;
        // one vector per thread at most: lane values are the vector trees,
        // combined by the butterfly and one balanced tree over warps
        *equivalent = (ta == tb) || (ta >= nvec && tb >= nvec);
        break;
    }
    default:
        *equivalent = a->chain_R == b->chain_R && a->launch_block == b->launch_block &&
                      a->chunk_log2 == b->chunk_log2;
        break;
    }
    return TCR_OK;
}

tcr_status tcr_device_faults(unsigned int *flags, int clear)
{
    if (!flags) return TCR_ERR_INVALID_ARG;
    if (current_device() < 0) return TCR_ERR_CUDA;
    unsigned int a = 0, g = 0;
    if (read_device_faults(&a, clear != 0) != cudaSuccess || read_gemm_faults(&g, clear != 0) != cudaSuccess)
        return TCR_ERR_CUDA;
    *flags = a | g;
    return TCR_OK;
}

const char *tcr_status_string(tcr_status status)
{
    switch (status) {
    case TCR_OK: return "success";
    case TCR_ERR_INVALID_ARG: return "invalid argument";
    case TCR_ERR_UNSUPPORTED: return "unsupported request";
    case TCR_ERR_CUDA: return "CUDA allocation or launch failure";
    default: return "unknown status";
    }
}

}  // extern "C"
