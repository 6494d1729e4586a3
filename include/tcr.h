/*
 * tcr.h -- tensor-core and fixed-order sum reduction on one GB300 GPU.
 *
 * The operation is the one stated by "GPU Tensor Cores for fast Arithmetic
 * Reductions" (arXiv 2001.05585), Abstract: the arithmetic reduction (sum)
 * of n numbers into one 32-bit floating-point result.  Inputs are binary16,
 * bfloat16 or binary32; every result is binary32.  Four ways of computing
 * it are offered (tcr_kind):
 *
 *   TCR_MMA_CHAIN     the page's method: the inputs are laid out as 16x16
 *                     tiles and multiplied by an all-ones matrix on the tensor
 *                     cores, R multiply-accumulates chained into one fp32
 *                     accumulator; each chain's sub-result is then added, in
 *                     fp32, into the final result (same Abstract: sub-results
 *                     of each chain of R MMAs kept as 32-bit floats, then all
 *                     reduced into a final 32-bit result).  The order inside
 *                     the tensor core is the hardware's, so results are held
 *                     to an error bound, not to bits:
 *                     |result - exact| <= 2^-20 * sum|x_i| + 1e-6.
 *                     Binary32 inputs are split exactly into three bfloat16
 *                     parts (x = hi + mid + lo, hi = x rounded toward zero,
 *                     the rest exact residuals) whose sums run on the
 *                     tensor cores, three MMAs per 256 inputs; the split
 *                     drops less than 2^-133 per input below 2^-110.
 *   TCR_SHUFFLE_TREE  the conventional GPU reduction the same Abstract
 *                     compares against, with its order declared (see
 *                     tcr_order_desc): grid-stride accumulation of 16-byte
 *                     vectors (8 inputs of 16 bits, 4 of binary32), a warp
 *                     butterfly, a tree over warps and a tree over blocks.  Bit-identical to the CPU emulation
 *                     of that order.
 *   TCR_MMA_CHAIN_TMEM  the same method on the fifth-generation tensor cores:
 *                     inputs staged into shared memory by bulk asynchronous
 *                     copies, tcgen05.mma (M = 128, N = 16, K = 16; one MMA
 *                     per 2048 inputs) with the accumulator in tensor memory,
 *                     R MMAs per chain, chain sub-results read out to fp32
 *                     registers.  Rows of 1024 k columns (k a divisor or
 *                     a multiple of 16) are read as the flat array they
 *                     are, 32 KiB at a time, each MMA lane group taking 1024
 *                     inputs of one row (a row is 8 k of D's lanes, or all
 *                     128 for k >= 16); other rows put 16 rows on an MMA
 *                     tile (8 lanes to a row, chains running along the row)
 *                     and reach shared memory by 3-D tensor-map or per-row
 *                     bulk copies.  A chain never spans two shared-memory
 *                     stages (8 MMAs for sums and flat rows, 16 for 16-row
 *                     tiles); when R does not divide that, a stage's last
 *                     chain is shorter.  The sum and the flat rows launch
 *                     one CTA per work unit and the resident CTAs take over
 *                     the units of those not yet started (cluster launch
 *                     control), so the result does not depend on which SM
 *                     runs which unit.  Same
 *                     error bound as TCR_MMA_CHAIN.  16-bit sums only: an
 *                     x that is not 16-byte aligned (or rows whose stride is
 *                     not), rows of fewer than 768 inputs (a 64 KiB stage of
 *                     them holds too little work per MMA chain), sums of
 *                     squares and binary32 inputs are reduced by the
 *                     TCR_MMA_CHAIN kernels instead.
 *   TCR_FIXED_ORDER   a balanced binary tree over index order, padded with
 *                     -0.0 to a power of two ("Taming Bitwise Behavior in
 *                     GPU Kernels with Tensor Core", arXiv 2609.11356,
 *                     Abstract: balanced-tree reduction, a descriptor of
 *                     reduction order, one bit-equivalence class).  The result
 *                     depends on the inputs and n only -- not on the launch
 *                     configuration, the block size or the GPU -- and is
 *                     bit-identical to the CPU emulation of that tree.
 *
 * All additions outside the tensor core are binary32, round to nearest
 * even, with no fused multiply-add and no flushing of subnormals.
 *
 * Memory and streams.  x and out are device pointers owned by the caller.
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL means the legacy
 * default stream): *out is valid once the stream reaches the point of the
 * call.  A call that needs scratch memory takes it from a library-owned,
 * stream-ordered pool on the current device (cudaMallocFromPoolAsync /
 * cudaFreeAsync on `stream`), so concurrent calls on different streams do
 * not share scratch.  The library keeps no other state between calls except
 * per-device launch-plan caches.  Every call runs on the current device.
 * Calls may come from several host threads at once, each on its own stream.
 * After one eager call of a kind on a device (which fills that device's
 * caches and sets the kernels' attributes), the reduction, rows, moments and
 * GEMM calls may be captured into a CUDA graph on a capturing stream; each
 * replay gives the eager call's bits.  (Not tcr_reduce_sum_noalloc, which
 * makes no such statement.)
 *
 * Kernel overlap.  A call's kernels are launched as programmatic dependents
 * of the kernel before them on the stream (programmatic stream
 * serialization): they may start, and run set-up that touches no global
 * memory, while that kernel finishes, and wait for it (griddepcontrol.wait)
 * before their first global memory access; they also let the next kernel
 * on the stream launch early.  A caller's kernel launched right after a
 * call without that attribute runs after the call's last kernel as usual;
 * one launched with it must execute griddepcontrol.wait
 * (cudaGridDependencySynchronize) before it reads the call's results.
 *
 * Shared memory and L1.  An SM keeps its shared-memory / L1 split while
 * CTAs stream onto it, so a kernel that needs a large split leaves the
 * next kernels on the stream a small L1.  The TCR_MMA_CHAIN_TMEM sum and
 * flat-rows kernels ask for the 164 KiB configuration (92 KiB of L1 left);
 * the 16-row tcgen05 rows kernel and tcr_gemm_splitk need 196-228 KiB
 * (28-60 KiB left), and streaming kernels that followed such a split on
 * the same SMs were measured about 14% slower.
 *
 * Errors.  Invalid arguments return TCR_ERR_INVALID_ARG before any GPU work
 * and leave *out untouched.  A CUDA error (allocation or launch) returns
 * TCR_ERR_CUDA; the CUDA error itself is left to cudaGetLastError /
 * cudaPeekAtLastError of the caller's runtime.
 */
#ifndef TCR_H
#define TCR_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TCR_API __attribute__((visibility("default")))
#else
#define TCR_API
#endif

typedef enum {
    TCR_OK = 0,
    TCR_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or mode field */
    TCR_ERR_UNSUPPORTED = 2,   /* well-formed request the library does not serve */
    TCR_ERR_CUDA = 3           /* a CUDA allocation or launch failed */
} tcr_status;

typedef enum {
    TCR_MMA_CHAIN = 0,
    TCR_SHUFFLE_TREE = 1,
    TCR_FIXED_ORDER = 2,
    TCR_MMA_CHAIN_TMEM = 3
} tcr_kind;

typedef enum {
    TCR_F16 = 0,    /* IEEE 754 binary16 */
    TCR_BF16 = 1,   /* bfloat16: the upper 16 bits of a binary32 */
    TCR_F32 = 2     /* IEEE 754 binary32 */
} tcr_dtype;

/*
 * How to reduce.
 *   kind           tcr_kind.
 *   R              TCR_MMA_CHAIN only: tensor-core MMAs per chain, 1..8, or
 *                  0 for the default, 4 (the Abstract of arXiv 2001.05585
 *                  finds R = 4 or 5 best for small thread blocks and R = 1
 *                  for large ones; on GB300 R = 4 is fastest at every block
 *                  size).  Ignored otherwise.
 *   block_threads  threads per CTA: 0 for the default (256) or one of 32,
 *                  64, 128, 256, 512, 1024.  For TCR_SHUFFLE_TREE it is part
 *                  of the declared order; for TCR_FIXED_ORDER it changes
 *                  only speed, never the result.
 *   dtype          tcr_dtype of the inputs.
 *   run_log2       TCR_FIXED_ORDER sums only (0 for every other call): 0
 *                  for the balanced tree over the inputs, or c in 1..16 for
 *                  the blocked-sequential-then-tree order -- runs of 2^c
 *                  consecutive inputs, each added left to right, then the
 *                  balanced tree over the run values (-0.0 pad).  c = 1 is
 *                  the plain tree (a run of two is a pair); c >= log2(n)
 *                  the plain left-to-right sum.  A second declared order in
 *                  the sense of "Taming Bitwise Behavior in GPU Kernels with
 *                  Tensor Core" (arXiv 2609.11356), Abstract, with the run
 *                  length chosen by the caller.  Each run is a serial chain:
 *                  the GPU runs n / 2^c of them in parallel, so long runs
 *                  on short inputs are slow.  Sums of squares with
 *                  run_log2 != 0 return TCR_ERR_UNSUPPORTED.
 */
typedef struct {
    int kind;
    int R;
    int block_threads;
    int dtype;
    int run_log2;
} tcr_mode;

/*
 * tcr_reduce_sum -- out[0] = sum of x[0 .. n-1].
 *   x       device pointer to n contiguous inputs of mode.dtype, aligned to
 *           the input size (2 bytes, or 4 for TCR_F32; any 16-byte
 *           misalignment is served by a slower load path with the same
 *           order).  May be NULL only when n == 0.
 *   n       number of inputs, 0 <= n < 2^40.  n == 0 writes +0.0.
 *   out     device pointer to one float, 4-byte aligned.
 *   mode    see tcr_mode.
 *   stream  cudaStream_t.
 * Launches one reduction kernel and, when it leaves more than one partial,
 * one combine kernel on the same stream; the partials live in pool scratch
 * of 4 bytes per partial (tcr_order_descriptor reports the count).
 */
TCR_API tcr_status tcr_reduce_sum(const void *x, size_t n, float *out, tcr_mode mode, void *stream);

/*
 * tcr_reduce_rows -- out[r] = sum of x[r*cols .. r*cols + cols-1], r < rows.
 *   x       device pointer to a row-major rows x cols matrix of inputs of
 *           mode.dtype (row stride = cols), aligned to the input size.  May
 *           be NULL only when rows * cols == 0.
 *   rows    number of rows (0 does nothing); cols: inputs per row (0 writes
 *           +0.0 to every out[r]).  rows * cols < 2^40.
 *   out     device pointer to rows floats, 4-byte aligned.
 * Each row is reduced exactly as tcr_reduce_sum would reduce it alone for
 * TCR_FIXED_ORDER and TCR_SHUFFLE_TREE (the order depends on cols only, never
 * on rows: results are batch invariant).  Short rows need no scratch and one
 * launch; long rows use per-row partials and a combine launch.  Rows of at
 * most 128 16-byte vectors (1024 16-bit or 512 binary32 inputs) are packed
 * several to a warp; when x or the row stride is not 16-byte aligned but
 * every row starts on a 4-byte boundary and is a whole number of 4-byte
 * words, those kernels read 8- or 4-byte words of the rows only; otherwise
 * they read whole 16-byte aligned granules that hold inputs of the matrix
 * -- up to 15 bytes before x or after its last input, never outside the
 * granules the data touches (an allocation from cudaMalloc is 256-byte
 * aligned, so such a granule lies inside it).
 */
TCR_API tcr_status tcr_reduce_rows(const void *x, size_t rows, size_t cols, float *out, tcr_mode mode,
                           void *stream);

/*
 * tcr_reduce_sum_squares, tcr_reduce_rows_sum_squares -- the sum of x_i^2
 * (over all inputs, or per row), a reduction with a fused pre-op in the
 * sense of the cascaded reductions named by the "RedFuser" title in the
 * first page's list of work built on the method.  Arguments, layout, modes
 * and errors are those of tcr_reduce_sum / tcr_reduce_rows.
 *   TCR_FIXED_ORDER, TCR_SHUFFLE_TREE  the same declared orders over the
 *                     leaves fl32(x_i * x_i) (one binary32 multiplication,
 *                     round to nearest; exact for binary16), bit-identical
 *                     to the CPU emulation of those orders.
 *   TCR_MMA_CHAIN     16-bit inputs: a dense contraction on the tensor
 *                     cores: for each 16 x 16 tile A, D = A * A^T holds the
 *                     rows' sums of squares on its diagonal (two m16n8k16
 *                     MMAs per tile, chains of R flushed to fp32).  Binary32
 *                     inputs: the leaves fl32(x_i * x_i), split and summed
 *                     as the sum does.  Error bound
 *                     |result - exact| <= 2^-20 * sum x_i^2 + 1e-6.
 *   TCR_MMA_CHAIN_TMEM  runs as TCR_MMA_CHAIN.
 * tcr_order_descriptor describes these calls as well: the order does not
 * depend on the leaves.
 */
TCR_API tcr_status tcr_reduce_sum_squares(const void *x, size_t n, float *out, tcr_mode mode,
                                          void *stream);
TCR_API tcr_status tcr_reduce_rows_sum_squares(const void *x, size_t rows, size_t cols,
                                               float *out, tcr_mode mode, void *stream);

/*
 * tcr_reduce_rows_moments -- for every row r < rows, in one pass over x:
 *   sums[r]            = the row's sum, as tcr_reduce_rows computes it, and
 *   sums_of_squares[r] = the row's sum of squares, as
 *                        tcr_reduce_rows_sum_squares computes it
 * (bit for bit in TCR_FIXED_ORDER and TCR_SHUFFLE_TREE: the same orders;
 * within the same bounds in TCR_MMA_CHAIN; TCR_MMA_CHAIN_TMEM runs as
 * TCR_MMA_CHAIN).  Two reductions of one input fused so that it is read
 * once: the cascaded reductions named by the "RedFuser" title in the first
 * page's list of work built on the method.  Arguments, layout and errors are
 * those of tcr_reduce_rows; sums and sums_of_squares are device arrays of
 * rows floats, 4-byte aligned.  A mode with run_log2 != 0 returns
 * TCR_ERR_UNSUPPORTED.
 *
 * tcr_reduce_rows_mean_var -- the same pass, then per row (n = cols as a
 * binary32, one rounding to nearest per operation):
 *   mean[r] = S1 / n,  var[r] = S2 / n - mean[r] * mean[r], or +0.0 where
 *   that is negative (rounding only)
 * from the row's sum S1 and sum of squares S2 above: the population
 * variance by the one-pass formula, exact to a few ulps of S2 / n when the
 * mean is small against the spread (|mean| large against the standard
 * deviation loses digits to cancellation).  cols == 0 gives NaN for both.
 */
TCR_API tcr_status tcr_reduce_rows_moments(const void *x, size_t rows, size_t cols, float *sums,
                                           float *sums_of_squares, tcr_mode mode, void *stream);
TCR_API tcr_status tcr_reduce_rows_mean_var(const void *x, size_t rows, size_t cols, float *mean,
                                            float *var, tcr_mode mode, void *stream);

/*
 * tcr_reduce_sum_noalloc -- tcr_reduce_sum for callers that must not
 * allocate device memory while they run: a service that reserved its whole
 * device-memory budget at start-up and treats any later allocation as a
 * fault, code running while another component owns the device allocator,
 * or a host thread with a deadline that cannot wait for the allocator.
 * The pages have no counterpart to this entry point; it is an interface
 * choice of this library.
 *
 * Same arguments as tcr_reduce_sum (caller-owned x and out), but the
 * partials live in one fixed array of 65536 floats (256 KiB) in device
 * memory, held by every GPU that loads the library until the process exits;
 * no cudaMalloc, cudaFree or other allocating call is made.
 *   - Serves TCR_FIXED_ORDER (run_log2 = 0) and TCR_MMA_CHAIN, with the work
 *     split of tcr_reduce_sum (one plan function serves both), so results
 *     are tcr_reduce_sum's bit for bit.  TCR_SHUFFLE_TREE, TCR_MMA_CHAIN_TMEM
 *     and a blocked order return TCR_ERR_UNSUPPORTED; malformed arguments
 *     return TCR_ERR_INVALID_ARG exactly as tcr_reduce_sum does.
 *   - n is limited to 65536 chunks of 2^(13 + log2(block_threads / 32))
 *     16-bit inputs (2^32 inputs at the default 256 threads, 2^29 at 32),
 *     half as many binary32 inputs; a larger n returns TCR_ERR_UNSUPPORTED
 *     before any GPU work.
 *   - The first call on each device, with that device current, looks up the
 *     array's device address and has the driver load every kernel this
 *     entry point can launch (the runtime otherwise loads a kernel at its
 *     first launch, and loading code takes device memory): later calls load
 *     nothing.  Make that first call before any stream capture.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents (nothing needs clearing: each call writes every partial it
 *     reads).  Calls that overlap on the GPU race on it: order them on one
 *     stream or with events.
 */
TCR_API tcr_status tcr_reduce_sum_noalloc(const void *x, size_t n, float *out, tcr_mode mode,
                                          void *stream);

/* Declared reduction orders (tcr_order_desc.order). */
typedef enum {
    TCR_ORDER_TENSOR_CORE = 0,      /* MMA_CHAIN: inner order is the tensor core's */
    TCR_ORDER_GRID_STRIDE = 1,      /* SHUFFLE_TREE: see tcr_order_desc */
    TCR_ORDER_BALANCED_TREE = 2,    /* FIXED_ORDER: balanced tree over index order */
    TCR_ORDER_BLOCKED_TREE = 3      /* FIXED_ORDER, run_log2 > 0: runs left to right, then the tree */
} tcr_order;

/*
 * The order a call reduces in, and how it is launched -- what the CPU
 * emulation needs to reproduce a result bit for bit (the descriptor of
 * reduction order of arXiv 2609.11356, Abstract, restated for 1-D sums and
 * rows).
 *
 *   order            tcr_order.
 *   segment_len      inputs per reduced segment (n, or cols).
 *   segments         number of results (1, or rows).
 *   vector_len       inputs per 16-byte vector leaf group (8 for 16-bit
 *                    inputs, 4 for binary32).
 *   team_threads     SHUFFLE_TREE: threads per block Bt of the team that
 *                    reduces one segment (32 means one warp per segment).
 *   team_blocks      SHUFFLE_TREE: blocks G per segment.  Thread g = b*Bt + t
 *                    accumulates vectors g, g + G*Bt, g + 2*G*Bt, ... into an
 *                    fp32 value that starts at -0.0; a warp combines its lanes
 *                    by the butterfly with offsets 16, 8, 4, 2, 1 (lane i adds
 *                    lane i^offset); a block is the balanced tree over its
 *                    warps; a segment is the balanced tree over its G blocks,
 *                    padded with -0.0.  A vector's value is the balanced tree
 *                    over its vector_len inputs, missing inputs being -0.0.
 *                    The team is one warp (32, 1) when the segment has at
 *                    most 1024 vectors, else Bt = block_threads and
 *                    G = ceil(vectors / (16 * Bt)).
 *   chain_R          MMA_CHAIN: MMAs per chain (after defaults).
 *   pad_negative_zero 1: padding inputs and absent subtrees are -0.0.
 *   launch_grid, launch_block, chunk_log2, partials, launches
 *                    the launch plan of the first (reduction) kernel, the
 *                    inputs per CTA work unit (log2; 0 if not chunked), the
 *                    number of fp32 partials written to scratch (0 if none)
 *                    and the number of kernel launches.  For FIXED_ORDER they
 *                    never change the result.
 *   dtype            tcr_dtype of the inputs (mode.dtype).
 *   run_log2         TCR_ORDER_BLOCKED_TREE: log2 of the run length (as given
 *                    in the mode); 0 otherwise.
 */
typedef struct {
    int kind;
    int order;
    size_t segment_len;
    size_t segments;
    int vector_len;
    int team_threads;
    int team_blocks;
    int chain_R;
    int pad_negative_zero;
    int launch_grid;
    int launch_block;
    int chunk_log2;
    size_t partials;
    int launches;
    int dtype;
    int run_log2;
} tcr_order_desc;

/*
 * tcr_order_descriptor -- fill *desc for the call tcr_reduce_sum(n) when
 * rows == 0, or tcr_reduce_rows(rows, cols) when rows > 0 (n is then
 * ignored).  Host only; queries the current device's SM count for the
 * launch plan.  Returns TCR_ERR_INVALID_ARG for the same arguments the
 * reduction would reject.
 */
TCR_API tcr_status tcr_order_descriptor(size_t n, size_t rows, size_t cols, tcr_mode mode,
                                tcr_order_desc *desc);

/*
 * tcr_order_equivalent -- *equivalent = 1 when the two described calls give
 * bit-identical results for every input, 0 when the descriptors cannot show
 * that.  Decided from the descriptors alone, in the spirit of the
 * bit-equivalence classes of "Taming Bitwise Behavior in GPU Kernels with
 * Tensor Core" (arXiv 2609.11356), Abstract (an autotuner restricted to one
 * class).  Same kind, dtype and segment_len are required; then
 *   TCR_FIXED_ORDER   equivalent when the run lengths agree once reduced to
 *                     what they do: runs of 1 or 2 inputs are the plain tree,
 *                     runs of at least the segment length the plain
 *                     left-to-right sum (the tree depends on the length and
 *                     the run length only);
 *   TCR_SHUFFLE_TREE  the block and grid trees are both balanced over power-
 *                     of-two warp counts, so together they are one balanced
 *                     tree over warp index: the order is fixed by the team
 *                     size T = team_threads * team_blocks alone, and by
 *                     nothing at all once T >= the number of vectors
 *                     (every thread then holds at most one);
 *   TCR_MMA_CHAIN(_TMEM) equivalent when chain_R, launch_block and chunk_log2
 *                     match (the tensor core's own order is fixed per shape).
 * Host only.  Returns TCR_ERR_INVALID_ARG for NULL pointers.
 */
TCR_API tcr_status tcr_order_equivalent(const tcr_order_desc *a, const tcr_order_desc *b,
                                        int *equivalent);

/*
 * Split-K GEMM with a declared K-partition combine -- the GEMM part of the
 * descriptor of reduction order of "Taming Bitwise Behavior in GPU Kernels
 * with Tensor Core" (arXiv 2609.11356), Abstract, which pins GEMM results
 * down by declaring how K is partitioned and how the partitions combine.
 *
 *   C (M x N, binary32, row-major) = A * W^T
 *   A: M x K, W: N x K, row-major binary16 or bfloat16 (dtype, both alike)
 *
 * K is cut into S splits of k_split columns (a multiple of 64; the last
 * split shorter).  P_s, the sum over split s, is one chain of tensor-core
 * MMAs accumulating in fp32 (the tensor core's own order inside, as in
 * TCR_MMA_CHAIN); C is the balanced binary32 tree over P_0 .. P_{S-1} in
 * split order (-0.0 pad), formed by a second kernel, never by atomics.  So
 * the bits of C depend only on (A, W, M, N, K, dtype, S, k_split) -- not on
 * the grid, the scheduling of CTAs or the GPU model -- and two calls with
 * equal descriptors give identical bits.  The MMAs run on pairs of SMs
 * (clusters of two CTAs issuing tcgen05.mma.cta_group::2 on 256 x 256
 * output tiles, each SM holding half of each operand tile) where the device
 * can co-schedule a pair, else one SM per 128 x 256 tile (also when the
 * environment variable TCR_GEMM_ONE_SM is set to a non-zero value); the
 * descriptor's tile_m, tile_n and launch_grid report which.  Error bound per element:
 *   |C - exact| <= (2^-22 * k_split / 16 + 2^-24 * ceil(log2 S)) * sum_k |a_ik w_jk| + 1e-30.
 *
 * tcr_gemm_descriptor -- fill *desc for a call (host only).
 *   splits  0 for the default rule -- with T the number of 128 x 256 output
 *           tiles, S = 1 when T >= 152, else min(32, floor(152 / T)): the
 *           most splits that keep the T x S work units within one wave of
 *           152 CTAs -- or the requested S in 1..64; either is then limited
 *           to ceil(K / 64) and reported as the effective S with its
 *           k_split (whole 64-column boxes per split, the last split
 *           shorter).  The rule depends on (M, N, K) only, never on the
 *           device, so the declared order is the same on every GPU.
 * tcr_gemm_splitk -- the GEMM.  A and W are device pointers, 16-byte
 *   aligned; C a device pointer, 4-byte aligned; M, N, K < 2^31 and K a
 *   multiple of 8 (the 16-byte row pitch of the tensor-map copies), else
 *   TCR_ERR_INVALID_ARG.  K == 0 writes +0.0 everywhere; S > 1 takes S x M x
 *   N floats of pool scratch and launches the combine.
 */
typedef struct {
    size_t M, N, K;
    int dtype;
    int splits;              /* effective S */
    size_t k_split;          /* K columns per split */
    int tile_m, tile_n, tile_k;
    int combine_order;       /* TCR_ORDER_BALANCED_TREE, over splits */
    size_t workspace_bytes;  /* pool scratch of the call */
    int launch_grid, launch_block;
    int launches;
} tcr_gemm_desc;

TCR_API tcr_status tcr_gemm_descriptor(size_t M, size_t N, size_t K, int splits, int dtype,
                                       tcr_gemm_desc *desc);
TCR_API tcr_status tcr_gemm_splitk(const void *A, const void *W, float *C, size_t M, size_t N,
                                   size_t K, int splits, int dtype, void *stream);

/*
 * tcr_device_faults -- the fault word of the current device: bit 0
 * (TCR_FAULT_PIPELINE_WAIT) is set when a wait inside a TCR_MMA_CHAIN_TMEM
 * or split-K GEMM kernel gave up after its limit of about one second (the kernel then
 * drained its own copies and tensor-core work, freed its tensor memory and
 * wrote NaN partials, so that call's result is NaN).  The word stays set
 * until cleared: clear != 0 resets it after reading.  Synchronous with
 * respect to the device (call it after the work in question has finished).
 * Returns TCR_ERR_INVALID_ARG for a NULL flags, TCR_ERR_CUDA if the device
 * cannot be read.
 */
#define TCR_FAULT_PIPELINE_WAIT 1u
TCR_API tcr_status tcr_device_faults(unsigned int *flags, int clear);

/*
 * tcr_read_probe -- a measurement aid, not part of the reduction method:
 * the read ceiling of the current GPU.  A kernel streams `bytes` bytes at x
 * in with the reduction kernels' 16-byte streaming loads (eight in flight
 * per thread) and writes the XOR of all their 32-bit words to *out (so the
 * loads cannot be optimised away); time it to learn what a read-only kernel
 * reaches on this GPU, beside the copy bandwidth that counts a read and a
 * write.  x: device pointer, 16-byte aligned; bytes a multiple of 16; out:
 * device word, 4-byte aligned (set to 0 first, on the stream, so the call is
 * a memset and one kernel launch).  Grid: ctas_per_sm CTAs (0: as many as
 * fit) of block_threads threads (0: 512; else a power of two in 32..1024)
 * on every SM, each thread striding over the whole input; or, for
 * ctas_per_sm = -1, one CTA per 8 x block_threads vectors (each thread eight
 * loads in flight, the block scheduler placing the CTAs -- the launch shape
 * of the reduction kernels).  TCR_ERR_INVALID_ARG on a bad argument,
 * TCR_ERR_CUDA if the device cannot be queried or the launch fails.
 * Asynchronous.
 */
TCR_API tcr_status tcr_read_probe(const void *x, size_t bytes, unsigned int *out, int ctas_per_sm,
                                  int block_threads, void *stream);

/* Static English text for a status code; never NULL. */
TCR_API const char *tcr_status_string(tcr_status status);

#ifdef __cplusplus
}
#endif

#endif /* TCR_H */
