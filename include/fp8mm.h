/*
 * fp8mm.h -- C ABI of the GB300 (sm_103a) FP8 scaled matrix multiply.
 *
 *   out[M,N] = bf16( (A[M,K] . B[K,N]) * (scale_a (x) scale_b) + bias[N] )
 *
 * A and B hold float8_e4m3fn codes; products are exact and accumulate in
 * fp32 on the tensor cores (tcgen05, accumulators in tensor memory); the
 * scale and the optional bias are applied to the fp32 sum, which is then
 * rounded once to bf16 (round to nearest even).
 *
 * Operation sources:
 *  - scaled_mm with per-tensor or row-wise scales, fp32 accumulation, output
 *    cast: gist "matmul_fp8.py" (FP8 Matmul), `matmul_fp8_kernel` and its
 *    scale epilogue; `torch._scaled_mm(a, b, scale_a, scale_b, out=...)` as
 *    called in `torch_scaled_mm`.
 *  - row-wise scales: x's scale of length M, y's of length N, TN layout only:
 *    PyTorch PR #125204 "fp8 row-scaling kernel for scaled_mm", Summary.
 *  - B column-major: gist "matmul_fp8.py", `benchmark()` (B is made
 *    column-major "for cuBLAS compatibility").
 *  - the bias epilogue: PyTorch PR #142045, Summary ("Limitations").
 *  - 16-byte aligned, contiguous operands; K * itemsize a multiple of 16 with
 *    out-of-range K zero-filled by TMA: PyTorch PR #142101, description and
 *    the review reply on K not divisible by the K block.
 *
 * Layout (all row-major, no padding, leading dimension = row length):
 *   A        e4m3fn [M, K], K contiguous.
 *   B        e4m3fn [K, N] column-major, i.e. the bytes of Bt[N, K] row-major.
 *   scale_a  fp32: 1 value (FP8MM_SCALE_TENSOR) or M values (FP8MM_SCALE_ROWWISE).
 *   scale_b  fp32: 1 value (FP8MM_SCALE_TENSOR) or N values (FP8MM_SCALE_ROWWISE).
 *   bias     bf16 [N], or NULL for none.
 *   out      bf16 [M, N], N contiguous.
 *
 * Constraints: M >= 0, N >= 0, K >= 16 and K % 16 == 0 (the TMA row pitch
 * of A and B must be a multiple of 16 bytes), A and B 16-byte aligned,
 * scale_a / scale_b / out 4-byte aligned, bias 2-byte aligned. M == 0 or
 * N == 0 is a no-op that returns FP8MM_OK (the pointers may then be NULL).
 * M, N <= 2^31 - 1, K <= 2^24.
 *
 * Ownership: the caller owns every buffer passed in; the library never keeps
 * or frees them. The library owns a per-device split-K workspace (fp32
 * partial tiles plus per-tile arrival counters) and the staging buffers of
 * fp8_scaled_mm_host, both grown on demand and kept until the process exits.
 * Each host thread keeps the TMA tensor maps of its last 32 operand and
 * output buffers (keyed on device, address, sizes, box, element type and
 * leading dimension: everything a map encodes), so repeated calls on the
 * same buffers skip encoding them; a buffer freed and reallocated at the
 * same address with the same shape gets the same, still correct, map.
 *
 * Logging: with FP8MM_LOG=1 in the environment, the first call of each
 * problem (device, batch, shape, scaling, element types, requested kernel)
 * prints one line on stderr naming the kernel chosen and whether the time
 * model, a tuned entry (fp8mm_autotune) or the caller chose it.
 *
 * Threading: calls may come from any host thread. Calls that use the split-K
 * workspace and run concurrently on different streams of one device race on
 * it; issue them on one stream.
 *
 * Errors: argument errors are found on the host before anything is enqueued
 * and come back as a negative fp8mm_status; nothing is launched then. A
 * failing CUDA call returns FP8MM_ERR_CUDA and fp8mm_last_cuda_error()
 * describes it. Kernels never trap: every wait inside them is bounded, and a
 * wait that runs out records FP8MM_ERR_TIMEOUT in a per-device status word
 * that fp8mm_device_status() reads.
 */
#ifndef FP8MM_H_
#define FP8MM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp8mm_scale_mode {
    FP8MM_SCALE_TENSOR = 0,   /* one fp32 per operand                          */
    FP8MM_SCALE_ROWWISE = 1   /* scale_a[M] per row of A, scale_b[N] per column of B */
} fp8mm_scale_mode;

typedef enum fp8mm_status {
    FP8MM_OK = 0,
    FP8MM_ERR_NULL = -1,      /* a required pointer is NULL                    */
    FP8MM_ERR_SHAPE = -2,     /* M, N or K out of range, or K % 16 != 0        */
    FP8MM_ERR_ALIGN = -3,     /* a pointer is not aligned as required          */
    FP8MM_ERR_MODE = -4,      /* unknown scale_mode or kernel variant          */
    FP8MM_ERR_CUDA = -5,      /* a CUDA call failed; see fp8mm_last_cuda_error() */
    FP8MM_ERR_NODEV = -6,     /* no CUDA device, or not an sm_103 device       */
    FP8MM_ERR_TIMEOUT = -7    /* a bounded in-kernel wait ran out              */
} fp8mm_status;

/* Kernel variants (fp8_scaled_mm_config). */
typedef enum fp8mm_variant {
    FP8MM_VARIANT_AUTO = 0,   /* heuristic choice (what fp8_scaled_mm uses)     */
    FP8MM_VARIANT_TILE = 1,   /* 128 x tile_n output tiles; tile rows over M    */
    FP8MM_VARIANT_SWAP = 2,   /* operands swapped: 128-row tiles over N, tile_n columns over M */
    FP8MM_VARIANT_PAIR = 3,   /* 2-SM MMA: a CTA pair computes 256 x tile_n tiles, with split-K
                                 or stream-K (split_k = -1) */
    FP8MM_VARIANT_SWAPK = 4,  /* SWAP tiles with K spread over a cluster of split_k CTAs,
                                 reduced through distributed shared memory (no workspace) */
    FP8MM_VARIANT_SWAPPAIR = 5 /* SWAP with 2-SM MMA: a CTA pair covers 256 rows of N and
                                  shares the tile_n rows of A (no split-K) */
} fp8mm_variant;

/*
 * out = bf16(A.B * (scale_a (x) scale_b) + bias), enqueued on `stream`
 * (a cudaStream_t; NULL = the legacy default stream). All pointers are device
 * pointers (or managed memory) of the current device. Asynchronous: returns
 * once the work is enqueued; no host synchronisation.
 */
int fp8_scaled_mm(const void *A, const void *B,
                  const float *scale_a, const float *scale_b, int scale_mode,
                  const void *bias, void *out,
                  int64_t M, int64_t N, int64_t K,
                  void *stream);

/*
 * Same operation with an explicit kernel choice (tests, tuning, benchmarks).
 *   variant   fp8mm_variant; AUTO ignores tile_n and split_k.
 *   tile_n    TILE: 128 or 256. SWAP: 16, 32, 64 or 128 (M is covered by
 *             ceil(M / tile_n) column tiles). PAIR: 128 or 256. SWAPK: as
 *             SWAP. SWAPPAIR: 16, 32, 64 or 128. 0 = heuristic.
 *   split_k   1 .. 16 K-slices per output tile (reduced deterministically in
 *             slice order by the last slice to arrive); SWAPPAIR takes 0 or 1;
 *             SWAPK takes the cluster size 2, 4 or 8 (0 = 4); PAIR also takes
 *             -1: stream-K, where the tiles of the last partial wave (plus one
 *             full wave) have their K blocks divided evenly over all CTA
 *             pairs and each such tile is finished by the pair holding its
 *             first K block, which adds the other pieces' fp32 partials in K
 *             order (deterministic). 0 = heuristic.
 * Returns FP8MM_ERR_MODE for an unsupported combination.
 */
int fp8_scaled_mm_config(const void *A, const void *B,
                         const float *scale_a, const float *scale_b, int scale_mode,
                         const void *bias, void *out,
                         int64_t M, int64_t N, int64_t K,
                         void *stream, int variant, int tile_n, int split_k);

/* Element types of fp8_scaled_mm_ex. */
typedef enum fp8mm_type {
    FP8MM_TYPE_E4M3 = 0,      /* float8_e4m3fn operand                          */
    FP8MM_TYPE_E5M2 = 1       /* float8_e5m2 operand                            */
} fp8mm_type;

typedef enum fp8mm_out_type {
    FP8MM_OUT_BF16 = 0,       /* bf16 output and bias                           */
    FP8MM_OUT_F16 = 1,        /* IEEE fp16 output and bias                      */
    FP8MM_OUT_F32 = 2,        /* IEEE fp32 output and bias (bias 4-byte aligned) */
    FP8MM_OUT_E4M3 = 3        /* float8_e4m3fn output, saturating at +-448; bf16 bias */
} fp8mm_out_type;

typedef struct fp8mm_options {
    int a_type;               /* fp8mm_type of A                                */
    int b_type;               /* fp8mm_type of B                                */
    int out_type;             /* fp8mm_out_type of out and bias                 */
    int variant;              /* fp8mm_variant (0 = heuristic)                  */
    int tile_n;               /* as in fp8_scaled_mm_config (0 = heuristic)     */
    int split_k;              /* as in fp8_scaled_mm_config (0 = heuristic)     */
    int64_t ldo;              /* elements between consecutive rows of out: 0 = N
                                 (contiguous), otherwise >= N, e.g. to write the
                                 product into columns of a wider matrix; batched
                                 items then sit M * ldo elements apart. Rows whose
                                 byte pitch is not a multiple of 16 are written
                                 with plain stores instead of TMA. */
} fp8mm_options;

/*
 * The operation with other element types: A and B each e4m3fn or e5m2
 * (mixed allowed; the tensor cores multiply them exactly and sum in fp32),
 * and the output bf16, fp16, fp32 or e4m3fn: one conversion of the fp32
 * result acc * scale + bias, round to nearest even. bf16 / fp16 / fp32
 * outputs take a bias of their own type; an e4m3fn output takes a bf16
 * bias, and values that round above 448 in magnitude (and infinities)
 * saturate to +-448 while NaN stays NaN (0x7F), as the hardware conversion
 * does. Sources: the gist "matmul_fp8.py", `benchmark()`, quantises to
 * float8_e4m3fn or float8_e5m2 and takes the output dtype as an argument,
 * and `matmul_fp8_kernel` casts the accumulator to the output's dtype
 * ("Cast the accumulator to output dtype (fp8)"). out is [M, N] row-major
 * with elements of 2, 2, 4 or 1 bytes. Layouts, alignment and the other
 * arguments as fp8_scaled_mm / _config; unknown type codes return
 * FP8MM_ERR_MODE; options == NULL returns FP8MM_ERR_NULL.
 */
int fp8_scaled_mm_ex(const void *A, const void *B,
                     const float *scale_a, const float *scale_b, int scale_mode,
                     const void *bias, void *out,
                     int64_t M, int64_t N, int64_t K,
                     void *stream, const fp8mm_options *options);

/*
 * Host-memory entry point: A, B, scale_a, scale_b, bias and out are HOST
 * pointers (pinned memory gives full copy bandwidth; pageable works). The
 * call copies the inputs to device staging buffers owned by the library
 * (grown on demand, kept per device), computes, copies the result back into
 * `out` and synchronises `stream` before returning. Internally A's rows and
 * B's columns are cut into up to 4 chunks each and out into the blocks they
 * form; the chunks arrive in a growing square (A chunk k, then B chunk k,
 * after which every block of row k and column k has its operands), so that
 * blocks are computed and copied back while later chunks arrive, on three
 * library streams; the work is ordered after everything already queued on
 * `stream`. Same layouts, constraints and result as fp8_scaled_mm within the
 * parity tolerance (each block runs the kernel fp8_scaled_mm would choose
 * for the block's shape; blocks start at multiples of 256 rows and columns).
 */
int fp8_scaled_mm_host(const void *A, const void *B,
                       const float *scale_a, const float *scale_b, int scale_mode,
                       const void *bias, void *out,
                       int64_t M, int64_t N, int64_t K,
                       void *stream);

/* Which dimension of an operand is contiguous in memory. */
typedef enum {
    FP8MM_MAJOR_K = 0,   /* K contiguous: A row-major [M, K]; B column-major [K, N] */
    FP8MM_MAJOR_MN = 1   /* M (for A) or N (for B) contiguous: A column-major; B row-major */
} fp8mm_major;

/*
 * fp8_scaled_mm_ex with either operand in either layout (the four layout
 * combinations of a matrix product). The pages pass transposed layouts of
 * A and B to their Triton matmul template as compile-time flags (PyTorch PR
 * #142101, "Additional notes"); their FP8 scaled_mm is TN only (PR #125204,
 * Summary). Here an MN-major operand is first transposed on the GPU into a
 * library-owned staging buffer (an HBM-bound byte transpose, one read and
 * one write of the operand), then the K-major kernels run. Scales keep their
 * meaning: row-wise scale_a has one value per row of A and scale_b one per
 * column of B, whatever the layout.
 *
 *   A        a_major K: [M, K] row-major; MN: [M, K] column-major (= At [K, M] row-major)
 *   B        b_major K: [K, N] column-major (= Bt [N, K]); MN: [K, N] row-major
 *   other arguments as fp8_scaled_mm_ex (options may be NULL).
 *
 * The staging buffers (M*K and N*K bytes) are grown on demand and kept per
 * device; growing them synchronises the device, so make a first call of the
 * largest shape before any stream capture. Calls on different streams of
 * one device that both transpose race on the staging buffers.
 */
int fp8_scaled_mm_layout(const void *A, int a_major, const void *B, int b_major,
                         const float *scale_a, const float *scale_b, int scale_mode,
                         const void *bias, void *out,
                         int64_t M, int64_t N, int64_t K,
                         void *stream, const fp8mm_options *options);

/*
 * Batched form: `batch` independent products of one shape,
 *
 *   out[b] = cast( (A[b] . B[b]) * (scale_a[b] (x) scale_b[b]) + bias )
 *
 * for b < batch, in one launch (the operands are read through 3-D TMA
 * tensor maps [batch, rows, K]). The pages name this case as the one that
 * 2-D-only TMA descriptors block (PyTorch PR #142101, "Additional notes",
 * the note on torch.bmm); each item follows fp8_scaled_mm exactly.
 *
 *   A        fp8 [batch, M, K]: items back to back, each row-major.
 *   B        fp8 [batch, K, N] with every item column-major, i.e. the bytes
 *            of Bt [batch, N, K] row-major.
 *   scale_a  fp32: batch values (FP8MM_SCALE_TENSOR, one per item) or
 *            batch * M values (ROWWISE, item b's at b * M).
 *   scale_b  fp32: batch or batch * N values, likewise.
 *   bias     [N] of the output type shared by every item, or NULL.
 *   out      [batch, M, N], items back to back, each row-major.
 *   options  element types and kernel choice as for fp8_scaled_mm_ex; NULL
 *            for e4m3 operands, bf16 output, automatic choice.
 *
 * Constraints as fp8_scaled_mm, plus batch >= 0 (0 is a no-op) and
 * batch * ceil(M/16) * ceil(N/128) * 16 < 2^31 (FP8MM_ERR_SHAPE otherwise).
 */
int fp8_scaled_bmm(const void *A, const void *B,
                   const float *scale_a, const float *scale_b, int scale_mode,
                   const void *bias, void *out,
                   int64_t batch, int64_t M, int64_t N, int64_t K,
                   void *stream, const fp8mm_options *options);

/*
 * Quantise bf16 data to fp8 codes with fp32 scales: the step that makes the
 * operands of fp8_scaled_mm (gist "matmul_fp8.py", `get_scale` and
 * `benchmark()`):
 *
 *   amax  = max |x|  over all of x (FP8MM_SCALE_TENSOR) or over each row
 *           (FP8MM_SCALE_ROWWISE)
 *   scale = amax / qmax, in fp32; qmax = 448 (e4m3fn) or 57344 (e5m2), the
 *           format's largest finite value (torch.finfo(dtype).max)
 *   q     = fp8(clamp(x / scale, -qmax, qmax)): fp32 division, correctly
 *           rounded; conversion rounds to nearest, ties to even
 *
 * For B pass Bt, i.e. B [K, N] column-major as the row-major [N, K] array:
 * its row-wise scales are then B's per-column scales, the layout
 * fp8_scaled_mm takes.
 *
 *   x      device bf16 [R, C], row-major, C contiguous; 16-byte aligned.
 *   R, C   R >= 0, C >= 0, C % 8 == 0. R == 0 or C == 0 is a no-op.
 *   scale_mode  FP8MM_SCALE_TENSOR or FP8MM_SCALE_ROWWISE.
 *   q_type FP8MM_TYPE_E4M3 or FP8MM_TYPE_E5M2.
 *   q      device fp8 [R, C] (output), 8-byte aligned.
 *   scale  device fp32 (output): 1 value, or R values (row-wise); 4-byte aligned.
 *
 * Cases the recipe leaves open: a zero scale (all elements +-0) gives the
 * codes of +-0 instead of the NaN of 0/0; every NaN encodes as 0x7F; a NaN
 * anywhere in the tensor (row) makes its scale NaN and all its codes NaN;
 * an infinity makes the scale inf, finite elements then encode as +-0.
 *
 * Asynchronous on `stream`. Row-wise is one kernel launch. Per-tensor is one
 * cooperative launch (one CTA per SM, a grid-wide amax exchange with a
 * bounded wait that records FP8MM_ERR_TIMEOUT in the device status word if it
 * runs out), or two launches (amax, then conversion) for tensors under 1 MB
 * and where the device cannot hold that grid at once
 * (fp8mm_describe_quant_plan reports which). It uses a small per-device scratch owned by the
 * library (per-CTA maxima, a call number and counters), so per-tensor calls
 * that overlap on the GPU on different streams of one device race on it.
 */
int fp8_quantize(const void *x, int64_t R, int64_t C, int scale_mode, int q_type,
                 void *q, float *scale, void *stream);

/*
 * The whole path from bf16 operands: quantise A [M, K] and B (column-major
 * [K, N], i.e. Bt [N, K] row-major) as fp8_quantize does, with scale_mode
 * for both, then out = fp8_scaled_mm_ex(A_q, B_q, scale_a, scale_b, ...).
 * The launches are chained on `stream` (programmatic dependent launch).
 *
 *   A, B      device bf16, 16-byte aligned; K % 16 == 0 as for fp8_scaled_mm.
 *   A_q, B_q  device fp8 outputs, [M, K] and Bt [N, K], 16-byte aligned;
 *             their element types are options->a_type / b_type.
 *   scale_a, scale_b  device fp32 outputs, 1 or M / N values.
 *   bias, out as fp8_scaled_mm_ex (out type options->out_type).
 *   options   may be NULL: e4m3 operands, bf16 out, automatic kernel choice.
 *
 * The caller owns A_q, B_q and the scales, which hold the quantised
 * operands afterwards (reusable as fp8_scaled_mm inputs).
 */
int fp8_scaled_mm_bf16(const void *A, const void *B, int scale_mode,
                       const void *bias, void *out,
                       int64_t M, int64_t N, int64_t K,
                       void *A_q, void *B_q, float *scale_a, float *scale_b,
                       void *stream, const fp8mm_options *options);

/*
 * Allocation-free variant of fp8_scaled_mm. The pages have no counterpart:
 * this is an addition for callers that cannot allocate device memory while
 * they run (for example code running inside a memory pool it does not own,
 * or a runtime whose device memory was partitioned up front), because
 * fp8_scaled_mm may cudaMalloc its split-K workspace on first use.
 *
 * Same arguments, layouts and result as fp8_scaled_mm. The split-K scratch
 * is a fixed array inside the library's device image (about 16.1 MiB, held
 * by every GPU that loads the library until the process exits): at most
 * 16 MiB of fp32 partial tiles and 64 KiB of arrival counters. A problem
 * whose kernel choice needs more is rejected with FP8MM_ERR_SHAPE and a
 * message in fp8mm_last_error(); nothing is launched then. The call makes
 * no cudaMalloc/cudaFree and uses no allocating library routine.
 *
 * The first call on a device does a one-time set-up (device checks and the
 * scratch array's device address); make that first call before any stream
 * capture. Every call on a device shares the scratch array and clears the
 * parts it needs on `stream` first; calls that overlap on the GPU race on
 * it. In-kernel wait timeouts of this entry point are not reported through
 * fp8mm_device_status().
 */
int fp8_scaled_mm_noalloc(const void *A, const void *B,
                          const float *scale_a, const float *scale_b, int scale_mode,
                          const void *bias, void *out,
                          int64_t M, int64_t N, int64_t K,
                          void *stream);

/*
 * Shape-keyed autotuning. The pages tune their kernels per problem shape
 * (gist "matmul_fp8.py", the `triton.autotune` configs keyed on M, N, K and
 * the scaling; PyTorch PR #130422, max-autotune of scaled_mm). Here the
 * candidates are the kernel configurations compiled into the library (pair
 * and 1-SM kernels with their split-K factors for M > 128; SWAP, cluster-K
 * and pair-SWAP kernels for M <= 128).
 *
 * fp8mm_autotune times every candidate for a (batch, M, N, K, scale_mode,
 * element types) problem on the current device and remembers the fastest;
 * from then on fp8_scaled_mm, _ex, _bmm, _layout, _bf16 and _host calls of
 * that shape with automatic kernel choice (variant FP8MM_VARIANT_AUTO) use
 * it. The operands are scratch buffers the call allocates, fills with
 * pseudo-random finite fp8 codes and frees (copies rotated so that they
 * exceed L2); each candidate runs 2 warm-up launches and is timed over 5
 * launches with CUDA events on `stream`; the call synchronises the device
 * and must not run during stream capture. options: element types only (NULL
 * for e4m3 operands and bf16 output); batch >= 1. Returns FP8MM_OK, an
 * argument error, FP8MM_ERR_CUDA, or FP8MM_ERR_TIMEOUT if a candidate's
 * bounded wait ran out. fp8_scaled_mm_noalloc ignores tuned choices (its
 * scratch bound is that of the built-in choice).
 */
int fp8mm_autotune(int64_t batch, int64_t M, int64_t N, int64_t K, int scale_mode,
                   const fp8mm_options *options, void *stream);

/* Forget every tuned choice of this process. */
int fp8mm_autotune_clear(void);

/* Number of tuned choices held. */
int fp8mm_autotune_count(void);

/*
 * Write the tuned choices to a text file (one line per shape: device
 * compute capability and SM count, batch, M, N, K, scale mode, element
 * types, then the kernel, tile_n, split and the measured microseconds), or
 * read such a file and add its entries (entries for other devices are kept
 * and only used on a matching device). Load returns the number of entries
 * read, or FP8MM_ERR_NULL / FP8MM_ERR_SHAPE (unreadable file or a malformed
 * line; entries before it are kept).
 */
int fp8mm_autotune_save(const char *path);
int fp8mm_autotune_load(const char *path);

/*
 * Grow the current device's split-K workspace to at least `bytes` now, so
 * that later calls do not allocate (for example before a CUDA graph
 * capture). The pages' persistent TMA scaled_mm template is launched with a
 * device workspace argument beside its operands (PyTorch PR #142045, review
 * of torch/_inductor/kernel/mm_scaled.py, `get_tma_workspace_arg`); here the
 * library owns that memory and holds the fp32 partial tiles of the split-K
 * reduction (gist "matmul_fp8.py", `matmul_fp8_kernel`, SPLIT_K).
 *   bytes  >= 0; FP8MM_ERR_SHAPE if negative. Growing synchronises the
 *          device (the old buffer may be in use) and frees the old buffer.
 * Returns FP8MM_OK, FP8MM_ERR_NODEV or FP8MM_ERR_CUDA (cudaMalloc failed;
 * fp8mm_last_cuda_error() says why).
 */
int fp8mm_reserve_workspace(int64_t bytes);

/*
 * Synchronise `stream`, then read and clear the current device's in-kernel
 * status word. Returns FP8MM_OK, FP8MM_ERR_TIMEOUT (a bounded wait ran out;
 * that launch's output is undefined, the split-K counters are reset here),
 * or FP8MM_ERR_CUDA.
 */
int fp8mm_device_status(void *stream);

/*
 * Test hook for the bounded in-kernel waits (failure detection without a GPU
 * fault). From the next launch on, in the 128-row kernels (TILE, SWAP), the
 * TMA producer of CTA 0 stops after `stop_after_kblocks` K blocks, so the
 * MMA thread's wait for the next block runs out; in the pair kernel's
 * stream-K schedule, the partials of CTA pair 1 are never flagged, so the
 * owner's wait for them runs out. Either way the kernel records
 * FP8MM_ERR_TIMEOUT in the device status word, releases its tensor memory
 * and returns; that launch's output is undefined. `wait_limit_cycles` > 0
 * replaces the wait budget of every kernel (default 4e9 clock64 cycles).
 * fp8mm_debug_inject(-1, 0) restores normal operation. Returns
 * FP8MM_ERR_SHAPE for out-of-range arguments. Not for production use.
 */
int fp8mm_debug_inject(int64_t stop_after_kblocks, int64_t wait_limit_cycles);

/*
 * Test hook for per-tensor quantisation (fp8_quantize, fp8_scaled_mm_bf16),
 * from the next call on: mode 0 is normal operation (one cooperative launch
 * with a grid-wide amax, falling back to two launches only when the device
 * cannot hold the grid at once); mode 1 always takes the two-launch form (an
 * amax kernel, then a convert kernel), so that it can be tested; mode 2
 * makes CTA 0 of the one-launch kernel withhold its share of the grid-wide
 * amax, so every CTA's bounded wait for it runs out: the kernel records
 * FP8MM_ERR_TIMEOUT in the device status word and returns without writing
 * codes or the scale. Returns FP8MM_ERR_MODE for other modes. Not for
 * production use.
 */
int fp8mm_debug_quant(int mode);

/*
 * Static description of a status code (never NULL; "unknown status" for a
 * code not in fp8mm_status). The codes report the operand conditions the
 * pages state for the TMA scaled_mm path, 16-byte aligned contiguous
 * operands and K * itemsize a multiple of 16 (PyTorch PR #142101,
 * description, and the review reply on K not divisible by the K block), and
 * the pages' rejection of an unknown scaling granularity (gist
 * "matmul_fp8.py", `get_scale`, which raises for anything but per-tensor and
 * per-row). The returned string is static; the caller must not free it.
 */
const char *fp8mm_status_string(int status);

/*
 * Detail of the last failure on this host thread, "" if none: set whenever
 * a call returns FP8MM_ERR_CUDA (the failing CUDA call with its error name
 * and message) or FP8MM_ERR_TIMEOUT from fp8mm_device_status (the wait that
 * ran out), and for the few argument errors that need more than a status
 * code (a tensor-map encoding the driver refused, a problem beyond
 * fp8_scaled_mm_noalloc's scratch). Thread-local; the pointer stays valid
 * until the next call on this thread. The pages raise Python exceptions
 * with a message at the same points (gist "matmul_fp8.py", `get_scale`).
 */
const char *fp8mm_last_cuda_error(void);

/* The same string as fp8mm_last_cuda_error (an alias kept for callers of
 * earlier builds). */
const char *fp8mm_last_error(void);

/* The kernel fp8_scaled_mm would launch for this problem, as text; for logs
 * and tests. Format: the variant ("tile", "swap", "pair", "swapk",
 * "swappair") followed by key=value fields: tile_n, split (K slices; the
 * cluster size for swapk), tiles (row tiles x column tiles per item), units
 * (work units dealt round-robin), grid (CTAs), and when they apply
 * stream_k_tiles (tiles whose K blocks are spread over all CTA pairs) and
 * group (tile rows per group of the tile order, when not 8). Example:
 * "pair tile_n=256 split=1 tiles=32x32 units=912 grid=152
 * stream_k_tiles=112 group=16". */
const char *fp8mm_describe_choice(int64_t M, int64_t N, int64_t K, int scale_mode);

/* The same for a batch of `batch` products (fp8_scaled_bmm); tiles are per
 * item, units count the whole batch. Both report a tuned choice
 * (fp8mm_autotune) for e4m3 operands and bf16 output when one is held. */
const char *fp8mm_describe_bmm_choice(int64_t batch, int64_t M, int64_t N, int64_t K, int scale_mode);

/* The automatic choice the time model makes for a device with `sms` SMs, in
 * the same format: no device is needed and tuned entries are not consulted
 * (the choice a device of that size makes before fp8mm_autotune). For tests
 * of the dispatch on any host and for planning. Returns "no-op or invalid
 * shape" for M, N <= 0, K < 16, batch <= 0 or sms < 2. The string is
 * thread-local and valid until the next describe call on this thread. */
const char *fp8mm_describe_model_choice(int64_t batch, int64_t M, int64_t N, int64_t K, int sms);

/* The launch plan fp8_quantize takes for bf16 [R, C] on a device with `sms`
 * SMs, without a device: "rows team=<lanes>x<warps> chunks=<groups per
 * thread>" or "rows long" (row-wise), "tensor one-launch grid=<CTAs>
 * tmem=<0|1> keep=<groups per CTA marked evict-last>" or "tensor
 * two-launch" (per-tensor; the one-launch form also falls back to two
 * launches on a device that cannot hold its grid at once). Returns "no-op or
 * invalid shape" for R, C <= 0, C % 8 != 0, sms < 1 or an unknown
 * scale_mode. Thread-local string, valid until the next describe call. */
const char *fp8mm_describe_quant_plan(int64_t R, int64_t C, int scale_mode, int sms);

#ifdef __cplusplus
}
#endif

#endif /* FP8MM_H_ */
