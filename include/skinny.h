/*
 * skinny.h -- C ABI of the GB300 (sm_103a) decode GEMM and reduce + residual +
 * RMSNorm library (libskinny.so).
 *
 * Two operations of a speculative-decoding drafter step, as the vLLM DSpark
 * drafter pages define them:
 *
 *   decode_gemm_bf16         out[M,N] = x[M,K] @ W[N,K]^T, BF16 operands, FP32
 *                            accumulation, one BF16 rounding
 *                            ("drafter/linears": module text, DraftGemm).
 *   reduce_residual_rmsnorm  TP BF16 partial rows summed in FP32 in rank order,
 *                            rounded once; residual added, rounded once; RMSNorm
 *                            of the result ("drafter/comm": module text, ArNorm;
 *                            "cutedsl/common/twoshot": reduce, whose one-GPU
 *                            stand-in lets TP local slots play the ranks).
 *
 * Conventions for every entry point below:
 *  - Pointers are DEVICE pointers (memory of the current CUDA device, from
 *    cudaMalloc / a PyTorch CUDA tensor) unless a comment says otherwise. The
 *    caller owns every buffer; the library keeps no pointer after a call returns.
 *  - BF16 values are IEEE bfloat16 (uint16 bit patterns in memory).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is
 *    enqueued on it; the call returns without waiting for the GPU.
 *  - Return value: SKINNY_OK (0) or a skinny_status code. On any nonzero code
 *    nothing was launched and no output was touched. Faults of the GPU work
 *    itself surface later, at a stream synchronisation, as CUDA errors.
 *  - Every wait inside a decode GEMM kernel is bounded (1 s). A kernel whose
 *    wait ran out records it in a device error word and in a host-mapped word;
 *    from then on every call that uses the decode GEMM's scratch on that device
 *    returns SKINNY_ERR_TIMEOUT without launching, until skinny_device_error()
 *    reads and clears the error (and re-arms the scratch). The output of the
 *    kernel that gave up is unspecified. The reduce kernel's wait for its
 *    cluster's sums of squares is bounded too (1 s); one that runs out leaves
 *    that call's output unspecified and is reported by skinny_device_error()
 *    (bit 128), without holding back later calls (the reduce keeps no state).
 *  - Nothing is allocated per call. decode_gemm_bf16 uses a per-device scratch
 *    area (split-K partial sums, published-partial flags, an error word, plus
 *    one page of host-mapped memory) that its first call on each device
 *    allocates; make that first call outside CUDA stream capture. All calls on
 *    one device share that scratch, whatever their stream: calls whose kernels
 *    may run at the same time (streams not ordered with each other by events or
 *    a common predecessor) race on it and give wrong results, so order them.
 *  - Launch settings: programmatic dependent launch and the decode GEMM's L2
 *    lead are process-wide settings (skinny_set_pdl, skinny_set_l2_prefetch)
 *    that the _ex entry points override per call (skinny_launch_opts), so code
 *    that wants its own settings never changes what other threads' calls see;
 *    the decode GEMM's prefetch after a reduce is a per-call setting only.
 *    None of them changes a result bit.
 *  - Calls are thread-safe on the host.
 */
#ifndef SKINNY_H
#define SKINNY_H

#include <stddef.h>

#if defined(__GNUC__)
#define SKINNY_API __attribute__((visibility("default")))
#else
#define SKINNY_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SKINNY_OK = 0,
    SKINNY_ERR_NULL = 1,     /* a required pointer is NULL */
    SKINNY_ERR_SHAPE = 2,    /* a size is outside the accepted range */
    SKINNY_ERR_ALIGN = 3,    /* a pointer is not aligned as required */
    SKINNY_ERR_DEVICE = 4,   /* no sm_103 device, or a pointer is not memory of it */
    SKINNY_ERR_LAUNCH = 5,   /* the CUDA launch itself failed */
    SKINNY_ERR_ALIAS = 6,    /* an output overlaps an input or the other output */
    SKINNY_ERR_CAPTURE = 7,  /* first call on a device made during stream capture */
    SKINNY_ERR_ALLOC = 8,    /* the one-time scratch allocation failed */
    SKINNY_ERR_TIMEOUT = 9,  /* a kernel's bounded internal wait ran out */
    SKINNY_ERR_ARG = 10      /* a scalar argument is invalid (eps, timeout, ...) */
} skinny_status;

/* Row width of every reduce + RMSNorm row: 7168 ("drafter/comm", ArNorm
 * docstring: the all-reduced rows are M x 7168 BF16; the mean divides by 7168). */
#define SKINNY_HIDDEN 7168
/* Largest row count of decode_gemm_bf16: the pages' engine keeps its speed for at
 * most 32 rows ("drafter/linears" module text); this library also serves 33..64
 * (the row cap of the pages' reduction buffers, "cutedsl/common/twoshot", cap=64). */
#define SKINNY_GEMM_MAX_M 64
/* Largest row count of reduce_residual_rmsnorm (the row cap of the pages'
 * reduction buffers, "cutedsl/common/twoshot", TwoShot: cap=64). */
#define SKINNY_REDUCE_MAX_M 64
/* Largest TP (number of partial slots) of reduce_residual_rmsnorm (TP8 on the
 * pages, "drafter/comm" module text). */
#define SKINNY_REDUCE_MAX_TP 8

/* Per-call launch settings of the _ex entry points. Each field is either a
 * value or SKINNY_OPT_DEFAULT, which takes the process-wide setting. */
#define SKINNY_OPT_DEFAULT (-1)
typedef struct {
    int pdl;          /* 1: programmatic dependent launch (see skinny_set_pdl), 0: off */
    int l2_prefetch;  /* decode GEMM deep-ring L2 lead in [0, 64] (see
                         skinny_set_l2_prefetch); ignored by the reduce */
    int l2_after_reduce;
    /* decode GEMM only, for the call that follows decode_gemm_bf16_reduce_rmsnorm
     * in the same stream (a layer chain's next first GEMM): weight blocks in
     * [0, 64] each CTA prefetches into L2, beyond its ring's first fill, as soon
     * as that call's reduce has seen its GEMM complete -- so that HBM streams
     * this GEMM's weights while the reduce runs, without slowing the previous
     * GEMM's last CTAs. The CTA waits at most 50 us for that signal, then goes
     * on without it. 0 or SKINNY_OPT_DEFAULT: off. Timing only: no result bit
     * depends on it. The signal is one word of the device's scratch, shared by
     * every stream like the split-K scratch; it stays set until the next
     * decode_gemm_bf16_reduce_rmsnorm's GEMM clears it, so a call that is not
     * behind one may prefetch at once. */
} skinny_launch_opts;

/*
 * decode_gemm_bf16 -- out[M,N] = x[M,K] @ W[N,K]^T
 *   ("drafter/linears": the module text fixes the precision -- BF16 inputs, an
 *    FP32 accumulator, a single rounding to BF16, the same arithmetic as cuBLAS
 *    with the order of the additions free; DraftGemm gives the product
 *    out[M, N] = x[M, K] @ weight[N, K]^T.)
 *
 *   x    [M, K] BF16, row-major (row stride K elements), 16-byte aligned.
 *   W    [N, K] BF16, row-major (each weight row is one output column), 16-byte
 *        aligned. Read exactly once from HBM.
 *   out  [M, N] BF16, row-major (row stride N elements), 2-byte aligned. Written
 *        once; must not overlap x or W.
 *   1 <= M <= 64;  N >= 1;  K >= 8 and K % 8 == 0 (16-byte row strides);
 *   ceil(N / 128) * ceil(K / 64) < 2^31 (a weight below 32 TiB).
 *   Ragged N (N % 128 != 0) and ragged K (K % 64 != 0) are handled exactly.
 *
 *   Every out element is the FP32 sum of the K products (split over K across
 *   CTAs, partial sums added in K order), rounded once to BF16 (nearest even).
 *   Deterministic: the same inputs on the same device give the same bits.
 *   Errors: SKINNY_ERR_NULL, _SHAPE, _ALIGN, _ALIAS, _DEVICE, _CAPTURE, _ALLOC,
 *   _LAUNCH as above; _TIMEOUT while an earlier kernel's wait that ran out is
 *   not yet cleared (see the conventions at the top).
 */
SKINNY_API int decode_gemm_bf16(const void *x, const void *W, void *out,
                     int M, int N, int K, void *stream);

/*
 * decode_gemm_bf16_ex -- decode_gemm_bf16 with per-call launch settings.
 *   opts: host pointer, or NULL for the process-wide settings. The settings
 *   change when and how the kernel's work is scheduled, never a result bit.
 *   Errors: as decode_gemm_bf16, plus SKINNY_ERR_ARG for a field out of range.
 */
SKINNY_API int decode_gemm_bf16_ex(const void *x, const void *W, void *out, int M, int N,
                                   int K, const skinny_launch_opts *opts, void *stream);

/*
 * decode_gemm_bf16_logits -- the lm_head logits with the epilogue fused
 *   ("drafter/linears", draft_logits: the lm_head GEMM, then the slice to
 *    org_vocab_size, then tanh(logits / soft_cap) * soft_cap if a soft cap is
 *    set, then logits * scale.)
 *
 *   x [M, K], W [N, K] as for decode_gemm_bf16; out [M, n_out] BF16 (row stride
 *   n_out). out[m][n] = BF16(scale * c(sum_k x[m,k] W[n,k])) for n < n_out, with
 *   c(v) = soft_cap * tanh(v / soft_cap) if soft_cap > 0, else v; the epilogue
 *   runs on the FP32 sum and rounds once (the pages apply it one BF16 tensor op
 *   at a time). Only the first n_out weight rows are read. 1 <= n_out <= N;
 *   soft_cap and scale finite. Other rules and errors as decode_gemm_bf16.
 */
SKINNY_API int decode_gemm_bf16_logits(const void *x, const void *W, void *out, int M,
                                       int N, int K, int n_out, float soft_cap, float scale,
                                       void *stream);

/*
 * decode_gemm_bf16_noalloc -- decode_gemm_bf16 that allocates no device memory
 *   The drafter pages have no counterpart to this entry point. It is for callers
 *   that cannot let a library call cudaMalloc: serving engines that hand all
 *   spare device memory to their own pool at start-up, so that a later
 *   allocation fails or forces the pool to give memory back; plug-ins that may
 *   only take memory from their host framework's allocator; loops that cannot
 *   afford cudaMalloc's implicit device synchronisation.
 *
 *   Same arguments, layouts, results and errors as decode_gemm_bf16 (the same
 *   kernel runs). The split-K scratch -- partial tiles, published-partial flags, error
 *   word -- lives instead in one static device array of the library, 5.2 MB,
 *   which every GPU that loads the library holds until the process exits. It has
 *   partial-tile slots for 160 CTAs of up to 32 rows: the call runs with
 *   min(SM count, 160) CTAs and rejects M > 32 with SKINNY_ERR_SHAPE.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   Each call first clears the flags and the error word with a
 *   cudaMemsetAsync on `stream`, then launches the kernel. All calls share the
 *   one array: calls whose GPU work may overlap (streams not ordered with each
 *   other on the same device) race and give wrong results; order them. A kernel
 *   wait that runs out still ends the kernel, but this entry point does not
 *   report it (the next call clears the word); the output is then unspecified.
 */
SKINNY_API int decode_gemm_bf16_noalloc(const void *x, const void *W, void *out,
                                        int M, int N, int K, void *stream);

/*
 * reduce_residual_rmsnorm -- the ArNorm row operation on TP local slots
 *   ("drafter/comm": the module text and the ArNorm kernel define the steps --
 *    the TP partial rows are added in FP32 from rank 0 upwards and rounded to
 *    BF16 once, the residual is added with a second BF16 rounding, and the
 *    RMSNorm of that new residual uses an FP32 sum of squares, the reciprocal
 *    square root of its mean over 7168 columns plus eps, and one rounding of
 *    x * rstd * gamma; the ArNorm docstring gives the argument list and, when no
 *    residual is given, makes the summed row itself the new residual.
 *    "cutedsl/common/twoshot": with a single owner the TP ranks can be local
 *    slots of one GPU, the stand-in used here.)
 *
 *   partials      [TP, M, 7168] BF16, contiguous (slot r = rank r's partial row),
 *                 16-byte aligned.
 *   residual      [M, 7168] BF16 or NULL (NULL: residual_out = the rounded sum).
 *   gamma         [7168] BF16, the RMSNorm weight.
 *   out           [M, 7168] BF16: RMSNorm(residual_out) * gamma.
 *   residual_out  [M, 7168] BF16: the new residual. May be the same pointer as
 *                 residual (in-place update); no other overlap between outputs
 *                 and inputs, or between the two outputs, is allowed.
 *   All pointers 16-byte aligned. 1 <= TP <= 8; 1 <= M <= 64; eps > 0, finite.
 *
 *   residual_out is bit-exact: s = p[0]; s = s + p[r] (FP32, r = 1..TP-1);
 *   a = BF16(s); h = residual ? BF16(a + residual) : a.
 *   out = BF16((h * rstd) * gamma), rstd = rsqrt(sum(h^2) / 7168 + eps), FP32.
 *   Errors: SKINNY_ERR_NULL, _SHAPE, _ALIGN, _ALIAS, _ARG, _DEVICE, _LAUNCH.
 */
SKINNY_API int reduce_residual_rmsnorm(const void *partials, int TP, const void *residual,
                            const void *gamma, void *out, void *residual_out,
                            int M, float eps, void *stream);

/* reduce_residual_rmsnorm with per-call launch settings (as decode_gemm_bf16_ex;
 * only opts->pdl applies). */
SKINNY_API int reduce_residual_rmsnorm_ex(const void *partials, int TP, const void *residual,
                                          const void *gamma, void *out, void *residual_out,
                                          int M, float eps, const skinny_launch_opts *opts,
                                          void *stream);

/*
 * decode_gemm_bf16_reduce_rmsnorm -- a row-parallel drafter linear whose output
 *   rows are this rank's partial of the TP all-reduce, with that all-reduce's
 *   local stand-in and the RMSNorm that follows ("drafter/comm" module text: each
 *   layer's row-parallel linear ends in the TP all-reduce fused with the next
 *   RMSNorm; ArNorm for the arithmetic; "drafter/linears" DraftGemm for the
 *   GEMM). Computes what decode_gemm_bf16(x, W, partials[0], M, 7168, K)
 *   followed by reduce_residual_rmsnorm(partials, TP, residual, gamma, out,
 *   residual_out, M, eps) compute, bit for bit, with two kernels instead of
 *   three phases: the GEMM leaves every split-K partial in the library's scratch
 *   without finishing any tile, and the reduce kernel adds each column's
 *   partials in K order (the GEMM's own order), rounds once into slot 0 and goes
 *   on with the rank-order sum, residual and RMSNorm.
 *
 *   x             [M, K] BF16 row-major; W [7168, K] BF16 row-major.
 *   partials      [TP, M, 7168] BF16, contiguous. Slot 0 is written with the
 *                 GEMM's rows; slots 1..TP-1 (the other ranks' rows) are read.
 *   residual      [M, 7168] BF16 or NULL; gamma [7168] BF16.
 *   out           [M, 7168] BF16: RMSNorm(residual_out) * gamma.
 *   residual_out  [M, 7168] BF16: the new residual; may be the same pointer as
 *                 residual (in place), no other overlap between any output and
 *                 any input or between outputs.
 *   All pointers 16-byte aligned. 1 <= M <= 64; 1 <= TP <= 8; K >= 8 and
 *   K % 8 == 0; eps > 0, finite. Needs at least 56 SMs. Uses the decode GEMM's
 *   per-device scratch, like decode_gemm_bf16 (same rules on streams). Its
 *   reduce also raises the signal a following decode GEMM's l2_after_reduce
 *   waits for (see skinny_launch_opts), and its GEMM lowers it.
 *   Errors: SKINNY_ERR_NULL, _SHAPE, _ALIGN, _ALIAS, _ARG, _DEVICE, _CAPTURE,
 *   _ALLOC, _LAUNCH, _TIMEOUT (as decode_gemm_bf16).
 */
SKINNY_API int decode_gemm_bf16_reduce_rmsnorm(const void *x, const void *W, void *partials,
                                               int TP, const void *residual, const void *gamma,
                                               void *out, void *residual_out, int M, int K,
                                               float eps, void *stream);

/* decode_gemm_bf16_reduce_rmsnorm with per-call launch settings (as
 * decode_gemm_bf16_ex). */
SKINNY_API int decode_gemm_bf16_reduce_rmsnorm_ex(const void *x, const void *W, void *partials,
                                                  int TP, const void *residual,
                                                  const void *gamma, void *out,
                                                  void *residual_out, int M, int K, float eps,
                                                  const skinny_launch_opts *opts, void *stream);

/* Largest TP and row count of gather_shards_bf16. */
#define SKINNY_GATHER_MAX_TP 64
#define SKINNY_GATHER_MAX_M 65535

/*
 * gather_shards_bf16 -- every rank's shard into the gathered rows, locally
 *   ("drafter/comm": Gather places each rank's [M, S] shard side by side in rows
 *    of TP * S columns, rank r starting at column r * S; gather_context builds
 *    [M, 7168] from [M, 7168 / TP], gather_logits [M, V] from [M, V / TP]. Here
 *    the TP shards are local slots, as in the pages' one-GPU stand-in of
 *    "cutedsl/common/twoshot".)
 *
 *   shards  [TP, M, S] BF16, contiguous (slot r = rank r's [M, S] shard).
 *   out     [M, TP * S] BF16: out[m][r * S + j] = shards[r][m][j]; must not
 *           overlap shards.
 *   1 <= TP <= 64, 1 <= M <= 65535, S >= 8 and S % 8 == 0 (16-byte fragments,
 *   as the pages' Gather requires), both pointers 16-byte aligned.
 *   A byte move: the values are copied unchanged (the local slots have no
 *   sentinel, so the pages' (+0, -0) -> (+0, +0) cleaning does not apply).
 *   Errors: SKINNY_ERR_NULL, _SHAPE, _ALIGN, _ALIAS, _DEVICE, _LAUNCH.
 */
SKINNY_API int gather_shards_bf16(const void *shards, int TP, int M, int S, void *out,
                                  void *stream);

/* Human-readable text of a skinny_status code (static storage). */
SKINNY_API const char *skinny_status_string(int status);

/*
 * skinny_device_error -- read and clear the error word of `device`
 *   Synchronises the device, then returns SKINNY_OK if no kernel of this library
 *   recorded a problem since the last read, else SKINNY_ERR_TIMEOUT, and writes
 *   the raw word (a bit set per waiting role that gave up; 64 if only the
 *   host-mapped word was set; 128 if a reduce_residual_rmsnorm cluster's
 *   exchange of its sums of squares ran out) to *word if word is not NULL. Clearing also
 *   re-arms the decode GEMM's scratch flags, so the next call starts clean and
 *   calls stop returning SKINNY_ERR_TIMEOUT. Host pointer: word.
 */
SKINNY_API int skinny_device_error(int device, int *word);

/*
 * skinny_set_pdl -- programmatic dependent launch (PDL) for later launches.
 *   enable != 0: kernels are launched with programmatic stream serialisation, so
 *   a kernel may start while its predecessor on the stream finishes. Each kernel
 *   then reads only data that belongs to the model -- the weight W of
 *   decode_gemm_bf16, gamma of reduce_residual_rmsnorm -- before waiting for its
 *   predecessor, and everything else after ("drafter/comm", ArNorm.kernel: gamma
 *   is loaded before the launch_dependents / wait pair, the rows after it). So
 *   with PDL on, W and gamma must not be written by any kernel that may still be
 *   running on the stream when the call is made (every kernel of this library
 *   lets its successor start early, so more than one predecessor can still be in
 *   flight): write weights before the chain of calls. Off by default. Returns
 *   the previous setting.
 */
SKINNY_API int skinny_set_pdl(int enable);

/*
 * skinny_set_l2_prefetch -- L2 lead of decode_gemm_bf16's deep ring, for later
 *   launches of every decode GEMM entry point. With PDL on, each CTA streams its
 *   first ring of weight tiles and prefetches `blocks` more 16 KB weight blocks
 *   into L2 before it waits for its predecessor (rings of 9 to 11 stages, used
 *   when M > 32 or a CTA streams at least 1 MiB, 1.5 MiB for M <= 16; the
 *   shallow ring keeps its own lead). A performance hint only: results are the same bits
 *   for every value. Measured
 *   on GB300: the default 6 suits a GEMM that follows another GEMM; 0 suits the
 *   layer chain, where each GEMM follows a short kernel (the reduce) or is
 *   followed by one, and early requests only slow the previous GEMM's last
 *   CTAs. blocks in [0, 64]. Returns the previous value, or -1 (setting
 *   unchanged) if blocks is out of range.
 */
SKINNY_API int skinny_set_l2_prefetch(int blocks);

/* ---- host-side planning (no GPU needed) ------------------------------------ */

/* How decode_gemm_bf16 splits a problem over `num_sms` CTAs: one whole 128-row
 * tile per CTA when the tiles fill at least 90 % of the SMs (no split-K), else
 * stream-K: the ceil(N/128) x ceil(K/64) weight blocks, in tile-major order, are
 * cut into `ctas` contiguous, equal-as-possible ranges. The ring depth follows
 * the weight bytes per CTA under the current PDL setting: the shallow ring (two
 * CTAs per SM) below 1 MiB (1.5 MiB for M <= 16) with PDL on and M <= 32, the
 * deep ring otherwise. */
typedef struct {
    int tiles;          /* ceil(N / 128): 128-row weight tiles */
    int kblocks;        /* ceil(K / 64): 64-wide K blocks per tile */
    long long blocks;   /* tiles * kblocks */
    int ctas;           /* CTAs launched: tiles, or min(num_sms, blocks) */
    int mma_n;          /* padded row count the MMA runs with: 16, 32 or 64 */
    int stages;         /* shared-memory pipeline stages per CTA */
    int smem_bytes;     /* dynamic shared memory per CTA */
    int split_tiles;    /* tiles whose K range spans more than one CTA */
} skinny_gemm_plan;

/* Fill *plan for (M, N, K) on a device with num_sms SMs. Host pointer: plan.
 * Returns SKINNY_ERR_SHAPE for shapes decode_gemm_bf16 rejects. */
SKINNY_API int skinny_gemm_plan_query(int M, int N, int K, int num_sms, skinny_gemm_plan *plan);

/* The pieces CTA `cta` of that plan computes: for each of at most max_pieces
 * pieces, the tile, its K-block range [kb0, kb1), and the scratch slot its
 * partial sum goes to (-1 for a tile the CTA covers whole). Host pointers.
 * Returns the number of pieces, or -1 on bad arguments. */
SKINNY_API int skinny_gemm_cta_pieces(int M, int N, int K, int num_sms, int cta, int *tile,
                           int *kb0, int *kb1, int *slot, int max_pieces);

/* ---- diagnostics ---------------------------------------------------------- */

/*
 * skinny_watchdog_selftest -- exercise the decode GEMM's bounded-wait path.
 *   Launches decode_gemm_bf16's kernel on (x, W, out, M, N, K) with its MMA
 *   role first waiting on a barrier that nothing ever completes, limited to
 *   timeout_ns nanoseconds (1e3 <= timeout_ns <= 2e9). The kernel records
 *   the timeout in the device error word, drains the copies it has in flight,
 *   frees its tensor memory and exits; out is left unspecified. Read the outcome
 *   with skinny_device_error(). For tests of the failure path only.
 */
SKINNY_API int skinny_watchdog_selftest(const void *x, const void *W, void *out, int M, int N,
                             int K, long long timeout_ns, void *stream);

/*
 * skinny_reduce_selftest -- exercise reduce_residual_rmsnorm's bounded wait.
 *   Checks its arguments as reduce_residual_rmsnorm does, then launches the
 *   reduce with one 8-CTA cluster per row in which the last CTA keeps its
 *   share of the row's sum of squares to itself: every CTA's wait for the
 *   cluster's sums runs out after timeout_ns nanoseconds (1e3 <= timeout_ns <=
 *   2e9), is recorded, and ends; out and residual_out are left unspecified.
 *   skinny_device_error() then reports bit 128 and clears it. No state outlives
 *   the call: the next reduce runs normally. For tests of the failure path
 *   only.
 */
SKINNY_API int skinny_reduce_selftest(const void *partials, int TP, const void *residual,
                                      const void *gamma, void *out, void *residual_out, int M,
                                      float eps, long long timeout_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SKINNY_H */
