// Launch interface between the C ABI (api.cu) and the kernel translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace skinny {

// Bits of the device error word (one per waiting role that gave up).
enum ErrorBits : int {
    kErrProducerWait = 1,   // TMA producer: a pipeline slot never came free
    kErrMmaFullWait = 2,    // MMA issuer: a stage's copies never landed
    kErrMmaAccWait = 4,     // MMA issuer: the epilogue never released an accumulator
    kErrEpilogueWait = 8,   // epilogue: an accumulator never completed
    kErrDrain = 16,         // teardown: in-flight copies or MMAs did not finish
    kErrSelftest = 32,      // the watchdog self-test's deliberate wait ran out
    kErrUnknown = 64,       // the host-mapped word was set but the device word was not
    kErrReduceExchange = 128,  // reduce: a cluster exchange wait ran out
};

struct GemmArgs {
    int M, N, K;
    uint16_t *out;          // [M, N] BF16 patterns
    float *partials;        // [2 * ctas][slot rows][128] FP32 split-K partial tiles
    int slot_floats;        // floats from one partial tile to the next
    unsigned *flags;        // [2 * ctas] "partial published" flags, zero between calls
    int *err;               // device error word
    int *host_err;          // host-mapped word set to 1 on any error, or nullptr
    unsigned long long wait_limit_ns;
    int selftest;           // 1: the MMA role waits on a barrier nothing completes
    // lm_head epilogue (logits = 1): v = soft_cap > 0 ? soft_cap * tanh(v / soft_cap)
    // : v; v *= scale; applied to the FP32 sum before the one BF16 rounding.
    int logits;
    float soft_cap, scale;
    // 1: every piece, whole tiles included, leaves its FP32 partial in its scratch
    // slot and nothing is finished here (no flags): the reduce kernel that follows
    // adds them (decode_gemm_bf16_reduce_rmsnorm).
    int publish_only;
    // Deep ring only: weight blocks each CTA prefetches into L2, beyond its ring's
    // first fill, before waiting on the previous kernel (skinny_set_l2_prefetch).
    int l2_lead;
    // The "GEMM before the reduce is complete" word of decode_gemm_bf16_reduce_rmsnorm
    // (set by its reduce, cleared by its GEMM), or nullptr. With l2_after_reduce > 0
    // the producer waits (bounded) for it to be set and then prefetches that many
    // more weight blocks into L2 before waiting on the previous kernel.
    unsigned *gemm_done;
    int l2_after_reduce;
    int clear_gemm_done;  // 1: clear the word once the previous kernel is complete
};

// Default and largest l2_lead. Measured on GB300: 6 suits back-to-back GEMMs
// (each CTA's early blocks arrive while the previous kernel's last CTAs finish);
// 0 suits a GEMM behind a short latency-bound kernel, such as the layer chain's
// reduce, where those requests only slow the previous GEMM's last CTAs.
constexpr int kL2LeadDefault = 6;
constexpr int kL2LeadMax = 64;

// Where the reduce kernel finds a publish-only GEMM's partials of the 7168
// slot-0 columns: the GEMM's geometry (tiles, K blocks, CTAs) and scratch.
struct SplitKPartials {
    const float *partials;  // [2 * ctas][slot_floats]
    int slot_floats;
    int M, N, K, ctas;
    unsigned *gemm_done;    // set to 1 once the GEMM is complete (or nullptr)
};

// Pipeline depth and shared memory of the decode GEMM for a padded row count,
// with the shallow or the deep ring (plan.cuh use_shallow_ring).
int gemm_stages(int mma_n, bool shallow);
int gemm_smem_bytes(int mma_n, bool shallow);

// Launch the decode GEMM: grid = ctas CTAs of 192 threads; pdl sets the
// programmatic-dependent-launch attribute, shallow picks the ring.
cudaError_t launch_decode_gemm(const CUtensorMap &w_map, const CUtensorMap &x_map,
                               const GemmArgs &args, int mma_n, int ctas, cudaStream_t stream,
                               bool pdl, bool shallow, int device);

// Split-K scratch held in a static device array (decode_gemm_bf16_noalloc).
constexpr int kStaticScratchCtas = 160;   // CTAs the array holds partial tiles for
constexpr int kStaticSlotRows = 32;       // rows of x a static partial tile holds

struct StaticScratch {
    float *partials;      // [2 * max_ctas][kStaticSlotRows][128] FP32
    unsigned *flags;      // [2 * max_ctas], contiguous with err
    int *err;             // error word, right after the flag space
    size_t zero_bytes;    // bytes from `flags` through `err` that must start at zero
    int max_ctas;
};

// Device addresses of the static scratch on the current device; the first call
// per device looks them up (cudaGetSymbolAddress).
cudaError_t static_scratch_for_current_device(StaticScratch *out);

// Launch reduce + residual + RMSNorm over rows of 7168: M clusters of
// ctas_per_row CTAs.
cudaError_t launch_reduce_rmsnorm(const void *partials, int TP, const void *residual,
                                  const void *gamma, void *out, void *residual_out, int M,
                                  float eps, int ctas_per_row, cudaStream_t stream, bool pdl);

// Finish a publish-only decode GEMM: out[M, N] = the partials added in K order,
// rounded once to BF16.
cudaError_t launch_splitk_finish(const SplitKPartials &fix, uint16_t *out, cudaStream_t stream,
                                 bool pdl);

// The same with slot 0 made from a publish-only GEMM's FP32 partials (added in
// K order, rounded once, and written to slot 0 of `partials`).
cudaError_t launch_reduce_rmsnorm_splitk(void *partials, int TP, const void *residual,
                                         const void *gamma, void *out, void *residual_out, int M,
                                         float eps, int ctas_per_row, const SplitKPartials &fix,
                                         cudaStream_t stream, bool pdl);

// The plain reduce with 8-CTA clusters whose last CTA keeps its sum of squares
// to itself, every exchange wait limited to limit_ns: the failure-path
// self-test (the waits run out, are recorded in the reduce's error word and
// end; the outputs are unspecified).
cudaError_t launch_reduce_rmsnorm_selftest(const void *partials, int TP, const void *residual,
                                           const void *gamma, void *out, void *residual_out,
                                           int M, float eps, unsigned long long limit_ns,
                                           cudaStream_t stream);

// The reduce kernel's own error word on the current device (nonzero: a
// cluster exchange wait ran out), cleared after reading if `clear`.
cudaError_t reduce_error_word(int *value, bool clear);

// Gather TP shards [TP, M, S] into rows [M, TP * S] (S a multiple of 8).
cudaError_t launch_gather(const void *shards, int TP, int M, int S, void *out,
                          cudaStream_t stream, bool pdl);

}  // namespace skinny
