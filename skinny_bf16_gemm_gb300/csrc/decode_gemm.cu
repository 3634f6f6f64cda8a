// Decode GEMM for GB300 (sm_103a): out[M, N] = x[M, K] @ W[N, K]^T, BF16 operands,
// FP32 accumulation, one BF16 rounding ("drafter/linears": module text and
// DraftGemm). M <= 64, so the time is the weight stream: every byte of W is read
// once from HBM by TMA and fed to the tensor cores while it is on chip.
//
// Persistent CTAs of 192 threads in three roles:
//   warp 0      TMA producer: W tiles [128 rows x 64 K] and x slices [MP x 64 K]
//               into a ring of STAGES shared-memory stages (128-byte swizzle);
//   warp 1      MMA issuer: tcgen05.mma kind::f16, M = 128 weight rows, N = MP
//               (x rows padded to 16, 32 or 64; the padding rows are TMA zero
//               fill), accumulating in tensor memory (two accumulator buffers);
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (TMEM lane = weight row =
//               output column n, column = output row m), one BF16 rounding and
//               the store (for whole tiles of 32/64 padded rows through the
//               idle ring, as 16-byte row pieces), or the split-K fix-up.
// Work split (plan.cuh): one whole 128-row tile per CTA when the tiles nearly fill
// the GPU, otherwise the ceil(N/128) x ceil(K/64) weight blocks dealt to one CTA
// per SM as equal contiguous ranges (stream-K). A tile whose K range is shared
// by several CTAs is finished by the CTA holding its first K blocks (for which it
// is the last piece): the others publish their FP32 partials behind a release
// flag, and the finisher adds them in K order, so the bits do not depend on
// timing. Ranges go to CTAs in reverse block order, so a finisher waits only on
// CTAs with lower block indices, which the GPU dispatched before it.
// Ring depth (plan.cuh use_shallow_ring): the deep ring, one CTA per SM, for
// long streams; the shallow ring for short ones under programmatic dependent
// launch, so that the next kernel's CTA shares the SM. Before waiting on the
// previous kernel in the stream the producer already streams the first STAGES
// weight tiles and prefetches more into L2 -- behind decode_gemm_bf16_reduce_rmsnorm
// optionally more again once that call's reduce has seen its GEMM complete:
// weights never depend on the previous kernel, x may.
// Every wait is bounded (wait_limit_ns); a role that gives up records a bit in
// the device error word, the CTA drains its in-flight copies and MMAs, frees its
// tensor memory and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace skinny {
namespace {

constexpr int kThreads = 192;
constexpr int kEpilogueThreads = 128;
constexpr int kWBytes = kBlockN * kBlockK * 2;
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s for copies already issued
// Weight blocks prefetched to L2, beyond the ring's first fill, before waiting
// on the previous kernel: 8 with the shallow ring, the caller's GemmArgs::l2_lead
// with the deep ring. Both short: the early requests share the SM and HBM with
// the previous kernel's last CTAs and slow them. Measured on GB300 for the
// shallow ring (its co-resident CTA is the previous kernel's): leads of 8-10
// beat 26 (most of a short range) by up to 1.4 us at N = 4096 and 3.5 us at
// N = 6144-7168 (K = 7168, 0.4-0.7 MB per CTA); 0-4 are slower again.
constexpr int kL2PrefetchShallow = 8;
// The longest a producer waits for the previous GEMM's completion signal before
// it goes on without the prefetch that depends on it (GemmArgs::l2_after_reduce).
constexpr uint64_t kAfterReduceWaitNs = 50000ull;
constexpr int kMaxShallowStages = 6;  // shallow rings have 5..6 stages, deep ones 9..11

// MP: padded row count (MMA N). STAGES: shared-memory ring depth. The deep ring
// (185-227 KB) keeps the most bytes in flight; the shallow one (~100-112 KB) lets
// the next kernel's CTAs be resident on the same SM while this one finishes, so
// with programmatic dependent launch they stream weights across the boundary
// (plan.cuh use_shallow_ring picks one by the weight bytes per CTA).
template <int MP, int STAGES>
struct Layout {
    static constexpr int kStages = STAGES;
    static constexpr int kAccCols = MP == 64 ? 64 : 32;  // TMEM columns per accumulator
    static constexpr int kTmemCols = 2 * kAccCols;       // two accumulator buffers
    static constexpr int kXBytes = MP * kBlockK * 2;
    static constexpr int kStageBytes = kWBytes + kXBytes;
    static constexpr int kBarOffset = kStages * kStageBytes;
    static constexpr int kNumBars = 2 * kStages + 7;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
    static constexpr int kBytes = kMiscOffset + 16;
    static constexpr int kDynamicBytes = kBytes + 1024;  // slack to align the base to 1024
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
};

enum WaitResult { kWaitDone = 1, kWaitTimeout = 0, kWaitAborted = -1 };

// Wait for completion of the barrier phase with `parity`, giving up after
// limit_ns or as soon as another role of this CTA has aborted.
__device__ __forceinline__ int bounded_wait(uint32_t bar, uint32_t parity,
                                            const volatile uint32_t *abort_flag,
                                            uint64_t limit_ns) {
    if (ptx::mbar_try_wait(bar, parity)) return kWaitDone;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (ptx::mbar_try_wait(bar, parity)) return kWaitDone;
        if ((spin & 15u) == 0) {
            if (*abort_flag) return kWaitAborted;
            if (ptx::global_timer_ns() - t0 > limit_ns) return kWaitTimeout;
        }
    }
}

// Record a problem: the bit in the device error word, and a nonzero word in the
// caller's host-mapped memory when there is one (the host reads it without
// synchronising, so the library's next call can report it).
__device__ __forceinline__ void record_error(const GemmArgs &a, int bit) {
    atomicOr(a.err, bit);
    if (a.host_err != nullptr) {
        *reinterpret_cast<volatile int *>(a.host_err) = 1;
        __threadfence_system();
    }
}

__device__ __forceinline__ void raise_error(const GemmArgs &a, volatile uint32_t *abort_flag,
                                            int bit) {
    record_error(a, bit);
    *abort_flag = 1u;
}

// Barrier-wide OR of a predicate over the epilogue's 128 threads (named barrier 1).
__device__ __forceinline__ bool epilogue_any(bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred a, b;\n\t"
        "setp.ne.u32 a, %1, 0;\n\t"
        "bar.red.or.pred b, 1, 128, a;\n\t"
        "selp.u32 %0, 1, 0, b;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(p))
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint16_t to_bf16_bits(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// The value an output element is rounded from: the FP32 sum itself, or for the
// lm_head logits ("drafter/linears", draft_logits) the soft-capped, scaled sum.
__device__ __forceinline__ float output_value(float v, const GemmArgs &a) {
    if (!a.logits) return v;
    if (a.soft_cap > 0.0f) v = __fmul_rn(tanhf(__fdiv_rn(v, a.soft_cap)), a.soft_cap);
    return __fmul_rn(v, a.scale);
}

// Store rows 0..M-1 of one tile's output (this thread's column n = tile * 128 +
// row; v[m] the values to round) through the idle ring: each thread puts its
// BF16 values in shared memory, then the 128 epilogue threads write 16-byte
// pieces of whole rows instead of one 2-byte store per row and thread. Needs
// 16-byte aligned rows (N a multiple of 8) and a ring nothing uses any more.
// Measured on GB300 for whole tiles of 32 and 64 padded rows with the deep
// ring: 0.3-0.6 us faster per call at N = 18432; no gain for 16 rows or on
// split tiles, and 0.2 us slower with the shallow ring, so only there.
template <int MP>
__device__ __forceinline__ void store_tile_staged(const float (&v)[MP], uint16_t *out, int M, int N,
                                                  int tile, int row, int etid, uint32_t stage) {
#pragma unroll
    for (int m = 0; m < MP; ++m)
        if (m < M)
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(stage + (m * kBlockN + row) * 2),
                         "h"(to_bf16_bits(v[m])) : "memory");
    ptx::named_barrier_sync(1, kEpilogueThreads);
    const int pieces = M * (kBlockN / 8);
    for (int i = etid; i < pieces; i += kEpilogueThreads) {
        const int m = i / (kBlockN / 8), c = i % (kBlockN / 8);
        const int n0 = tile * kBlockN + c * 8;
        if (n0 < N) {
            uint4 w;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                         : "r"(stage + (m * kBlockN + c * 8) * 2) : "memory");
            *reinterpret_cast<uint4 *>(out + static_cast<size_t>(m) * N + n0) = w;
        }
    }
}

template <int MP, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap w_map,
                       const __grid_constant__ CUtensorMap x_map, const GemmArgs args) {
    using L = Layout<MP, STAGES>;
    constexpr int S = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t bar_full = sbase + L::kBarOffset;   // + 8 s
    const uint32_t bar_empty = bar_full + 8 * S;       // + 8 s
    const uint32_t bar_acc_full = bar_empty + 8 * S;   // + 8 b
    const uint32_t bar_acc_empty = bar_acc_full + 16;  // + 8 b
    const uint32_t bar_drain = bar_acc_empty + 16;
    const uint32_t bar_never = bar_drain + 8;
    const uint32_t bar_fix = bar_never + 8;             // split-K fix-up bulk copies
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + L::kMiscOffset);
    // misc[0]: tensor-memory base, misc[1]: abort flag

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const GemmGeometry g = make_geometry(args.M, args.N, args.K, gridDim.x);
    // This CTA's range of weight blocks (plan.cuh: reverse block order, so the
    // split-K finisher below waits only on CTAs with lower block indices).
    const int cta = range_of_block(g, static_cast<int>(blockIdx.x));
    const uint64_t limit = args.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);
            ptx::mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_acc_full + 8 * b, 1);
            ptx::mbar_init(bar_acc_empty + 8 * b, kEpilogueThreads);
        }
        ptx::mbar_init(bar_drain, 1);
        ptx::mbar_init(bar_never, 1);
        ptx::mbar_init(bar_fix, 1);
        misc[1] = 0u;
        ptx::fence_barrier_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(sbase + L::kMiscOffset, L::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = misc[0];
    volatile uint32_t *abort_flag = misc + 1;

    // The next kernel in the stream may launch now: its CTAs take SMs as they
    // free up (beside this one with the shallow ring), set up and stream their
    // first weights while this grid runs, and wait for it before touching
    // anything it writes.
    ptx::pdl_launch_dependents();

    // This CTA's blocks [b0, b1). Block indices stay below 2^31 (the host rejects
    // larger problems), so after the two 64-bit divisions of the range ends all
    // the plan arithmetic here is 32-bit.
    const long long b0 = cta_begin(g, cta);
    const long long b1 = cta_begin(g, cta + 1);
    const int total = static_cast<int>(b1 - b0);
    const BlockCursor start = {static_cast<int>(b0) / g.kblocks,
                               static_cast<int>(b0) - (static_cast<int>(b0) / g.kblocks) * g.kblocks};
    const int pieces = total > 0 ? (static_cast<int>(b1) - 1) / g.kblocks - start.t + 1 : 0;
    // Piece q of this CTA's range (plan.cuh cta_piece, from the range ends above).
    auto piece_of = [&](int q) {
        Piece p;
        p.tile = start.t + q;
        const int t0 = p.tile * g.kblocks;
        p.kb0 = static_cast<int>(b0) > t0 ? static_cast<int>(b0) - t0 : 0;
        p.kb1 = (static_cast<int>(b1) < t0 + g.kblocks ? static_cast<int>(b1) : t0 + g.kblocks) - t0;
        return p;
    };

    // Producer bookkeeping kept for the drain (lane 0 of warp 0).
    uint32_t armed = 0, armed_parity = 0;
    // MMA bookkeeping for the drain (lane 0 of warp 1).
    bool mma_issued = false;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            ptx::prefetch_tensormap(&w_map);
            ptx::prefetch_tensormap(&x_map);
            const uint64_t pol_w = ptx::policy_evict_first();
            const uint64_t pol_x = ptx::policy_evict_last();
            const int npre = total < S ? total : S;
            // Fresh stages: arm them and stream weights before the predecessor ends.
            BlockCursor w = start;
            for (int j = 0; j < npre; ++j) {
                const uint32_t st = sbase + j * L::kStageBytes;
                ptx::mbar_arrive_expect_tx(bar_full + 8 * j, L::kStageBytes);
                armed |= 1u << j;
                ptx::tma_load_2d(st, &w_map, bar_full + 8 * j, w.kb * kBlockK, w.t * kBlockN, pol_w);
                w.next(g.kblocks);
            }
            // The blocks after the ring's worth go to L2 ahead of time.
            const int lead = STAGES <= kMaxShallowStages ? kL2PrefetchShallow : args.l2_lead;
            const int npf = total - npre < lead ? total - npre : lead;
            BlockCursor pf = w;
            for (int j = 0; j < npf; ++j) {
                ptx::tma_prefetch_l2_2d(&w_map, pf.kb * kBlockK, pf.t * kBlockN);
                pf.next(g.kblocks);
            }
            if (args.l2_after_reduce > 0) {
                // Behind a reduce whose GEMM is complete, HBM would idle until this
                // kernel's wait returns: prefetch more now. Not earlier, where the
                // requests would slow that GEMM's last CTAs.
                const uint64_t t0 = ptx::global_timer_ns();
                bool go = ptx::ld_acquire_gpu(args.gemm_done) != 0u;
                while (!go && ptx::global_timer_ns() - t0 < kAfterReduceWaitNs) {
                    __nanosleep(128);
                    go = ptx::ld_acquire_gpu(args.gemm_done) != 0u;
                }
                if (go) {
                    const int rest = total - npre - npf;
                    const int more = rest < args.l2_after_reduce ? rest : args.l2_after_reduce;
                    for (int j = 0; j < more; ++j) {
                        ptx::tma_prefetch_l2_2d(&w_map, pf.kb * kBlockK, pf.t * kBlockN);
                        pf.next(g.kblocks);
                    }
                }
            }
            ptx::pdl_wait();  // x may be the predecessor's output
            BlockCursor xc = start;
            for (int j = 0; j < npre; ++j) {
                const uint32_t st = sbase + j * L::kStageBytes;
                ptx::tma_load_2d(st + kWBytes, &x_map, bar_full + 8 * j, xc.kb * kBlockK, 0, pol_x);
                xc.next(g.kblocks);
            }
            int s = npre % S;
            uint32_t ph = npre == S ? 1u : 0u;
            for (int j = npre; j < total; ++j) {
                const int r = bounded_wait(bar_empty + 8 * s, ph ^ 1u, abort_flag, limit);
                if (r != kWaitDone) {
                    if (r == kWaitTimeout) raise_error(args, abort_flag, kErrProducerWait);
                    break;
                }
                const uint32_t st = sbase + s * L::kStageBytes;
                ptx::mbar_arrive_expect_tx(bar_full + 8 * s, L::kStageBytes);
                armed |= 1u << s;
                armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
                ptx::tma_load_2d(st, &w_map, bar_full + 8 * s, w.kb * kBlockK, w.t * kBlockN, pol_w);
                ptx::tma_load_2d(st + kWBytes, &x_map, bar_full + 8 * s, w.kb * kBlockK, 0, pol_x);
                w.next(g.kblocks);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBlockN, MP);
            ptx::pdl_wait();  // start the bounded waits' clocks after the predecessor
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            if (args.selftest) {
                // Wait on a barrier nothing ever completes: exercises the bounded wait.
                const int r = bounded_wait(bar_never, 0, abort_flag, limit);
                if (r == kWaitTimeout) raise_error(args, abort_flag, kErrSelftest);
                ok = false;
            }
            for (int q = 0; ok && q < pieces; ++q) {
                const Piece p = piece_of(q);
                const int b = q & 1;
                const uint32_t aph = (q >> 1) & 1;
                int r = bounded_wait(bar_acc_empty + 8 * b, aph ^ 1u, abort_flag, limit);
                if (r != kWaitDone) {
                    if (r == kWaitTimeout) raise_error(args, abort_flag, kErrMmaAccWait);
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * L::kAccCols;
                for (int kb = p.kb0; kb < p.kb1; ++kb) {
                    r = bounded_wait(bar_full + 8 * s, ph, abort_flag, limit);
                    if (r != kWaitDone) {
                        if (r == kWaitTimeout) raise_error(args, abort_flag, kErrMmaFullWait);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t st = sbase + s * L::kStageBytes;
                    const uint64_t a_desc = ptx::smem_desc_sw128_kmajor(st);
                    const uint64_t b_desc = ptx::smem_desc_sw128_kmajor(st + kWBytes);
#pragma unroll
                    for (int k = 0; k < kBlockK / 16; ++k) {
                        // +32 bytes along K per step: +2 in the address field (>> 4).
                        ptx::mma_bf16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc,
                                      (kb > p.kb0 || k > 0) ? 1u : 0u);
                    }
                    mma_issued = true;
                    ptx::mma_commit(bar_empty + 8 * s);  // stage free once these MMAs finish
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(bar_acc_full + 8 * b);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (128 threads) ----------------
        ptx::pdl_wait();  // scratch and out may still be in use by the predecessor
        if (args.clear_gemm_done && blockIdx.x == 0 && threadIdx.x == 64) atomicExch(args.gemm_done, 0u);
        const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
        const int row = quarter * 32 + lane;       // weight row within the tile
        const int etid = threadIdx.x - 64;
        const int slot_bytes = g.M * kBlockN * static_cast<int>(sizeof(float));
        const int ring_slots = L::kRingBytes / slot_bytes;
        const float *staging = reinterpret_cast<const float *>(smem);
        uint32_t fix_phase = 0;
        bool fix_pending = false;
        // Whole tiles of 32 or 64 padded rows, deep ring, 16-byte aligned output
        // rows: the last piece's tile goes out through the ring.
        constexpr bool kStagedOut = MP >= 32 && STAGES > kMaxShallowStages;
        const bool staged = kStagedOut && (reinterpret_cast<uintptr_t>(args.out) & 15) == 0 &&
                            (g.N & 7) == 0;

        // Finish split tile t. This CTA holds the tile's first K blocks, so the
        // tile is its last piece: its own partial is in registers and the ring
        // is free. Wait until the other contributors have published their
        // partials, pull them into the ring with bulk copies (all in flight at
        // once), add in K (= CTA) order and round once. false = aborted.
        auto finish_tile = [&](int t, int first, int last, const float *own,
                               int first_peer_slot) -> bool {
            float sum[MP];
#pragma unroll
            for (int m = 0; m < MP; ++m) sum[m] = own[m];
            for (int c0 = first + 1; c0 <= last;) {
                const int c1 = last + 1 < c0 + ring_slots ? last + 1 : c0 + ring_slots;
                const int n_in = c1 - c0;
                // The barrier expects every copy of this chunk; one thread per
                // contributor waits for its flag and starts its copy at once, so
                // early partials are on their way while late ones are published.
                if (etid == 0)
                    ptx::mbar_arrive_expect_tx(bar_fix, static_cast<uint32_t>(n_in * slot_bytes));
                fix_pending = true;
                int r = kWaitDone;
                int slot = 0;
                if (etid < n_in) {
                    const int c = c0 + etid;
                    slot = c0 == first + 1 ? first_peer_slot : partial_slot(g, c, t);
                    const unsigned *flag = args.flags + slot;
                    // Acquire loads: the partial behind the flag is visible once it is 1.
                    if (ptx::ld_acquire_gpu(flag) == 0u) {
                        const uint64_t t0 = ptx::global_timer_ns();
                        for (uint32_t spin = 1; ptx::ld_acquire_gpu(flag) == 0u; ++spin) {
                            if ((spin & 15u) == 0) {
                                if (*abort_flag) { r = kWaitAborted; break; }
                                if (ptx::global_timer_ns() - t0 > limit) { r = kWaitTimeout; break; }
                            }
                        }
                    }
                    if (r == kWaitDone) {
                        ptx::fence_proxy_async_global();  // the bulk copy reads what was acquired
                        ptx::bulk_load(sbase + etid * slot_bytes,
                                       args.partials + static_cast<size_t>(slot) * args.slot_floats,
                                       slot_bytes, bar_fix);
                    }
                }
                if (r == kWaitTimeout) raise_error(args, abort_flag, kErrEpilogueWait);
                if (epilogue_any(r != kWaitDone)) return false;
                r = bounded_wait(bar_fix, fix_phase, abort_flag, limit);
                if (r == kWaitTimeout) raise_error(args, abort_flag, kErrEpilogueWait);
                if (epilogue_any(r != kWaitDone)) return false;
                fix_pending = false;
                fix_phase ^= 1u;
                for (int c = c0; c < c1; ++c) {
                    const float *src = staging + static_cast<size_t>(c - c0) * g.M * kBlockN + row;
#pragma unroll
                    for (int m = 0; m < MP; ++m)
                        if (m < g.M) sum[m] = __fadd_rn(sum[m], src[m * kBlockN]);
                }
                // The partials are consumed: re-arm their flags for the next call.
                if (etid < n_in) args.flags[slot] = 0u;
                ptx::named_barrier_sync(1, kEpilogueThreads);  // the ring is refilled next
                c0 = c1;
            }
            const int n = t * kBlockN + row;
            if (n < g.N) {
#pragma unroll
                for (int m = 0; m < MP; ++m)
                    if (m < g.M)
                        args.out[static_cast<size_t>(m) * g.N + n] = to_bf16_bits(output_value(sum[m], args));
            }
            return true;
        };

        for (int q = 0; q < pieces; ++q) {
            const Piece p = piece_of(q);
            // The plan's arithmetic (64-bit divisions) before the wait, not on
            // the split-K tail after it.
            int first, last;
            tile_contributors(g, p.tile, first, last);
            const int my_slot = 2 * cta + (p.tile == start.t ? 0 : 1);  // plan.cuh partial_slot
            const int first_peer_slot =
                first + 1 + etid <= last ? partial_slot(g, first + 1 + etid, p.tile) : 0;
            const int b = q & 1;
            const uint32_t aph = (q >> 1) & 1;
            const int r = bounded_wait(bar_acc_full + 8 * b, aph, abort_flag, limit);
            if (r == kWaitTimeout) raise_error(args, abort_flag, kErrEpilogueWait);
            if (epilogue_any(r != kWaitDone)) break;
            ptx::tc_fence_after_sync();
            float acc[MP];
            {
                const uint32_t taddr =
                    tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * L::kAccCols;
#pragma unroll
                for (int c = 0; c < MP; c += 16) {
                    uint32_t v[16];
                    ptx::tmem_ld16(taddr + c, v);
                    ptx::tmem_ld_wait(v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[c + i] = __uint_as_float(v[i]);
                }
            }
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar_acc_empty + 8 * b);  // the MMA may reuse this buffer

            const int n = p.tile * kBlockN + row;
            if (p.kb0 == 0 && p.kb1 == g.kblocks && !args.publish_only) {
                // Whole tile in this CTA: round once and store.
                if (kStagedOut && staged && q == pieces - 1) {
#pragma unroll
                    for (int m = 0; m < MP; ++m) acc[m] = output_value(acc[m], args);
                    store_tile_staged<MP>(acc, args.out, g.M, g.N, p.tile, row, etid, sbase);
                    continue;
                }
                if (n < g.N) {
#pragma unroll
                    for (int m = 0; m < MP; ++m)
                        if (m < g.M)
                            args.out[static_cast<size_t>(m) * g.N + n] =
                                to_bf16_bits(output_value(acc[m], args));
                }
                continue;
            }
            if (first == cta && !args.publish_only) {
                // The tile starts in this CTA's range: this CTA finishes it.
                if (!finish_tile(p.tile, first, last, acc, first_peer_slot)) break;
                continue;
            }
            // Publish this CTA's partial: the values, then a release flag. The
            // finishing CTA reads them with bulk copies (the async proxy).
            float *mine = args.partials + static_cast<size_t>(my_slot) * args.slot_floats;
#pragma unroll
            for (int m = 0; m < MP; ++m)
                if (m < g.M) __stcg(mine + m * kBlockN + row, acc[m]);
            if (args.publish_only) continue;  // read by the next kernel, after this grid
            ptx::fence_proxy_async_global();
            ptx::named_barrier_sync(1, kEpilogueThreads);
            // One release store after the barrier covers every thread's stores of
            // the partial (the barrier orders them before it).
            if (etid == 0) {
                ptx::st_release_gpu(args.flags + my_slot, 1u);
            }
        }
        if (fix_pending) {
            // Copies still in flight must land before the CTA's memory is released.
            const uint64_t t0 = ptx::global_timer_ns();
            while (!ptx::mbar_try_wait(bar_fix, fix_phase)) {
                if (ptx::global_timer_ns() - t0 > kDrainLimitNs) {
                    record_error(args, kErrDrain);
                    break;
                }
            }
        }
    }

    // ---------------- teardown ----------------
    __syncthreads();
    if (*abort_flag) {
        // Nothing may still write this CTA's shared or tensor memory when it exits.
        if (warp == 0 && lane == 0) {
            for (int s = 0; s < S; ++s) {
                if (!(armed & (1u << s))) continue;
                const uint32_t par = (armed_parity >> s) & 1u;
                const uint64_t t0 = ptx::global_timer_ns();
                while (!ptx::mbar_try_wait(bar_full + 8 * s, par)) {
                    if (ptx::global_timer_ns() - t0 > kDrainLimitNs) {
                        record_error(args, kErrDrain);
                        break;
                    }
                }
            }
        }
        if (warp == 1 && lane == 0 && mma_issued) {
            ptx::mma_commit(bar_drain);
            const uint64_t t0 = ptx::global_timer_ns();
            while (!ptx::mbar_try_wait(bar_drain, 0)) {
                if (ptx::global_timer_ns() - t0 > kDrainLimitNs) {
                    record_error(args, kErrDrain);
                    break;
                }
            }
        }
        __syncthreads();
    }
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

template <int MP, int STAGES>
cudaError_t launch_variant(const CUtensorMap &w_map, const CUtensorMap &x_map,
                           const GemmArgs &args, int ctas, cudaStream_t stream, bool pdl,
                           int device) {
    using L = Layout<MP, STAGES>;
    static bool configured[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (!configured[device]) {
        cudaError_t e = cudaFuncSetAttribute(decode_gemm_kernel<MP, STAGES>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             L::kDynamicBytes);
        if (e != cudaSuccess) return e;
        configured[device] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kDynamicBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_gemm_kernel<MP, STAGES>, w_map, x_map, args);
}

// Deep rings: about 185 KB for 16 rows, near the 227 KB a CTA may use for 32 and
// 64 rows (their x slices take a larger share of each stage). Measured on GB300:
// 12 stages for 16 rows gain alone but lose inside the layer chain.
constexpr int kDeepStages16 = 10, kDeepStages32 = 11, kDeepStages64 = 9;
// Shallow rings sized so two CTAs fit on one SM (about 112 and 104 KB). Rows of
// x above 32 always take the deep ring (plan.cuh): a 4-stage shallow ring for
// them measured 0.6-1 us slower on GB300 even on short streams.
constexpr int kShallowStages16 = 6, kShallowStages32 = 5;
static_assert(kShallowStages16 <= kMaxShallowStages && kDeepStages64 > kMaxShallowStages,
              "ring classes must stay apart");

}  // namespace

int gemm_stages(int mma_n, bool shallow) {
    if (mma_n == 64) return kDeepStages64;
    if (shallow) return mma_n == 16 ? kShallowStages16 : kShallowStages32;
    return mma_n == 16 ? kDeepStages16 : kDeepStages32;
}

int gemm_smem_bytes(int mma_n, bool shallow) {
    if (mma_n == 16)
        return shallow ? Layout<16, kShallowStages16>::kDynamicBytes : Layout<16, kDeepStages16>::kDynamicBytes;
    if (mma_n == 32)
        return shallow ? Layout<32, kShallowStages32>::kDynamicBytes : Layout<32, kDeepStages32>::kDynamicBytes;
    return Layout<64, kDeepStages64>::kDynamicBytes;
}

cudaError_t launch_decode_gemm(const CUtensorMap &w_map, const CUtensorMap &x_map,
                               const GemmArgs &args, int mma_n, int ctas, cudaStream_t stream,
                               bool pdl, bool shallow, int device) {
    if (mma_n == 16) {
        if (shallow) return launch_variant<16, kShallowStages16>(w_map, x_map, args, ctas, stream, pdl, device);
        return launch_variant<16, kDeepStages16>(w_map, x_map, args, ctas, stream, pdl, device);
    }
    if (mma_n == 32) {
        if (shallow) return launch_variant<32, kShallowStages32>(w_map, x_map, args, ctas, stream, pdl, device);
        return launch_variant<32, kDeepStages32>(w_map, x_map, args, ctas, stream, pdl, device);
    }
    return launch_variant<64, kDeepStages64>(w_map, x_map, args, ctas, stream, pdl, device);
}

}  // namespace skinny

// ---- scratch in a static device array (for decode_gemm_bf16_noalloc) -----------------
//
// The same kernel can run with its split-K scratch in this file-scope array
// instead of memory from cudaMalloc. Sized for kStaticScratchCtas CTAs with
// partial tiles of up to 32 rows: 2 slots per CTA, then one flag per slot, then
// the error word. Every GPU that loads the library holds it until the process
// exits.
namespace skinny {
namespace {

constexpr size_t kStaticPartialBytes =
    static_cast<size_t>(2) * kStaticScratchCtas * kStaticSlotRows * kBlockN * sizeof(float);
constexpr size_t kStaticFlagBytes = 2048;  // >= 2 * kStaticScratchCtas flags, 256-aligned
constexpr size_t kStaticScratchBytes = kStaticPartialBytes + kStaticFlagBytes + 256;
static_assert(2 * kStaticScratchCtas * sizeof(unsigned) <= kStaticFlagBytes, "flag space");

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mutex;
void *g_static_base[64] = {};

}  // namespace

cudaError_t static_scratch_for_current_device(StaticScratch *out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_base[dev] == nullptr) {
        // Host code sees g_static_scratch only as a stand-in symbol; the array's
        // device address has to be looked up, once per device, with it current.
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        g_static_base[dev] = p;
    }
    char *base = static_cast<char *>(g_static_base[dev]);
    out->partials = reinterpret_cast<float *>(base);
    out->flags = reinterpret_cast<unsigned *>(base + kStaticPartialBytes);
    out->err = reinterpret_cast<int *>(base + kStaticPartialBytes + kStaticFlagBytes);
    out->zero_bytes = kStaticFlagBytes + sizeof(int);  // flags and error word
    out->max_ctas = kStaticScratchCtas;
    return cudaSuccess;
}

}  // namespace skinny
