// Reduce + residual + RMSNorm over rows of 7168 BF16 values on GB300 (sm_103a)
// ("drafter/comm": module text and ArNorm; "cutedsl/common/twoshot": reduce).
//
// Per element of row m, column c (bit-exact):
//   s = p[0][m][c]; s = s + p[r][m][c] for r = 1..TP-1      (FP32, round to nearest)
//   a = BF16(s);  h = residual ? BF16(a + residual[m][c]) : a  ->  residual_out
// then per row: rstd = rsqrt(sum_c h^2 / 7168 + eps) (FP32) and
//   out[m][c] = BF16((h * rstd) * gamma[c]).
//
// Layout: one cluster of C CTAs per row (grid C x M; C = 1: one CTA, no cluster,
// whose 896 threads cover the row); CTA r of the cluster owns
// the 896 / C 16-byte fragments (8 BF16 each) r*896/C .. ; thread t owns one
// fragment, so a whole row's TP + 1 loads per thread are in flight at once. The
// row's sum of squares: an FMA chain over the thread's 8 values, a warp butterfly,
// the warps in order, then the C CTA sums exchanged through distributed shared
// memory and added in CTA order (every CTA gets the same bits). Each CTA sends its
// sum to every peer with st.async, which completes bytes on the peer's mbarrier,
// and waits on its own: measured on GB300, 0.3-0.4 us faster per call than
// remote stores followed by a full cluster barrier (the layer chain's step
// 1.5 us faster). The wait is bounded; one that runs out is recorded in a
// device word skinny_device_error() reports.
// With programmatic dependent launch, gamma (a weight) is loaded before waiting
// for the previous kernel; the partial rows and the residual after.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace skinny {
namespace {

constexpr int kHidden = 7168;
constexpr uint64_t kExchangeLimitNs = 1000000000ull;  // 1 s for the CTA sums
__device__ int g_reduce_err;  // nonzero: a cluster exchange wait ran out
constexpr int kRowFrags = kHidden / 8;  // 896 fragments of 16 bytes
constexpr int kMaxTP = 8;

template <int C>
struct ReduceShape {
    static constexpr int kFrags = kRowFrags / C;               // fragments per CTA
    static constexpr int kThreads = (kFrags + 31) / 32 * 32;   // whole warps
    static constexpr int kWarps = kThreads / 32;
    static_assert(kRowFrags % C == 0, "row fragments must split evenly");
};

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t bf16_bits(float v) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    f[0] = lo_bf16(v.x); f[1] = hi_bf16(v.x);
    f[2] = lo_bf16(v.y); f[3] = hi_bf16(v.y);
    f[4] = lo_bf16(v.z); f[5] = hi_bf16(v.z);
    f[6] = lo_bf16(v.w); f[7] = hi_bf16(v.w);
}

__device__ __forceinline__ uint4 pack8(const uint32_t (&b)[8]) {
    return make_uint4(b[0] | (b[1] << 16), b[2] | (b[3] << 16), b[4] | (b[5] << 16),
                      b[6] | (b[7] << 16));
}

// FIX: slot 0 is not read but made here from a publish-only decode GEMM's FP32
// partials ("drafter/linears": FP32 split-K partials, one BF16 rounding): the
// partials of the fragment's 8 columns added in K order and rounded once, as the
// GEMM's own finisher would; the result is also stored to slot 0.
// TEST (the failure-path self-test only): the last CTA of each cluster keeps
// its sum to itself, so that every wait of the cluster runs out, after limit_ns
// instead of the regular limit.
template <int C, bool RES, bool FIX, bool TEST = false>
__global__ void __launch_bounds__(ReduceShape<C>::kThreads)
    reduce_rmsnorm_kernel(const uint4 *partials, int TP, const uint4 *residual,
                          const uint4 *__restrict__ gamma, uint4 *__restrict__ out,
                          uint4 *residual_out, int M, float eps, uint4 *slot0,
                          SplitKPartials fix, unsigned long long limit_ns) {
    using R = ReduceShape<C>;
    __shared__ float warp_sums[R::kWarps];
    __shared__ float parts[C];

    const int tid = threadIdx.x;
    const int rank = C > 1 ? static_cast<int>(blockIdx.x) : 0;  // cluster spans x
    const int row = blockIdx.y;
    const bool active = tid < R::kFrags;
    const int frag = rank * R::kFrags + tid;
    const size_t row_off = static_cast<size_t>(row) * kRowFrags + frag;

    __shared__ alignas(8) unsigned long long recv_bar;  // the C CTA sums arrived
    if constexpr (C > 1) {
        // Each CTA's sum goes to every peer with st.async, completing bytes on the
        // peer's barrier; the barriers must be initialised (and published to the
        // cluster) before any peer may send.
        if (tid == 0) {
            ptx::mbar_init(ptx::smem_addr(&recv_bar), 1);
            ptx::fence_barrier_init();
        }
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    }

    uint4 gw = make_uint4(0, 0, 0, 0);
    if (active) gw = __ldg(gamma + frag);
    // The next kernel may launch now: a decode GEMM that follows sets up and
    // streams its first weights while this kernel waits and runs.
    // FIX: the plan arithmetic of this thread's tile (64-bit divisions) and the
    // addresses of its first partials before the wait, off the path from the
    // GEMM's end to this kernel's first load (measured on GB300: the layer
    // chain's step 1.6 us faster). Up to kU contributors' partials are loaded
    // together (fewer with 896-thread CTAs, whose register budget is smaller).
    constexpr int kU = C == 1 ? 2 : 4;
    int fx_first = 0, fx_last = -1, fx_t = 0;
    const float *fx_src[kU];
    GemmGeometry fx_g = {};
    if constexpr (FIX) {
        fx_g = make_geometry(fix.M, fix.N, fix.K, fix.ctas);
        const int col = frag * 8;
        fx_t = col / kBlockN;
        tile_contributors(fx_g, fx_t, fx_first, fx_last);
#pragma unroll
        for (int q = 0; q < kU; ++q)
            fx_src[q] = fx_first + q <= fx_last
                            ? fix.partials + static_cast<size_t>(partial_slot(fx_g, fx_first + q, fx_t)) * fix.slot_floats +
                                  row * kBlockN + (col % kBlockN)
                            : nullptr;
    }
    ptx::pdl_launch_dependents();
    ptx::pdl_wait();  // the partial rows may be the previous kernel's output
    if constexpr (FIX) {
        // The GEMM is complete: a decode GEMM waiting behind this kernel may
        // prefetch its weights now (GemmArgs::l2_after_reduce).
        if (fix.gemm_done != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0)
            atomicExch(fix.gemm_done, 1u);
    }

    float h[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float ss = 0.0f;
    if (active) {
        uint4 pv[kMaxTP];
#pragma unroll
        for (int r = 0; r < kMaxTP; ++r)
            if (r < TP && (!FIX || r > 0))
                pv[r] = __ldcs(partials + static_cast<size_t>(r) * M * kRowFrags + row_off);
        uint4 rv = make_uint4(0, 0, 0, 0);
        if constexpr (RES) rv = __ldcs(residual + row_off);

        float s[8];
        if constexpr (FIX) {
            const GemmGeometry &g = fx_g;
            const int col = frag * 8;
            const int t = fx_t;
            const int first = fx_first, last = fx_last;
            float a[8];
            for (int c0 = first; c0 <= last; c0 += kU) {
                float4 v[kU][2];
#pragma unroll
                for (int q = 0; q < kU; ++q) {
                    if (c0 + q <= last) {
                        const float4 *src = reinterpret_cast<const float4 *>(
                            c0 == first ? fx_src[q]
                                        : fix.partials + static_cast<size_t>(partial_slot(g, c0 + q, t)) * fix.slot_floats +
                                              row * kBlockN + (col % kBlockN));
                        v[q][0] = __ldcg(src);
                        v[q][1] = __ldcg(src + 1);
                    }
                }
#pragma unroll
                for (int q = 0; q < kU; ++q) {
                    if (c0 + q > last) break;
                    const float u[8] = {v[q][0].x, v[q][0].y, v[q][0].z, v[q][0].w,
                                        v[q][1].x, v[q][1].y, v[q][1].z, v[q][1].w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) a[j] = c0 + q == first ? u[j] : __fadd_rn(a[j], u[j]);
                }
            }
            uint32_t s0[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                s0[j] = bf16_bits(a[j]);
                s[j] = __uint_as_float(s0[j] << 16);
            }
            slot0[row_off] = pack8(s0);
        } else {
            unpack8(pv[0], s);  // the sum starts from slot 0 (keeps -0)
        }
#pragma unroll
        for (int r = 1; r < kMaxTP; ++r) {
            if (r < TP) {
                float t[8];
                unpack8(pv[r], t);
#pragma unroll
                for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], t[j]);
            }
        }
        uint32_t hb[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) hb[j] = bf16_bits(s[j]);
        if constexpr (RES) {
            float res[8];
            unpack8(rv, res);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                hb[j] = bf16_bits(__fadd_rn(__uint_as_float(hb[j] << 16), res[j]));
        }
        residual_out[row_off] = pack8(hb);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            h[j] = __uint_as_float(hb[j] << 16);
            ss = __fmaf_rn(h[j], h[j], ss);
        }
    }

    // Row sum of squares: warp butterfly, warps in order, CTAs in order.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, o));
    if ((tid & 31) == 0) warp_sums[tid >> 5] = ss;
    __syncthreads();
    if constexpr (C > 1) {
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        const uint32_t bar = ptx::smem_addr(&recv_bar);
        if (tid == 0) {
            float block = warp_sums[0];
#pragma unroll
            for (int w = 1; w < R::kWarps; ++w) block = __fadd_rn(block, warp_sums[w]);
            ptx::mbar_arrive_expect_tx(bar, C * 4);
            const uint32_t local = ptx::smem_addr(&parts[rank]);
#pragma unroll
            for (int peer = 0; peer < C; ++peer)
                if (!TEST || rank != C - 1)
                    asm volatile(
                    "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                        ptx::map_to_cluster_rank(local, peer)),
                    "r"(__float_as_uint(block)), "r"(ptx::map_to_cluster_rank(bar, peer))
                    : "memory");
        }
        // Every CTA's sum has landed here (bounded wait: a sum that never comes
        // is recorded and the row's output is unspecified).
        if (!ptx::mbar_try_wait(bar, 0)) {
            const uint64_t t0 = ptx::global_timer_ns();
            for (uint32_t spin = 1; !ptx::mbar_try_wait(bar, 0); ++spin) {
                if ((spin & 15u) == 0 &&
                    ptx::global_timer_ns() - t0 > (TEST ? limit_ns : kExchangeLimitNs)) {
                    if (tid == 0) atomicOr(&g_reduce_err, 1);
                    break;
                }
            }
        }
    } else {
        if (tid == 0) {
            float block = warp_sums[0];
            for (int w = 1; w < R::kWarps; ++w) block = __fadd_rn(block, warp_sums[w]);
            parts[0] = block;
        }
        __syncthreads();
    }
    float total = parts[0];
#pragma unroll
    for (int c = 1; c < C; ++c) total = __fadd_rn(total, parts[c]);
    const float rstd = rsqrtf(__fadd_rn(__fdiv_rn(total, static_cast<float>(kHidden)), eps));

    if (active) {
        float g[8];
        unpack8(gw, g);
        uint32_t ob[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) ob[j] = bf16_bits(__fmul_rn(__fmul_rn(h[j], rstd), g[j]));
        out[row_off] = pack8(ob);
    }
}

template <int C, bool RES, bool FIX, bool TEST = false>
cudaError_t launch_c(const void *partials, int TP, const void *residual, const void *gamma,
                     void *out, void *residual_out, int M, float eps, cudaStream_t stream,
                     bool pdl, const SplitKPartials &fix,
                     unsigned long long limit_ns = kExchangeLimitNs) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, M, 1);
    cfg.blockDim = dim3(ReduceShape<C>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (C > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = C;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, reduce_rmsnorm_kernel<C, RES, FIX, TEST>,
                              static_cast<const uint4 *>(partials), TP,
                              static_cast<const uint4 *>(residual),
                              static_cast<const uint4 *>(gamma), static_cast<uint4 *>(out),
                              static_cast<uint4 *>(residual_out), M, eps,
                              const_cast<uint4 *>(static_cast<const uint4 *>(partials)), fix,
                              limit_ns);
}

template <int C, bool FIX>
cudaError_t launch_res(const void *partials, int TP, const void *residual, const void *gamma,
                       void *out, void *residual_out, int M, float eps, cudaStream_t stream,
                       bool pdl, const SplitKPartials &fix) {
    if (residual)
        return launch_c<C, true, FIX>(partials, TP, residual, gamma, out, residual_out, M, eps,
                                      stream, pdl, fix);
    return launch_c<C, false, FIX>(partials, TP, residual, gamma, out, residual_out, M, eps,
                                   stream, pdl, fix);
}

template <bool FIX>
cudaError_t launch_any(const void *partials, int TP, const void *residual, const void *gamma,
                       void *out, void *residual_out, int M, float eps, int ctas_per_row,
                       cudaStream_t stream, bool pdl, const SplitKPartials &fix) {
    switch (ctas_per_row) {
        case 1: return launch_res<1, FIX>(partials, TP, residual, gamma, out, residual_out, M, eps, stream, pdl, fix);
        case 2: return launch_res<2, FIX>(partials, TP, residual, gamma, out, residual_out, M, eps, stream, pdl, fix);
        case 4: return launch_res<4, FIX>(partials, TP, residual, gamma, out, residual_out, M, eps, stream, pdl, fix);
        case 8: return launch_res<8, FIX>(partials, TP, residual, gamma, out, residual_out, M, eps, stream, pdl, fix);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_reduce_rmsnorm(const void *partials, int TP, const void *residual,
                                  const void *gamma, void *out, void *residual_out, int M,
                                  float eps, int ctas_per_row, cudaStream_t stream, bool pdl) {
    const SplitKPartials none = {};
    return launch_any<false>(partials, TP, residual, gamma, out, residual_out, M, eps,
                             ctas_per_row, stream, pdl, none);
}

cudaError_t launch_reduce_rmsnorm_splitk(void *partials, int TP, const void *residual,
                                         const void *gamma, void *out, void *residual_out, int M,
                                         float eps, int ctas_per_row, const SplitKPartials &fix,
                                         cudaStream_t stream, bool pdl) {
    return launch_any<true>(partials, TP, residual, gamma, out, residual_out, M, eps,
                            ctas_per_row, stream, pdl, fix);
}

cudaError_t launch_reduce_rmsnorm_selftest(const void *partials, int TP, const void *residual,
                                           const void *gamma, void *out, void *residual_out,
                                           int M, float eps, unsigned long long limit_ns,
                                           cudaStream_t stream) {
    const SplitKPartials none = {};
    if (residual)
        return launch_c<8, true, false, true>(partials, TP, residual, gamma, out, residual_out, M,
                                              eps, stream, false, none, limit_ns);
    return launch_c<8, false, false, true>(partials, TP, residual, gamma, out, residual_out, M,
                                           eps, stream, false, none, limit_ns);
}

cudaError_t reduce_error_word(int *value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_reduce_err, sizeof(int));
    if (e != cudaSuccess || !clear || *value == 0) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_reduce_err, &zero, sizeof(int));
}

}  // namespace skinny
