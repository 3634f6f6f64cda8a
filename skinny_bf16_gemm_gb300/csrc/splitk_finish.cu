// Split-K finish of a publish-only decode GEMM ("drafter/linears": FP32 split-K
// partials, one BF16 rounding): every output column's partials, added in K order
// -- the first contributor's (lowest K blocks) first, as the GEMM's own
// finisher adds them, so the bits are the same -- and rounded once.
//
// One thread per 8 consecutive output columns of one row (all in one 128-column
// tile): two 16-byte loads per contributor, up to 4 contributors in flight, one
// 16-byte store (scalar stores at a ragged right edge or an unaligned out).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace skinny {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads)
    splitk_finish_kernel(SplitKPartials fix, uint16_t *__restrict__ out, int vector_out) {
    ptx::pdl_launch_dependents();
    const int frag = blockIdx.x * kThreads + threadIdx.x;
    const int m = blockIdx.y;
    const int col = frag * 8;
    ptx::pdl_wait();  // the partials are the previous kernel's output
    if (col >= fix.N) return;
    const GemmGeometry g = make_geometry(fix.M, fix.N, fix.K, fix.ctas);
    const int t = col / kBlockN;
    int first, last;
    tile_contributors(g, t, first, last);
    float a[8];
    for (int c0 = first; c0 <= last; c0 += 4) {
        float4 v[4][2];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (c0 + q <= last) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    fix.partials + static_cast<size_t>(partial_slot(g, c0 + q, t)) * fix.slot_floats +
                    m * kBlockN + (col % kBlockN));
                v[q][0] = __ldcg(src);
                v[q][1] = __ldcg(src + 1);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (c0 + q > last) break;
            const float u[8] = {v[q][0].x, v[q][0].y, v[q][0].z, v[q][0].w,
                                v[q][1].x, v[q][1].y, v[q][1].z, v[q][1].w};
#pragma unroll
            for (int j = 0; j < 8; ++j) a[j] = c0 + q == first ? u[j] : __fadd_rn(a[j], u[j]);
        }
    }
    uint16_t b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = __bfloat16_as_ushort(__float2bfloat16_rn(a[j]));
    uint16_t *dst = out + static_cast<size_t>(m) * fix.N + col;
    if (vector_out && col + 8 <= fix.N) {
        *reinterpret_cast<uint4 *>(dst) =
            make_uint4(b[0] | (static_cast<uint32_t>(b[1]) << 16), b[2] | (static_cast<uint32_t>(b[3]) << 16),
                       b[4] | (static_cast<uint32_t>(b[5]) << 16), b[6] | (static_cast<uint32_t>(b[7]) << 16));
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (col + j < fix.N) dst[j] = b[j];
    }
}

}  // namespace

cudaError_t launch_splitk_finish(const SplitKPartials &fix, uint16_t *out, cudaStream_t stream,
                                 bool pdl) {
    const int frags = (fix.N + 7) / 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((frags + kThreads - 1) / kThreads, fix.M, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const int vector_out = (fix.N % 8 == 0 && (reinterpret_cast<uintptr_t>(out) % 16) == 0) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, splitk_finish_kernel, fix, out, vector_out);
}

}  // namespace skinny
