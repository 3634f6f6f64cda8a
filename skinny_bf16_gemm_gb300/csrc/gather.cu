// Local gather of TP shards on GB300 (sm_103a) ("drafter/comm": Gather, and the
// gather_context / gather_logits users): out[m][r*S + j] = shards[r][m][j].
// A byte move bound by HBM: every thread copies one 16-byte fragment (8 BF16),
// consecutive threads take consecutive fragments of a gathered row, so both the
// reads (within a shard row) and the writes are fully coalesced. The local
// slots have no sentinel, so nothing is rewritten on the way.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace skinny {
namespace {

constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(const uint4 *__restrict__ shards, uint4 *__restrict__ out, int TP, int M,
                  int frags_per_shard) {
    const int row_frags = TP * frags_per_shard;
    const int f = blockIdx.x * kGatherThreads + threadIdx.x;  // fragment of the gathered row
    const int m = blockIdx.y;
    ptx::pdl_launch_dependents();
    ptx::pdl_wait();  // the shards may be the previous kernel's output
    if (f >= row_frags) return;
    const int r = f / frags_per_shard;
    const int j = f - r * frags_per_shard;
    out[static_cast<size_t>(m) * row_frags + f] =
        __ldcs(shards + (static_cast<size_t>(r) * M + m) * frags_per_shard + j);
}

}  // namespace

cudaError_t launch_gather(const void *shards, int TP, int M, int S, void *out,
                          cudaStream_t stream, bool pdl) {
    const int frags = S / 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((TP * frags + kGatherThreads - 1) / kGatherThreads, M, 1);
    cfg.blockDim = dim3(kGatherThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gather_kernel, static_cast<const uint4 *>(shards),
                              static_cast<uint4 *>(out), TP, M, frags);
}

}  // namespace skinny
