// Test support only: blocks that hold shared memory on their SMs for a bounded
// time, so that a kernel launched beside them cannot place a CTA on those SMs.
// Each block's first thread sleeps in short naps until `ns` nanoseconds have
// passed on the global timer; nothing else is read or written.
#include <cuda_runtime.h>

__global__ void occupy_kernel(unsigned long long ns) {
    extern __shared__ unsigned char held[];
    if (threadIdx.x == 0) {
        held[0] = 1;
        unsigned long long t0, t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
        do {
            __nanosleep(1000);
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        } while (t - t0 < ns);
    }
}

extern "C" int occupy_launch(int blocks, int smem_bytes, unsigned long long ns, void *stream) {
    if (blocks < 1 || smem_bytes < 1 || ns > 1000000000ull) return -1;
    if (cudaFuncSetAttribute(occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes) != cudaSuccess)
        return -2;
    occupy_kernel<<<blocks, 32, smem_bytes, static_cast<cudaStream_t>(stream)>>>(ns);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}
