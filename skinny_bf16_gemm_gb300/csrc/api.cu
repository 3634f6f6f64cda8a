// The library's C ABI (include/skinny.h): argument checks, the per-device state
// (SM count, split-K scratch, error word), TMA descriptor encoding and launches.
// Every check runs before any launch; a rejected call touches nothing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "plan.cuh"
#include "skinny.h"

namespace skinny {
namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per internal wait

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int major = 0, minor = 0;
    // Split-K scratch of the decode GEMM, sized for one CTA per SM.
    void *scratch = nullptr;
    float *partials = nullptr;
    unsigned *flags = nullptr;
    int *err = nullptr;
    size_t flag_bytes = 0;
    // decode_gemm_bf16_reduce_rmsnorm's "its GEMM is complete" word (in the
    // scratch's last 256 bytes, after the error word).
    unsigned *gemm_done = nullptr;
    // A host-mapped word the decode GEMM sets when one of its waits runs out:
    // the host reads it without synchronising, so the next call can refuse to
    // run on scratch a kernel left half used (host_err) -- and the kernel's
    // address of it (host_err_dev).
    int *host_err = nullptr;
    int *host_err_dev = nullptr;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
bool g_pdl = false;  // programmatic dependent launch, opt-in (skinny_set_pdl)
int g_l2_lead = kL2LeadDefault;  // decode GEMM deep-ring L2 lead (skinny_set_l2_prefetch)

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) {
        cudaGetLastError();
        return SKINNY_ERR_DEVICE;
    }
    return SKINNY_OK;
}

// Device properties (once per device). Caller holds g_mutex.
int device_state_locked(int dev, DeviceState **out) {
    DeviceState &d = g_devices[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return SKINNY_ERR_DEVICE;
        }
        d.ready = true;
    }
    // The kernels are built for sm_103a only.
    if (d.major != 10 || d.minor != 3) return SKINNY_ERR_DEVICE;
    *out = &d;
    return SKINNY_OK;
}

int device_state(int dev, DeviceState **out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    return device_state_locked(dev, out);
}

// The decode GEMM's scratch: allocated and zeroed once per device.
int ensure_scratch(int dev, cudaStream_t stream, DeviceState **out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState *d = nullptr;
    int st = device_state_locked(dev, &d);
    if (st != SKINNY_OK) return st;
    if (d->scratch == nullptr) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
            cudaGetLastError();
            return SKINNY_ERR_LAUNCH;
        }
        if (cap != cudaStreamCaptureStatusNone) return SKINNY_ERR_CAPTURE;
        const size_t partial_bytes = static_cast<size_t>(2) * d->sms * kSlotFloats * sizeof(float);
        const size_t flag_bytes = (static_cast<size_t>(2) * d->sms * sizeof(unsigned) + 255) / 256 * 256;
        const size_t bytes = partial_bytes + flag_bytes + 256;
        void *p = nullptr;
        if (cudaMalloc(&p, bytes) != cudaSuccess) {
            cudaGetLastError();
            return SKINNY_ERR_ALLOC;
        }
        if (cudaMemset(p, 0, bytes) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(p);
            return SKINNY_ERR_ALLOC;
        }
        void *h = nullptr, *hd = nullptr;
        if (cudaHostAlloc(&h, 256, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(p);
            return SKINNY_ERR_ALLOC;
        }
        if (cudaHostGetDevicePointer(&hd, h, 0) != cudaSuccess) {
            cudaGetLastError();
            cudaFreeHost(h);
            cudaFree(p);
            return SKINNY_ERR_ALLOC;
        }
        std::memset(h, 0, 256);
        d->host_err = static_cast<int *>(h);
        d->host_err_dev = static_cast<int *>(hd);
        d->scratch = p;
        d->partials = static_cast<float *>(p);
        d->flags = reinterpret_cast<unsigned *>(static_cast<char *>(p) + partial_bytes);
        d->err = reinterpret_cast<int *>(static_cast<char *>(p) + partial_bytes + flag_bytes);
        d->flag_bytes = flag_bytes;
        d->gemm_done = reinterpret_cast<unsigned *>(d->err) + 32;
    }
    *out = d;
    return SKINNY_OK;
}

int encoder(EncodeTiledFn *fn) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_encode == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || p == nullptr) {
            cudaGetLastError();
            return SKINNY_ERR_DEVICE;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(p);
    }
    *fn = g_encode;
    return SKINNY_OK;
}

// The pointer must be device (or managed) memory of device `dev`.
int check_device_pointer(const void *p, int dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_DEVICE;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return SKINNY_ERR_DEVICE;
    if (a.device != dev) return SKINNY_ERR_DEVICE;
    return SKINNY_OK;
}

bool overlaps(const void *a, size_t an, const void *b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 2-D BF16 tensor map over a row-major [rows, cols] array, box [box_rows, 64].
int encode_2d(EncodeTiledFn enc, CUtensorMap *map, const void *base, uint64_t rows,
              uint64_t cols, uint32_t box_rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), box_rows};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                     strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SKINNY_OK : SKINNY_ERR_LAUNCH;
}

int gemm_shape_ok(int M, int N, int K) {
    if (M < 1 || M > kMaxM || N < 1 || K < 8 || (K % 8) != 0) return SKINNY_ERR_SHAPE;
    // The kernel counts 128 x 64 weight blocks in 32-bit integers (a weight of
    // 2^31 blocks would be 32 TiB).
    const long long blocks = static_cast<long long>((N + kBlockN - 1) / kBlockN) *
                             ((K + kBlockK - 1) / kBlockK);
    if (blocks >= (1ll << 31)) return SKINNY_ERR_SHAPE;
    return SKINNY_OK;
}

int mma_n_for(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

// SKINNY_ERR_TIMEOUT while a decode GEMM on this device has recorded a wait that
// ran out and skinny_device_error() has not cleared it: the split-K scratch
// may hold flags that kernel never consumed, so nothing that uses it runs.
int pending_timeout(const DeviceState *d) {
    if (d->host_err != nullptr && *reinterpret_cast<volatile const int *>(d->host_err) != 0)
        return SKINNY_ERR_TIMEOUT;
    return SKINNY_OK;
}

// The launch settings of one call: the caller's options where given, else the
// process-wide settings (skinny_set_pdl, skinny_set_l2_prefetch).
struct LaunchSettings {
    bool pdl;
    int l2_lead;
    int l2_after_reduce;
};

int resolve_settings(const skinny_launch_opts *opts, LaunchSettings *out) {
    if (opts != nullptr) {
        if (opts->pdl < SKINNY_OPT_DEFAULT || opts->pdl > 1) return SKINNY_ERR_ARG;
        if (opts->l2_prefetch < SKINNY_OPT_DEFAULT || opts->l2_prefetch > kL2LeadMax)
            return SKINNY_ERR_ARG;
        if (opts->l2_after_reduce < SKINNY_OPT_DEFAULT || opts->l2_after_reduce > kL2LeadMax)
            return SKINNY_ERR_ARG;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    out->pdl = g_pdl;
    out->l2_lead = g_l2_lead;
    out->l2_after_reduce = 0;
    if (opts != nullptr) {
        if (opts->pdl != SKINNY_OPT_DEFAULT) out->pdl = opts->pdl != 0;
        if (opts->l2_prefetch != SKINNY_OPT_DEFAULT) out->l2_lead = opts->l2_prefetch;
        if (opts->l2_after_reduce > 0) out->l2_after_reduce = opts->l2_after_reduce;
    }
    return SKINNY_OK;
}

int gemm_launch(const void *x, const void *W, void *out, int M, int N, int K, void *stream,
                const skinny_launch_opts *opts, int selftest, unsigned long long limit_ns,
                int logits = 0, float soft_cap = 0.0f, float scale = 1.0f) {
    if (!x || !W || !out) return SKINNY_ERR_NULL;
    int st = gemm_shape_ok(M, N, K);
    if (st) return st;
    if (!aligned(x, 16) || !aligned(W, 16) || !aligned(out, 2)) return SKINNY_ERR_ALIGN;
    const size_t xb = static_cast<size_t>(M) * K * 2, wb = static_cast<size_t>(N) * K * 2,
                 ob = static_cast<size_t>(M) * N * 2;
    if (overlaps(out, ob, x, xb) || overlaps(out, ob, W, wb)) return SKINNY_ERR_ALIAS;
    LaunchSettings ls;
    if ((st = resolve_settings(opts, &ls))) return st;
    int dev;
    if ((st = current_device(&dev))) return st;
    if ((st = check_device_pointer(x, dev)) || (st = check_device_pointer(W, dev)) ||
        (st = check_device_pointer(out, dev)))
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceState *d = nullptr;
    if ((st = ensure_scratch(dev, s, &d))) return st;
    if ((st = pending_timeout(d))) return st;
    EncodeTiledFn enc;
    if ((st = encoder(&enc))) return st;
    const int mma_n = mma_n_for(M);
    alignas(64) CUtensorMap w_map, x_map;
    if ((st = encode_2d(enc, &w_map, W, N, K, kBlockN))) return st;
    if ((st = encode_2d(enc, &x_map, x, M, K, mma_n))) return st;
    const GemmGeometry g = make_geometry(M, N, K, choose_ctas(N, d->sms));
    GemmArgs a = {};
    a.M = M;
    a.N = N;
    a.K = K;
    a.out = static_cast<uint16_t *>(out);
    a.partials = d->partials;
    a.slot_floats = kSlotFloats;
    a.flags = d->flags;
    a.err = d->err;
    a.host_err = d->host_err_dev;
    a.wait_limit_ns = limit_ns;
    a.selftest = selftest;
    a.logits = logits;
    a.soft_cap = soft_cap;
    a.scale = scale;
    const bool pdl = ls.pdl;
    a.l2_lead = ls.l2_lead;
    a.gemm_done = d->gemm_done;
    a.l2_after_reduce = ls.l2_after_reduce;
    // Split tiles of 64-row accumulators, every CTA within at most two tiles (two
    // scratch slots), plain output: the GEMM only publishes its partials and a
    // small kernel finishes them (same order, same bits). A finisher CTA would
    // pull 32 KB partial slots through its ring and add 64 rows per thread; the
    // finish kernel spreads that over every column. Measured on GB300: 2 µs
    // faster at M = 64, N = 7168, K = 14336; slower for 16 and 32 rows, where the
    // extra kernel boundary costs more than the in-kernel finish.
    int split = 0;
    for (int t = 0; t < g.tiles && !split; ++t) {
        int first, last;
        tile_contributors(g, t, first, last);
        split = first != last;
    }
    if (split && mma_n == 64 && g.ctas >= g.tiles && !logits && !selftest) {
        a.publish_only = 1;
        cudaError_t e = launch_decode_gemm(w_map, x_map, a, mma_n, g.ctas, s, pdl,
                                           use_shallow_ring(g, pdl), dev);
        if (e == cudaSuccess) {
            SplitKPartials fix = {};
            fix.partials = d->partials;
            fix.slot_floats = kSlotFloats;
            fix.M = M;
            fix.N = N;
            fix.K = K;
            fix.ctas = g.ctas;
            e = launch_splitk_finish(fix, static_cast<uint16_t *>(out), s, pdl);
        }
        if (e != cudaSuccess) {
            cudaGetLastError();
            return SKINNY_ERR_LAUNCH;
        }
        return SKINNY_OK;
    }
    cudaError_t e = launch_decode_gemm(w_map, x_map, a, mma_n, g.ctas, s, pdl,
                                       use_shallow_ring(g, pdl), dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_LAUNCH;
    }
    return SKINNY_OK;
}

// decode_gemm_bf16 with its split-K scratch in the static device array of
// decode_gemm.cu: no device memory is allocated on this path.
int gemm_launch_static(const void *x, const void *W, void *out, int M, int N, int K,
                       void *stream) {
    if (!x || !W || !out) return SKINNY_ERR_NULL;
    int st = gemm_shape_ok(M, N, K);
    if (st) return st;
    if (M > kStaticSlotRows) return SKINNY_ERR_SHAPE;  // the static partial tiles hold 32 rows
    if (!aligned(x, 16) || !aligned(W, 16) || !aligned(out, 2)) return SKINNY_ERR_ALIGN;
    const size_t xb = static_cast<size_t>(M) * K * 2, wb = static_cast<size_t>(N) * K * 2,
                 ob = static_cast<size_t>(M) * N * 2;
    if (overlaps(out, ob, x, xb) || overlaps(out, ob, W, wb)) return SKINNY_ERR_ALIAS;
    int dev;
    if ((st = current_device(&dev))) return st;
    DeviceState *d = nullptr;
    if ((st = device_state(dev, &d))) return st;
    if ((st = check_device_pointer(x, dev)) || (st = check_device_pointer(W, dev)) ||
        (st = check_device_pointer(out, dev)))
        return st;
    StaticScratch sc;
    if (static_scratch_for_current_device(&sc) != cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_DEVICE;
    }
    EncodeTiledFn enc;
    if ((st = encoder(&enc))) return st;
    const int mma_n = mma_n_for(M);
    alignas(64) CUtensorMap w_map, x_map;
    if ((st = encode_2d(enc, &w_map, W, N, K, kBlockN))) return st;
    if ((st = encode_2d(enc, &x_map, x, M, K, mma_n))) return st;
    // At most as many CTAs as the array has partial-tile slots for.
    const int ctas = choose_ctas(N, d->sms);
    const GemmGeometry g = make_geometry(M, N, K, ctas < sc.max_ctas ? ctas : sc.max_ctas);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: the published-partial flags
    // and the error word must start this call at zero.
    if (cudaMemsetAsync(sc.flags, 0, sc.zero_bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_LAUNCH;
    }
    GemmArgs a = {};
    a.M = M;
    a.N = N;
    a.K = K;
    a.out = static_cast<uint16_t *>(out);
    a.partials = sc.partials;
    a.slot_floats = kStaticSlotRows * kBlockN;
    a.flags = sc.flags;
    a.err = sc.err;
    a.wait_limit_ns = kWaitLimitNs;
    a.selftest = 0;
    a.logits = 0;
    a.soft_cap = 0.0f;
    a.scale = 1.0f;
    bool pdl;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        pdl = g_pdl;
        a.l2_lead = g_l2_lead;
    }
    cudaError_t e = launch_decode_gemm(w_map, x_map, a, mma_n, g.ctas, s, pdl,
                                       use_shallow_ring(g, pdl), dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_LAUNCH;
    }
    return SKINNY_OK;
}

// CTAs per row of the reduce. An 8-CTA cluster per row spreads a few rows, or
// heavy ones, over many SMs; with enough light rows one 896-thread CTA per row is
// faster (no cluster exchange). Loads per thread = TP partial fragments plus the
// residual's. Chosen from a sweep of 1, 2, 4 and 8 CTAs per row over TP in
// {2, 4, 8}, M in {1, .., 64}, residual or not, on GB300.
int reduce_ctas_per_row(int M, int TP, bool residual) {
    const int loads = TP + (residual ? 1 : 0);
    if ((M >= 32 && loads <= 8) || (M >= 16 && loads <= 4)) return 1;
    return 8;
}

// The reduce's argument checks that need no device: pointers, shapes, eps,
// alignment, aliasing.
int reduce_arg_checks(const void *partials, int TP, const void *residual, const void *gamma,
                      const void *out, const void *residual_out, int M, float eps) {
    if (!partials || !gamma || !out || !residual_out) return SKINNY_ERR_NULL;
    if (TP < 1 || TP > SKINNY_REDUCE_MAX_TP || M < 1 || M > SKINNY_REDUCE_MAX_M)
        return SKINNY_ERR_SHAPE;
    if (!(eps > 0.0f) || !std::isfinite(eps)) return SKINNY_ERR_ARG;
    if (!aligned(partials, 16) || !aligned(gamma, 16) || !aligned(out, 16) ||
        !aligned(residual_out, 16) || (residual && !aligned(residual, 16)))
        return SKINNY_ERR_ALIGN;
    const size_t row = static_cast<size_t>(M) * SKINNY_HIDDEN * 2;
    const size_t pb = row * TP, gb = SKINNY_HIDDEN * 2;
    if (overlaps(out, row, residual_out, row) || overlaps(out, row, partials, pb) ||
        overlaps(out, row, gamma, gb) || overlaps(residual_out, row, partials, pb) ||
        overlaps(residual_out, row, gamma, gb) || (residual && overlaps(out, row, residual, row)))
        return SKINNY_ERR_ALIAS;
    // residual_out may be residual itself (element-wise in-place), nothing else.
    if (residual && residual != residual_out && overlaps(residual_out, row, residual, row))
        return SKINNY_ERR_ALIAS;
    return SKINNY_OK;
}

// The current device, and the reduce's pointers on it.
int reduce_device_checks(const void *partials, const void *residual, const void *gamma,
                         const void *out, const void *residual_out, int *dev) {
    int st;
    if ((st = current_device(dev))) return st;
    DeviceState *d = nullptr;
    if ((st = device_state(*dev, &d))) return st;
    if ((st = check_device_pointer(partials, *dev)) || (st = check_device_pointer(gamma, *dev)) ||
        (st = check_device_pointer(out, *dev)) || (st = check_device_pointer(residual_out, *dev)) ||
        (residual && (st = check_device_pointer(residual, *dev))))
        return st;
    return SKINNY_OK;
}

}  // namespace
}  // namespace skinny

using namespace skinny;

extern "C" {

int decode_gemm_bf16(const void *x, const void *W, void *out, int M, int N, int K, void *stream) {
    return gemm_launch(x, W, out, M, N, K, stream, nullptr, 0, kWaitLimitNs);
}

int decode_gemm_bf16_ex(const void *x, const void *W, void *out, int M, int N, int K,
                        const skinny_launch_opts *opts, void *stream) {
    return gemm_launch(x, W, out, M, N, K, stream, opts, 0, kWaitLimitNs);
}

int decode_gemm_bf16_noalloc(const void *x, const void *W, void *out, int M, int N, int K,
                             void *stream) {
    return gemm_launch_static(x, W, out, M, N, K, stream);
}

int decode_gemm_bf16_reduce_rmsnorm_ex(const void *x, const void *W, void *partials, int TP,
                                       const void *residual, const void *gamma, void *out,
                                       void *residual_out, int M, int K, float eps,
                                       const skinny_launch_opts *opts, void *stream) {
    constexpr int N = SKINNY_HIDDEN;
    if (!x || !W || !partials || !gamma || !out || !residual_out) return SKINNY_ERR_NULL;
    if (M < 1 || M > SKINNY_REDUCE_MAX_M || TP < 1 || TP > SKINNY_REDUCE_MAX_TP) return SKINNY_ERR_SHAPE;
    int st = gemm_shape_ok(M, N, K);
    if (st) return st;
    if (!(eps > 0.0f) || !std::isfinite(eps)) return SKINNY_ERR_ARG;
    if (!aligned(x, 16) || !aligned(W, 16) || !aligned(partials, 16) || !aligned(gamma, 16) ||
        !aligned(out, 16) || !aligned(residual_out, 16) || (residual && !aligned(residual, 16)))
        return SKINNY_ERR_ALIGN;
    const size_t xb = static_cast<size_t>(M) * K * 2, wb = static_cast<size_t>(N) * K * 2;
    const size_t row = static_cast<size_t>(M) * N * 2, pb = row * TP, gb = N * 2;
    // Slot 0 of partials, out and residual_out are written; residual_out may be
    // residual itself (element-wise in place), nothing else may overlap.
    if (overlaps(partials, pb, x, xb) || overlaps(partials, pb, W, wb) ||
        overlaps(partials, pb, gamma, gb) || overlaps(out, row, x, xb) ||
        overlaps(out, row, W, wb) || overlaps(out, row, partials, pb) ||
        overlaps(out, row, gamma, gb) || overlaps(out, row, residual_out, row) ||
        overlaps(residual_out, row, x, xb) || overlaps(residual_out, row, W, wb) ||
        overlaps(residual_out, row, partials, pb) || overlaps(residual_out, row, gamma, gb) ||
        (residual && (overlaps(out, row, residual, row) || overlaps(partials, pb, residual, row) ||
                      (residual != residual_out && overlaps(residual_out, row, residual, row)))))
        return SKINNY_ERR_ALIAS;
    LaunchSettings ls;
    if ((st = resolve_settings(opts, &ls))) return st;
    int dev;
    if ((st = current_device(&dev))) return st;
    if ((st = check_device_pointer(x, dev)) || (st = check_device_pointer(W, dev)) ||
        (st = check_device_pointer(partials, dev)) || (st = check_device_pointer(gamma, dev)) ||
        (st = check_device_pointer(out, dev)) || (st = check_device_pointer(residual_out, dev)) ||
        (residual && (st = check_device_pointer(residual, dev))))
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceState *d = nullptr;
    if ((st = ensure_scratch(dev, s, &d))) return st;
    if ((st = pending_timeout(d))) return st;
    const GemmGeometry g = make_geometry(M, N, K, choose_ctas(N, d->sms));
    // The scratch holds two partial slots per CTA: every CTA's range must touch
    // at most two tiles, which at least one CTA per tile guarantees.
    if (g.ctas < g.tiles) return SKINNY_ERR_DEVICE;
    EncodeTiledFn enc;
    if ((st = encoder(&enc))) return st;
    const int mma_n = mma_n_for(M);
    alignas(64) CUtensorMap w_map, x_map;
    if ((st = encode_2d(enc, &w_map, W, N, K, kBlockN))) return st;
    if ((st = encode_2d(enc, &x_map, x, M, K, mma_n))) return st;
    const bool pdl = ls.pdl;
    const int l2_lead = ls.l2_lead;
    GemmArgs a = {};
    a.M = M;
    a.N = N;
    a.K = K;
    a.out = static_cast<uint16_t *>(partials);
    a.partials = d->partials;
    a.slot_floats = kSlotFloats;
    a.flags = d->flags;
    a.err = d->err;
    a.host_err = d->host_err_dev;
    a.wait_limit_ns = kWaitLimitNs;
    a.scale = 1.0f;
    a.publish_only = 1;
    a.l2_lead = l2_lead;
    a.gemm_done = d->gemm_done;
    a.clear_gemm_done = 1;
    if (launch_decode_gemm(w_map, x_map, a, mma_n, g.ctas, s, pdl, use_shallow_ring(g, pdl), dev) !=
        cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_LAUNCH;
    }
    SplitKPartials fix = {};
    fix.partials = d->partials;
    fix.slot_floats = kSlotFloats;
    fix.gemm_done = d->gemm_done;
    fix.M = M;
    fix.N = N;
    fix.K = K;
    fix.ctas = g.ctas;
    // The same CTAs per row as reduce_residual_rmsnorm: the same order of the sum
    // of squares, so out is bit-identical to the two separate calls.
    const int cpr = reduce_ctas_per_row(M, TP, residual != nullptr);
    if (launch_reduce_rmsnorm_splitk(partials, TP, residual, gamma, out, residual_out, M, eps, cpr,
                                     fix, s, pdl) != cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_LAUNCH;
    }
    return SKINNY_OK;
}

int decode_gemm_bf16_reduce_rmsnorm(const void *x, const void *W, void *partials, int TP,
                                    const void *residual, const void *gamma, void *out,
                                    void *residual_out, int M, int K, float eps, void *stream) {
    return decode_gemm_bf16_reduce_rmsnorm_ex(x, W, partials, TP, residual, gamma, out,
                                              residual_out, M, K, eps, nullptr, stream);
}

int decode_gemm_bf16_logits(const void *x, const void *W, void *out, int M, int N, int K,
                            int n_out, float soft_cap, float scale, void *stream) {
    if (n_out < 1 || n_out > N) return SKINNY_ERR_SHAPE;
    if (!std::isfinite(soft_cap) || !std::isfinite(scale)) return SKINNY_ERR_ARG;
    // Only the first n_out weight rows are read: the same GEMM with N = n_out.
    return gemm_launch(x, W, out, M, n_out, K, stream, nullptr, 0, kWaitLimitNs, 1,
                       soft_cap > 0.0f ? soft_cap : 0.0f, scale);
}

int skinny_watchdog_selftest(const void *x, const void *W, void *out, int M, int N, int K,
                             long long timeout_ns, void *stream) {
    if (timeout_ns < 1000 || timeout_ns > 2000000000LL) return SKINNY_ERR_ARG;
    return gemm_launch(x, W, out, M, N, K, stream, nullptr, 1,
                       static_cast<unsigned long long>(timeout_ns));
}

int reduce_residual_rmsnorm_ex(const void *partials, int TP, const void *residual,
                               const void *gamma, void *out, void *residual_out, int M, float eps,
                               const skinny_launch_opts *opts, void *stream) {
    LaunchSettings ls;
    int dev, st;
    if ((st = reduce_arg_checks(partials, TP, residual, gamma, out, residual_out, M, eps)) ||
        (st = resolve_settings(opts, &ls)) ||
        (st = reduce_device_checks(partials, residual, gamma, out, residual_out, &dev)))
        return st;
    cudaError_t e = launch_reduce_rmsnorm(partials, TP, residual, gamma, out, residual_out, M, eps,
                                          reduce_ctas_per_row(M, TP, residual != nullptr),
                                          static_cast<cudaStream_t>(stream), ls.pdl);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_LAUNCH;
    }
    return SKINNY_OK;
}

int skinny_reduce_selftest(const void *partials, int TP, const void *residual, const void *gamma,
                           void *out, void *residual_out, int M, float eps, long long timeout_ns,
                           void *stream) {
    if (timeout_ns < 1000 || timeout_ns > 2000000000LL) return SKINNY_ERR_ARG;
    int dev, st;
    if ((st = reduce_arg_checks(partials, TP, residual, gamma, out, residual_out, M, eps)) ||
        (st = reduce_device_checks(partials, residual, gamma, out, residual_out, &dev)))
        return st;
    cudaError_t e = launch_reduce_rmsnorm_selftest(partials, TP, residual, gamma, out,
                                                   residual_out, M, eps,
                                                   static_cast<unsigned long long>(timeout_ns),
                                                   static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_LAUNCH;
    }
    return SKINNY_OK;
}

int reduce_residual_rmsnorm(const void *partials, int TP, const void *residual,
                            const void *gamma, void *out, void *residual_out, int M, float eps,
                            void *stream) {
    return reduce_residual_rmsnorm_ex(partials, TP, residual, gamma, out, residual_out, M, eps,
                                      nullptr, stream);
}

int gather_shards_bf16(const void *shards, int TP, int M, int S, void *out, void *stream) {
    if (!shards || !out) return SKINNY_ERR_NULL;
    if (TP < 1 || TP > SKINNY_GATHER_MAX_TP || M < 1 || M > SKINNY_GATHER_MAX_M || S < 8 ||
        (S % 8) != 0 || static_cast<long long>(TP) * S > (1LL << 30))
        return SKINNY_ERR_SHAPE;
    if (!aligned(shards, 16) || !aligned(out, 16)) return SKINNY_ERR_ALIGN;
    const size_t bytes = static_cast<size_t>(TP) * M * S * 2;
    if (overlaps(out, bytes, shards, bytes)) return SKINNY_ERR_ALIAS;
    int dev, st;
    if ((st = current_device(&dev))) return st;
    DeviceState *d = nullptr;
    if ((st = device_state(dev, &d))) return st;
    if ((st = check_device_pointer(shards, dev)) || (st = check_device_pointer(out, dev))) return st;
    bool pdl;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        pdl = g_pdl;
    }
    if (launch_gather(shards, TP, M, S, out, static_cast<cudaStream_t>(stream), pdl) != cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_LAUNCH;
    }
    return SKINNY_OK;
}

const char *skinny_status_string(int status) {
    switch (status) {
        case SKINNY_OK: return "ok";
        case SKINNY_ERR_NULL: return "a required pointer is NULL";
        case SKINNY_ERR_SHAPE: return "a size is outside the accepted range";
        case SKINNY_ERR_ALIGN: return "a pointer is not aligned as required";
        case SKINNY_ERR_DEVICE: return "no sm_103 device, or a pointer is not memory of the current device";
        case SKINNY_ERR_LAUNCH: return "the CUDA launch failed";
        case SKINNY_ERR_ALIAS: return "an output overlaps an input or the other output";
        case SKINNY_ERR_CAPTURE: return "first call on this device made during stream capture";
        case SKINNY_ERR_ALLOC: return "scratch allocation failed";
        case SKINNY_ERR_TIMEOUT: return "a kernel's bounded internal wait ran out";
        case SKINNY_ERR_ARG: return "a scalar argument is invalid";
        default: return "unknown status";
    }
}

int skinny_device_error(int device, int *word) {
    if (device < 0 || device >= kMaxDevices) return SKINNY_ERR_DEVICE;
    if (word) *word = 0;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) {
        cudaGetLastError();
        return SKINNY_ERR_DEVICE;
    }
    if (cudaSetDevice(device) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        cudaSetDevice(prev);
        return SKINNY_ERR_DEVICE;
    }
    int value = 0;
    int st = SKINNY_OK;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceState &d = g_devices[device];
        if (d.scratch) {
            if (cudaMemcpy(&value, d.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
                cudaGetLastError();
                st = SKINNY_ERR_DEVICE;
            } else if (value != 0 || *reinterpret_cast<volatile int *>(d.host_err) != 0) {
                // A kernel gave up part-way: clear the words and the partial flags,
                // which lets later calls run again.
                if (cudaMemset(d.err, 0, sizeof(int)) != cudaSuccess ||
                    cudaMemset(d.flags, 0, d.flag_bytes) != cudaSuccess) {
                    cudaGetLastError();
                    st = SKINNY_ERR_DEVICE;
                } else {
                    if (value == 0) value = kErrUnknown;
                    *reinterpret_cast<volatile int *>(d.host_err) = 0;
                }
            }
        }
    }
    // The reduce kernel's own word (its cluster exchange waits).
    int reduce_word = 0;
    if (st == SKINNY_OK && reduce_error_word(&reduce_word, true) != cudaSuccess) {
        cudaGetLastError();
        st = SKINNY_ERR_DEVICE;
    }
    if (reduce_word) value |= kErrReduceExchange;
    cudaSetDevice(prev);
    if (word) *word = value;
    if (st != SKINNY_OK) return st;
    return value ? SKINNY_ERR_TIMEOUT : SKINNY_OK;
}

int skinny_set_pdl(int enable) {
    std::lock_guard<std::mutex> lock(g_mutex);
    const int prev = g_pdl ? 1 : 0;
    g_pdl = enable != 0;
    return prev;
}

int skinny_set_l2_prefetch(int blocks) {
    if (blocks < 0 || blocks > kL2LeadMax) return -1;
    std::lock_guard<std::mutex> lock(g_mutex);
    const int prev = g_l2_lead;
    g_l2_lead = blocks;
    return prev;
}

int skinny_gemm_plan_query(int M, int N, int K, int num_sms, skinny_gemm_plan *plan) {
    if (!plan) return SKINNY_ERR_NULL;
    if (num_sms < 1) return SKINNY_ERR_ARG;
    int st = gemm_shape_ok(M, N, K);
    if (st) return st;
    const GemmGeometry g = make_geometry(M, N, K, choose_ctas(N, num_sms));
    plan->tiles = g.tiles;
    plan->kblocks = g.kblocks;
    plan->blocks = g.blocks;
    plan->ctas = g.ctas;
    plan->mma_n = mma_n_for(M);
    bool pdl;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        pdl = g_pdl;
    }
    plan->stages = gemm_stages(plan->mma_n, use_shallow_ring(g, pdl));
    plan->smem_bytes = gemm_smem_bytes(plan->mma_n, use_shallow_ring(g, pdl));
    int split = 0;
    for (int t = 0; t < g.tiles; ++t) {
        int first, last;
        tile_contributors(g, t, first, last);
        split += first != last;
    }
    plan->split_tiles = split;
    return SKINNY_OK;
}

int skinny_gemm_cta_pieces(int M, int N, int K, int num_sms, int cta, int *tile, int *kb0,
                           int *kb1, int *slot, int max_pieces) {
    if (!tile || !kb0 || !kb1 || !slot || num_sms < 1 || gemm_shape_ok(M, N, K)) return -1;
    const GemmGeometry g = make_geometry(M, N, K, choose_ctas(N, num_sms));
    if (cta < 0 || cta >= g.ctas) return -1;
    const int r = range_of_block(g, cta);
    const int n = cta_piece_count(g, r);
    for (int q = 0; q < n && q < max_pieces; ++q) {
        const Piece p = cta_piece(g, r, q);
        tile[q] = p.tile;
        kb0[q] = p.kb0;
        kb1[q] = p.kb1;
        const bool whole = p.kb0 == 0 && p.kb1 == g.kblocks;
        slot[q] = whole ? -1 : partial_slot(g, r, p.tile);
    }
    return n;
}

}  // extern "C"
