"""Python binding of libskinny.so (include/skinny.h): argument marshalling only.

Every computation runs in the library's CUDA kernels; this module checks that
PyTorch tensors have the shapes and dtypes the C ABI documents, passes their
device pointers and the current CUDA stream, and turns nonzero status codes into
``SkinnyError``. There is no fallback: if the library is missing, importing the
operations raises.

    decode_gemm_bf16(x, W, out)                      out = x @ W^T (BF16)
    reduce_residual_rmsnorm(partials, residual, gamma, out, residual_out, eps)
    gather_shards_bf16(shards, out)                  TP shards side by side
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(PKG, "libskinny.so")
HIDDEN = 7168
GEMM_MAX_M = 64
REDUCE_MAX_M = 64
REDUCE_MAX_TP = 8

STATUS = {
    0: "SKINNY_OK", 1: "SKINNY_ERR_NULL", 2: "SKINNY_ERR_SHAPE", 3: "SKINNY_ERR_ALIGN",
    4: "SKINNY_ERR_DEVICE", 5: "SKINNY_ERR_LAUNCH", 6: "SKINNY_ERR_ALIAS",
    7: "SKINNY_ERR_CAPTURE", 8: "SKINNY_ERR_ALLOC", 9: "SKINNY_ERR_TIMEOUT",
    10: "SKINNY_ERR_ARG",
}


class SkinnyError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_string(status)})")


class LaunchOpts(ctypes.Structure):
    """skinny_launch_opts: per-call settings, -1 = the process-wide one (for
    l2_after_reduce: off)."""
    _fields_ = [("pdl", ctypes.c_int), ("l2_prefetch", ctypes.c_int),
                ("l2_after_reduce", ctypes.c_int)]


def _opts(pdl, l2_prefetch, l2_after_reduce=None):
    """A LaunchOpts for the given keywords, or None if all are None (the call
    then goes to the plain entry point and the process-wide settings)."""
    if pdl is None and l2_prefetch is None and l2_after_reduce is None:
        return None
    return LaunchOpts(-1 if pdl is None else int(bool(pdl)),
                      -1 if l2_prefetch is None else int(l2_prefetch),
                      -1 if l2_after_reduce is None else int(l2_after_reduce))


class GemmPlan(ctypes.Structure):
    _fields_ = [("tiles", ctypes.c_int), ("kblocks", ctypes.c_int),
                ("blocks", ctypes.c_longlong), ("ctas", ctypes.c_int),
                ("mma_n", ctypes.c_int), ("stages", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("split_tiles", ctypes.c_int)]


_lib = None


def load_library(path: str = LIBRARY):
    """Load libskinny.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} is missing: build it with "
                      "`python -m skinny_bf16_gemm_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    op = ctypes.POINTER(LaunchOpts)
    lib.decode_gemm_bf16.argtypes = [vp, vp, vp, i32, i32, i32, vp]
    lib.decode_gemm_bf16.restype = i32
    lib.decode_gemm_bf16_ex.argtypes = [vp, vp, vp, i32, i32, i32, op, vp]
    lib.decode_gemm_bf16_ex.restype = i32
    lib.reduce_residual_rmsnorm.argtypes = [vp, i32, vp, vp, vp, vp, i32, f32, vp]
    lib.reduce_residual_rmsnorm.restype = i32
    lib.reduce_residual_rmsnorm_ex.argtypes = [vp, i32, vp, vp, vp, vp, i32, f32, op, vp]
    lib.reduce_residual_rmsnorm_ex.restype = i32
    lib.decode_gemm_bf16_logits.argtypes = [vp, vp, vp, i32, i32, i32, i32, f32, f32, vp]
    lib.decode_gemm_bf16_logits.restype = i32
    lib.decode_gemm_bf16_reduce_rmsnorm.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32,
                                                    f32, vp]
    lib.decode_gemm_bf16_reduce_rmsnorm.restype = i32
    lib.decode_gemm_bf16_reduce_rmsnorm_ex.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32,
                                                       f32, op, vp]
    lib.decode_gemm_bf16_reduce_rmsnorm_ex.restype = i32
    lib.gather_shards_bf16.argtypes = [vp, i32, i32, i32, vp, vp]
    lib.gather_shards_bf16.restype = i32
    lib.skinny_status_string.argtypes = [i32]
    lib.skinny_status_string.restype = ctypes.c_char_p
    lib.skinny_device_error.argtypes = [i32, ctypes.POINTER(i32)]
    lib.skinny_device_error.restype = i32
    lib.skinny_set_pdl.argtypes = [i32]
    lib.skinny_set_pdl.restype = i32
    lib.skinny_set_l2_prefetch.argtypes = [i32]
    lib.skinny_set_l2_prefetch.restype = i32
    lib.skinny_gemm_plan_query.argtypes = [i32, i32, i32, i32, ctypes.POINTER(GemmPlan)]
    lib.skinny_gemm_plan_query.restype = i32
    ip = ctypes.POINTER(i32)
    lib.skinny_gemm_cta_pieces.argtypes = [i32, i32, i32, i32, i32, ip, ip, ip, ip, i32]
    lib.skinny_gemm_cta_pieces.restype = i32
    lib.skinny_watchdog_selftest.argtypes = [vp, vp, vp, i32, i32, i32, ctypes.c_longlong, vp]
    lib.skinny_watchdog_selftest.restype = i32
    lib.skinny_reduce_selftest.argtypes = [vp, i32, vp, vp, vp, vp, i32, f32, ctypes.c_longlong, vp]
    lib.skinny_reduce_selftest.restype = i32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().skinny_status_string(int(status)).decode()


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != 0:
        raise SkinnyError(status, where)


def _bf16_cuda(t, name, shape=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor (got {t.dtype} on {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def decode_gemm_bf16(x, W, out, stream=None, pdl=None, l2_prefetch=None, l2_after_reduce=None):
    """out[M, N] = x[M, K] @ W[N, K]^T on the current (or given) stream.

    x, W, out: contiguous CUDA bfloat16 tensors. Returns ``out``. pdl and
    l2_prefetch, when given, are this call's launch settings (decode_gemm_bf16_ex)
    instead of the process-wide ones; l2_after_reduce (weight blocks, 0..64) is
    for a call right behind decode_gemm_bf16_reduce_rmsnorm (see skinny.h).
    """
    _bf16_cuda(x, "x")
    _bf16_cuda(W, "W")
    if x.dim() != 2 or W.dim() != 2 or x.shape[1] != W.shape[1]:
        raise ValueError(f"x {tuple(x.shape)} and W {tuple(W.shape)} must be [M,K] and [N,K]")
    M, K = x.shape
    N = W.shape[0]
    _bf16_cuda(out, "out", (M, N))
    o = _opts(pdl, l2_prefetch, l2_after_reduce)
    lib = load_library()
    if o is None:
        st = lib.decode_gemm_bf16(x.data_ptr(), W.data_ptr(), out.data_ptr(), M, N, K,
                                  _stream_handle(stream))
    else:
        st = lib.decode_gemm_bf16_ex(x.data_ptr(), W.data_ptr(), out.data_ptr(), M, N, K,
                                     ctypes.byref(o), _stream_handle(stream))
    _check(st, "decode_gemm_bf16")
    return out


def decode_gemm_bf16_logits(x, W, out, soft_cap=0.0, scale=1.0, stream=None):
    """lm_head logits out[M, n_out] = scale * cap * tanh((x @ W[:n_out]^T) / cap)
    (no tanh if soft_cap <= 0); n_out = out.shape[1] <= W.shape[0]. Returns out."""
    _bf16_cuda(x, "x")
    _bf16_cuda(W, "W")
    _bf16_cuda(out, "out")
    if x.dim() != 2 or W.dim() != 2 or out.dim() != 2 or x.shape[1] != W.shape[1] \
            or out.shape[0] != x.shape[0]:
        raise ValueError("x [M,K], W [N,K] and out [M,n_out] do not fit together")
    M, K = x.shape
    N, n_out = W.shape[0], out.shape[1]
    st = load_library().decode_gemm_bf16_logits(x.data_ptr(), W.data_ptr(), out.data_ptr(), M,
                                                N, K, n_out, float(soft_cap), float(scale),
                                                _stream_handle(stream))
    _check(st, "decode_gemm_bf16_logits")
    return out


def reduce_residual_rmsnorm(partials, residual, gamma, out, residual_out, eps=1e-6,
                            stream=None, pdl=None):
    """(out, residual_out) of the rank-order reduce + residual + RMSNorm.

    partials [TP, M, 7168], residual [M, 7168] or None, gamma [7168],
    out and residual_out [M, 7168]; all contiguous CUDA bfloat16. pdl, when
    given, is this call's setting (reduce_residual_rmsnorm_ex).
    """
    _bf16_cuda(partials, "partials")
    if partials.dim() != 3 or partials.shape[2] != HIDDEN:
        raise ValueError(f"partials must be [TP, M, {HIDDEN}], got {tuple(partials.shape)}")
    TP, M, _ = partials.shape
    if residual is not None:
        _bf16_cuda(residual, "residual", (M, HIDDEN))
    _bf16_cuda(gamma, "gamma", (HIDDEN,))
    _bf16_cuda(out, "out", (M, HIDDEN))
    _bf16_cuda(residual_out, "residual_out", (M, HIDDEN))
    args = (partials.data_ptr(), TP, None if residual is None else residual.data_ptr(),
            gamma.data_ptr(), out.data_ptr(), residual_out.data_ptr(), M, float(eps))
    o = _opts(pdl, None)
    if o is None:
        st = load_library().reduce_residual_rmsnorm(*args, _stream_handle(stream))
    else:
        st = load_library().reduce_residual_rmsnorm_ex(*args, ctypes.byref(o),
                                                       _stream_handle(stream))
    _check(st, "reduce_residual_rmsnorm")
    return out, residual_out


def decode_gemm_bf16_reduce_rmsnorm(x, W, partials, residual, gamma, out, residual_out,
                                    eps=1e-6, stream=None, pdl=None, l2_prefetch=None):
    """The row-parallel linear with the reduce + residual + RMSNorm after it.

    x [M, K], W [7168, K]; partials [TP, M, 7168] (slot 0 receives x @ W^T,
    slots 1.. are read); residual [M, 7168] or None; gamma [7168]; out and
    residual_out [M, 7168]; all contiguous CUDA bfloat16. Returns
    (out, residual_out), bit for bit those of decode_gemm_bf16 followed by
    reduce_residual_rmsnorm. pdl and l2_prefetch as for decode_gemm_bf16.
    """
    _bf16_cuda(x, "x")
    _bf16_cuda(W, "W")
    _bf16_cuda(partials, "partials")
    if x.dim() != 2 or W.dim() != 2 or tuple(W.shape) != (HIDDEN, x.shape[1]):
        raise ValueError(f"x must be [M, K] and W [{HIDDEN}, K]")
    M, K = x.shape
    if partials.dim() != 3 or tuple(partials.shape[1:]) != (M, HIDDEN):
        raise ValueError(f"partials must be [TP, {M}, {HIDDEN}], got {tuple(partials.shape)}")
    TP = partials.shape[0]
    if residual is not None:
        _bf16_cuda(residual, "residual", (M, HIDDEN))
    _bf16_cuda(gamma, "gamma", (HIDDEN,))
    _bf16_cuda(out, "out", (M, HIDDEN))
    _bf16_cuda(residual_out, "residual_out", (M, HIDDEN))
    args = (x.data_ptr(), W.data_ptr(), partials.data_ptr(), TP,
            None if residual is None else residual.data_ptr(), gamma.data_ptr(), out.data_ptr(),
            residual_out.data_ptr(), M, K, float(eps))
    o = _opts(pdl, l2_prefetch)
    if o is None:
        st = load_library().decode_gemm_bf16_reduce_rmsnorm(*args, _stream_handle(stream))
    else:
        st = load_library().decode_gemm_bf16_reduce_rmsnorm_ex(*args, ctypes.byref(o),
                                                               _stream_handle(stream))
    _check(st, "decode_gemm_bf16_reduce_rmsnorm")
    return out, residual_out


def gather_shards_bf16(shards, out, stream=None):
    """out[M, TP*S] = the TP shards [TP, M, S] side by side (rank r at columns r*S..).

    shards, out: contiguous CUDA bfloat16 tensors. Returns ``out``.
    """
    _bf16_cuda(shards, "shards")
    if shards.dim() != 3:
        raise ValueError(f"shards must be [TP, M, S], got {tuple(shards.shape)}")
    TP, M, S = shards.shape
    _bf16_cuda(out, "out", (M, TP * S))
    st = load_library().gather_shards_bf16(shards.data_ptr(), TP, M, S, out.data_ptr(),
                                           _stream_handle(stream))
    _check(st, "gather_shards_bf16")
    return out


def device_error(device=None):
    """(status, word): read and clear the library's device error word."""
    import torch
    dev = torch.cuda.current_device() if device is None else int(device)
    word = ctypes.c_int(0)
    st = load_library().skinny_device_error(dev, ctypes.byref(word))
    return st, word.value


def set_pdl(enable: bool) -> bool:
    """Enable or disable programmatic dependent launch; returns the old setting."""
    return bool(load_library().skinny_set_pdl(1 if enable else 0))


def set_l2_prefetch(blocks: int) -> int:
    """Weight blocks the decode GEMM's deep ring prefetches to L2 before its PDL
    wait (skinny_set_l2_prefetch); returns the old value."""
    prev = load_library().skinny_set_l2_prefetch(int(blocks))
    if prev < 0:
        raise ValueError(f"l2 prefetch blocks must be in [0, 64], got {blocks}")
    return prev


def gemm_plan(M, N, K, num_sms) -> GemmPlan:
    plan = GemmPlan()
    _check(load_library().skinny_gemm_plan_query(M, N, K, num_sms, ctypes.byref(plan)),
           "skinny_gemm_plan_query")
    return plan


def gemm_cta_pieces(M, N, K, num_sms, cta, max_pieces=64):
    """[(tile, kb0, kb1, slot)] of one CTA of the decode GEMM's work split."""
    arrs = [(ctypes.c_int * max_pieces)() for _ in range(4)]
    n = load_library().skinny_gemm_cta_pieces(M, N, K, num_sms, cta, *arrs, max_pieces)
    if n < 0:
        raise ValueError("bad arguments to skinny_gemm_cta_pieces")
    return [tuple(a[i] for a in arrs) for i in range(min(n, max_pieces))]


def watchdog_selftest(x, W, out, timeout_ns, stream=None):
    """Launch the decode GEMM with a wait that can never complete (see skinny.h)."""
    M, K = x.shape
    N = W.shape[0]
    st = load_library().skinny_watchdog_selftest(x.data_ptr(), W.data_ptr(), out.data_ptr(),
                                                 M, N, K, int(timeout_ns),
                                                 _stream_handle(stream))
    _check(st, "skinny_watchdog_selftest")


def reduce_selftest(partials, residual, gamma, out, residual_out, eps, timeout_ns, stream=None):
    """Launch the reduce with a cluster exchange that can never complete (see skinny.h)."""
    _bf16_cuda(partials, "partials")
    if partials.dim() != 3 or partials.shape[2] != HIDDEN:
        raise ValueError(f"partials must be [TP, M, {HIDDEN}], got {tuple(partials.shape)}")
    TP, M, _ = partials.shape
    if residual is not None:
        _bf16_cuda(residual, "residual", (M, HIDDEN))
    _bf16_cuda(gamma, "gamma", (HIDDEN,))
    _bf16_cuda(out, "out", (M, HIDDEN))
    _bf16_cuda(residual_out, "residual_out", (M, HIDDEN))
    st = load_library().skinny_reduce_selftest(
        partials.data_ptr(), TP, residual.data_ptr() if residual is not None else None,
        gamma.data_ptr(), out.data_ptr(), residual_out.data_ptr(), M, float(eps),
        int(timeout_ns), _stream_handle(stream))
    _check(st, "skinny_reduce_selftest")
