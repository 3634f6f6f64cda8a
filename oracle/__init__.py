"""CPU oracle for the decode GEMM and the reduce + residual + RMSNorm.

TEST INFRASTRUCTURE ONLY: the plain, slow, obviously correct definitions the CUDA
path is checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library
(``skinny_bf16_gemm_gb300``) never imports it, and this package imports nothing
from the library. The arithmetic lives in ``oracle.c``; this module only moves
numpy arrays of BF16 bit patterns (``uint16``) in and out.

What each function follows (the vLLM DSpark drafter pages):

* ``decode_gemm`` -- "drafter/linears", module text and ``DraftGemm``:
  out[M,N] = x[M,K] @ weight[N,K]^T, BF16 operands, FP32 accumulation, one BF16
  rounding, cuBLAS's arithmetic in any order of additions. Reading: the exact
  product sum (binary64 here) rounded once to BF16, ties to even.
* ``reduce_residual`` -- "drafter/comm", ``ArNorm`` docstring and kernel, and
  "cutedsl/common/twoshot" ``reduce``: FP32 sum of the TP partials in rank order
  0..TP-1 from slot 0, one BF16 rounding, FP32 add of the residual, one BF16
  rounding. Bit-exact by definition.
* ``rmsnorm`` -- "drafter/comm" module text (a sum of squares in FP32, the
  reciprocal square root of its mean over 7168 columns plus eps, the product
  x * rstd * gamma rounded once) and ``ArNorm.kernel``'s last block.
  Evaluated in binary64 and rounded once.
* ``decode_gemm_logits`` -- "drafter/linears", ``draft_logits``: the lm_head GEMM
  sliced to its first n_out (org_vocab_size) columns, optional tanh soft cap,
  scale; binary64, one rounding (the fused-epilogue reading of the pages' BF16
  ops).
* ``gather_shards`` -- "drafter/comm", ``Gather`` docstring and module text:
  every rank's [M, S] shard at columns r*S.. of the [M, TP*S] row; a byte move.
* ``rmsnorm_f32_steps`` -- diagnostic: the same formula in the binary32 steps the
  kernel lists; never a parity reference.
"""
import ctypes
import os

import numpy as np

from . import build as _build

HIDDEN = 7168  # the row width of every ArNorm row ("drafter/comm", ArNorm docstring)

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i32p = ctypes.POINTER(ctypes.c_int)
        lib.oracle_bf16_from_f64.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_f64.restype = ctypes.c_uint16
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_decode_gemm.argtypes = [u16p, u16p, u16p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int]
        lib.oracle_decode_gemm.restype = None
        lib.oracle_bf16_from_f64_array.argtypes = [ctypes.POINTER(ctypes.c_double), u16p,
                                                    ctypes.c_long]
        lib.oracle_bf16_from_f64_array.restype = None
        f64p = ctypes.POINTER(ctypes.c_double)
        lib.oracle_decode_gemm_f64.argtypes = [u16p, u16p, f64p, f64p, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int,
                                               ctypes.c_int]
        lib.oracle_decode_gemm_f64.restype = None
        lib.oracle_reduce_residual.argtypes = [u16p, ctypes.c_int, u16p, u16p,
                                               ctypes.c_int, ctypes.c_int]
        lib.oracle_reduce_residual.restype = None
        for name in ("oracle_rmsnorm", "oracle_rmsnorm_f32_steps"):
            fn = getattr(lib, name)
            fn.argtypes = [u16p, u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_float]
            fn.restype = None
        lib.oracle_decode_gemm_logits.argtypes = [u16p, u16p, u16p, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                  ctypes.c_double, ctypes.c_int]
        lib.oracle_decode_gemm_logits.restype = None
        lib.oracle_gather_shards.argtypes = [u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, u16p]
        lib.oracle_gather_shards.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _u16(a, shape=None):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def bf16_from_f64(v: float) -> int:
    """Nearest BF16 pattern to the binary64 value ``v`` (ties to even)."""
    return int(_load().oracle_bf16_from_f64(float(v)))


def bf16_to_f64(bits: int) -> float:
    """The value of a BF16 pattern, exactly."""
    return float(_load().oracle_bf16_to_f64(int(bits) & 0xFFFF))


def bf16_from_f64_array(v) -> np.ndarray:
    """Element-wise ``bf16_from_f64`` over an array of binary64 values."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_bf16_from_f64_array(v.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                       _ptr(out), v.size)
    return out


def decode_gemm_f64(x, W, cols=None, threads=0):
    """(sum, abs_sum): the unrounded binary64 sums behind ``decode_gemm`` and
    sum_k |x[m,k] W[n,k]| beside each, [M, len(cols)] (all columns if None)."""
    x = _u16(x)
    W = _u16(W)
    M, K = x.shape
    N, K2 = W.shape
    if K2 != K:
        raise ValueError("x and W disagree on K")
    c = np.arange(N, dtype=np.int32) if cols is None else np.ascontiguousarray(cols, np.int32)
    if c.size and (c.min() < 0 or c.max() >= N):
        raise ValueError("column index out of range")
    s = np.empty((M, c.size), dtype=np.float64)
    a = np.empty((M, c.size), dtype=np.float64)
    f64p = ctypes.POINTER(ctypes.c_double)
    _load().oracle_decode_gemm_f64(_ptr(x), _ptr(W), s.ctypes.data_as(f64p),
                                   a.ctypes.data_as(f64p), M, N, K,
                                   c.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), c.size,
                                   threads)
    return s, a


def decode_gemm(x, W, cols=None, threads=0):
    """BF16 patterns out[M, N] (or out[M, len(cols)]) of x[M, K] @ W[N, K]^T.

    ``cols`` selects output columns (weight rows) for sampled checks of
    full-size problems; ``threads`` caps OpenMP (0 = its default).
    """
    x = _u16(x)
    W = _u16(W)
    M, K = x.shape
    N, K2 = W.shape
    if K2 != K:
        raise ValueError("x and W disagree on K")
    if cols is None:
        out = np.empty((M, N), dtype=np.uint16)
        _load().oracle_decode_gemm(_ptr(x), _ptr(W), _ptr(out), M, N, K, None, 0, threads)
        return out
    c = np.ascontiguousarray(cols, dtype=np.int32)
    if c.size and (c.min() < 0 or c.max() >= N):
        raise ValueError("column index out of range")
    out = np.empty((M, c.size), dtype=np.uint16)
    _load().oracle_decode_gemm(_ptr(x), _ptr(W), _ptr(out), M, N, K,
                               c.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), c.size,
                               threads)
    return out


def decode_gemm_logits(x, W, n_out=None, soft_cap=0.0, scale=1.0, threads=0):
    """BF16 patterns [M, n_out] of scale * cap * tanh((x @ W[:n_out]^T) / cap)
    (no tanh when soft_cap <= 0), binary64, one rounding."""
    x = _u16(x)
    W = _u16(W)
    M, K = x.shape
    N, K2 = W.shape
    if K2 != K:
        raise ValueError("x and W disagree on K")
    n_out = N if n_out is None else int(n_out)
    if not 1 <= n_out <= N:
        raise ValueError("n_out out of range")
    out = np.empty((M, n_out), dtype=np.uint16)
    _load().oracle_decode_gemm_logits(_ptr(x), _ptr(W), _ptr(out), M, N, K, n_out,
                                      float(soft_cap), float(scale), threads)
    return out


def reduce_residual(partials, residual=None):
    """BF16 patterns residual_out[M, width] of the rank-order reduce (+ residual)."""
    p = _u16(partials)
    TP, M, width = p.shape
    res = None if residual is None else _u16(residual, (M, width))
    out = np.empty((M, width), dtype=np.uint16)
    _load().oracle_reduce_residual(_ptr(p), TP, None if res is None else _ptr(res),
                                   _ptr(out), M, width)
    return out


def rmsnorm(h, gamma, eps):
    """BF16 patterns of RMSNorm(h) * gamma, binary64 evaluation, one rounding."""
    h = _u16(h)
    M, width = h.shape
    g = _u16(gamma, (width,))
    out = np.empty((M, width), dtype=np.uint16)
    _load().oracle_rmsnorm(_ptr(h), _ptr(g), _ptr(out), M, width, float(eps))
    return out


def rmsnorm_f32_steps(h, gamma, eps):
    """Diagnostic binary32-step RMSNorm (see module docstring)."""
    h = _u16(h)
    M, width = h.shape
    g = _u16(gamma, (width,))
    out = np.empty((M, width), dtype=np.uint16)
    _load().oracle_rmsnorm_f32_steps(_ptr(h), _ptr(g), _ptr(out), M, width, float(eps))
    return out


def reduce_residual_rmsnorm(partials, residual, gamma, eps):
    """(out, residual_out): the whole row op -- reduce, residual, then RMSNorm."""
    h = reduce_residual(partials, residual)
    return rmsnorm(h, gamma, eps), h


def gather_shards(shards):
    """[M, TP * S] rows from [TP, M, S] shards, rank r at columns r*S.."""
    sh = _u16(shards)
    TP, M, S = sh.shape
    out = np.empty((M, TP * S), dtype=np.uint16)
    _load().oracle_gather_shards(_ptr(sh), TP, M, S, _ptr(out))
    return out


def max_threads() -> int:
    """Threads OpenMP gives the GEMM loop (what a timing of it actually used)."""
    return int(_load().oracle_max_threads())
