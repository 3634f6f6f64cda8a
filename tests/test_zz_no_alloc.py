"""decode_gemm_bf16_noalloc against decode_gemm_bf16, on the GPU, through the C ABI.

The allocation-free entry point serves callers that must not have a library call
cudaMalloc behind their back -- code running during a strict CUDA graph capture,
serving engines that hand all spare device memory to their own pool, plug-ins
tied to their host framework's allocator. It runs the same kernel with its
split-K scratch in one static device array that every call reuses, so it is
checked here call after call against the regular entry point, within the decode
GEMM tolerance the other tests use. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import compare
import skinny_bf16_gemm_gb300 as sk
import workloads
from gpu_helpers import gemm_inputs_device

pytestmark = pytest.mark.gpu


def _entry_point():
    fn = sk.load_library().decode_gemm_bf16_noalloc
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


# Shapes whose tiles are split across many CTAs (the scratch is used) and one
# with ragged N and K tails; M spans both MMA widths.
@pytest.mark.parametrize("M,N,K", [(16, 2048, 7168), (32, 640, 1000), (3, 4096, 7168)])
def test_noalloc_matches_regular_entry_point_twice(cuda_ok, M, N, K):
    fn = _entry_point()
    x, W = gemm_inputs_device(M, N, K, workloads.seed_for("noalloc", M, N, K))
    ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    sk.decode_gemm_bf16(x, W, ref)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs = []
    for _ in range(2):  # the second call reuses the scratch the first one left
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        status = fn(x.data_ptr(), W.data_ptr(), out.data_ptr(), M, N, K, stream)
        assert status == 0, sk.status_string(status)
        outs.append(out)
    torch.cuda.synchronize()
    exact, abs_sum = oracle.decode_gemm_f64(workloads.bits(x), workloads.bits(W))
    want = workloads.bits(ref)
    for out in outs:
        rep = compare.gemm_check(workloads.bits(out), want, exact, abs_sum)
        assert rep["ok"], rep
    assert np.array_equal(workloads.bits(outs[0]), workloads.bits(outs[1]))


def test_noalloc_rejects_rows_beyond_its_slots(cuda_ok):
    fn = _entry_point()
    x = torch.zeros(33, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(33, 16, dtype=torch.bfloat16, device="cuda")
    assert fn(x.data_ptr(), W.data_ptr(), out.data_ptr(), 33, 16, 64, None) == 2
