"""decode_gemm_bf16_noalloc on the GPU, through the C ABI, against the regular
entry point and the oracle.

Some callers cannot let a library allocate device memory behind their back: a
serving engine that hands all spare device memory to its own pool at start-up
(a later cudaMalloc fails, or forces the pool to give memory back), a plug-in
that may only take memory from its host framework's allocator, a loop that
cannot afford cudaMalloc's implicit device synchronisation. The allocation-free
entry point runs the same kernel with its split-K scratch in one static device
array that every call reuses, so each call here is checked twice: bit for bit
against decode_gemm_bf16 (same kernel, same work split whenever the GPU has at
most 160 SMs, as a GB300 does), and within the decode GEMM tolerance against the
oracle. Two calls in a row show that a call starts clean from the array's
previous contents. This file is collected last on purpose.
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

STATIC_MAX_CTAS = 160  # CTAs the static array holds partial tiles for


def _entry_point():
    fn = sk.load_library().decode_gemm_bf16_noalloc
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


# Shapes whose tiles are split across many CTAs (the scratch is used) and one
# with ragged N and K tails; M spans both MMA widths.
@pytest.mark.parametrize("M,N,K", [(16, 2048, 7168), (32, 640, 1000), (3, 4096, 7168)])
def test_noalloc_matches_regular_entry_point_and_oracle_twice(cuda_ok, M, N, K):
    fn = _entry_point()
    x, W = gemm_inputs_device(M, N, K, workloads.seed_for("noalloc", M, N, K))
    ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    sk.decode_gemm_bf16(x, W, ref)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs = []
    for _ in range(2):  # the second call starts from what the first left in the array
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        status = fn(x.data_ptr(), W.data_ptr(), out.data_ptr(), M, N, K, stream)
        assert status == 0, sk.status_string(status)
        outs.append(out)
    torch.cuda.synchronize()
    xb, wb = workloads.bits(x), workloads.bits(W)
    want = oracle.decode_gemm(xb, wb)
    exact, abs_sum = oracle.decode_gemm_f64(xb, wb)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    same_split = sk.gemm_plan(M, N, K, sms).ctas <= STATIC_MAX_CTAS
    for out in outs:
        got = workloads.bits(out)
        rep = compare.gemm_check(got, want, exact, abs_sum)
        assert rep["ok"], rep
        if same_split:
            assert compare.bits_equal(got, workloads.bits(ref)), compare.first_mismatch(
                got, workloads.bits(ref))
    assert np.array_equal(workloads.bits(outs[0]), workloads.bits(outs[1]))


def test_noalloc_rejects_rows_beyond_its_slots(cuda_ok):
    fn = _entry_point()
    x = torch.zeros(33, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(33, 16, dtype=torch.bfloat16, device="cuda")
    assert fn(x.data_ptr(), W.data_ptr(), out.data_ptr(), 33, 16, 64, None) == 2
