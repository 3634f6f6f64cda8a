"""Forward progress of the split-K hand-off without co-residency, on the GPU.

A test-only kernel (tests/cuda/occupy.cu, built here with nvcc) holds 120 KB of
shared memory on each of 100 SMs for a bounded 30 ms, so a decode GEMM launched
beside it finds room for its CTAs (185 KB with the deep ring, 112 KB with the
shallow one) on the other SMs only and runs in waves. A tile's finisher waits
only on CTAs with lower block indices (ranges dealt in reverse block order),
which the GPU dispatched before it, so the call completes -- with the bits of
the same call on an idle GPU and no recorded wait that ran out. Every wait in
both kernels is bounded: a mistake here shows as a timeout, not a hang."""
import ctypes
import os
import subprocess
import time

import pytest
import torch

import skinny_bf16_gemm_gb300 as sk
import workloads
from gpu_helpers import gemm_inputs_device

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def occupy(cuda_ok, tmp_path_factory):
    out = str(tmp_path_factory.mktemp("occupy") / "libocc.so")
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", "-o", out, os.path.join(HERE, "cuda", "occupy.cu")],
                   check=True)
    lib = ctypes.CDLL(out)
    lib.occupy_launch.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_ulonglong, ctypes.c_void_p]
    lib.occupy_launch.restype = ctypes.c_int
    return lib


def _timed_gemm(x, W, out, stream, pdl):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        sk.decode_gemm_bf16(x, W, out, stream=stream, pdl=pdl)
        b.record(stream)
    return a, b


@pytest.mark.parametrize("M,N,K,pdl", [(4, 2048, 7168, True), (16, 7168, 18432, False)])
def test_split_k_completes_with_most_sms_held(occupy, M, N, K, pdl):
    x, W = gemm_inputs_device(M, N, K, workloads.seed_for("occupy", M, N, K))
    gemm_stream, hold_stream = torch.cuda.Stream(), torch.cuda.Stream()
    ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        a, b = _timed_gemm(x, W, ref, gemm_stream, pdl)
    torch.cuda.synchronize()
    idle_ms = a.elapsed_time(b)
    assert sk.device_error() == (0, 0)

    out = torch.full_like(ref, 7.0)
    assert occupy.occupy_launch(100, 120 * 1024, 30_000_000, ctypes.c_void_p(hold_stream.cuda_stream)) == 0
    time.sleep(0.002)  # the holding blocks are resident before the GEMM launches
    a, b = _timed_gemm(x, W, out, gemm_stream, pdl)
    torch.cuda.synchronize()
    held_ms = a.elapsed_time(b)
    assert sk.device_error() == (0, 0)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # Evidence that the GEMM really ran on the remaining SMs, in waves.
    assert held_ms > 1.5 * idle_ms, (held_ms, idle_ms)
