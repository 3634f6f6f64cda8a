"""GPU parity of decode_gemm_bf16_logits (the lm_head GEMM with the slice, tanh
soft cap and scale of "drafter/linears", draft_logits, fused into its epilogue),
through the C ABI, against the oracle's binary64 logits rounded once.

Tolerance: the decode GEMM's (oracle/compare.py), with the cancellation floor
carried through the epilogue (|d/dv scale*cap*tanh(v/cap)| <= |scale|)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare
import skinny_bf16_gemm_gb300 as sk
import workloads
from gpu_helpers import Guarded, gemm_inputs_device, sample_columns

pytestmark = pytest.mark.gpu


def run_logits(x, W, n_out, cap, scale):
    out = Guarded((x.shape[0], n_out))
    sk.decode_gemm_bf16_logits(x, W, out.tensor, cap, scale)
    torch.cuda.synchronize()
    out.check()
    assert sk.device_error() == (0, 0)
    return out.tensor


def check(x, W_rows, got, cap, scale):
    xb, wb = workloads.bits(x), workloads.bits(W_rows)
    ref = oracle.decode_gemm_logits(xb, wb, wb.shape[0], cap, scale)
    s, a = oracle.decode_gemm_f64(xb, wb)
    v = np.tanh(s / cap) * cap if cap > 0 else s
    rep = compare.gemm_check(got, ref, v * scale, a * abs(scale))
    assert rep["ok"], rep
    return rep


@pytest.mark.parametrize("M,N,K,n_out,cap,scale", [
    (4, 1000, 7168, 900, 30.0, 0.5), (16, 300, 200, 300, 0.0, 2.0), (1, 129, 72, 100, 1.0, 1.0),
    (32, 512, 1024, 512, 5.0, -0.25), (64, 257, 520, 250, 30.0, 1.0),
    (8, 2048, 7168, 2000, 30.0, 0.5)])  # the last one runs the cluster plan on a GB300
def test_logits_small_full(cuda_ok, M, N, K, n_out, cap, scale):
    x, W = gemm_inputs_device(M, N, K, workloads.seed_for("logits", M, N, K))
    x = (x.float() * 8).to(torch.bfloat16)  # logits of a few units: the cap bends them
    got = run_logits(x, W, n_out, cap, scale)
    check(x, W[:n_out], workloads.bits(got), cap, scale)


@pytest.mark.parametrize("M", [1, 8, 32])
def test_logits_lm_head_sampled(cuda_ok, M):
    """The lm_head shape (N = 20480, K = 7168) sliced to 20000 columns, cap 30."""
    N, K, n_out, cap, scale = 20480, 7168, 20000, 30.0, 0.5
    x, W = gemm_inputs_device(M, N, K, workloads.seed_for("lm_head_logits", M))
    x = (x.float() * 8).to(torch.bfloat16)
    got = workloads.bits(run_logits(x, W, n_out, cap, scale))
    cols = sample_columns(n_out, seed=M)
    idx = torch.as_tensor(cols, device=W.device, dtype=torch.long)
    check(x, W[idx], got[:, cols], cap, scale)


def test_logits_without_epilogue_equal_the_gemm(cuda_ok):
    x, W = gemm_inputs_device(8, 1024, 7168, 5)
    plain = torch.empty(8, 1024, dtype=torch.bfloat16, device="cuda")
    sk.decode_gemm_bf16(x, W, plain)
    got = run_logits(x, W, 1000, 0.0, 1.0)
    assert torch.equal(got.view(torch.int16), plain[:, :1000].view(torch.int16))


def test_logits_rejects_bad_arguments(cuda_ok):
    lib = sk.load_library()
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(4, 16, dtype=torch.bfloat16, device="cuda")
    f = lib.decode_gemm_bf16_logits
    assert f(x.data_ptr(), W.data_ptr(), out.data_ptr(), 4, 16, 64, 17, 0.0, 1.0, None) == 2
    assert f(x.data_ptr(), W.data_ptr(), out.data_ptr(), 4, 16, 64, 0, 0.0, 1.0, None) == 2
    assert f(x.data_ptr(), W.data_ptr(), out.data_ptr(), 4, 16, 64, 8, float("nan"), 1.0, None) == 10
    assert f(x.data_ptr(), W.data_ptr(), out.data_ptr(), 4, 16, 64, 8, 0.0, float("inf"), None) == 10


# Cases drawn once from a seeded generator (random.Random(20480): M from the row
# classes, N and n_out <= N any, K any multiple of 8 up to 9600, a cap of 0, 1,
# 5 or 30, a scale of 1, 0.5, -0.25 or 2), kept literal.
RANDOM_LOGITS = [(3, 16243, 776, 695, 0.0, 0.5), (64, 1791, 2976, 1534, 0.0, 1.0),
                 (1, 7103, 2936, 5327, 1.0, 0.5), (3, 14649, 8816, 2591, 5.0, 1.0),
                 (32, 15619, 304, 8576, 0.0, 2.0), (64, 231, 7672, 23, 1.0, 0.5),
                 (3, 12435, 1560, 9775, 30.0, 1.0), (1, 14338, 2296, 5809, 0.0, 1.0),
                 (3, 2608, 8656, 2087, 30.0, 1.0), (8, 18002, 1544, 15828, 0.0, 1.0)]


@pytest.mark.parametrize("M,N,K,n_out,cap,scale", RANDOM_LOGITS)
def test_logits_random_cases_every_element(cuda_ok, M, N, K, n_out, cap, scale):
    x, W = gemm_inputs_device(M, N, K, workloads.seed_for("logits random", M, N, K))
    x = (x.float() * 8).to(torch.bfloat16)
    got = run_logits(x, W, n_out, cap, scale)
    check(x, W[:n_out], workloads.bits(got), cap, scale)
