"""The decode GEMM's bounded waits on the GPU: a wait that can never complete ends
with a recorded status instead of a hang, the kernel cleans up after itself
(in-flight copies drained, tensor memory freed), later calls that use the
split-K scratch report the timeout (SKINNY_ERR_TIMEOUT, nothing launched) until
the error is read and cleared, and the context stays usable -- the next regular
call returns the right bits. Nothing here faults or traps."""
import pytest
import torch

import skinny_bf16_gemm_gb300 as sk
import workloads
from gpu_helpers import gemm_inputs_device

pytestmark = pytest.mark.gpu

SELFTEST_BIT = 32  # the self-test's deliberate wait ran out


def _gemm(x, W):
    out = torch.empty(x.shape[0], W.shape[0], dtype=torch.bfloat16, device="cuda")
    sk.decode_gemm_bf16(x, W, out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("M,N,K", [(4, 2048, 7168), (32, 18432, 7168)])
def test_bounded_wait_reports_and_recovers(cuda_ok, M, N, K):
    x, W = gemm_inputs_device(M, N, K, workloads.seed_for("watchdog", M, N, K))
    ref = _gemm(x, W)
    assert sk.device_error() == (0, 0)

    junk = torch.empty_like(ref)
    sk.watchdog_selftest(x, W, junk, timeout_ns=2_000_000)  # 2 ms limit
    torch.cuda.synchronize()
    # The timeout is visible to the host without reading the error word: calls
    # that would use the scratch refuse to launch.
    untouched = torch.full_like(ref, 3.0)
    with pytest.raises(sk.SkinnyError) as e:
        sk.decode_gemm_bf16(x, W, untouched)
    assert e.value.status == 9
    with pytest.raises(sk.SkinnyError) as e:
        sk.decode_gemm_bf16(x, W, untouched, pdl=True, l2_prefetch=0)
    assert e.value.status == 9
    torch.cuda.synchronize()
    assert bool((untouched.float() == 3.0).all())
    status, word = sk.device_error()
    assert status == 9, sk.status_string(status)
    assert word & SELFTEST_BIT

    again = _gemm(x, W)
    assert sk.device_error() == (0, 0)
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))


def test_selftest_rejects_out_of_range_limits(cuda_ok):
    x, W = gemm_inputs_device(1, 16, 64, 3)
    out = torch.empty(1, 16, dtype=torch.bfloat16, device="cuda")
    for bad in (0, 999, 3_000_000_000):
        with pytest.raises(sk.SkinnyError):
            sk.watchdog_selftest(x, W, out, timeout_ns=bad)


REDUCE_EXCHANGE_BIT = 128  # a reduce cluster's wait for its CTA sums ran out


def test_reduce_exchange_wait_reports_and_recovers(cuda_ok):
    """The reduce's bounded wait for its cluster's sums of squares: a cluster
    whose last CTA never sends its sum ends every wait after the limit, the
    host reads bit 128 once, and the next reduce returns the right bits."""
    TP, M = 8, 16
    inp = workloads.reduce_inputs(TP, M, workloads.seed_for("reduce watchdog", TP, M), True,
                                  device=torch.device("cuda"))
    out = torch.empty(M, workloads.HIDDEN, dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(out)
    sk.reduce_residual_rmsnorm(inp.partials, inp.residual, inp.gamma, out, rout, 1e-6)
    torch.cuda.synchronize()
    ref, rref = out.clone(), rout.clone()
    assert sk.device_error() == (0, 0)

    junk, rjunk = torch.empty_like(out), torch.empty_like(rout)
    sk.reduce_selftest(inp.partials, inp.residual, inp.gamma, junk, rjunk, 1e-6,
                       timeout_ns=5_000_000)  # 5 ms limit
    torch.cuda.synchronize()
    status, word = sk.device_error()
    assert status == 9, sk.status_string(status)
    assert word == REDUCE_EXCHANGE_BIT
    assert sk.device_error() == (0, 0)

    out.zero_()
    rout.zero_()
    sk.reduce_residual_rmsnorm(inp.partials, inp.residual, inp.gamma, out, rout, 1e-6)
    torch.cuda.synchronize()
    assert sk.device_error() == (0, 0)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(rout.view(torch.int16), rref.view(torch.int16))


def test_reduce_selftest_rejects_out_of_range_limits(cuda_ok):
    TP, M = 8, 1
    inp = workloads.reduce_inputs(TP, M, 5, False, device=torch.device("cuda"))
    out = torch.empty(M, workloads.HIDDEN, dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(out)
    for bad in (0, 999, 3_000_000_000):
        with pytest.raises(sk.SkinnyError):
            sk.reduce_selftest(inp.partials, None, inp.gamma, out, rout, 1e-6, timeout_ns=bad)
