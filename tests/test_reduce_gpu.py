"""GPU parity of reduce_residual_rmsnorm with the oracle, through the C ABI.

residual_out must be bit-exact (sign of zero included); out within one BF16 ulp
("drafter/comm": the rank-order FP32 sum, one rounding, residual add, one
rounding; RMSNorm rounded once)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare
import skinny_bf16_gemm_gb300 as sk
import workloads
from gpu_helpers import Guarded

pytestmark = pytest.mark.gpu

HIDDEN = 7168


def run_reduce(partials, residual, gamma, eps=1e-6, in_place=False):
    TP, M, _ = partials.shape
    out = Guarded((M, HIDDEN))
    if in_place:
        res_out = residual
    else:
        res_out = Guarded((M, HIDDEN))
    sk.reduce_residual_rmsnorm(partials, residual, gamma, out.tensor,
                               res_out if in_place else res_out.tensor, eps)
    torch.cuda.synchronize()
    out.check()
    if not in_place:
        res_out.check()
        return out.tensor, res_out.tensor
    return out.tensor, res_out


def check_against_oracle(inp, out, res_out, eps=1e-6):
    p = workloads.bits(inp.partials)
    r = None if inp.residual is None else workloads.bits(inp.residual)
    want_h = oracle.reduce_residual(p, r)
    got_h = workloads.bits(res_out)
    mism = compare.first_mismatch(got_h, want_h)
    assert mism is None, f"residual_out not bit-exact at {mism}"
    want_o = oracle.rmsnorm(want_h, workloads.bits(inp.gamma), eps)
    d = compare.ulp_distance(workloads.bits(out), want_o)
    assert not compare.is_nonfinite(workloads.bits(out)).any()
    assert int(d.max()) <= 1, compare.histogram(d)
    return compare.histogram(d)


SWEEP = [(tp, m, res) for tp in (2, 4, 8) for m in (1, 4, 8, 16, 32, 64) for res in (True, False)]


@pytest.mark.parametrize("TP,M,res", SWEEP)
def test_reduce_sweep(cuda_ok, TP, M, res):
    inp = workloads.reduce_inputs(TP, M, workloads.seed_for("reduce", TP, M, res), res,
                                  device="cuda")
    out, res_out = run_reduce(inp.partials, inp.residual, inp.gamma)
    check_against_oracle(inp, out, res_out)


@pytest.mark.parametrize("TP,M", [(1, 1), (1, 5), (3, 2), (5, 7), (7, 63), (8, 64)])
def test_reduce_odd_shapes(cuda_ok, TP, M):
    for res in (True, False):
        inp = workloads.reduce_inputs(TP, M, workloads.seed_for("odd", TP, M, res), res,
                                      device="cuda")
        out, res_out = run_reduce(inp.partials, inp.residual, inp.gamma)
        check_against_oracle(inp, out, res_out)


def test_reduce_pr1_case(cuda_ok):
    """PR1: TP=8, M=4, residual given, eps=1e-6, seed 0."""
    inp = workloads.reduce_inputs(8, 4, 0, True, device="cuda")
    out, res_out = run_reduce(inp.partials, inp.residual, inp.gamma)
    check_against_oracle(inp, out, res_out)


def test_tp1_without_residual_is_identity(cuda_ok):
    inp = workloads.reduce_inputs(1, 3, 5, False, device="cuda")
    p = inp.partials.clone()
    p.view(torch.int16)[0, 0, :64] = int(np.int16(np.uint16(0x8000).view(np.int16)))
    _, res_out = run_reduce(p, None, inp.gamma)
    assert torch.equal(res_out.view(torch.int16), p[0].view(torch.int16))


def test_stored_golden_columns(cuda_ok):
    """The stored order / signed-zero / overflow columns, placed into full rows
    (one column each, the rest random), are reproduced bit for bit."""
    from oracle_pins import read_cases
    rows = read_cases("reduce_cases.txt")
    for i, row in enumerate(rows):
        slots_s, res_s, want_s = [p.strip() for p in row.split("|")]
        slots = [int(t, 16) for t in slots_s.split()]
        TP = len(slots)
        has_res = res_s != "-"
        inp = workloads.reduce_inputs(TP, 2, workloads.seed_for("golden", i), has_res)
        p = workloads.bits(inp.partials).copy()
        col = 37 + 101 * i
        p[:, 1, col] = slots
        r = None
        if has_res:
            r = workloads.bits(inp.residual).copy()
            r[1, col] = int(res_s, 16)
        pt = workloads.from_bits(p).cuda()
        rt = None if r is None else workloads.from_bits(r).cuda()
        _, res_out = run_reduce(pt, rt, inp.gamma.cuda())
        got = workloads.bits(res_out)
        assert int(got[1, col]) == int(want_s, 16), f"case {row}"
        mism = compare.first_mismatch(got, oracle.reduce_residual(p, r))
        assert mism is None


def test_in_place_residual(cuda_ok):
    inp = workloads.reduce_inputs(4, 8, 17, True, device="cuda")
    want = oracle.reduce_residual(workloads.bits(inp.partials), workloads.bits(inp.residual))
    res = inp.residual.clone()
    out, res_out = run_reduce(inp.partials, res, inp.gamma, in_place=True)
    assert compare.first_mismatch(workloads.bits(res_out), want) is None


def test_order_sensitive_rows(cuda_ok):
    """Rows built so that the FP32 sum depends on the order of the slots: only the
    rank order 0..TP-1 gives the oracle's bits."""
    rng = np.random.default_rng(3)
    TP, M = 8, 4
    big = (rng.standard_normal((M, HIDDEN)) * 64).astype(np.float32)
    parts = np.zeros((TP, M, HIDDEN), dtype=np.float32)
    parts[0] = big
    parts[1] = -big
    parts[2:] = rng.standard_normal((TP - 2, M, HIDDEN)).astype(np.float32) * 2.0 ** -12
    # shuffle which slot holds the big pair per column
    for c in range(0, HIDDEN, 3):
        perm = rng.permutation(TP)
        parts[:, :, c] = parts[perm, :, c]
    p = workloads.to_bf16(parts)
    inp = workloads.ReduceInputs(p.cuda(), None, workloads.to_bf16(
        np.ones(HIDDEN, dtype=np.float32)).cuda())
    out, res_out = run_reduce(inp.partials, None, inp.gamma)
    check_against_oracle(inp, out, res_out)
    # the reversed-order sum differs on many columns: the test can see order
    rev = oracle.reduce_residual(workloads.bits(p)[::-1].copy())
    assert int((rev != workloads.bits(res_out)).sum()) > 100


def test_repeat_calls_identical(cuda_ok):
    inp = workloads.reduce_inputs(8, 16, 9, True, device="cuda")
    a = run_reduce(inp.partials, inp.residual, inp.gamma)
    b = run_reduce(inp.partials, inp.residual, inp.gamma)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))


def test_rejects_host_memory(cuda_ok):
    inp = workloads.reduce_inputs(2, 1, 1, True)
    outs = torch.empty(2, 1, HIDDEN, dtype=torch.bfloat16)  # host memory
    lib = sk.load_library()
    st = lib.reduce_residual_rmsnorm(inp.partials.data_ptr(), 2, inp.residual.data_ptr(),
                                     inp.gamma.data_ptr(), outs[0].data_ptr(),
                                     outs[1].data_ptr(), 1, 1e-6, None)
    assert st == 4
