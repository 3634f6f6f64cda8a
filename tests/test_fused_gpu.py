"""GPU parity of decode_gemm_bf16_reduce_rmsnorm: the row-parallel linear and the
TP reduce + residual + RMSNorm after it ("drafter/comm" module text: the
linear's TP all-reduce is fused with the RMSNorm that follows; ArNorm for the
arithmetic; "drafter/linears" DraftGemm for the GEMM), computed by a
publish-only GEMM and a reduce that finishes the split-K sums itself.

Against the two library calls it replaces: slot 0, residual_out and out bit for
bit (the same partials added in the same order, then the same reduce). Against
the oracle on the GPU's own inputs: slot 0 within the GEMM tolerance,
residual_out bit for bit, out within one ulp."""
import pytest
import torch

import oracle
from oracle import compare
import skinny_bf16_gemm_gb300 as sk
import workloads
from gpu_helpers import Guarded, check_gemm_full, check_gemm_sampled, sample_columns

pytestmark = pytest.mark.gpu

H = 7168
EPS = 1e-6


def inputs(M, K, TP, residual, seed):
    g = workloads.gemm_inputs(M, H, K, workloads.seed_for("fused-gemm", seed, M, K))
    r = workloads.reduce_inputs(TP, M, workloads.seed_for("fused-reduce", seed, M, TP), residual)
    return (g.x.cuda(), g.W.cuda(), r.partials.cuda(),
            None if r.residual is None else r.residual.cuda(), r.gamma.cuda())


def run_fused(x, W, partials, residual, gamma, in_place=False):
    M = x.shape[0]
    out = Guarded((M, H))
    rout = None if in_place else Guarded((M, H))
    sk.decode_gemm_bf16_reduce_rmsnorm(x, W, partials, residual, gamma, out.tensor,
                                       residual if in_place else rout.tensor, EPS)
    torch.cuda.synchronize()
    out.check()
    if rout is not None:
        rout.check()
    st, word = sk.device_error()
    assert st == 0 and word == 0, f"device error word {word}"
    return out.tensor, (residual if in_place else rout.tensor)


def run_two_calls(x, W, partials, residual, gamma):
    M = x.shape[0]
    sk.decode_gemm_bf16(x, W, partials[0])
    out = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(out)
    sk.reduce_residual_rmsnorm(partials, residual, gamma, out, rout, EPS)
    torch.cuda.synchronize()
    return out, rout


def same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


CASES = [(16, 18432, 8, True), (4, 7168, 8, True), (1, 1000, 2, False), (16, 64, 8, True),
         (7, 520, 1, True), (13, 2048, 4, False), (16, 14336, 8, False), (32, 7168, 8, True),
         (64, 4096, 2, True), (48, 18432, 8, False)]


@pytest.mark.parametrize("M,K,TP,res", CASES)
@pytest.mark.parametrize("pdl", [False, True])
def test_fused_equals_two_calls_and_oracle(cuda_ok, M, K, TP, res, pdl):
    x, W, partials, residual, gamma = inputs(M, K, TP, res, 0)
    prev = sk.set_pdl(pdl)
    try:
        pu = partials.clone()
        out_u, rout_u = run_two_calls(x, W, pu, residual, gamma)
        pf = partials.clone()
        out_f, rout_f = run_fused(x, W, pf, residual, gamma)
    finally:
        sk.set_pdl(prev)
    assert same_bits(pf, pu), "slots differ from decode_gemm_bf16's (or untouched slots moved)"
    assert same_bits(rout_f, rout_u), "residual_out differs"
    assert same_bits(out_f, out_u), "out differs"
    if pdl:
        return  # the oracle comparison below is the same for both settings
    if K <= 2048:
        check_gemm_full(x, W, pf[0])
    else:
        check_gemm_sampled(x, W, pf[0], sample_columns(H, count=256, seed=M))
    want_h = oracle.reduce_residual(workloads.bits(pf),
                                    None if residual is None else workloads.bits(residual))
    mism = compare.first_mismatch(workloads.bits(rout_f), want_h)
    assert mism is None, f"residual_out not bit-exact at {mism}"
    want_o = oracle.rmsnorm(want_h, workloads.bits(gamma), EPS)
    d = compare.ulp_distance(workloads.bits(out_f), want_o)
    assert int(d.max()) <= 1, compare.histogram(d)


def test_fused_in_place_residual_and_repeat(cuda_ok):
    x, W, partials, residual, gamma = inputs(16, 7168, 8, True, 1)
    out_a, rout_a = run_fused(x, W, partials.clone(), residual, gamma)
    res2 = residual.clone()
    out_b, rout_b = run_fused(x, W, partials.clone(), res2, gamma, in_place=True)
    assert same_bits(out_b, out_a) and same_bits(rout_b, rout_a)
    out_c, rout_c = run_fused(x, W, partials.clone(), residual, gamma)
    assert same_bits(out_c, out_a) and same_bits(rout_c, rout_a)


def test_fused_interleaved_with_plain_calls(cuda_ok):
    """The publish-only GEMM leaves no state behind: plain decode GEMMs before and
    after it (sharing the scratch) give the same bits as alone."""
    x, W, partials, residual, gamma = inputs(16, 18432, 8, True, 3)
    alone = torch.empty(16, H, dtype=torch.bfloat16, device="cuda")
    sk.decode_gemm_bf16(x, W, alone)
    torch.cuda.synchronize()
    prev = sk.set_pdl(True)
    try:
        outs = []
        for _ in range(3):
            o = torch.empty_like(alone)
            sk.decode_gemm_bf16(x, W, o)
            run_fused(x, W, partials.clone(), residual, gamma)
            outs.append(o)
        torch.cuda.synchronize()
    finally:
        sk.set_pdl(prev)
    for o in outs:
        assert same_bits(o, alone)


# Cases drawn once from a seeded generator (random.Random(7168): M from the row
# classes, K any multiple of 8 up to 19200, TP in 1..8, a residual or not), kept
# literal so that every run checks the same ones.
RANDOM_CASES = [(33, 10040, 6, True), (41, 9192, 8, True), (2, 4040, 6, True),
                (16, 9616, 6, False), (17, 11760, 7, True), (57, 12000, 7, True),
                (64, 14832, 6, False), (17, 6240, 5, True), (23, 10608, 5, False),
                (23, 6968, 4, True), (16, 8264, 4, True), (33, 13320, 3, True),
                (32, 16704, 5, True), (23, 1088, 7, False), (9, 32, 5, False),
                (32, 17128, 7, False)]


@pytest.mark.parametrize("i", range(len(RANDOM_CASES)))
def test_fused_random_cases_equal_two_calls(cuda_ok, i):
    """The fused call against the two calls it replaces, bit for bit (slots,
    residual_out, out), with PDL on every second case; residual_out against the
    oracle on the GPU's own slot 0."""
    M, K, TP, res = RANDOM_CASES[i]
    x, W, partials, residual, gamma = inputs(M, K, TP, res, 100 + i)
    prev = sk.set_pdl(i % 2 == 1)
    try:
        pu = partials.clone()
        out_u, rout_u = run_two_calls(x, W, pu, residual, gamma)
        pf = partials.clone()
        out_f, rout_f = run_fused(x, W, pf, residual, gamma)
    finally:
        sk.set_pdl(prev)
    assert same_bits(pf, pu) and same_bits(rout_f, rout_u) and same_bits(out_f, out_u)
    want_h = oracle.reduce_residual(workloads.bits(pf),
                                    None if residual is None else workloads.bits(residual))
    assert compare.first_mismatch(workloads.bits(rout_f), want_h) is None
