"""GPU parity of the synthetic drafter layer chain, run the way the benchmark
times it: 3 layers of M = 16 rows, GEMM 7168 -> 18432, GEMM 18432 -> 7168 into
slot 0 of the TP = 8 partial rows, reduce + residual + RMSNorm, full-size weights
(264 MB per GEMM), all calls on one stream with programmatic dependent launch, so
each kernel overlaps the one before it ("drafter/comm" module text; "drafter/
linears" DraftGemm).

Every intermediate is kept in its own buffer and each stage is checked against
the oracle on the GPU's own inputs to that stage: the GEMMs on sampled output
columns (tolerance of oracle/compare.py), the reduce's residual_out bit for bit
and its RMSNorm output within one BF16 ulp, on whole rows."""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare
import skinny_bf16_gemm_gb300 as sk
from skinny_bf16_gemm_gb300.chain import LayerChain
import workloads
from gpu_helpers import check_gemm_sampled, sample_columns

pytestmark = pytest.mark.gpu

CFG = workloads.CHAIN


@pytest.fixture(scope="module")
def chain_inputs(cuda_ok):
    return workloads.chain_inputs(CFG, workloads.seed_for("chain-test"), device="cuda")


def check_reduce(partials, residual, gamma, out, res_out, eps):
    want_h = oracle.reduce_residual(workloads.bits(partials), workloads.bits(residual))
    mism = compare.first_mismatch(workloads.bits(res_out), want_h)
    assert mism is None, f"residual_out not bit-exact at {mism}"
    want_o = oracle.rmsnorm(want_h, workloads.bits(gamma), eps)
    d = compare.ulp_distance(workloads.bits(out), want_o)
    assert int(d.max()) <= 1, compare.histogram(d)


def test_chain_step_with_pdl_matches_oracle_stage_by_stage(chain_inputs):
    inp = chain_inputs
    bf = dict(dtype=torch.bfloat16, device="cuda")
    L, M = CFG.layers, CFG.M
    partials = []
    for l in range(L):
        buf = torch.empty(CFG.TP, M, CFG.hidden, **bf)
        buf[1:].copy_(inp.peers[l])
        partials.append(buf)
    h1 = [torch.empty(M, CFG.ffn, **bf) for _ in range(L)]
    outs = [torch.empty(M, CFG.hidden, **bf) for _ in range(L)]
    ress = [torch.empty(M, CFG.hidden, **bf) for _ in range(L)]
    torch.cuda.synchronize()
    prev = sk.set_pdl(True)
    try:
        # The benchmark's launch sequence, uninterrupted by any other kernel.
        x, res = inp.x0, inp.residual0
        for l in range(L):
            sk.decode_gemm_bf16(x, inp.W1[l], h1[l])
            sk.decode_gemm_bf16(h1[l], inp.W2[l], partials[l][0])
            sk.reduce_residual_rmsnorm(partials[l], res, inp.gamma[l], outs[l], ress[l], CFG.eps)
            x, res = outs[l], ress[l]
        torch.cuda.synchronize()
    finally:
        sk.set_pdl(prev)
    st, word = sk.device_error()
    assert st == 0 and word == 0
    x, res = inp.x0, inp.residual0
    for l in range(L):
        check_gemm_sampled(x, inp.W1[l], h1[l], sample_columns(CFG.ffn, count=256, seed=l))
        check_gemm_sampled(h1[l], inp.W2[l], partials[l][0],
                           sample_columns(CFG.hidden, count=256, seed=100 + l))
        check_reduce(partials[l], res, inp.gamma[l], outs[l], ress[l], CFG.eps)
        x, res = outs[l], ress[l]


@pytest.mark.parametrize("fused", [False, True])
def test_chain_eager_and_graph_replay_give_the_same_bits(chain_inputs, fused):
    """LayerChain (the benchmark's driver): an eager step with PDL, a second eager
    step and a CUDA-graph replay of the step all produce identical rows -- also
    fused, where each first GEMM waits (bounded) for the reduce's signal and
    prefetches after it, inside the graph too."""
    inp = chain_inputs
    chain = LayerChain(inp.W1, inp.W2, inp.peers, inp.gamma, CFG.M, CFG.eps, pdl=True,
                       fused=fused)
    chain.x.copy_(inp.x0)
    chain.res_in.copy_(inp.residual0)
    a_out, a_res = (t.clone() for t in chain.run())
    b_out, b_res = (t.clone() for t in chain.run())
    g_out, g_res = chain.capture()
    chain.replay()
    torch.cuda.synchronize()
    for got in (b_out, g_out):
        assert torch.equal(got.view(torch.int16), a_out.view(torch.int16))
    for got in (b_res, g_res):
        assert torch.equal(got.view(torch.int16), a_res.view(torch.int16))
    assert not compare.is_nonfinite(workloads.bits(a_out)).any()


def test_fused_chain_equals_unfused_chain(chain_inputs):
    """The chain with decode_gemm_bf16_reduce_rmsnorm for each layer's second GEMM
    and reduce gives the unfused chain's rows bit for bit, with or without PDL,
    whatever the decode GEMM's L2 lead and its prefetch after the reduce; the
    chain's per-call settings leave the process-wide ones as the caller set them."""
    inp = chain_inputs
    rows = []
    for fused, lead, pdl, after in ((False, 6, True, 16), (True, 0, True, 16),
                                    (True, 0, True, 0), (True, 6, False, 64),
                                    (False, 0, False, 16), (True, 0, False, 16)):
        chain = LayerChain(inp.W1, inp.W2, inp.peers, inp.gamma, CFG.M, CFG.eps, fused=fused,
                           l2_prefetch=lead, pdl=pdl, l2_after_reduce=after)
        chain.x.copy_(inp.x0)
        chain.res_in.copy_(inp.residual0)
        prev = sk.set_pdl(not pdl)
        prev_lead = sk.set_l2_prefetch(9)
        try:
            out, res = (t.clone() for t in chain.run())
            torch.cuda.synchronize()
            assert sk.set_l2_prefetch(prev_lead) == 9
            assert sk.set_pdl(prev) == (not pdl)
        finally:
            sk.set_pdl(prev)
            sk.set_l2_prefetch(prev_lead)
        rows.append((out, res))
    o0, r0 = rows[0]
    for o1, r1 in rows[1:]:
        assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
        assert torch.equal(r0.view(torch.int16), r1.view(torch.int16))
