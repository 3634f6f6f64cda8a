"""Shared pieces of the GPU parity tests: guard-banded outputs, seeded inputs
copied to the device, and the oracle comparisons."""
import numpy as np
import torch

import oracle
from oracle import compare
import workloads

CANARY = 0x5A5A
GUARD = 4096  # elements of canary before and after every output


class Guarded:
    """A contiguous CUDA bf16 tensor of `shape` inside a larger buffer whose
    guard bands hold a canary pattern; ``check()`` asserts they are untouched."""

    def __init__(self, shape, device="cuda", fill=None):
        n = int(np.prod(shape))
        self.n = n
        self.buf = torch.empty(n + 2 * GUARD, dtype=torch.int16, device=device)
        self.buf.fill_(CANARY)
        inner = self.buf[GUARD:GUARD + n]
        if fill is not None:
            inner.copy_(fill.reshape(-1).view(torch.int16))
        self.tensor = inner.view(torch.bfloat16).view(*shape)

    def check(self):
        head = self.buf[:GUARD].cpu().numpy()
        tail = self.buf[GUARD + self.n:].cpu().numpy()
        assert np.all(head == CANARY) and np.all(tail == CANARY), "guard band overwritten"


def gemm_inputs_device(M, N, K, seed, kind="normal"):
    """(x, W) on the GPU, generated from the seeded host generator."""
    inp = workloads.gemm_inputs(M, N, K, seed, kind=kind)
    return inp.x.cuda(), inp.W.cuda()


def check_gemm_full(x, W, out, exact_bits_required=False):
    """Compare a whole GEMM result with the oracle. Returns the report dict."""
    xb, wb = workloads.bits(x), workloads.bits(W)
    got = workloads.bits(out)
    ref = oracle.decode_gemm(xb, wb)
    if exact_bits_required:
        mism = compare.first_mismatch(got, ref)
        assert mism is None, f"not bit-exact: {mism}"
        return {"ok": True}
    s, a = oracle.decode_gemm_f64(xb, wb)
    rep = compare.gemm_check(got, ref, s, a)
    assert rep["ok"], rep
    return rep


def check_gemm_sampled(x, W, out, cols):
    """Compare the selected output columns of a (large) GEMM with the oracle."""
    cols = np.asarray(cols, dtype=np.int32)
    xb = workloads.bits(x)
    wsel = workloads.bits(W[torch.as_tensor(cols, device=W.device, dtype=torch.long)])
    got = workloads.bits(out)[:, cols]
    idx = np.arange(cols.size, dtype=np.int32)
    ref = oracle.decode_gemm(xb, wsel, cols=idx)
    s, a = oracle.decode_gemm_f64(xb, wsel, cols=idx)
    rep = compare.gemm_check(got, ref, s, a)
    assert rep["ok"], rep
    return rep


def sample_columns(N, count=384, seed=0):
    """Stratified output columns of an N-column GEMM: in every 128-column tile
    (one MMA's weight rows) one random column in each 32-column quarter (one
    epilogue warp's TMEM lanes), plus `count` uniformly random columns and both
    ends of the first tile and of the matrix."""
    rng = np.random.default_rng(seed)
    base = {0, 1, 127, 128, N - 1, N - 2}
    for t0 in range(0, N, 128):
        for q0 in range(t0, min(t0 + 128, N), 32):
            base.add(int(rng.integers(q0, min(q0 + 32, N))))
    base |= set(int(c) for c in rng.integers(0, N, size=count))
    return np.array(sorted(c for c in base if 0 <= c < N), dtype=np.int32)
