"""GPU parity of gather_shards_bf16 with the oracle (bit-exact: a byte move),
through the C ABI, on the pages' gather shapes ("drafter/comm": gather_context
[M, 7168/TP] -> [M, 7168]; gather_logits [M, V/TP] -> [M, V])."""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare
import skinny_bf16_gemm_gb300 as sk
import workloads
from gpu_helpers import Guarded

pytestmark = pytest.mark.gpu

# The configs' shapes, edge sizes, and ten drawn once from a seeded generator
# (random.Random(20480) after the logits cases: TP 1..8, M 1..64, S any multiple
# of 8 up to 3200), kept literal.
SHAPES = [(8, m, 896) for m in (1, 16, 64)] + [(8, m, 2560) for m in (1, 8, 32, 64)] + [
    (3, 5, 40), (1, 2, 8), (64, 2, 16), (2, 300, 136)] + [
    (2, 52, 3184), (5, 12, 272), (4, 33, 184), (1, 50, 64), (6, 41, 1720), (8, 20, 1560),
    (8, 38, 504), (1, 8, 2712), (6, 5, 1520), (6, 12, 2744)]


@pytest.mark.parametrize("TP,M,S", SHAPES)
def test_gather_matches_oracle(cuda_ok, TP, M, S):
    rng = np.random.default_rng(workloads.seed_for("gather", TP, M, S))
    bits = rng.integers(0, 1 << 16, size=(TP, M, S), dtype=np.uint64).astype(np.uint16)
    bits[0, 0, :2] = [0x0000, 0x8000]  # the sentinel pair passes through unchanged
    shards = workloads.from_bits(bits).cuda()
    out = Guarded((M, TP * S))
    sk.gather_shards_bf16(shards, out.tensor)
    torch.cuda.synchronize()
    out.check()
    assert compare.first_mismatch(workloads.bits(out.tensor), oracle.gather_shards(bits)) is None


def test_gather_rejects_bad_arguments(cuda_ok):
    lib = sk.load_library()
    a = torch.zeros(8, 4, 64, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(4, 512, dtype=torch.bfloat16, device="cuda")
    assert lib.gather_shards_bf16(a.data_ptr(), 8, 4, 60, b.data_ptr(), None) == 2   # S % 8
    assert lib.gather_shards_bf16(a.data_ptr() + 2, 8, 4, 64, b.data_ptr(), None) == 3
    assert lib.gather_shards_bf16(a.data_ptr(), 8, 4, 64, a.data_ptr(), None) == 6
    host = torch.zeros(4, 512, dtype=torch.bfloat16)
    assert lib.gather_shards_bf16(a.data_ptr(), 8, 4, 64, host.data_ptr(), None) == 4
