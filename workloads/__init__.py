"""Seeded synthetic inputs for the decode GEMM and the reduce + RMSNorm.

The one module both sides use: it draws random numbers and rounds them to BF16
with PyTorch's own conversion (round to nearest even) and holds none of the
method's arithmetic. The oracle and the CUDA path both take what it makes.

Distributions follow the drafter pages' workloads (vLLM DSpark drafter,
"drafter/linears" and "drafter/comm"): activations x ~ N(0, 1); weights
W ~ N(0, 1/K) (a unit-variance output per row); TP partial rows and residual
rows ~ N(0, 1); RMSNorm weight gamma ~ 1 + N(0, 0.1); eps = 1e-6. The pages use
no dataset: every input is synthetic.

Host draws use numpy's PCG64 + ziggurat normals (integer state, the same on
x86_64 and aarch64). Device draws (the benchmark's large weights) use a seeded
torch CUDA generator; they feed timing only, never a stored expected value.
"""
from dataclasses import dataclass, field
import hashlib

import numpy as np
import torch

HIDDEN = 7168  # ArNorm row width ("drafter/comm")


def seed_for(*parts) -> int:
    """A stable 63-bit seed from any tuple of labels (config id, M, N, ...)."""
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _normal_f32(rng: np.random.Generator, shape, std=1.0, mean=0.0) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return a


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 numpy array -> CPU BF16 tensor (PyTorch's round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """A BF16 tensor's 16-bit patterns as a numpy uint16 array (CPU copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray) -> torch.Tensor:
    """numpy uint16 patterns -> CPU BF16 tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16)


@dataclass
class GemmInputs:
    x: torch.Tensor  # [M, K] bf16
    W: torch.Tensor  # [N, K] bf16


def gemm_inputs(M, N, K, seed, device="cpu", kind="normal") -> GemmInputs:
    """x ~ N(0,1) [M,K], W ~ N(0,1/K) [N,K] in BF16.

    kind="int": x, W uniform integers in [-4, 4] (exact in BF16), used where every
    partial sum must be exact in FP32.
    """
    if kind == "int":
        rng = np.random.Generator(np.random.PCG64(seed))
        x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
        w = rng.integers(-4, 5, size=(N, K)).astype(np.float32)
        return GemmInputs(to_bf16(x).to(device), to_bf16(w).to(device))
    if kind != "normal":
        raise ValueError(kind)
    if str(device).startswith("cuda"):
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
        w = torch.randn(N, K, generator=g, device=device, dtype=torch.float32)
        w.mul_(1.0 / np.sqrt(K))
        return GemmInputs(x.to(torch.bfloat16), w.to(torch.bfloat16))
    rng = np.random.Generator(np.random.PCG64(seed))
    x = _normal_f32(rng, (M, K))
    w = _normal_f32(rng, (N, K), std=1.0 / np.sqrt(K))
    return GemmInputs(to_bf16(x), to_bf16(w))


@dataclass
class ReduceInputs:
    partials: torch.Tensor          # [TP, M, 7168] bf16
    residual: torch.Tensor | None   # [M, 7168] bf16 or None
    gamma: torch.Tensor             # [7168] bf16
    eps: float = 1e-6


def reduce_inputs(TP, M, seed, residual=True, width=HIDDEN, device="cpu") -> ReduceInputs:
    """Partials and residual ~ N(0,1), gamma ~ 1 + N(0, 0.1), eps = 1e-6."""
    rng = np.random.Generator(np.random.PCG64(seed))
    p = _normal_f32(rng, (TP, M, width))
    r = _normal_f32(rng, (M, width)) if residual else None
    g = _normal_f32(rng, (width,), std=0.1, mean=1.0)
    return ReduceInputs(to_bf16(p).to(device),
                        None if r is None else to_bf16(r).to(device),
                        to_bf16(g).to(device))


# ---- the pages' workloads ------------------------------------------------------

@dataclass(frozen=True)
class GemmShape:
    M: int
    N: int
    K: int

    def weight_bytes(self):
        return 2 * self.N * self.K

    def algorithmic_bytes(self):
        """Weight read once + x read once + out written once (BF16)."""
        return 2 * self.N * self.K + 2 * self.M * self.K + 2 * self.M * self.N

    def flops(self):
        return 2 * self.M * self.N * self.K


@dataclass(frozen=True)
class ReduceShape:
    TP: int
    M: int
    residual: bool = True
    width: int = HIDDEN

    def algorithmic_bytes(self):
        """TP partial rows + residual rows (if any) + out + residual_out + gamma."""
        rows = self.TP * self.M + (self.M if self.residual else 0) + 2 * self.M
        return 2 * self.width * rows + 2 * self.width


# PR1 reference case: decode GEMM M=4, N=2048, K=7168; reduce TP=8, M=4.
PR1_GEMM = GemmShape(4, 2048, 7168)
PR1_REDUCE = ReduceShape(8, 4, True)

# Reduce + residual + RMSNorm sweep.
REDUCE_SWEEP = [ReduceShape(tp, m, res) for tp in (2, 4, 8) for m in (1, 4, 8, 16, 32, 64)
                for res in (True, False)]

# Decode GEMM sweep, K = 7168.
GEMM_SWEEP = [GemmShape(m, n, 7168) for m in (1, 2, 4, 8, 16, 24, 32)
              for n in (4096, 12288, 18432)]

# Wider shapes beyond the pages' 32 rows: M up to 64 (the row cap) and the TP1
# down projection's K = 14336 ("drafter/linears", warp_eligible).
GEMM_WIDER = ([GemmShape(m, 18432, 7168) for m in (48, 64)] + [GemmShape(64, 20480, 7168)]
              + [GemmShape(m, 7168, 14336) for m in (16, 32, 64)])

# Vocab-shard lm_head GEMM.
LM_HEAD = [GemmShape(m, 20480, 7168) for m in (1, 8, 32)]


@dataclass(frozen=True)
class ChainConfig:
    """Synthetic drafter layer chain: per layer GEMM [M,K]->[M,F], GEMM [M,F]->[M,K]
    into slot 0 of the [TP, M, K] partials, then reduce + residual + RMSNorm."""
    layers: int = 3
    M: int = 16
    hidden: int = HIDDEN
    ffn: int = 18432
    TP: int = 8
    eps: float = 1e-6

    def gemm1(self):
        return GemmShape(self.M, self.ffn, self.hidden)

    def gemm2(self):
        return GemmShape(self.M, self.hidden, self.ffn)

    def reduce(self):
        return ReduceShape(self.TP, self.M, True, self.hidden)

    def layer_bytes(self):
        return (self.gemm1().algorithmic_bytes() + self.gemm2().algorithmic_bytes()
                + self.reduce().algorithmic_bytes())

    def step_bytes(self):
        return self.layers * self.layer_bytes()

    def weight_bytes(self):
        return self.layers * (self.gemm1().weight_bytes() + self.gemm2().weight_bytes())


CHAIN = ChainConfig()


@dataclass
class ChainInputs:
    W1: list          # per layer [ffn, hidden] bf16
    W2: list          # per layer [hidden, ffn] bf16
    peers: list       # per layer [TP-1, M, hidden] bf16: the other ranks' partial rows
    gamma: list       # per layer [hidden] bf16
    x0: torch.Tensor  # [M, hidden] bf16
    residual0: torch.Tensor  # [M, hidden] bf16
    cfg: ChainConfig = field(default_factory=ChainConfig)


def chain_inputs(cfg: ChainConfig, seed, device="cpu") -> ChainInputs:
    """Seeded chain inputs. W1 ~ N(0, 1/hidden), W2 ~ N(0, 1/ffn), peer partial
    slots, x0 and residual0 ~ N(0,1), gamma ~ 1 + N(0, 0.1)."""
    W1, W2, peers, gamma = [], [], [], []
    for layer in range(cfg.layers):
        a = gemm_inputs(cfg.M, cfg.ffn, cfg.hidden, seed_for(seed, "W1", layer), device)
        b = gemm_inputs(cfg.M, cfg.hidden, cfg.ffn, seed_for(seed, "W2", layer), device)
        r = reduce_inputs(cfg.TP - 1, cfg.M, seed_for(seed, "peers", layer), True,
                          cfg.hidden, "cpu")
        W1.append(a.W)
        W2.append(b.W)
        peers.append(r.partials.to(device))
        gamma.append(r.gamma.to(device))
    first = reduce_inputs(1, cfg.M, seed_for(seed, "x0"), True, cfg.hidden, "cpu")
    return ChainInputs(W1, W2, peers, gamma, first.partials[0].to(device),
                       first.residual.to(device), cfg)
