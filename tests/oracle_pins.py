"""Pins: checks that tie an implementation of the method to what the pages and the
mathematics fix, independently of the implementation itself.

Each ``pin_*`` takes the implementation under test as callables with the oracle's
signatures (BF16 patterns in numpy uint16) and returns None on success or a
string saying what failed. ``tests/test_oracle.py`` runs every pin on the oracle
(all must pass) and on deliberately broken variants (each must be caught by at
least one pin), which shows the pins can see the mistakes they are meant to.

Sources of the expected values: the exact rational model (tests/exact_model.py),
PyTorch's float32 -> bfloat16 conversion (a library round-to-nearest-even),
closed forms, invariants, and the stored cases under tests/golden/.
"""
from dataclasses import dataclass
from fractions import Fraction
import decimal
import os
from typing import Callable

import numpy as np
import torch

import exact_model as em

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
HIDDEN = 7168


@dataclass
class Impl:
    """The functions a pin may call (the oracle's signatures)."""
    bf16_from_f64_array: Callable
    decode_gemm: Callable          # (x_bits, W_bits) -> out_bits
    reduce_residual: Callable      # (partials_bits, residual_bits|None) -> bits
    rmsnorm: Callable              # (h_bits, gamma_bits, eps) -> bits
    gather_shards: Callable = None  # (shards_bits [TP, M, S]) -> bits [M, TP*S]
    decode_gemm_logits: Callable = None  # (x, W, n_out, soft_cap, scale) -> bits [M, n_out]


def oracle_impl():
    import oracle
    return Impl(oracle.bf16_from_f64_array, oracle.decode_gemm, oracle.reduce_residual,
                oracle.rmsnorm, oracle.gather_shards, oracle.decode_gemm_logits)


# ---- helpers -----------------------------------------------------------------

def f32_to_bf16_torch(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_of(values) -> np.ndarray:
    """Patterns of float values that are already exactly on the BF16 grid."""
    a = np.asarray(values, dtype=np.float32)
    u = a.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("values not on the BF16 grid")
    return (u >> 16).astype(np.uint16)


def bits_to_f64(b) -> np.ndarray:
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):  # NaN patterns stay NaN
        return u.view(np.float32).astype(np.float64)


def random_bf16(rng, shape, std=1.0) -> np.ndarray:
    return f32_to_bf16_torch(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def read_cases(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line)
    return rows


# ---- BF16 rounding -------------------------------------------------------------

def pin_round_golden(impl: Impl):
    """Stored edge cases (ties, subnormals, overflow, the double-rounding trap):
    the stored value, the exact model and the implementation must all agree."""
    rows = read_cases("bf16_round_cases.txt")
    vals = np.array([float.fromhex(r.split()[0]) for r in rows])
    want = np.array([int(r.split()[1], 16) for r in rows], dtype=np.uint16)
    got = impl.bf16_from_f64_array(vals)
    for v, w, g in zip(vals, want, got):
        if v == 0:
            model = 0x8000 if np.signbit(v) else 0
        else:
            model = em.to_bits_bf16(em.round_ne(Fraction(float(v)), em.BF16))
        if model != int(w):
            return f"stored case {v!r}: file 0x{int(w):04x}, exact model 0x{model:04x}"
        if int(g) != int(w):
            return f"round({v!r}) = 0x{int(g):04x}, expected 0x{int(w):04x}"
    return None


def pin_round_vs_torch(impl: Impl, n=200_000, seed=1):
    """Random binary32 values across every exponent (subnormals and overflow
    included): rounding them must equal PyTorch's float32 -> bfloat16."""
    rng = np.random.default_rng(seed)
    u = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    got = impl.bf16_from_f64_array(f.astype(np.float64))
    want = f32_to_bf16_torch(f)
    bad = np.nonzero(got != want)[0]
    if bad.size:
        i = bad[0]
        return f"round({f[i]!r}) = 0x{int(got[i]):04x}, torch 0x{int(want[i]):04x}"
    return None


def pin_round_doubles_vs_model(impl: Impl, n=3000, seed=2):
    """Random binary64 values (not binary32 values: the double-rounding trap is
    live) against the exact rational model."""
    rng = np.random.default_rng(seed)
    mant = rng.random(n) + 1.0
    exps = rng.integers(-140, 130, size=n)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    v = sign * np.ldexp(mant, exps)
    # Put a third of them one binary64 step away from a BF16 tie.
    k = n // 3
    base = np.ldexp(np.floor(np.ldexp(mant[:k], 7)) + 0.5, exps[:k] - 7)
    v[:k] = np.nextafter(base, np.where(rng.random(k) < 0.5, 0.0, np.inf)) * sign[:k]
    got = impl.bf16_from_f64_array(v)
    for x, g in zip(v, got):
        r = em.round_ne(Fraction(float(x)), em.BF16)
        want = em.to_bits_bf16(r, negative_zero=bool(x < 0)) if r == 0 else em.to_bits_bf16(r)
        if int(g) != want:
            return f"round({float(x).hex()}) = 0x{int(g):04x}, exact 0x{want:04x}"
    return None


# ---- decode GEMM -------------------------------------------------------------------

def pin_gemm_exact_tiny(impl: Impl, seed=3):
    """Tiny random problems against the exact rational sum rounded once
    (brute force). Shapes small enough for Fractions; not square, so a transposed
    operand cannot pass."""
    rng = np.random.default_rng(seed)
    for (M, N, K) in [(1, 16, 128), (3, 16, 128), (2, 5, 40), (4, 3, 7)]:
        x = random_bf16(rng, (M, K))
        W = random_bf16(rng, (N, K), std=1.0 / np.sqrt(K))
        got = impl.decode_gemm(x, W)
        xv = [[Fraction(float(v)) for v in row] for row in bits_to_f64(x)]
        wv = [[Fraction(float(v)) for v in row] for row in bits_to_f64(W)]
        want = np.array(em.gemm_exact_bits(xv, wv), dtype=np.uint16)
        if got.shape != want.shape or not np.array_equal(got, want):
            return f"exact GEMM {M}x{N}x{K} differs"
    return None


def pin_gemm_integers(impl: Impl, seed=4):
    """Integer operands in [-4, 4] with K = 7168: the exact sums are integers whose
    BF16 rounding is computed with integer arithmetic and the exact model."""
    rng = np.random.default_rng(seed)
    M, N, K = 3, 24, HIDDEN
    xi = rng.integers(-4, 5, size=(M, K))
    wi = rng.integers(-4, 5, size=(N, K))
    x = bf16_bits_of(xi)
    W = bf16_bits_of(wi)
    got = impl.decode_gemm(x, W)
    exact = xi.astype(np.int64) @ wi.astype(np.int64).T
    want = np.array([[em.bf16_of_rational(int(v)) for v in row] for row in exact],
                    dtype=np.uint16)
    if not np.array_equal(got, want):
        i = tuple(np.argwhere(got != want)[0])
        return f"integer GEMM at {i}: 0x{int(got[i]):04x} vs exact 0x{int(want[i]):04x}"
    return None


def pin_gemm_ties(impl: Impl):
    """Rows built so that the exact dot product sits on, or a hair off, a BF16
    rounding tie: only a single round-to-nearest-even of the exact sum gives the
    exact model's answer (rounding through binary32 first, truncating, or breaking
    ties away from zero all miss some of them)."""
    K = HIDDEN
    x = np.zeros((1, K), dtype=np.float32)
    x[0, :4] = 1.0
    rows = [
        [1.0, 2.0 ** -8, 2.0 ** -30, 0.0],       # just above the 1 + 2^-8 tie
        [1.0, 2.0 ** -8, -2.0 ** -30, 0.0],      # just below it
        [1.0, 2.0 ** -8, 0.0, 0.0],              # on it: even is 1.0
        [1.0, 3 * 2.0 ** -8, 0.0, 0.0],          # on the next one: even is 1 + 2^-6
        [-1.0, -(2.0 ** -8), -(2.0 ** -30), 0.0],  # negative mirror
        [256.0, 1.0, 2.0 ** -20, 0.0],           # 257 + tiny: above the 256/258 tie
        [256.0, 1.0, 0.0, 0.0],                  # 257: tie, even is 256
        [1.0, 2.0 ** -9, 2.0 ** -9, 2.0 ** -40],  # 1 + 2^-8 + 2^-40 built from parts
    ]
    W = np.zeros((len(rows), K), dtype=np.float32)
    for i, r in enumerate(rows):
        W[i, :4] = r
    xb, wb = bf16_bits_of(x), bf16_bits_of(W)
    got = impl.decode_gemm(xb, wb)[0]
    for i, r in enumerate(rows):
        want = em.bf16_of_rational(sum(Fraction(v) for v in r))
        if int(got[i]) != want:
            return f"tie row {i}: 0x{int(got[i]):04x} vs exact 0x{want:04x}"
    return None


def pin_gemm_identity(impl: Impl, seed=5):
    """W = [I | 0] (N = 40 rows selecting the first 40 of K = 96 columns): out = x's
    first 40 columns, exactly (every other term is an exact zero)."""
    rng = np.random.default_rng(seed)
    M, N, K = 5, 40, 96
    x = random_bf16(rng, (M, K))
    w = np.zeros((N, K), dtype=np.float32)
    w[np.arange(N), np.arange(N)] = 1.0
    got = impl.decode_gemm(x, bf16_bits_of(w))
    want = x[:, :N].copy()
    want[want == 0x8000] = 0  # -0 * 1 + (+0) = +0
    if not np.array_equal(got, want):
        return "W = [I|0] does not reproduce x"
    return None


def pin_gemm_invariants(impl: Impl, seed=6):
    """Negating W negates out bit for bit (RNE is symmetric); scaling W by 2 scales
    out by 2 exactly; row m of an M-row call equals a 1-row call on row m."""
    rng = np.random.default_rng(seed)
    M, N, K = 6, 64, 512
    x = random_bf16(rng, (M, K))
    W = random_bf16(rng, (N, K), std=1.0 / np.sqrt(K))
    base = impl.decode_gemm(x, W)
    neg = impl.decode_gemm(x, W ^ np.uint16(0x8000))
    nz = (base & 0x7FFF) != 0
    if not np.array_equal(neg[nz], base[nz] ^ np.uint16(0x8000)):
        return "negating W does not negate out"
    w2 = f32_to_bf16_torch(bits_to_f64(W).astype(np.float32) * 2)
    two = impl.decode_gemm(x, w2)
    if not np.array_equal(bits_to_f64(two), 2 * bits_to_f64(base)):
        return "scaling W by 2 does not scale out by 2"
    for m in (0, M - 1):
        one = impl.decode_gemm(x[m:m + 1], W)
        if not np.array_equal(one[0], base[m]):
            return f"row {m} depends on the other rows"
    return None


# ---- reduce + residual -------------------------------------------------------------

def pin_reduce_golden(impl: Impl):
    """Stored order, signed-zero, overflow and double-rounding columns: file, exact
    model and implementation must agree."""
    for row in read_cases("reduce_cases.txt"):
        slots_s, res_s, want_s = [p.strip() for p in row.split("|")]
        slots = [int(t, 16) for t in slots_s.split()]
        res = None if res_s == "-" else int(res_s, 16)
        want = int(want_s, 16)
        model = em.reduce_bits(slots, res)
        if model != want:
            return f"stored case {slots_s}|{res_s}: file 0x{want:04x}, model 0x{model:04x}"
        p = np.array(slots, dtype=np.uint16).reshape(len(slots), 1, 1)
        r = None if res is None else np.array([[res]], dtype=np.uint16)
        got = int(impl.reduce_residual(p, r)[0, 0])
        if got != want:
            return f"reduce {slots_s}|{res_s} = 0x{got:04x}, expected 0x{want:04x}"
    return None


def _order_sensitive_columns(rng, count, TP):
    """Random columns whose rank-order binary32 sum rounds to a different BF16 than
    the reverse order does (found by search with the exact model)."""
    cols = []
    if TP < 3:
        return cols  # two binary32 addends commute: the order cannot matter
    for _ in range(200 * count):
        if len(cols) == count:
            break
        big = rng.standard_normal() * 8
        vals = np.array([big, -big] + list(rng.standard_normal(TP - 2) * 2.0 ** -rng.integers(
            6, 20, size=TP - 2)), dtype=np.float32)
        rng.shuffle(vals)
        b = [int(v) for v in f32_to_bf16_torch(vals)]
        if em.reduce_bits(b) != em.reduce_bits(b[::-1]):
            cols.append(b)
    return cols


def pin_reduce_random(impl: Impl, seed=7):
    """Random rows (TP = 2, 3, 5, 8; with and without residual) plus columns chosen
    so that the summation order changes the BF16 result, against the exact
    binary32-step model column by column."""
    rng = np.random.default_rng(seed)
    for TP in (2, 3, 5, 8):
        width = 48
        p = random_bf16(rng, (TP, 1, width))
        sens = _order_sensitive_columns(rng, 16, TP)
        for j, col in enumerate(sens):
            p[:, 0, j] = col
        for with_res in (False, True):
            r = random_bf16(rng, (1, width)) if with_res else None
            got = impl.reduce_residual(p, r)
            for c in range(width):
                want = em.reduce_bits([int(v) for v in p[:, 0, c]],
                                      None if r is None else int(r[0, c]))
                if int(got[0, c]) != want:
                    return (f"TP={TP} residual={with_res} column {c}: 0x{int(got[0, c]):04x} "
                            f"vs exact 0x{want:04x}")
    return None


def pin_reduce_identities(impl: Impl, seed=8):
    """TP = 1 without residual is the identity (signed zeros included), and
    residual = None gives the same row as a residual of -0 (x + -0 = x for every x,
    -0 included), i.e. the rounded rank-order sum itself."""
    rng = np.random.default_rng(seed)
    M, width = 3, HIDDEN
    p1 = random_bf16(rng, (1, M, width))
    p1[0, 0, :8] = 0x8000
    if not np.array_equal(impl.reduce_residual(p1, None), p1[0]):
        return "TP = 1 is not the identity"
    p = random_bf16(rng, (4, M, width))
    a = impl.reduce_residual(p, None)
    negz = np.full((M, width), 0x8000, dtype=np.uint16)
    if not np.array_equal(impl.reduce_residual(p, negz), a):
        return "a residual of -0 changes the result"
    return None


# ---- RMSNorm -------------------------------------------------------------------------

def _exact_rms_bits(h_vals, g_vals, eps):
    """BF16 of h * g / sqrt(mean(h^2) + eps) with 60-digit decimal arithmetic."""
    ctx = decimal.Context(prec=60)
    ss = sum((Fraction(v) ** 2 for v in h_vals), Fraction(0))
    arg = ss / len(h_vals) + Fraction(eps)
    d = ctx.divide(decimal.Decimal(arg.numerator), decimal.Decimal(arg.denominator))
    rstd = ctx.divide(decimal.Decimal(1), d.sqrt(ctx))
    out = []
    for v, g in zip(h_vals, g_vals):
        y = ctx.multiply(ctx.multiply(decimal.Decimal(v), rstd), decimal.Decimal(g))
        out.append(em.to_bits_bf16(em.round_ne(Fraction(y), em.BF16),
                                   negative_zero=(y == 0 and (v < 0) != (g < 0))))
    return out


def pin_rmsnorm_closed_forms(impl: Impl):
    """Rows with closed-form answers: constant rows (v / sqrt(v^2 + eps)), a row whose
    mean square is comparable to eps (eps must sit inside the root, the mean must
    divide by 7168), one spike, alternating signs; zero row gives zeros."""
    eps = np.float32(1e-6)
    rows = [
        np.full(HIDDEN, 1.0), np.full(HIDDEN, 2.0), np.full(HIDDEN, 2.0 ** -10),
        np.where(np.arange(HIDDEN) % 2 == 0, 3.0, -3.0),
        np.concatenate([[1.0], np.zeros(HIDDEN - 1)]),
        np.linspace(-4, 4, HIDDEN),
    ]
    gammas = [np.ones(HIDDEN), np.full(HIDDEN, 0.5), np.ones(HIDDEN), np.ones(HIDDEN),
              np.ones(HIDDEN), np.linspace(0.5, 1.5, HIDDEN)]
    for h, g in zip(rows, gammas):
        hb = f32_to_bf16_torch(h.astype(np.float32))[None, :]
        gb = f32_to_bf16_torch(g.astype(np.float32))
        got = impl.rmsnorm(hb, gb, float(eps))[0]
        want = _exact_rms_bits([float(v) for v in bits_to_f64(hb[0])],
                               [float(v) for v in bits_to_f64(gb)], float(eps))
        if not np.array_equal(got, np.array(want, dtype=np.uint16)):
            i = int(np.argwhere(got != np.array(want, dtype=np.uint16))[0][0])
            return f"closed form row {h[:2]}...: col {i} 0x{int(got[i]):04x} vs 0x{want[i]:04x}"
    zero = np.zeros((1, HIDDEN), dtype=np.uint16)
    if np.any((impl.rmsnorm(zero, f32_to_bf16_torch(np.ones(HIDDEN, np.float32)),
                            float(eps)) & 0x7FFF) != 0):
        return "a zero row does not give zeros"
    return None


def pin_rmsnorm_invariants(impl: Impl, seed=9):
    """With eps = 0, scaling a row by 2 changes nothing (bit for bit); a constant
    gamma = c gives an output whose RMS is |c| to within BF16 rounding."""
    rng = np.random.default_rng(seed)
    h = random_bf16(rng, (4, HIDDEN))
    g = f32_to_bf16_torch((1 + 0.1 * rng.standard_normal(HIDDEN)).astype(np.float32))
    a = impl.rmsnorm(h, g, 0.0)
    h2 = f32_to_bf16_torch(bits_to_f64(h).astype(np.float32) * 2)
    if not np.array_equal(impl.rmsnorm(h2, g, 0.0), a):
        return "RMSNorm(2h) != RMSNorm(h) with eps = 0"
    for c in (0.75, -2.0):
        gc = f32_to_bf16_torch(np.full(HIDDEN, c, np.float32))
        out = bits_to_f64(impl.rmsnorm(h, gc, 1e-6))
        rms = np.sqrt((out ** 2).mean(axis=1))
        if np.any(np.abs(rms - abs(c)) > abs(c) * 2.0 ** -8):
            return f"constant gamma {c}: rms {rms}"
    return None


# ---- lm_head logits epilogue ---------------------------------------------------------

def _decimal_tanh(q: Fraction, ctx) -> decimal.Decimal:
    """tanh of a rational via exp in decimal arithmetic: (e^(2q) - 1) / (e^(2q) + 1)."""
    d = ctx.divide(decimal.Decimal(q.numerator), decimal.Decimal(q.denominator))
    e = ctx.exp(ctx.multiply(decimal.Decimal(2), d))
    return ctx.divide(ctx.subtract(e, decimal.Decimal(1)), ctx.add(e, decimal.Decimal(1)))


def pin_logits_closed_forms(impl: Impl):
    """One nonzero product per output, so the dot product is exact (a*b): the result
    must be BF16(scale * cap * tanh(a*b / cap)) with tanh from exp in 60-digit
    decimal arithmetic, rounded once; large a*b saturates to +-cap*scale."""
    ctx = decimal.Context(prec=60)
    K = 64
    cases = [(1.5, 2.0, 30.0, 1.0), (0.75, -3.0, 30.0, 0.5), (8.0, 8.0, 30.0, 1.0),
             (3.0, 5.0, 4.0, 2.0), (256.0, 64.0, 30.0, 1.0), (-0.125, 0.25, 1.0, 3.0)]
    # Random products (BF16 operands) near the cap, where one rounding at the end
    # and a rounding after every step disagree often.
    rng = np.random.default_rng(16)
    ab = bits_to_f64(random_bf16(rng, (40, 2), std=6.0))
    cases += [(float(a), float(b), 30.0, 0.7) for a, b in ab]
    for a, b, cap, scale in cases:
        x = np.zeros((1, K), dtype=np.float32)
        W = np.zeros((2, K), dtype=np.float32)
        x[0, 5] = a
        W[0, 5] = b
        W[1, 7] = 1.0  # second column: exactly 0
        got = impl.decode_gemm_logits(bf16_bits_of(x), bf16_bits_of(W), 2, cap, scale)
        t = _decimal_tanh(Fraction(a) * Fraction(b) / Fraction(cap), ctx)
        v = Fraction(ctx.multiply(ctx.multiply(t, decimal.Decimal(cap)), decimal.Decimal(scale)))
        want = em.to_bits_bf16(em.round_ne(v, em.BF16))
        if int(got[0, 0]) != want:
            return f"a={a} b={b} cap={cap} scale={scale}: 0x{int(got[0, 0]):04x} vs 0x{want:04x}"
        if int(got[0, 1]) & 0x7FFF:
            return "tanh(0) * cap * scale is not zero"
    return None


def pin_logits_reduce_to_gemm(impl: Impl, seed=14):
    """No cap, scale 1: the first n_out columns of the plain GEMM, bit for bit; no
    cap, scale 4: exactly four times those values (a power of two)."""
    rng = np.random.default_rng(seed)
    M, N, K = 3, 200, 256
    x = random_bf16(rng, (M, K))
    W = random_bf16(rng, (N, K), std=1.0 / 16)
    full = oracle_gemm = impl.decode_gemm(x, W)
    got = impl.decode_gemm_logits(x, W, 150, 0.0, 1.0)
    if got.shape != (M, 150) or not np.array_equal(got, full[:, :150]):
        return "no-cap scale-1 logits are not the GEMM's first n_out columns"
    four = impl.decode_gemm_logits(x, W, N, 0.0, 4.0)
    if not np.array_equal(bits_to_f64(four), 4 * bits_to_f64(oracle_gemm)):
        return "scale 4 is not exactly four times the GEMM"
    return None


def pin_logits_odd_and_sliced(impl: Impl, seed=15):
    """tanh is odd: negating W negates every logit; the slice keeps the leading
    columns (a smaller n_out is a prefix of a larger one)."""
    rng = np.random.default_rng(seed)
    M, N, K = 2, 96, 128
    x = random_bf16(rng, (M, K))
    W = random_bf16(rng, (N, K), std=0.5)
    a = impl.decode_gemm_logits(x, W, N, 5.0, 0.75)
    b = impl.decode_gemm_logits(x, W ^ np.uint16(0x8000), N, 5.0, 0.75)
    nz = (a & 0x7FFF) != 0
    if not np.array_equal(b[nz], a[nz] ^ np.uint16(0x8000)):
        return "negating W does not negate the logits"
    if not np.array_equal(impl.decode_gemm_logits(x, W, 40, 5.0, 0.75), a[:, :40]):
        return "n_out = 40 is not the first 40 columns"
    if np.any(np.abs(bits_to_f64(a)) > 5.0 * 0.75 * (1 + 2.0 ** -8)):
        return "a soft-capped logit exceeds cap * scale"
    return None


# ---- gather ---------------------------------------------------------------------------

def pin_gather_placement(impl: Impl, seed=12):
    """Every element of the gathered row names where it came from: with shard
    values encoding (rank, row, column), out[m][c] must be rank c // S, row m,
    column c % S -- the pages' "rank r's at columns r S ..". Sentinel-like words
    (+0, -0) pass through unchanged."""
    TP, M, S = 4, 3, 24
    r, m, j = np.meshgrid(np.arange(TP), np.arange(M), np.arange(S), indexing="ij")
    code = (r * 64 + m * 16 + (j % 16)).astype(np.float32)  # small integers: exact in BF16
    code[:, :, 16:] += 0.5 * (j[:, :, 16:] // 16)  # keep columns >= 16 distinct
    shards = f32_to_bf16_torch(code)
    shards[1, 2, 5] = 0x8000   # the -0 half of the sentinel pair stays
    shards[1, 2, 4] = 0x0000
    got = impl.gather_shards(shards)
    if got.shape != (M, TP * S):
        return f"shape {got.shape}"
    for mm in range(M):
        for c in range(TP * S):
            if int(got[mm, c]) != int(shards[c // S, mm, c % S]):
                return f"out[{mm}][{c}] is not shard[{c // S}][{mm}][{c % S}]"
    return None


def pin_gather_inverse(impl: Impl, seed=13):
    """Cutting the gathered rows back into TP column blocks returns the shards
    (the gather is a bijection of positions); TP = 1 is the identity."""
    rng = np.random.default_rng(seed)
    for TP, M, S in [(8, 4, 896), (8, 2, 2560), (1, 3, 64), (3, 5, 40)]:
        shards = rng.integers(0, 1 << 16, size=(TP, M, S), dtype=np.uint64).astype(np.uint16)
        got = impl.gather_shards(shards)
        back = got.reshape(M, TP, S).transpose(1, 0, 2)
        if not np.array_equal(back, shards):
            return f"TP={TP} M={M} S={S}: not the inverse of the column split"
    return None


PINS = {
    "round_golden": pin_round_golden,
    "round_vs_torch": pin_round_vs_torch,
    "round_doubles": pin_round_doubles_vs_model,
    "gemm_exact_tiny": pin_gemm_exact_tiny,
    "gemm_integers": pin_gemm_integers,
    "gemm_ties": pin_gemm_ties,
    "gemm_identity": pin_gemm_identity,
    "gemm_invariants": pin_gemm_invariants,
    "reduce_golden": pin_reduce_golden,
    "reduce_random": pin_reduce_random,
    "reduce_identities": pin_reduce_identities,
    "rmsnorm_closed_forms": pin_rmsnorm_closed_forms,
    "rmsnorm_invariants": pin_rmsnorm_invariants,
    "logits_closed_forms": pin_logits_closed_forms,
    "logits_reduce_to_gemm": pin_logits_reduce_to_gemm,
    "logits_odd_and_sliced": pin_logits_odd_and_sliced,
    "gather_placement": pin_gather_placement,
    "gather_inverse": pin_gather_inverse,
}
