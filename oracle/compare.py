"""Distances between BF16 results, and the tolerance checks the tests apply.

Test infrastructure (part of the oracle package). Works on BF16 bit patterns
(numpy ``uint16``).

ulp distance: every BF16 pattern is placed on a monotone integer line (positive
patterns as they are, negative ones mirrored below zero, so +0 and -0 are both 0)
and the distance is the difference of the two positions. One step on that line is
one BF16 ulp at the magnitude of the values involved.

Decode GEMM tolerance. The stated bar is "within 1 BF16 ulp of the FP64 result
rounded to BF16 on >= 99.99 % of elements and within 2 ulp on all" for an FP32
accumulation. An FP32 accumulation of K products carries a rounding noise of
order u32 * sqrt(steps) * S, where S = sum_k |x_k w_k| and u32 = 2^-24; an output
that cancels to below about 2^8 times that noise has no meaningful BF16 ulp of
its own (the noise exceeds its ulp no matter how the sum is ordered, cuBLAS's
included). The reading used here: an output whose exact value is at least
``floor = FLOOR_SCALE * S`` is judged in ulps at its own magnitude (the literal
bar); one below the floor is judged in ulps at the floor's magnitude. With
FLOOR_SCALE = 2^-11 the floor sits near 2^8 times the sqrt(K) noise for
K <= 18432, so every output large enough to be resolved by FP32 accumulation is
held to the literal bar. The literal counts are reported beside the verdict.
"""
import math

import numpy as np

FLOOR_SCALE = 2.0 ** -11


def ordinal(b) -> np.ndarray:
    """Position of each BF16 pattern on the monotone integer line."""
    b = np.asarray(b, dtype=np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def is_nonfinite(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b & 0x7F80) == 0x7F80


def ulp_distance(a, b) -> np.ndarray:
    """|ordinal(a) - ordinal(b)| element-wise (int64)."""
    return np.abs(ordinal(a).astype(np.int64) - ordinal(b).astype(np.int64))


def bf16_values(b) -> np.ndarray:
    """BF16 patterns -> float64 values (exact)."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def bf16_ulp_at(v) -> np.ndarray:
    """Spacing of the BF16 grid at magnitude |v| (2^(e-7) for |v| in [2^e, 2^(e+1)),
    2^-133 in the subnormal range)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.exp2(e - 7.0)


def histogram(d, top=4) -> dict:
    """{0: count, 1: count, ..., 'more': count} of integer distances."""
    d = np.asarray(d).ravel()
    out = {str(i): int((d == i).sum()) for i in range(top)}
    out["more"] = int((d >= top).sum())
    return out


def gemm_check(got_bits, ref_bits, exact, abs_sum, floor_scale=FLOOR_SCALE):
    """Judge a decode GEMM result against the oracle.

    got_bits, ref_bits: BF16 patterns (result, oracle); exact: the oracle's
    unrounded binary64 sums; abs_sum: sum_k |x_k w_k| per output.
    Returns a dict with the verdict and the literal statistics.
    """
    got_bits = np.asarray(got_bits, dtype=np.uint16)
    ref_bits = np.asarray(ref_bits, dtype=np.uint16)
    n = got_bits.size
    literal = ulp_distance(got_bits, ref_bits)
    floor = floor_scale * np.asarray(abs_sum, dtype=np.float64)
    small = np.abs(exact) < floor
    judged = literal.astype(np.float64)
    if small.any():
        gv = bf16_values(got_bits)[small]
        rv = bf16_values(ref_bits)[small]
        judged[small] = np.minimum(judged[small],
                                   np.abs(gv - rv) / bf16_ulp_at(floor[small]))
    nonfinite = int(is_nonfinite(got_bits).sum())
    within1 = float((judged <= 1).sum()) / max(n, 1)
    ok = nonfinite == 0 and within1 >= 0.9999 and (n == 0 or judged.max() <= 2)
    return {
        "ok": bool(ok),
        "n": int(n),
        "nonfinite": nonfinite,
        "within1_frac": within1,
        "max_judged": float(judged.max()) if n else 0.0,
        "below_floor": int(small.sum()),
        "literal_hist": histogram(literal),
        "literal_within1_frac": float((literal <= 1).sum()) / max(n, 1),
        "literal_max": int(literal.max()) if n else 0,
    }


def bits_equal(a, b) -> bool:
    """Bit-for-bit equality of two pattern arrays (the sign of zero counts)."""
    a = np.asarray(a, dtype=np.uint16)
    b = np.asarray(b, dtype=np.uint16)
    return a.shape == b.shape and bool(np.array_equal(a, b))


def within_ulps(a, b, ulps=1) -> bool:
    """Every element within ``ulps`` BF16 ulps, none non-finite in ``a``."""
    return (not is_nonfinite(a).any()) and int(ulp_distance(a, b).max(initial=0)) <= ulps


def first_mismatch(a, b):
    """(index tuple, a bits, b bits) of the first differing element, or None."""
    a = np.asarray(a, dtype=np.uint16)
    b = np.asarray(b, dtype=np.uint16)
    diff = np.argwhere(a != b)
    if diff.size == 0:
        return None
    i = tuple(int(v) for v in diff[0])
    return i, hex(int(a[i])), hex(int(b[i]))


def fp32_accumulation_noise(K: int, abs_sum: float) -> float:
    """Order of the rounding noise of an FP32 sum of K terms of total size abs_sum."""
    return (2.0 ** -24) * math.sqrt(max(K, 1)) * abs_sum
