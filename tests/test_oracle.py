"""The oracle against its pins, and the pins against planted mistakes (CPU only).

Every pin must pass on the oracle. Every mutant -- the oracle with one plausible
mistake planted on the CPU side (a dropped term, a wrong sign or index, a
transposed operand, a wrong order, a missing or extra rounding, eps in the wrong
place, the wrong width) -- must fail at least one pin of its group.
"""
import numpy as np
import pytest

import oracle
from oracle_pins import PINS, Impl, oracle_impl, f32_to_bf16_torch, bits_to_f64

HIDDEN = 7168


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin_holds_on_oracle(name):
    assert PINS[name](oracle_impl()) is None


# ---- mutants: one planted mistake each ----------------------------------------------

def _with(**overrides):
    base = oracle_impl()
    return Impl(**{**base.__dict__, **overrides})


def _round_via_f32(v):
    with np.errstate(over="ignore"):  # out-of-range values become infinities
        f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return f32_to_bf16_torch(f)


def _round_truncate(v):
    with np.errstate(over="ignore"):  # out-of-range values become infinities
        f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _round_ties_away(v):
    v = np.asarray(v, dtype=np.float64)
    out = oracle.bf16_from_f64_array(v)
    # Where the input sits exactly half-way, move away from zero instead.
    lo = bits_to_f64(out)
    ulp = np.abs(bits_to_f64(out + np.uint16(1)) - lo)
    tie = np.abs(np.abs(v) - np.abs(lo)) == ulp / 2
    return np.where(tie & (np.abs(v) > np.abs(lo)), out + np.uint16(1), out).astype(np.uint16)


def _gemm_from_sums(round_fn):
    def gemm(x, W):
        s, _ = oracle.decode_gemm_f64(x, W)
        return round_fn(s)
    return gemm


def _rms_numpy(eps_inside=True, width=HIDDEN, use_gamma=True, use_eps=True):
    def rms(h, g, eps):
        hv = bits_to_f64(h)
        gv = bits_to_f64(g) if use_gamma else np.ones(h.shape[1])
        ss = (hv * hv).sum(axis=1, keepdims=True)
        e = float(np.float32(eps)) if use_eps else 0.0
        rstd = 1.0 / np.sqrt(ss / width + e) if eps_inside else 1.0 / np.sqrt(ss / width) + e
        return oracle.bf16_from_f64_array(hv * rstd * gv)
    return rms


def _reduce_bf16_each_step(p, r):
    p = np.asarray(p)
    acc = p[0].copy()
    for k in range(1, p.shape[0]):
        s = bits_to_f64(acc).astype(np.float32) + bits_to_f64(p[k]).astype(np.float32)
        acc = oracle.bf16_from_f64_array(s.astype(np.float64))
    if r is None:
        return acc
    return oracle.reduce_residual(acc[None], r)


def _reduce_f64(p, r):
    s = bits_to_f64(p).sum(axis=0)
    a = oracle.bf16_from_f64_array(s)
    return a if r is None else oracle.reduce_residual(a[None], r)


def _reduce_fused_residual(p, r):
    if r is None:
        return oracle.reduce_residual(p, None)
    s = bits_to_f64(p[0]).astype(np.float32)
    for k in range(1, p.shape[0]):
        s = s + bits_to_f64(p[k]).astype(np.float32)
    return oracle.bf16_from_f64_array((s + bits_to_f64(r).astype(np.float32)).astype(np.float64))


def _logits_numpy(x, W, n_out, cap, scale, div=True, mul=True, round_steps=False):
    """Deliberately broken variants of the logits epilogue (on the oracle's sums)."""
    s, _ = oracle.decode_gemm_f64(x, W[:n_out])
    r = (lambda v: bits_to_f64(oracle.bf16_from_f64_array(v))) if round_steps else (lambda v: v)
    v = r(s)
    if cap > 0:
        v = r(np.tanh(r(v / cap if div else v)))
        v = r(v * cap) if mul else v
    return oracle.bf16_from_f64_array(v * scale)


def _transposed_weight(x, W):
    N, K = W.shape
    return oracle.decode_gemm(x, np.ascontiguousarray(W.reshape(K, N).T))


MUTANTS = {
    # (group, implementation)
    "round_via_binary32": ("round", lambda: _with(bf16_from_f64_array=_round_via_f32)),
    "round_truncate": ("round", lambda: _with(bf16_from_f64_array=_round_truncate)),
    "round_ties_away": ("round", lambda: _with(bf16_from_f64_array=_round_ties_away)),
    "gemm_drop_last_k": ("gemm", lambda: _with(
        decode_gemm=lambda x, W: oracle.decode_gemm(x[:, :-1], W[:, :-1]))),
    "gemm_transposed_weight": ("gemm", lambda: _with(decode_gemm=_transposed_weight)),
    "gemm_sign": ("gemm", lambda: _with(
        decode_gemm=lambda x, W: oracle.decode_gemm(x, W) ^ np.uint16(0x8000))),
    "gemm_wrong_row": ("gemm", lambda: _with(
        decode_gemm=lambda x, W: oracle.decode_gemm(np.roll(x, 1, axis=0), W))),
    "gemm_double_rounding": ("gemm", lambda: _with(decode_gemm=_gemm_from_sums(_round_via_f32))),
    "gemm_truncating_round": ("gemm", lambda: _with(decode_gemm=_gemm_from_sums(_round_truncate))),
    "reduce_from_zero": ("reduce", lambda: _with(reduce_residual=lambda p, r: oracle.reduce_residual(
        np.concatenate([np.zeros_like(p[:1]), p]), r))),
    "reduce_reverse_order": ("reduce", lambda: _with(
        reduce_residual=lambda p, r: oracle.reduce_residual(p[::-1], r))),
    "reduce_drop_last_slot": ("reduce", lambda: _with(
        reduce_residual=lambda p, r: oracle.reduce_residual(p[:-1] if len(p) > 1 else p, r))),
    "reduce_binary64_sum": ("reduce", lambda: _with(reduce_residual=_reduce_f64)),
    "reduce_bf16_each_add": ("reduce", lambda: _with(reduce_residual=_reduce_bf16_each_step)),
    "reduce_fused_residual": ("reduce", lambda: _with(reduce_residual=_reduce_fused_residual)),
    "rms_eps_outside_root": ("rmsnorm", lambda: _with(rmsnorm=_rms_numpy(eps_inside=False))),
    "rms_no_eps": ("rmsnorm", lambda: _with(rmsnorm=_rms_numpy(use_eps=False))),
    "rms_width_off_by_one": ("rmsnorm", lambda: _with(rmsnorm=_rms_numpy(width=HIDDEN - 1))),
    "rms_no_gamma": ("rmsnorm", lambda: _with(rmsnorm=_rms_numpy(use_gamma=False))),
    "rms_sum_not_mean": ("rmsnorm", lambda: _with(rmsnorm=_rms_numpy(width=1))),
    "logits_no_division_by_cap": ("logits", lambda: _with(
        decode_gemm_logits=lambda x, W, n, cap, sc: _logits_numpy(x, W, n, cap, sc, div=False))),
    "logits_no_times_cap": ("logits", lambda: _with(
        decode_gemm_logits=lambda x, W, n, cap, sc: _logits_numpy(x, W, n, cap, sc, mul=False))),
    "logits_scale_ignored": ("logits", lambda: _with(
        decode_gemm_logits=lambda x, W, n, cap, sc: _logits_numpy(x, W, n, cap, 1.0))),
    "logits_slice_from_end": ("logits", lambda: _with(
        decode_gemm_logits=lambda x, W, n, cap, sc: _logits_numpy(x, W[W.shape[0] - n:], n, cap, sc))),
    "logits_bf16_between_ops": ("logits", lambda: _with(
        decode_gemm_logits=lambda x, W, n, cap, sc: _logits_numpy(x, W, n, cap, sc, round_steps=True))),
    "gather_rank_major_rows": ("gather", lambda: _with(
        gather_shards=lambda sh: np.ascontiguousarray(sh).reshape(sh.shape[1], -1))),
    "gather_reversed_ranks": ("gather", lambda: _with(
        gather_shards=lambda sh: oracle.gather_shards(sh[::-1].copy()))),
    "gather_drops_a_column": ("gather", lambda: _with(
        gather_shards=lambda sh: np.concatenate(
            [oracle.gather_shards(sh)[:, 1:], oracle.gather_shards(sh)[:, :1] * 0], axis=1))),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    group, make = MUTANTS[name]
    impl = make()
    caught = []
    for pin_name, pin in PINS.items():
        if not pin_name.startswith(group):
            continue
        try:
            result = pin(impl)
        except Exception as exc:  # a crash on the pin's inputs also exposes the mistake
            result = f"raised {type(exc).__name__}"
        if result:
            caught.append(pin_name)
    assert caught, f"no {group} pin catches mutant {name}"


def test_rmsnorm_binary32_steps_within_one_ulp():
    """The binary32-step evaluation of RMSNorm (the kernel's own precision) stays
    within one BF16 ulp of the binary64 oracle on random rows."""
    from oracle.compare import ulp_distance
    rng = np.random.default_rng(10)
    h = f32_to_bf16_torch(rng.standard_normal((16, HIDDEN)).astype(np.float32))
    g = f32_to_bf16_torch((1 + 0.1 * rng.standard_normal(HIDDEN)).astype(np.float32))
    a = oracle.rmsnorm(h, g, 1e-6)
    b = oracle.rmsnorm_f32_steps(h, g, 1e-6)
    assert int(ulp_distance(a, b).max()) <= 1


def test_gemm_sampled_columns_match_full():
    """The sampled-column mode (used for full-size checks) returns exactly the
    selected columns of the full product."""
    rng = np.random.default_rng(11)
    x = f32_to_bf16_torch(rng.standard_normal((4, 256)).astype(np.float32))
    W = f32_to_bf16_torch((rng.standard_normal((96, 256)) / 16).astype(np.float32))
    full = oracle.decode_gemm(x, W)
    cols = np.array([0, 5, 95, 17, 17])
    assert np.array_equal(oracle.decode_gemm(x, W, cols=cols), full[:, cols])
    s, a = oracle.decode_gemm_f64(x, W, cols=cols)
    assert np.array_equal(oracle.bf16_from_f64_array(s), full[:, cols])
    assert np.all(a >= np.abs(s))
