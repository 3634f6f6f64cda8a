"""The C ABI without a GPU: it builds, exports every declared symbol, rejects bad
arguments before touching CUDA, and its decode-GEMM work split covers every
weight block exactly once (the host planner shares its code with the kernel)."""
import ctypes
import os
import re

import pytest

import skinny_bf16_gemm_gb300 as sk
from skinny_bf16_gemm_gb300 import build as skbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "skinny.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "pages_facts.txt")


@pytest.fixture(scope="module")
def lib():
    skbuild.build()
    return sk.load_library()


def declared_functions():
    names = []
    for line in open(HEADER):
        m = re.match(r"^SKINNY_API\s+[\w\s\*]*?\b(\w+)\s*\(", line)
        if m:
            names.append(m.group(1))
    return names


def pages_facts():
    facts = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].split()
        if len(line) == 2:
            facts[line[0]] = int(line[1], 0)
    return facts


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"decode_gemm_bf16", "reduce_residual_rmsnorm", "skinny_status_string"} <= set(names)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in skinny.h but not exported"


def test_only_declared_symbols_are_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", sk.LIBRARY], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == set(declared_functions())


def test_status_strings(lib):
    for code in range(11):
        assert sk.status_string(code) != "unknown status"
    assert sk.status_string(999) == "unknown status"


def test_header_constants_match_the_pages():
    facts = pages_facts()
    text = open(HEADER).read()
    consts = dict(re.findall(r"#define (SKINNY_\w+) (\d+)", text))
    assert int(consts["SKINNY_HIDDEN"]) == facts["hidden"] == sk.HIDDEN
    # The pages' engine serves up to 32 rows; the library serves up to the row cap.
    assert facts["warp_rows"] <= int(consts["SKINNY_GEMM_MAX_M"]) == facts["twoshot_cap"]
    assert int(consts["SKINNY_GEMM_MAX_M"]) == sk.GEMM_MAX_M
    assert int(consts["SKINNY_REDUCE_MAX_M"]) == facts["twoshot_cap"] == sk.REDUCE_MAX_M
    # The ArNorm geometry the pages print: 8 CTAs x 112 fragments x 8 BF16 = 7168.
    assert facts["ar_ctas"] * facts["ar_frags_per_cta"] * facts["fragment_bf16"] == facts["hidden"]
    assert facts["ar_cols_per_cta"] == facts["ar_frags_per_cta"] * facts["fragment_bf16"]


def _gate(n, k, facts):
    """The pages' warp split-K shape gate (drafter/linears, warp_eligible)."""
    if n % facts["gate_n_multiple"] or k % facts["gate_k_multiple"]:
        return False
    tiles = facts["gate_max_k_tiles"]
    return k // 128 <= tiles or (k % 256 == 0 and k // 256 <= tiles)


def test_accepted_shapes_cover_the_pages_gate(lib):
    """Every (N, K) the pages' gate serves is accepted here (plus K = 18432 of the
    layer chain, which the gate refuses); the gate's own example holds."""
    facts = pages_facts()
    assert facts["tp1_down_k"] // 256 == facts["tp1_down_k_tiles"]
    assert _gate(7168, facts["tp1_down_k"], facts)
    assert not _gate(7168, 18432, facts)
    for n in (16, 2048, 4096, 7168, 12288, 18432, 20480):
        for k in (128, 7168, 14336, 18432):
            for m in (1, 32, 64):
                sk.gemm_plan(m, n, k, 152)


@pytest.mark.parametrize("args,code", [
    ((0, 16, 64), 2), ((65, 16, 64), 2), ((4, 0, 64), 2), ((4, 16, 0), 2), ((4, 16, 12), 2),
])
def test_gemm_rejects_shapes_before_cuda(lib, args, code):
    M, N, K = args
    buf = ctypes.create_string_buffer(1 << 16)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
    assert lib.decode_gemm_bf16(p, p + 8192, p + 16384, M, N, K, None) == code


def test_gemm_rejects_null_alignment_alias_before_cuda(lib):
    buf = ctypes.create_string_buffer(1 << 20)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
    assert lib.decode_gemm_bf16(None, p, p + 65536, 4, 16, 64, None) == 1
    assert lib.decode_gemm_bf16(p, None, p + 65536, 4, 16, 64, None) == 1
    assert lib.decode_gemm_bf16(p, p + 4096, None, 4, 16, 64, None) == 1
    assert lib.decode_gemm_bf16(p + 8, p + 4096, p + 65536, 4, 16, 64, None) == 3
    assert lib.decode_gemm_bf16(p, p + 4104, p + 65536, 4, 16, 64, None) == 3
    assert lib.decode_gemm_bf16(p, p + 4096, p + 65537, 4, 16, 64, None) == 3
    # out overlapping x, out overlapping W
    assert lib.decode_gemm_bf16(p, p + 4096, p + 256, 4, 16, 64, None) == 6
    assert lib.decode_gemm_bf16(p, p + 4096, p + 4096 + 512, 4, 16, 64, None) == 6


def test_reduce_rejects_before_cuda(lib):
    buf = ctypes.create_string_buffer(1 << 22)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
    row = 7168 * 2
    part, res, gam, out, rout = p, p + 8 * row * 2, p + 10 * row * 2, p + 11 * row * 2, p + 13 * row * 2
    f = lib.reduce_residual_rmsnorm
    assert f(None, 8, res, gam, out, rout, 2, 1e-6, None) == 1
    assert f(part, 8, res, None, out, rout, 2, 1e-6, None) == 1
    assert f(part, 0, res, gam, out, rout, 2, 1e-6, None) == 2
    assert f(part, 9, res, gam, out, rout, 2, 1e-6, None) == 2
    assert f(part, 8, res, gam, out, rout, 0, 1e-6, None) == 2
    assert f(part, 8, res, gam, out, rout, 65, 1e-6, None) == 2
    assert f(part, 8, res, gam, out, rout, 2, 0.0, None) == 10
    assert f(part, 8, res, gam, out, rout, 2, float("nan"), None) == 10
    assert f(part, 8, res, gam, out, rout, 2, float("inf"), None) == 10
    assert f(part + 2, 8, res, gam, out, rout, 2, 1e-6, None) == 3
    assert f(part, 8, res, gam, out + 8, rout, 2, 1e-6, None) == 3
    assert f(part, 8, res, gam, out, out, 2, 1e-6, None) == 6          # out == residual_out
    assert f(part, 8, res, gam, part, rout, 2, 1e-6, None) == 6        # out over partials
    assert f(part, 8, res, gam, out, res + 16, 2, 1e-6, None) == 6     # partial residual overlap


def test_fused_rejects_before_cuda(lib):
    buf = ctypes.create_string_buffer(1 << 23)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
    MB = 1 << 20
    x, W, part, res, gam, out, rout = p, p + 65536, p + 2 * MB, p + 3 * MB, p + 3 * MB + 65536, \
        p + 4 * MB, p + 5 * MB
    f = lib.decode_gemm_bf16_reduce_rmsnorm
    names = ["x", "W", "part", "TP", "res", "gam", "out", "rout", "M", "K", "eps", "s"]
    ok = dict(zip(names, (x, W, part, 8, res, gam, out, rout, 2, 64, 1e-6, None)))

    def call(**kw):
        args = dict(ok)
        args.update(kw)
        return f(*[args[n] for n in names])
    for name in ("x", "W", "part", "gam", "out", "rout"):
        assert call(**{name: None}) == 1
    assert call(M=0) == 2 and call(M=65) == 2
    assert call(TP=0) == 2 and call(TP=9) == 2
    assert call(K=60) == 2 and call(K=0) == 2
    assert call(eps=0.0) == 10 and call(eps=float("nan")) == 10
    assert call(x=x + 8) == 3 and call(part=part + 2) == 3 and call(out=out + 8) == 3
    assert call(out=rout) == 6                          # out == residual_out
    assert call(out=part + 256) == 6                    # out over the slots
    assert call(part=W + 4096) == 6                     # slot 0 written over W
    assert call(rout=res + 16) == 6                     # partial residual overlap


def test_gather_rejects_before_cuda(lib):
    buf = ctypes.create_string_buffer(1 << 20)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
    f = lib.gather_shards_bf16
    assert f(None, 8, 4, 64, p + 65536, None) == 1
    assert f(p, 8, 4, 64, None, None) == 1
    assert f(p, 0, 4, 64, p + 65536, None) == 2
    assert f(p, 65, 4, 64, p + 65536, None) == 2
    assert f(p, 8, 0, 64, p + 65536, None) == 2
    assert f(p, 8, 4, 12, p + 65536, None) == 2
    assert f(p, 8, 4, 0, p + 65536, None) == 2
    assert f(p + 8, 8, 4, 64, p + 65536, None) == 3
    assert f(p, 8, 4, 64, p + 2048, None) == 6


def test_calls_without_a_device_report_device_error(lib):
    """With valid arguments but no CUDA device the call fails cleanly."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    buf = ctypes.create_string_buffer(1 << 20)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
    assert lib.decode_gemm_bf16(p, p + 4096, p + 65536, 4, 16, 64, None) == 4


SHAPES = [(1, 16, 64, 152), (4, 2048, 7168, 152), (16, 18432, 7168, 152), (16, 18432, 7168, 148),
          (16, 7168, 18432, 152), (32, 20480, 7168, 152), (3, 200, 136, 152),
          (8, 128, 64, 152), (5, 12288, 7168, 148), (2, 4096, 7168, 7), (1, 1, 8, 152),
          (32, 1000, 1000, 152), (7, 300, 4096, 64), (64, 18432, 7168, 152),
          (48, 7168, 14336, 152), (33, 130, 72, 152), (8, 65536, 2048, 152),
          (3, 40000, 1000, 152)]


def _random_shapes(count, seed=20261202):
    # Seeded shapes across the accepted range: any M in 1..64, any N, K a
    # multiple of 8, and SM counts from tiny to a full GB300.
    import random
    r = random.Random(seed)
    out = []
    for _ in range(count):
        out.append((r.randint(1, 64), r.choice([r.randint(1, 300), r.randint(1, 30000)]),
                    8 * r.choice([r.randint(1, 40), r.randint(1, 2600)]),
                    r.choice([1, 3, 7, 64, 148, 152])))
    return out


SHAPES += _random_shapes(40)


@pytest.mark.parametrize("M,N,K,expect_shallow", [
    (4, 2048, 7168, True), (16, 4096, 7168, True), (32, 4096, 7168, True),
    (16, 12288, 7168, True), (16, 7168, 14336, True), (17, 12288, 7168, False),
    (32, 7168, 14336, False), (16, 18432, 7168, False), (16, 7168, 18432, False),
    (64, 18432, 7168, False), (64, 7168, 14336, False), (3, 200, 136, True),
    (64, 4096, 7168, False), (33, 2048, 7168, False), (48, 200, 136, False)])
def test_ring_depth_follows_weight_bytes_per_cta(lib, M, N, K, expect_shallow):
    """With programmatic dependent launch the shallow ring (two CTAs per SM) is
    taken below 1 MiB of weights per CTA (1.5 MiB for up to 16 rows, never for
    more than 32), the deep ring (more bytes in flight) above; without it always
    the deep ring."""
    prev = sk.set_pdl(False)
    try:
        deep = sk.gemm_plan(M, N, K, 152)
        sk.set_pdl(True)
        plan = sk.gemm_plan(M, N, K, 152)
    finally:
        sk.set_pdl(prev)
    per_cta = plan.blocks * 128 * 64 * 2 / plan.ctas
    limit = 0 if M > 32 else (1.5 if M <= 16 else 1) * 2 ** 20
    assert (per_cta < limit) == expect_shallow
    if expect_shallow:
        assert plan.stages < deep.stages
        assert 2 * (plan.smem_bytes + 1024) <= 233472  # two CTAs fit on an SM
    else:
        assert (plan.stages, plan.smem_bytes) == (deep.stages, deep.smem_bytes)
        assert deep.smem_bytes > 233472 // 2


@pytest.mark.parametrize("M,N,K,sms", SHAPES)
def test_work_split_covers_every_block_once(lib, M, N, K, sms):
    plan = sk.gemm_plan(M, N, K, sms)
    assert plan.tiles == -(-N // 128) and plan.kblocks == -(-K // 64)
    assert plan.blocks == plan.tiles * plan.kblocks
    # One whole tile per CTA when the tiles fill at least 90 % of the SMs, else
    # one CTA per SM (never more CTAs than weight blocks).
    tiles = -(-N // 128)
    want = tiles if tiles <= sms and 10 * tiles >= 9 * sms else min(sms, plan.blocks)
    assert plan.ctas == want
    if plan.ctas == tiles:
        assert plan.split_tiles == 0
    assert plan.mma_n == (16 if M <= 16 else (32 if M <= 32 else 64))
    assert plan.smem_bytes <= 232448
    seen = {}
    per_cta = []
    contributors = {}
    slots = set()
    for c in range(plan.ctas):
        pieces = sk.gemm_cta_pieces(M, N, K, sms, c, max_pieces=plan.tiles + 1)
        assert pieces, f"CTA {c} has no work"
        n_blocks = 0
        for (t, kb0, kb1, slot) in pieces:
            assert 0 <= kb0 < kb1 <= plan.kblocks
            for kb in range(kb0, kb1):
                assert (t, kb) not in seen, f"block {(t, kb)} twice"
                seen[(t, kb)] = c
            n_blocks += kb1 - kb0
            whole = kb0 == 0 and kb1 == plan.kblocks
            assert (slot == -1) == whole
            if not whole:
                assert slot not in slots and 0 <= slot < 2 * plan.ctas
                slots.add(slot)
            contributors.setdefault(t, []).append(c)
        per_cta.append(n_blocks)
    assert len(seen) == plan.blocks
    # Balanced: every CTA streams the same number of blocks, give or take one.
    assert max(per_cta) - min(per_cta) <= 1
    # Contributors of a tile are consecutive CTAs; ranges go to CTAs in reverse
    # block order, so along K the block index falls. The finisher (the CTA holding
    # the tile's first K blocks) is distinct for every shared tile.
    finishers = []
    for t, cs in contributors.items():
        cs = sorted(cs)
        assert cs == list(range(cs[0], cs[0] + len(cs)))
        order = [seen[(t, kb)] for kb in range(plan.kblocks)]
        assert order == sorted(order, reverse=True)
        if len(cs) > 1:
            finishers.append(seen[(t, 0)])
    assert len(finishers) == len(set(finishers)) == plan.split_tiles


@pytest.mark.parametrize("M,N,K,sms", SHAPES)
def test_split_k_waits_point_to_lower_block_indices(lib, M, N, K, sms):
    """Every wait of the split-K fix-up goes from a tile's finisher to the
    tile's other contributors. The finisher is the CTA for which the tile is its
    last piece and which holds the tile's first K blocks; every CTA it waits for
    has a lower block index. Blocks are dispatched in index order, so each CTA
    waited for is running or done before its waiter starts, and the kernel makes
    progress even when only some of its CTAs fit on the GPU at once."""
    plan = sk.gemm_plan(M, N, K, sms)
    pieces = {c: sk.gemm_cta_pieces(M, N, K, sms, c, max_pieces=plan.tiles + 1)
              for c in range(plan.ctas)}
    by_tile = {}
    for c, ps in pieces.items():
        for q, (t, kb0, kb1, slot) in enumerate(ps):
            by_tile.setdefault(t, []).append((c, q, kb0, kb1))
    edges = 0
    for t, entries in by_tile.items():
        if len(entries) == 1:
            continue
        finisher = [e for e in entries if e[2] == 0]
        assert len(finisher) == 1
        c_fin, q_fin = finisher[0][0], finisher[0][1]
        assert q_fin == len(pieces[c_fin]) - 1, "a finisher finishes its last piece"
        for c, q, kb0, kb1 in entries:
            if c != c_fin:
                assert c < c_fin, (t, c, c_fin)
                edges += 1
    assert (edges > 0) == (plan.split_tiles > 0)


def test_l2_prefetch_setting_round_trips_and_rejects_out_of_range(lib):
    """skinny_set_l2_prefetch returns the previous lead, accepts [0, 64] and
    leaves the setting unchanged (returning -1) outside it."""
    prev = lib.skinny_set_l2_prefetch(0)
    try:
        assert 0 <= prev <= 64
        assert lib.skinny_set_l2_prefetch(64) == 0
        assert lib.skinny_set_l2_prefetch(-1) == -1
        assert lib.skinny_set_l2_prefetch(65) == -1
        assert lib.skinny_set_l2_prefetch(6) == 64
        with pytest.raises(ValueError):
            sk.set_l2_prefetch(100)
        assert sk.set_l2_prefetch(3) == 6
    finally:
        lib.skinny_set_l2_prefetch(prev)


def test_default_l2_prefetch_is_six(lib):
    prev = lib.skinny_set_l2_prefetch(6)
    lib.skinny_set_l2_prefetch(prev)
    # A fresh process starts at the library default.
    import subprocess, sys
    code = ("import skinny_bf16_gemm_gb300 as sk; lib = sk.load_library(); "
            "print(lib.skinny_set_l2_prefetch(0))")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "6"


def test_ex_entry_points_validate_options_before_cuda(lib):
    """The per-call launch settings are checked before anything touches CUDA:
    a field out of range is SKINNY_ERR_ARG; SKINNY_OPT_DEFAULT (-1) or NULL
    takes the process-wide setting (here the call then fails for lack of a
    device, or runs on a GPU machine)."""
    import torch
    buf = ctypes.create_string_buffer(1 << 22)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
    bad = [sk.LaunchOpts(2, 0), sk.LaunchOpts(-2, 0), sk.LaunchOpts(1, 65),
           sk.LaunchOpts(0, -2), sk.LaunchOpts(1, 0, 65), sk.LaunchOpts(1, 0, -2)]
    row = 7168 * 2
    part, res, gam, out, rout = p, p + 8 * row * 2, p + 10 * row * 2, p + 11 * row * 2, \
        p + 13 * row * 2
    for o in bad:
        r = ctypes.byref(o)
        assert lib.decode_gemm_bf16_ex(p, p + 4096, p + 65536, 4, 16, 64, r, None) == 10
        assert lib.reduce_residual_rmsnorm_ex(part, 8, res, gam, out, rout, 2, 1e-6, r,
                                              None) == 10
        assert lib.decode_gemm_bf16_reduce_rmsnorm_ex(p, p + 65536, p + (2 << 20), 8, None,
                                                      p + (3 << 20), p + (4 << 20),
                                                      p + (5 << 20), 2, 64, 1e-6, r, None) == 10
    if not torch.cuda.is_available():
        for o in (None, ctypes.byref(sk.LaunchOpts(-1, -1)), ctypes.byref(sk.LaunchOpts(1, 0))):
            assert lib.decode_gemm_bf16_ex(p, p + 4096, p + 65536, 4, 16, 64, o, None) == 4
    # Shape errors still come first.
    assert lib.decode_gemm_bf16_ex(p, p + 4096, p + 65536, 0, 16, 64,
                                   ctypes.byref(sk.LaunchOpts(1, 0)), None) == 2


def test_selftests_check_their_limits_before_cuda(lib):
    """Both failure-path self-tests reject a wait limit outside [1 us, 2 s] with
    SKINNY_ERR_ARG before touching CUDA; the reduce's also checks its other
    arguments as reduce_residual_rmsnorm does."""
    import torch
    buf = ctypes.create_string_buffer(1 << 22)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
    row = 7168 * 2
    part, res, gam, out, rout = p, p + 8 * row * 2, p + 10 * row * 2, p + 11 * row * 2, \
        p + 13 * row * 2
    for bad in (0, 999, 3_000_000_000):
        assert lib.skinny_watchdog_selftest(p, p + 4096, p + 65536, 4, 16, 64, bad, None) == 10
        assert lib.skinny_reduce_selftest(part, 8, res, gam, out, rout, 2, 1e-6, bad, None) == 10
    assert lib.skinny_reduce_selftest(part, 9, res, gam, out, rout, 2, 1e-6, 10**6, None) == 2
    assert lib.skinny_reduce_selftest(None, 8, res, gam, out, rout, 2, 1e-6, 10**6, None) == 1
    assert lib.skinny_reduce_selftest(part, 8, res, gam, out, out, 2, 1e-6, 10**6, None) == 6
    if not torch.cuda.is_available():
        assert lib.skinny_reduce_selftest(part, 8, res, gam, out, rout, 2, 1e-6, 10**6, None) == 4


def test_process_settings_are_thread_safe_and_ex_calls_leave_them(lib):
    """Two host threads: one flips the process-wide settings, the other makes
    _ex calls with its own settings. The _ex calls never change the process-wide
    settings, and the setters stay consistent under contention."""
    import threading
    prev_pdl, prev_lead = lib.skinny_set_pdl(0), lib.skinny_set_l2_prefetch(5)
    stop = threading.Event()
    seen = []

    def flipper():
        k = 0
        while not stop.is_set():
            lib.skinny_set_pdl(k & 1)
            lib.skinny_set_l2_prefetch(5)
            k += 1

    def caller():
        buf = ctypes.create_string_buffer(1 << 20)
        p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
        o = ctypes.byref(sk.LaunchOpts(1, 64))
        for _ in range(2000):
            seen.append(lib.decode_gemm_bf16_ex(p, p + 4096, p + 65536, 0, 16, 64, o, None))

    t1, t2 = threading.Thread(target=flipper), threading.Thread(target=caller)
    t1.start()
    t2.start()
    t2.join()
    stop.set()
    t1.join()
    try:
        assert set(seen) == {2}
        assert lib.skinny_set_l2_prefetch(5) == 5  # never the _ex calls' 64
    finally:
        lib.skinny_set_pdl(prev_pdl)
        lib.skinny_set_l2_prefetch(prev_lead)


def test_gemm_rejects_block_counts_beyond_32_bits(lib):
    """The kernel counts 128 x 64 weight blocks in 32-bit integers: a shape with
    2^31 blocks or more is rejected before anything else happens."""
    buf = ctypes.create_string_buffer(1 << 16)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
    N, K = 2 ** 31 - 128, 2 ** 20 * 8  # ceil(N/128) * ceil(K/64) >= 2^31
    assert lib.decode_gemm_bf16(p, p + 8192, p + 16384, 4, N, K, None) == 2
    plan = sk.GemmPlan()
    assert lib.skinny_gemm_plan_query(4, N, K, 152, ctypes.byref(plan)) == 2
