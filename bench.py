"""Benchmark: the synthetic drafter layer chain on GB300, one JSON line.

One step = one pass of the whole hot path: 3 drafter layers, each a decode GEMM
[16, 7168] -> [16, 18432], a decode GEMM [16, 18432] -> [16, 7168] into slot 0 of
the [8, 16, 7168] partial rows, and reduce + residual + RMSNorm over the 8 slots.
Metric: achieved HBM GB/s = algorithmic bytes of the step / step time. The
weights (1.585 GB) are far larger than L2 (~126 MB), so every step streams them
from HBM; nothing is flushed in between.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (oracle/, test infrastructure) on a bounded
sample of the same workload on the host cores. N > 1 (torchrun, one rank per GPU)
runs independent replicas: the path has no exchange step on one node.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "achieved HBM GB/s (and % of GB300 peak) for decode GEMM and reduce+RMSNorm"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_gemm_traffic.json")
GEMM_SOURCES = ["skinny_bf16_gemm_gb300/csrc/decode_gemm.cu", "skinny_bf16_gemm_gb300/csrc/ptx.cuh",
                "skinny_bf16_gemm_gb300/csrc/plan.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--pdl", type=int, default=1, help="programmatic dependent launch")
    ap.add_argument("--graph", type=int, default=0, help="replay the step as a CUDA graph")
    ap.add_argument("--fused", type=int, default=1,
                    help="each layer's second GEMM and reduce + RMSNorm through "
                         "decode_gemm_bf16_reduce_rmsnorm (bit-identical; 0: the two calls)")
    ap.add_argument("--l2-prefetch", type=int, default=0,
                    help="weight blocks each decode GEMM CTA (deep ring) prefetches to L2 "
                         "before its PDL wait, in the chain (library default 6)")
    ap.add_argument("--l2-after-reduce", type=int, default=16,
                    help="with --fused 1: weight blocks each first GEMM's CTA prefetches to L2 "
                         "once the reduce before it has seen its GEMM complete (0: off)")
    ap.add_argument("--e2e-group", type=int, default=4,
                    help="end-to-end timing: steps per group of buffer sets whose inputs go up "
                         "together (one cross-stream wait per group)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="per-config GB/s of every GEMM and reduce config instead of the chain")
    ap.add_argument("--sweep-calls", type=int, default=200)
    ap.add_argument("--configs", type=int, default=1,
                    help="add the per-config block (every GEMM / reduce / gather config of "
                         "the workloads, with the oracle per config kind) to the line")
    ap.add_argument("--profile", action="store_true",
                    help="a few launches of each chain kernel, for ncu captures")
    ap.add_argument("--profile-configs", action="store_true",
                    help="two launches of every GEMM / reduce / gather config, for a per-call "
                         "ncu launch list")
    ap.add_argument("--config-filter", default="",
                    help="with --profile-configs: only configs whose label contains this")
    return ap.parse_args()


def dist_info():
    from skinny_bf16_gemm_gb300.replicas import rank_info
    return rank_info()


def workload_config(cfg, extra=None):
    c = {"workload": "synthetic drafter layer chain (3 layers: 16x7168->18432 GEMM, "
                     "16x18432->7168 GEMM, reduce+residual+RMSNorm TP=8 M=16)",
         "layers": cfg.layers, "M": cfg.M, "hidden": cfg.hidden, "ffn": cfg.ffn, "TP": cfg.TP,
         "weight_bytes": cfg.weight_bytes(), "step_bytes": cfg.step_bytes(),
         "l2_policy": "inputs larger than L2 (1.585 GB of weights streamed per step)"}
    if extra:
        c.update(extra)
    return c


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def gemm_source_hash():
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(shape_key):
    """DRAM bytes per launch of the decode GEMM from the committed ncu summary,
    or None if absent or taken on a different version of the kernel."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("source_hash") != gemm_source_hash():
        return None
    entry = t.get("per_launch_bytes", {}).get(shape_key)
    return None if entry is None else float(entry)


def host_lead(stream):
    """A ~1 ms spin on the stream just before a timed region's start event, so
    that the host has enqueued the first timed kernels by the time the event
    is reached: the region then times the GPU's work, not Python's first
    launches after the synchronisation."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)


def keep_streaming(device, seconds):
    """Device-to-device copies of a 256 MB buffer for about `seconds` (host
    time): keeps HBM and the SMs busy while the host waits on something."""
    src = torch.empty(1 << 28, dtype=torch.uint8, device=device)
    dst = torch.empty_like(src)
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(50):
            dst.copy_(src)
        torch.cuda.synchronize()
    del src, dst


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---- the oracle as the CPU baseline / reference arm ------------------------------

def host_cores():
    """Host cores this process may run on: the thread count every all-core oracle
    timing passes explicitly (OpenMP keeps the last count it was given)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_chain_sample(inp_bits, cfg, cols1, cols2, threads=0):
    """One chain step by the oracle on sampled GEMM output columns. The reduce and
    RMSNorm run on full rows; the sampled columns of GEMM2 fill slot 0 where
    computed (the rest of slot 0 keeps the previous values). Returns the
    algorithmic bytes the sample covers."""
    import oracle
    x = inp_bits["x0"]
    res = inp_bits["res0"]
    M, H, F = cfg.M, cfg.hidden, cfg.ffn
    h1 = np.zeros((M, F), dtype=np.uint16)
    slot0 = np.zeros((M, H), dtype=np.uint16)
    nbytes = 0
    for l in range(cfg.layers):
        W1 = inp_bits["W1"][l]
        W2 = inp_bits["W2"][l]
        h1[:, cols1] = oracle.decode_gemm(x, W1[cols1], cols=np.arange(len(cols1)), threads=threads)
        slot0[:, cols2] = oracle.decode_gemm(h1, W2[cols2], cols=np.arange(len(cols2)),
                                             threads=threads)
        p = np.concatenate([slot0[None], inp_bits["peers"][l]], axis=0)
        out, res = oracle.reduce_residual_rmsnorm(p, res, inp_bits["gamma"][l], cfg.eps)
        x = out
        nbytes += (2 * len(cols1) * H + 2 * M * H + 2 * M * len(cols1)
                   + 2 * len(cols2) * F + 2 * M * F + 2 * M * len(cols2)
                   + cfg.reduce().algorithmic_bytes())
    return nbytes


def host_chain_bits(cfg, seed):
    """Chain inputs as BF16 patterns on the host, from the seeded generator."""
    inp = workloads.chain_inputs(cfg, seed, device="cpu")
    return {"W1": [workloads.bits(w) for w in inp.W1], "W2": [workloads.bits(w) for w in inp.W2],
            "peers": [workloads.bits(p) for p in inp.peers],
            "gamma": [workloads.bits(g) for g in inp.gamma],
            "x0": workloads.bits(inp.x0), "res0": workloads.bits(inp.residual0)}


def _gemm_literal_report(got_bits, ref, ssum, asum):
    """The decode GEMM tolerance verdict plus the literal ulp statistics."""
    from oracle import compare
    rep = compare.gemm_check(got_bits, ref, ssum, asum)
    lit = compare.ulp_distance(got_bits, ref)
    small = np.abs(ssum) < compare.FLOOR_SCALE * asum
    keep = ("ok", "n", "within1_frac", "max_judged", "below_floor", "literal_hist",
            "literal_within1_frac", "literal_max")
    out = {k: rep[k] for k in keep}
    out["literal_gt2_above_floor"] = int(((lit > 2) & ~small).sum())
    out["literal_gt2_below_floor"] = int(((lit > 2) & small).sum())
    return out


def chain_parity(inp, cfg, sk):
    """The oracle beside the GPU on the timed chain's own inputs (part of the CPU
    baseline leg): every output element of layer 0's two GEMMs, judged by the
    GEMM tolerance with the literal ulp histogram, and cuBLAS (torch.mm) on the
    same inputs judged the same way; then layer 0's reduce + residual + RMSNorm
    on whole rows (residual bit for bit, out in ulps)."""
    import oracle
    from oracle import compare
    dev = inp.x0.device
    h1 = torch.empty(cfg.M, cfg.ffn, dtype=torch.bfloat16, device=dev)
    parts = torch.empty(cfg.TP, cfg.M, cfg.hidden, dtype=torch.bfloat16, device=dev)
    parts[1:].copy_(inp.peers[0])
    out = torch.empty(cfg.M, cfg.hidden, dtype=torch.bfloat16, device=dev)
    rout = torch.empty_like(out)
    sk.decode_gemm_bf16(inp.x0, inp.W1[0], h1)
    sk.decode_gemm_bf16(h1, inp.W2[0], parts[0])
    sk.reduce_residual_rmsnorm(parts, inp.residual0, inp.gamma[0], out, rout, cfg.eps)
    cub1 = torch.mm(inp.x0, inp.W1[0].t())
    cub2 = torch.mm(h1, inp.W2[0].t())  # the same input as our second GEMM
    torch.cuda.synchronize()
    report = {"gemm_columns": "all"}
    for name, x, W, y, c in (("gemm1", inp.x0, inp.W1[0], h1, cub1),
                             ("gemm2", h1, inp.W2[0], parts[0], cub2)):
        xb, wb = workloads.bits(x), workloads.bits(W)
        ref = oracle.decode_gemm(xb, wb)
        ssum, asum = oracle.decode_gemm_f64(xb, wb)
        report[name] = _gemm_literal_report(workloads.bits(y), ref, ssum, asum)
        report[name + "_cublas"] = _gemm_literal_report(workloads.bits(c), ref, ssum, asum)
    want_h = oracle.reduce_residual(workloads.bits(parts), workloads.bits(inp.residual0))
    want_o = oracle.rmsnorm(want_h, workloads.bits(inp.gamma[0]), cfg.eps)
    d = compare.ulp_distance(workloads.bits(out), want_o)
    report["reduce"] = {"residual_bit_exact": compare.bits_equal(workloads.bits(rout), want_h),
                        "out_ulp_hist": compare.histogram(d), "out_ulp_max": int(d.max())}
    return report


def time_oracle(cfg, budget_s, steps=None, warmup=0, seed=0, threads=None):
    """Time the oracle on the chain workload on the host cores (all of them, or
    `threads`).

    Each step covers sampled GEMM output columns sized to about budget_s of CPU
    work (all columns if a whole step fits). steps=None: repeat steps until about
    budget_s has elapsed in total (at least one)."""
    import oracle
    from oracle import build as obuild
    obuild.build()
    bits = host_chain_bits(cfg, seed)
    threads = host_cores() if threads is None else threads
    probe = 64
    t0 = time.perf_counter()
    oracle_chain_sample(bits, cfg, np.arange(probe), np.arange(probe), threads)
    per_col = (time.perf_counter() - t0) / probe
    n = int(max(16, budget_s / max(per_col, 1e-9)))
    rng = np.random.default_rng(seed)
    cols1 = np.sort(rng.choice(cfg.ffn, size=min(cfg.ffn, n), replace=False)).astype(np.int32)
    cols2 = np.sort(rng.choice(cfg.hidden, size=min(cfg.hidden, n), replace=False)).astype(np.int32)
    for _ in range(warmup):
        oracle_chain_sample(bits, cfg, cols1, cols2, threads)
    done, nbytes = 0, 0
    t0 = time.perf_counter()
    while True:
        nbytes += oracle_chain_sample(bits, cfg, cols1, cols2, threads)
        done += 1
        dt = time.perf_counter() - t0
        if (steps is not None and done >= steps) or (steps is None and dt >= budget_s):
            break
    sample = (f"{len(cols1)} of {cfg.ffn} GEMM1 and {len(cols2)} of {cfg.hidden} GEMM2 output "
              f"columns per layer (oracle FP64 dot products), full reduce+RMSNorm rows, "
              f"{cfg.layers} layers per step; {done} step(s) in {dt:.1f} s")
    return {"value": nbytes / dt / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": sample, "seconds": dt, "steps": done}


def run_reference(args, rank, world, cfg):
    if rank != 0:
        return 0
    total = max(1, args.steps + args.warmup)
    budget = max(0.02, min(10.0, 150.0 / total))
    r = time_oracle(cfg, budget, steps=max(1, args.steps), warmup=args.warmup)
    line = {"metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * r["seconds"] / r["steps"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "impl": "reference", "config": workload_config(cfg),
            "cpu_baseline": {"value": r["value"], "unit": UNIT, "cores": r["cores"],
                             "kind": "oracle", "sample": r["sample"]},
            "e2e": {"value": r["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- per-config sweep ----------------------------------------------------------------

def _l2_bytes():
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 126 * 2 ** 20


def _rotation(nbytes):
    """Copies of a buffer so that the rotation spans at least 3x L2."""
    return max(2, -(-3 * _l2_bytes() // max(nbytes, 1)))


def _time_calls(fn, calls, copies, stream):
    """Device time per call of `calls` back-to-back calls (rotating through the
    buffer copies), captured once as a CUDA graph so host launch overhead does
    not enter the number; the graph is replayed five times, timed with CUDA events; the median is kept."""
    for i in range(min(copies, 8)):
        fn(i % copies)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i in range(calls):
                fn(i % copies)
    stream.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(5):
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / calls)
    del graph
    return statistics.median(times)


GATHER_CONFIGS = [(8, m, 896) for m in (1, 16, 64)] + [(8, m, 2560) for m in (1, 8, 32, 64)]


def _entry(peak, nb, t_ms, **fields):
    gbs = nb / (t_ms * 1e-3) / 1e9
    fields.update({"us": t_ms * 1e3, "GBps": gbs, "frac_measured": gbs / peak,
                   "frac_nominal_8000": gbs / 8000.0, "bytes": nb})
    return fields


def measure_configs(sk, calls, peak):
    """Per-call time of every GEMM, reduce and gather config (PR1, the reduce
    sweep with and without residual, the GEMM sweep, lm_head, the wider shapes,
    the chain's two GEMMs and the local gather), each from a CUDA graph of
    `calls` back-to-back calls rotating through buffer copies that span at least
    3x L2 (median of 5 replays); cuBLAS (torch.mm) timed the same way beside
    every GEMM."""
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    out_sets = {"pr1": {}, "gemm_sweep": [], "lm_head": [], "wider": [], "chain_gemms": [],
                "reduce_sweep": [], "gather": []}
    gemms = ([("pr1", workloads.PR1_GEMM)] + [("gemm_sweep", g) for g in workloads.GEMM_SWEEP]
             + [("lm_head", g) for g in workloads.LM_HEAD]
             + [("wider", g) for g in workloads.GEMM_WIDER]
             + [("chain_gemms", workloads.CHAIN.gemm1()), ("chain_gemms", workloads.CHAIN.gemm2())])
    for label, g in gemms:
        copies = _rotation(g.weight_bytes())
        gen = torch.Generator(device=dev)
        gen.manual_seed(workloads.seed_for("sweep", g.M, g.N, g.K))
        Ws = [(torch.randn(g.N, g.K, device=dev, generator=gen) / g.K ** 0.5).to(torch.bfloat16)
              for _ in range(copies)]
        x = torch.randn(g.M, g.K, device=dev, generator=gen).to(torch.bfloat16)
        out = torch.empty(g.M, g.N, device=dev, dtype=torch.bfloat16)
        ours = _time_calls(lambda i: sk.decode_gemm_bf16(x, Ws[i], out), calls, copies, stream)
        cub = _time_calls(lambda i: torch.mm(x, Ws[i].t(), out=out), calls, copies, stream)
        nb = g.algorithmic_bytes()
        e = _entry(peak, nb, ours, M=g.M, N=g.N, K=g.K, cublas_us=cub * 1e3,
                   cublas_GBps=nb / (cub * 1e-3) / 1e9, rotation_copies=copies)
        if label == "pr1":
            out_sets["pr1"]["gemm"] = e
        else:
            out_sets[label].append(e)
        del Ws
        torch.cuda.empty_cache()
    reduces = [("pr1", workloads.PR1_REDUCE)] + [("reduce_sweep", r) for r in workloads.REDUCE_SWEEP]
    for label, r in reduces:
        per = 2 * r.width * r.M * (r.TP + 1)
        copies = _rotation(per)
        parts = [torch.randn(r.TP, r.M, r.width, device=dev).to(torch.bfloat16)
                 for _ in range(copies)]
        ress = [torch.randn(r.M, r.width, device=dev).to(torch.bfloat16) if r.residual else None
                for _ in range(copies)]
        gamma = (1 + 0.1 * torch.randn(r.width, device=dev)).to(torch.bfloat16)
        out = torch.empty(r.M, r.width, device=dev, dtype=torch.bfloat16)
        rout = torch.empty_like(out)
        t = _time_calls(lambda i: sk.reduce_residual_rmsnorm(parts[i], ress[i], gamma, out, rout),
                        calls, copies, stream)
        e = _entry(peak, r.algorithmic_bytes(), t, TP=r.TP, M=r.M, residual=r.residual,
                   rotation_copies=copies)
        if label == "pr1":
            out_sets["pr1"]["reduce"] = e
        else:
            out_sets[label].append(e)
        del parts, ress
        torch.cuda.empty_cache()
    for TP, M, S in GATHER_CONFIGS:
        per = 2 * TP * M * S
        copies = _rotation(per)
        shards = [torch.randn(TP, M, S, device=dev).to(torch.bfloat16) for _ in range(copies)]
        out = torch.empty(M, TP * S, device=dev, dtype=torch.bfloat16)
        t = _time_calls(lambda i: sk.gather_shards_bf16(shards[i], out), calls, copies, stream)
        out_sets["gather"].append(_entry(peak, 2 * per, t, TP=TP, M=M, S=S,
                                         set="context" if S == 896 else "logits",
                                         rotation_copies=copies))
        del shards
        torch.cuda.empty_cache()
    return out_sets


def oracle_configs(budget_s=2.0, seed=0):
    """The oracle timed on the host cores on each config kind of the report:
    PR1's GEMM and reduce whole, the reduce sweep and the gathers whole, the
    GEMM sweep, lm_head and wider shapes on sampled output columns (the bytes
    counted are those of the sample). Each kind repeats for about budget_s."""
    import oracle
    threads = host_cores()
    rng = np.random.default_rng(seed)

    def gemm_job(shapes, cols):
        jobs = []
        for g in shapes:
            n = min(cols, g.N)
            inp = workloads.gemm_inputs(g.M, n, g.K, workloads.seed_for("oracle-cfg", g.M, g.N, g.K))
            jobs.append((workloads.bits(inp.x), workloads.bits(inp.W),
                         2 * n * g.K + 2 * g.M * g.K + 2 * g.M * n))
        def run():
            nb = 0
            for xb, wb, b in jobs:
                oracle.decode_gemm(xb, wb, threads=threads)
                nb += b
            return nb
        every = all(cols >= g.N for g in shapes)
        what = "all output columns" if every else f"{cols} output columns each"
        return run, f"{len(shapes)} shape(s), {what}", threads

    def reduce_job(shapes):
        jobs = []
        for r in shapes:
            inp = workloads.reduce_inputs(r.TP, r.M, workloads.seed_for("oracle-cfg", r.TP, r.M),
                                          r.residual)
            jobs.append((workloads.bits(inp.partials),
                         None if inp.residual is None else workloads.bits(inp.residual),
                         workloads.bits(inp.gamma), r.algorithmic_bytes()))
        def run():
            nb = 0
            for p, res, gam, b in jobs:
                oracle.reduce_residual_rmsnorm(p, res, gam, 1e-6)
                nb += b
            return nb
        return run, f"{len(shapes)} config(s), whole rows (single-threaded oracle)", 1

    def gather_job():
        jobs = [(rng.integers(0, 1 << 16, size=(TP, M, S), dtype=np.uint16), 4 * TP * M * S)
                for TP, M, S in GATHER_CONFIGS]
        def run():
            nb = 0
            for sh, b in jobs:
                oracle.gather_shards(sh)
                nb += b
            return nb
        return run, f"{len(GATHER_CONFIGS)} config(s), whole rows (single-threaded oracle)", 1

    kinds = {
        "pr1_gemm": gemm_job([workloads.PR1_GEMM], 1 << 30),
        "pr1_reduce": reduce_job([workloads.PR1_REDUCE]),
        "reduce_sweep": reduce_job(workloads.REDUCE_SWEEP),
        "gemm_sweep": gemm_job(workloads.GEMM_SWEEP, 64),
        "lm_head": gemm_job(workloads.LM_HEAD, 256),
        "wider": gemm_job(workloads.GEMM_WIDER, 64),
        "gather": gather_job(),
    }
    out = {}
    for name, (run, sample, cores) in kinds.items():
        run()  # warm
        nb, reps, t0 = 0, 0, time.perf_counter()
        while True:
            nb += run()
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s:
                break
        out[name] = {"GBps": nb / dt / 1e9, "cores": cores, "kind": "oracle",
                     "sample": f"{sample}; {reps} pass(es) in {dt:.2f} s"}
    return out


def configs_report(sk, calls, peak, peak_kind, device_index, pdl=True, with_oracle=True):
    """The per-config block of the benchmark line: GPU per-call figures under a
    clock record, with the oracle's GB/s per config kind beside them."""
    clocks = ClockSampler(device_index)
    prev = sk.set_pdl(pdl)
    try:
        clocks.start()
        time.sleep(0.3)
        sets = measure_configs(sk, calls, peak)
        torch.cuda.synchronize()
    finally:
        sk.set_pdl(prev)
    sets["clocks"] = clocks.stop()
    sets["peak_gbs"] = peak
    sets["peak_source"] = peak_kind
    sets["timing"] = (f"CUDA graph of {calls} back-to-back calls per config rotating through "
                      "buffer copies spanning >= 3x L2, median of 5 replays, CUDA events; "
                      f"PDL {'on' if pdl else 'off'}")
    if with_oracle:
        sets["oracle"] = oracle_configs()
    return sets


def run_sweep(args):
    import __graft_entry__
    __graft_entry__.build()
    import skinny_bf16_gemm_gb300 as sk
    peak, peak_kind = measured_peaks()
    rep = configs_report(sk, args.sweep_calls, peak, peak_kind, torch.cuda.current_device(),
                         pdl=bool(args.pdl), with_oracle=not args.no_cpu_baseline)
    rep["calls_per_config"] = args.sweep_calls
    print(json.dumps({"configs": rep}), flush=True)
    return 0


def run_profile_configs(args):
    """Every GEMM, reduce and gather config of the sweep, launched twice each
    (eagerly, one config's buffers at a time), for a per-call ncu launch list
    with cold caches. Prints the launch order, one label per launch pair."""
    import __graft_entry__
    __graft_entry__.build()
    import skinny_bf16_gemm_gb300 as sk
    sk.set_pdl(bool(args.pdl))
    dev = torch.device("cuda", 0)
    labels = []
    gemms = ([("gemm pr1", workloads.PR1_GEMM)] + [("gemm sweep", g) for g in workloads.GEMM_SWEEP]
             + [("gemm lm_head", g) for g in workloads.LM_HEAD]
             + [("gemm wider", g) for g in workloads.GEMM_WIDER]
             + [("gemm chain", workloads.CHAIN.gemm1()), ("gemm chain", workloads.CHAIN.gemm2())])
    for label, g in gemms:
        name = f"{label} M={g.M} N={g.N} K={g.K}"
        if args.config_filter not in name:
            continue
        inp = workloads.gemm_inputs(g.M, g.N, g.K, workloads.seed_for("cold", g.M, g.N, g.K),
                                    device=dev)
        out = torch.empty(g.M, g.N, device=dev, dtype=torch.bfloat16)
        for _ in range(2):
            sk.decode_gemm_bf16(inp.x, inp.W, out)
        torch.cuda.synchronize()
        labels.append({"label": name, "kernel": "decode_gemm", "bytes": g.algorithmic_bytes()})
        del inp
        torch.cuda.empty_cache()
    reduces = [("reduce pr1", workloads.PR1_REDUCE)] + [("reduce sweep", r) for r in workloads.REDUCE_SWEEP]
    for label, r in reduces:
        name = f"{label} TP={r.TP} M={r.M} res={int(r.residual)}"
        if args.config_filter not in name:
            continue
        inp = workloads.reduce_inputs(r.TP, r.M, workloads.seed_for("cold", r.TP, r.M), r.residual,
                                      device=dev)
        out = torch.empty(r.M, r.width, device=dev, dtype=torch.bfloat16)
        rout = torch.empty_like(out)
        for _ in range(2):
            sk.reduce_residual_rmsnorm(inp.partials, inp.residual, inp.gamma, out, rout, 1e-6)
        torch.cuda.synchronize()
        labels.append({"label": name, "kernel": "reduce_rmsnorm", "bytes": r.algorithmic_bytes()})
    for TP, M, S in GATHER_CONFIGS:
        name = f"gather TP={TP} M={M} S={S}"
        if args.config_filter not in name:
            continue
        shards = torch.randn(TP, M, S, device=dev).to(torch.bfloat16)
        out = torch.empty(M, TP * S, device=dev, dtype=torch.bfloat16)
        for _ in range(2):
            sk.gather_shards_bf16(shards, out)
        torch.cuda.synchronize()
        labels.append({"label": name, "kernel": "gather", "bytes": 4 * TP * M * S})
    st, word = sk.device_error(0)
    print(json.dumps({"profile_configs": labels, "device_error": word}), flush=True)
    return 0 if st == 0 else 1


def run_profile(args):
    """Three launches each of the chain's two decode GEMMs and its reduce, on the
    chain's shapes (weights 264 MB each, larger than L2), PDL and L2 lead as the
    chain runs them, then three of the chain's fused second call, for ncu
    captures."""
    import __graft_entry__
    __graft_entry__.build()
    import skinny_bf16_gemm_gb300 as sk
    sk.set_pdl(bool(args.pdl))
    sk.set_l2_prefetch(args.l2_prefetch)
    cfg = workloads.CHAIN
    dev = torch.device("cuda", 0)
    g1, g2 = cfg.gemm1(), cfg.gemm2()
    a = workloads.gemm_inputs(g1.M, g1.N, g1.K, 1, device=dev)
    b = workloads.gemm_inputs(g2.M, g2.N, g2.K, 2, device=dev)
    r = workloads.reduce_inputs(cfg.TP, cfg.M, 3, True, cfg.hidden, device=dev)
    h1 = torch.empty(g1.M, g1.N, dtype=torch.bfloat16, device=dev)
    out = torch.empty(cfg.M, cfg.hidden, dtype=torch.bfloat16, device=dev)
    res_out = torch.empty_like(out)
    for _ in range(3):
        sk.decode_gemm_bf16(a.x, a.W, h1)
        sk.decode_gemm_bf16(b.x, b.W, r.partials[0])
        sk.reduce_residual_rmsnorm(r.partials, r.residual, r.gamma, out, res_out, cfg.eps)
    # Then the chain's second call as the chain makes it: the second GEMM in
    # publish-only mode and the reduce kernel's split-K variant.
    for _ in range(3):
        sk.decode_gemm_bf16_reduce_rmsnorm(b.x, b.W, r.partials, r.residual, r.gamma, out, res_out,
                                           cfg.eps)
    torch.cuda.synchronize()
    st, word = sk.device_error(0)
    print(json.dumps({"profile": "chain kernels x3, then the fused call x3", "device_error": word}),
          flush=True)
    return 0 if st == 0 else 1


# ---- our arm ------------------------------------------------------------------------

def main():
    args = parse()
    rank, world, local = dist_info()
    cfg = workloads.CHAIN
    if args.impl == "reference":
        return run_reference(args, rank, world, cfg)
    if args.sweep:
        return run_sweep(args)
    if args.profile:
        return run_profile(args)
    if args.profile_configs:
        return run_profile_configs(args)

    import __graft_entry__
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        if rank == 0:
            __graft_entry__.build()
        dist.barrier()
    else:
        torch.cuda.set_device(local)
        __graft_entry__.build()
    import skinny_bf16_gemm_gb300 as sk
    from skinny_bf16_gemm_gb300.chain import LayerChain

    device = torch.device("cuda", local)
    from skinny_bf16_gemm_gb300.replicas import replica_seed
    inp = workloads.chain_inputs(cfg, replica_seed(workloads.seed_for("chain"), rank), device=device)
    chain = LayerChain(inp.W1, inp.W2, inp.peers, inp.gamma, cfg.M, cfg.eps, device=device,
                       fused=bool(args.fused), l2_prefetch=args.l2_prefetch,
                       pdl=bool(args.pdl), l2_after_reduce=args.l2_after_reduce)
    chain.x.copy_(inp.x0)
    chain.res_in.copy_(inp.residual0)
    sk.set_pdl(bool(args.pdl))
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def step():
        return chain.replay() if chain.graph is not None else chain.run()

    # The clock sampler needs a moment to start; the GPU streams plain device
    # copies meanwhile (not chain steps) instead of idling, so that the warm-up
    # and timed steps do not begin on a GPU coming out of an idle spell.
    clocks = ClockSampler(local)
    clocks.start()
    keep_streaming(device, 0.3)

    # Warm-up (eager), then optionally capture the step as one graph.
    for _ in range(max(args.warmup, 3)):
        chain.run()
    torch.cuda.synchronize()
    if args.graph:
        chain.capture()
        for _ in range(3):
            chain.replay()
        torch.cuda.synchronize()
    st, word = sk.device_error(local)
    if st != 0:
        raise RuntimeError(f"device error word {word} during warm-up")

    # ---- timed region: K steps, inputs resident ----
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    host_lead(stream)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clock_info = clocks.stop()
    from skinny_bf16_gemm_gb300 import replicas
    ms = replicas.slowest_ms(e0.elapsed_time(e1), device=device)
    ms_per_step = ms / args.steps
    value = replicas.aggregate_throughput(cfg.step_bytes(), args.steps, ms, world)
    st, word = sk.device_error(local)
    if st != 0:
        raise RuntimeError(f"device error word {word} in the timed region")

    # ---- per-kernel durations: each kernel back to back on the same stream ----
    # The chain's own launch sequence with the reduce calls left out (and then
    # the reduces alone, replayed from a CUDA graph), timed with CUDA events
    # around the whole loop: the
    # average launch duration of a kernel as it runs in a stream (programmatic
    # dependent launch on, as in the timed region). Events around every single
    # launch would serialise the kernels and add each launch's gap.
    kernel_steps = max(1, min(args.steps, 400))

    # The chain's launch settings, passed with every call.
    kopts = dict(pdl=bool(args.pdl), l2_prefetch=args.l2_prefetch)

    def gemm_only():
        x = chain.x
        for l in range(cfg.layers):
            sk.decode_gemm_bf16(x, chain.W1[l], chain.h1, **kopts)
            sk.decode_gemm_bf16(chain.h1, chain.W2[l], chain.partials[l][0], **kopts)

    def reduce_only():
        for l in range(cfg.layers):
            sk.reduce_residual_rmsnorm(chain.partials[l], chain.res_in, chain.gamma[l],
                                       chain.outs[l % 2], chain.res[l % 2], cfg.eps,
                                       pdl=kopts["pdl"])

    def loop_ms(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        host_lead(stream)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def graph_ms(fn, reps):
        # A kernel of a few microseconds launched from Python is host-bound:
        # capture the launches once and time the graph's replay instead.
        fn()
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for _ in range(reps):
                    fn()
        stream.wait_stream(side)
        graph.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    gemm_launches = kernel_steps * 2 * cfg.layers
    gemm_ms = loop_ms(gemm_only, kernel_steps) / gemm_launches
    reduce_reps = 100
    reduce_ms = graph_ms(reduce_only, reduce_reps) / (reduce_reps * cfg.layers)
    g1 = cfg.gemm1()
    gemm_bytes = g1.algorithmic_bytes()  # GEMM1 and GEMM2 move the same bytes
    peak, peak_kind = measured_peaks()
    achieved = gemm_bytes / (gemm_ms * 1e-3) / 1e9
    traffic = recorded_traffic("chain_gemm")

    # ---- end to end through the public API: host inputs in, host result out ----
    # Steps go in groups of G, each step with its own buffer set (sharing the
    # weights), two groups' sets in all, and a copy stream: group k+1's inputs go
    # up while group k computes, and each step's result rows come back once its
    # group is done. Every step copies its own inputs in and its rows out inside
    # the timed region; one event per group (not per step) keeps the compute
    # stream's kernels chained under programmatic dependent launch.
    G = max(1, args.e2e_group)
    pin = dict(pin_memory=True)
    host_x = inp.x0.cpu().pin_memory()
    host_res = inp.residual0.cpu().pin_memory()
    host_peers = [p.cpu().pin_memory() for p in inp.peers]
    host_out = [torch.empty(cfg.M, cfg.hidden, dtype=torch.bfloat16, **pin) for _ in range(2 * G)]
    host_res_out = [torch.empty(cfg.M, cfg.hidden, dtype=torch.bfloat16, **pin) for _ in range(2 * G)]
    h2d = (host_x.numel() + host_res.numel() + sum(p.numel() for p in host_peers)) * 2
    d2h = (host_out[0].numel() + host_res_out[0].numel()) * 2
    # At least 200 steps (at most 500): the copy pipeline's fill and drain are a
    # few steps' worth, so a short run would mostly time those.
    e2e_steps = max(200, min(args.steps, 500)) // G * G
    chains = [chain] + [LayerChain(inp.W1, inp.W2, inp.peers, inp.gamma, cfg.M, cfg.eps,
                                   device=device, fused=bool(args.fused),
                                   l2_prefetch=args.l2_prefetch, pdl=bool(args.pdl),
                                   l2_after_reduce=args.l2_after_reduce)
                        for _ in range(2 * G - 1)]
    copy_stream = torch.cuda.Stream()
    inputs_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def upload(k):
        with torch.cuda.stream(copy_stream):
            for j in range(G):
                c = chains[(k % 2) * G + j]
                c.x.copy_(host_x, non_blocking=True)
                c.res_in.copy_(host_res, non_blocking=True)
                for l in range(cfg.layers):
                    c.partials[l][1:].copy_(host_peers[l], non_blocking=True)
            inputs_ready[k % 2].record(copy_stream)

    def e2e_steps_run(n):
        groups = n // G
        upload(0)
        last = None
        for k in range(groups):
            stream.wait_event(inputs_ready[k % 2])
            rows = [chains[(k % 2) * G + j].run() for j in range(G)]
            done[k % 2].record(stream)
            with torch.cuda.stream(copy_stream):
                if k + 1 < groups:
                    if k >= 1:  # the other group's buffer sets must be free
                        copy_stream.wait_event(done[(k + 1) % 2])
                    upload(k + 1)
                copy_stream.wait_event(done[k % 2])
                for j, (out, res) in enumerate(rows):
                    host_out[(k % 2) * G + j].copy_(out, non_blocking=True)
                    host_res_out[(k % 2) * G + j].copy_(res, non_blocking=True)
            last = (k % 2) * G + G - 1
        stream.wait_stream(copy_stream)
        return last

    e2e_steps_run(2 * G)
    torch.cuda.synchronize()
    barrier()
    host_lead(stream)
    e0.record(stream)
    last = e2e_steps_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    # Every step has the same inputs: the rows read back must be the device path's.
    ref_out, ref_res = chain.run()
    torch.cuda.synchronize()
    if not (torch.equal(host_out[last].view(torch.int16), ref_out.cpu().view(torch.int16)) and
            torch.equal(host_res_out[last].view(torch.int16), ref_res.cpu().view(torch.int16))):
        raise RuntimeError("end-to-end result rows differ from the device-resident run")
    e2e_value = world * cfg.step_bytes() / (e2e_ms * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/K) weights)",
        "impl": "ours",
        "config": workload_config(cfg, {"pdl": bool(args.pdl), "graph": bool(args.graph),
                                        "fused_gemm_reduce": bool(args.fused),
                                        "l2_prefetch_blocks": args.l2_prefetch,
                                        "l2_after_reduce_blocks":
                                            args.l2_after_reduce if args.fused else 0,
                                        "parallelism": "replicas" if world > 1 else "single"}),
        "hbm_frac_of_measured": value / peak,
        "hbm_frac_of_nominal_8000": value / 8000.0,
        "roofline": {"bound": "hbm", "kernel": "decode_gemm_bf16 (chain shapes)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6800 GB/s",
                     "algorithmic_bytes_per_launch": gemm_bytes,
                     "avg_launch_ms": gemm_ms, "launches_timed": gemm_launches,
                     "timing": "back-to-back launches of the chain's 6 GEMMs (decode_gemm_bf16), "
                               "CUDA events around the loop, PDL and L2 lead as in the timed region"},
        "kernels": {"decode_gemm_avg_us": gemm_ms * 1e3, "reduce_rmsnorm_avg_us": reduce_ms * 1e3,
                    "reduce_algorithmic_bytes": cfg.reduce().algorithmic_bytes(),
                    "reduce_gbs": cfg.reduce().algorithmic_bytes() / (reduce_ms * 1e-3) / 1e9},
        "clocks": clock_info,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps},
        "gpu_launches": args.steps * chain.launches_per_step(),
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = {k: v for k, v in time_oracle(cfg, 10.0).items()
                                if k in ("value", "unit", "cores", "kind", "sample")}
        one = time_oracle(cfg, 5.0, threads=1)
        line["cpu_baseline"]["one_thread"] = {"value": one["value"], "sample": one["sample"]}
        line["parity"] = chain_parity(inp, cfg, sk)
    if rank == 0 and args.configs:
        line["configs"] = configs_report(sk, args.sweep_calls, peak, peak_kind, local,
                                         pdl=bool(args.pdl),
                                         with_oracle=world == 1 and not args.no_cpu_baseline)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
