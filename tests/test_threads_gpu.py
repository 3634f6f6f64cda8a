"""Host threads and the library on the GPU, through the C ABI.

Two host threads of a fresh process start at the same moment and make plain
decode GEMM and reduce + RMSNorm calls on one stream, while a third thread flips
the process-wide launch settings; a layer chain with its own per-call settings
runs beside them. Every result must equal, bit for bit, the same call made alone
afterwards: the first-call set-up (device state, split-K scratch, tensor-map
encoder) is shared safely, and launch settings never change a bit."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import json, threading
import torch
import skinny_bf16_gemm_gb300 as sk
import workloads
from skinny_bf16_gemm_gb300.chain import LayerChain

torch.cuda.set_device(0)
dev = torch.device("cuda", 0)
stream = torch.cuda.default_stream(dev)
# Split-K shapes (the scratch is used) and one whole-tile shape.
jobs = [(4, 2048, 7168, 1), (16, 7168, 4608, 2), (32, 640, 1000, 3), (8, 18432, 1024, 4)]
inputs = [workloads.gemm_inputs(M, N, K, seed, device=dev) for (M, N, K, seed) in jobs]
red = workloads.reduce_inputs(8, 16, 5, True, device=dev)
cfg = workloads.ChainConfig(layers=2, M=16, ffn=2048)
cin = workloads.chain_inputs(cfg, 6, device=dev)
torch.cuda.synchronize()
reps = 12
go = threading.Barrier(3)
stop = threading.Event()
results = {0: [], 1: []}

def worker(t):
    torch.cuda.set_device(0)
    with torch.cuda.stream(stream):
        go.wait()
        for r in range(reps):
            i = (t + r) % len(jobs)
            g = inputs[i]
            out = torch.empty(g.x.shape[0], g.W.shape[0], dtype=torch.bfloat16, device=dev)
            sk.decode_gemm_bf16(g.x, g.W, out)
            y = torch.empty(16, sk.HIDDEN, dtype=torch.bfloat16, device=dev)
            h = torch.empty_like(y)
            sk.reduce_residual_rmsnorm(red.partials, red.residual, red.gamma, y, h, red.eps)
            results[t].append((i, out, y, h))

def flipper():
    go.wait()
    k = 0
    while not stop.is_set():
        sk.set_pdl(bool(k & 1))
        sk.set_l2_prefetch((7 * k) % 65)
        k += 1

ts = [threading.Thread(target=worker, args=(t,)) for t in (0, 1)]
tf = threading.Thread(target=flipper)
for t in ts + [tf]:
    t.start()
for t in ts:
    t.join()
# A chain with its own settings while the flipper still runs.
chain = LayerChain(cin.W1, cin.W2, cin.peers, cin.gamma, cfg.M, cfg.eps, device=dev,
                   fused=True, l2_prefetch=0, pdl=True)
chain.x.copy_(cin.x0)
chain.res_in.copy_(cin.residual0)
c_out, c_res = (t.clone() for t in chain.run())
stop.set()
tf.join()
torch.cuda.synchronize()
status, word = sk.device_error(0)

# The same calls alone, with the settings fixed.
sk.set_pdl(False)
sk.set_l2_prefetch(6)
mism = 0
for t in (0, 1):
    for i, out, y, h in results[t]:
        g = inputs[i]
        ref = torch.empty_like(out)
        sk.decode_gemm_bf16(g.x, g.W, ref)
        mism += int(not torch.equal(ref.view(torch.int16), out.view(torch.int16)))
        ry, rh = torch.empty_like(y), torch.empty_like(h)
        sk.reduce_residual_rmsnorm(red.partials, red.residual, red.gamma, ry, rh, red.eps)
        mism += int(not torch.equal(ry.view(torch.int16), y.view(torch.int16)))
        mism += int(not torch.equal(rh.view(torch.int16), h.view(torch.int16)))
alone = LayerChain(cin.W1, cin.W2, cin.peers, cin.gamma, cfg.M, cfg.eps, device=dev,
                   fused=False, l2_prefetch=6, pdl=False)
alone.x.copy_(cin.x0)
alone.res_in.copy_(cin.residual0)
a_out, a_res = alone.run()
torch.cuda.synchronize()
chain_same = torch.equal(a_out.view(torch.int16), c_out.view(torch.int16)) and \
    torch.equal(a_res.view(torch.int16), c_res.view(torch.int16))
print(json.dumps({"calls": sum(len(v) for v in results.values()), "mismatches": mism,
                  "chain_same": chain_same, "status": status, "word": word}))
'''


def test_two_host_threads_share_the_library_safely(cuda_ok):
    p = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, capture_output=True, text=True,
                       timeout=600, env=dict(os.environ, PYTHONPATH=ROOT))
    assert p.returncode == 0, p.stderr[-3000:]
    rep = json.loads(p.stdout.strip().splitlines()[-1])
    assert rep["calls"] == 24
    assert rep["mismatches"] == 0, rep
    assert rep["chain_same"], rep
    assert (rep["status"], rep["word"]) == (0, 0), rep
