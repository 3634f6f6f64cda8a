"""The drafter layer chain on the two library calls.

Per layer l ("drafter/comm" module text: each draft layer's row-parallel linear
ends in a TP all-reduce fused with the following RMSNorm; here the other ranks'
partial rows are local slots, the one-GPU stand-in of "cutedsl/common/twoshot"):

    h1              = x @ W1[l]^T                      decode_gemm_bf16  [M, F]
    partials[l][0]  = h1 @ W2[l]^T                     decode_gemm_bf16  [M, H]
    out, residual   = reduce_residual_rmsnorm(partials[l], residual, gamma[l])
    x               = out

Slots 1..TP-1 of partials[l] hold the other ranks' rows. With fused=True the
second GEMM and the reduce + residual + RMSNorm are one call,
decode_gemm_bf16_reduce_rmsnorm (bit-identical results, two kernels instead of a
split-K fix-up inside the GEMM plus a reduce). Every step of the chain runs in
the library's kernels; this class only owns the device buffers and orders the
calls on one stream (optionally as one CUDA graph). Every call carries the
chain's own launch settings (the library's _ex entry points), so the chain never
changes the process-wide ones other code sees: programmatic dependent launch
(pdl, on by default) and the decode GEMM's L2 lead (l2_prefetch, 0 by default:
measured on GB300, each GEMM of the chain runs behind or ahead of a short
kernel, and weight prefetches issued before the PDL wait only slow the previous
GEMM's last CTAs there; chain step 0.7-0.8 % faster than with the default 6).
With fused=True each first GEMM also prefetches l2_after_reduce weight blocks
per CTA (16 by default) into L2 as soon as the reduce before it has seen the
second GEMM complete: HBM then streams while the reduce runs (measured on
GB300: chain step 250.8 -> 247.8 us; timing only, the same bits).
"""
import torch

from . import decode_gemm_bf16, decode_gemm_bf16_reduce_rmsnorm, reduce_residual_rmsnorm


class LayerChain:
    def __init__(self, W1, W2, peers, gamma, M, eps=1e-6, device="cuda", fused=False,
                 l2_prefetch=0, pdl=True, l2_after_reduce=16):
        self.layers = len(W1)
        self.fused = fused
        self.l2_prefetch = l2_prefetch
        self.l2_after_reduce = l2_after_reduce if fused else None
        self.pdl = bool(pdl)
        self.W1, self.W2, self.gamma = W1, W2, gamma
        self.M, self.eps = M, eps
        self.F, self.H = W1[0].shape
        self.TP = peers[0].shape[0] + 1
        bf = dict(dtype=torch.bfloat16, device=device)
        # One [TP, M, H] partial buffer per layer: slot 0 is written by the
        # second GEMM, slots 1.. are the other ranks' rows.
        self.partials = []
        for p in peers:
            buf = torch.empty(self.TP, M, self.H, **bf)
            buf[1:].copy_(p)
            self.partials.append(buf)
        self.h1 = torch.empty(M, self.F, **bf)
        self.x = torch.empty(M, self.H, **bf)          # step input
        self.res_in = torch.empty(M, self.H, **bf)     # step residual input
        self.outs = [torch.empty(M, self.H, **bf) for _ in range(2)]
        self.res = [torch.empty(M, self.H, **bf) for _ in range(2)]
        self.graph = None

    def launches_per_step(self) -> int:
        return 3 * self.layers

    def run(self, stream=None, on_launch=None):
        """Enqueue one step reading self.x / self.res_in; returns (out, residual).

        on_launch(kind, layer, phase) is called with phase 'before' / 'after'
        around every launch (used to bracket kernels with timing events)."""
        gemm_opts = dict(pdl=self.pdl, l2_prefetch=self.l2_prefetch)
        x, res = self.x, self.res_in
        for l in range(self.layers):
            if on_launch:
                on_launch("gemm", l, "before")
            decode_gemm_bf16(x, self.W1[l], self.h1, stream, l2_after_reduce=self.l2_after_reduce,
                             **gemm_opts)
            if on_launch:
                on_launch("gemm", l, "after")
                on_launch("gemm", l, "before")
            out, res_out = self.outs[l % 2], self.res[l % 2]
            if self.fused:
                decode_gemm_bf16_reduce_rmsnorm(self.h1, self.W2[l], self.partials[l], res,
                                                self.gamma[l], out, res_out, self.eps, stream,
                                                **gemm_opts)
                if on_launch:
                    on_launch("gemm", l, "after")
            else:
                decode_gemm_bf16(self.h1, self.W2[l], self.partials[l][0], stream, **gemm_opts)
                if on_launch:
                    on_launch("gemm", l, "after")
                    on_launch("reduce", l, "before")
                reduce_residual_rmsnorm(self.partials[l], res, self.gamma[l], out, res_out,
                                        self.eps, stream, pdl=self.pdl)
                if on_launch:
                    on_launch("reduce", l, "after")
            x, res = out, res_out
        return x, res

    def capture(self):
        """Capture one step as a CUDA graph (after at least one eager step), with
        the chain's launch settings."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                self.graph_out = self.run()
        torch.cuda.current_stream().wait_stream(s)
        self.graph = g
        return self.graph_out

    def replay(self):
        self.graph.replay()
        return self.graph_out
