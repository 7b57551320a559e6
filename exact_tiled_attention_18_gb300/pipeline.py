"""Training step on a batch held in pinned host memory, with the copies hidden.

Heads are independent, so a batch can be cut into chunks of consecutive
(batch, head) pairs (rows of the [B*H, N, d] view, contiguous in host and
device memory) whose host->device copies, kernels and device->host copies run
on three streams:
while chunk k computes, chunk k+1's inputs come in and chunk k-1's results go
out (the copy engines and the SMs work at the same time).  Every computation
is the C ABI's forward and backward (fa_fwd, fa_bwd) on each chunk; this
module only orders copies and calls.
"""

from __future__ import annotations

from . import binding


class HostStepPipeline:
    """Forward + backward of [B, H, N, d] attention whose inputs (q, k, v, dO)
    live in pinned host memory and whose results (O, LSE, dQ, dK, dV) go back
    to pinned host memory.

    ``chunks`` pieces of B*H/chunks (batch, head) pairs each are in flight at
    once; device buffers for each piece are allocated once here and reused by
    every ``step``.
    """

    def __init__(self, B: int, H: int, N: int, d: int, causal: bool, scale: float, chunks: int = 2,
                 device=None, backward: bool = True):
        import torch
        if chunks < 1 or (B * H) % chunks != 0:
            raise ValueError("chunks must divide B*H")
        self.B, self.H, self.N, self.d = B, H, N, d
        self.causal, self.scale, self.backward = causal, scale, backward
        self.chunks = chunks
        self.ch = B * H // chunks  # (batch, head) pairs per chunk
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.s_in = torch.cuda.Stream(self.device)
        self.s_cmp = torch.cuda.Stream(self.device)
        self.s_out = torch.cuda.Stream(self.device)
        shp = (1, self.ch, N, d)  # one "batch" of ch heads
        bf, f32 = torch.bfloat16, torch.float32
        self.bufs = []
        for _ in range(chunks):
            b = {n: torch.empty(shp, dtype=bf, device=self.device) for n in ("q", "k", "v")}
            b["o"] = torch.empty(shp, dtype=f32, device=self.device)
            b["lse"] = torch.empty((1, self.ch, N), dtype=f32, device=self.device)
            if backward:
                b["do"] = torch.empty(shp, dtype=bf, device=self.device)
                for n in ("dq", "dk", "dv"):
                    b[n] = torch.empty(shp, dtype=f32, device=self.device)
                b["ws"] = torch.empty(binding.fa_bwd_workspace_bytes(1, self.ch, N) // 4, dtype=f32,
                                      device=self.device)
            self.bufs.append(b)
        # per chunk: inputs consumed by the kernels / results copied out
        self.in_free = [None] * chunks
        self.out_free = [None] * chunks

    def step(self, host_in: dict, host_out: dict):
        """Queue one step: host_in holds pinned q, k, v (and do), host_out
        pinned o, lse (and dq, dk, dv), all [B, H, ...] and contiguous (a
        chunk is a row range of their [B*H, ...] view; anything else raises).
        Returns at once; the results are in host_out after ``synchronize()``."""
        import torch
        ins = ("q", "k", "v") + (("do",) if self.backward else ())
        outs = ("o", "lse") + (("dq", "dk", "dv") if self.backward else ())
        BH = self.B * self.H

        def rows(t):  # the [B*H, ...] view of a [B, H, ...] host tensor
            return t.view((BH,) + tuple(t.shape[2:]))

        for c in range(self.chunks):
            sl = slice(c * self.ch, (c + 1) * self.ch)
            b = self.bufs[c]
            with torch.cuda.stream(self.s_in):
                if self.in_free[c] is not None:
                    self.s_in.wait_event(self.in_free[c])
                for n in ins:
                    b[n][0].copy_(rows(host_in[n])[sl], non_blocking=True)
                arrived = torch.cuda.Event()
                arrived.record(self.s_in)
            with torch.cuda.stream(self.s_cmp):
                self.s_cmp.wait_event(arrived)
                if self.out_free[c] is not None:
                    self.s_cmp.wait_event(self.out_free[c])
                binding.forward(b["q"], b["k"], b["v"], causal=self.causal, scale=self.scale,
                                out=(b["o"], b["lse"]))
                if self.backward:
                    binding.backward(b["q"], b["k"], b["v"], b["o"], b["lse"], b["do"], causal=self.causal,
                                     scale=self.scale, workspace=b["ws"], out=(b["dq"], b["dk"], b["dv"]))
                done = torch.cuda.Event()
                done.record(self.s_cmp)
                self.in_free[c] = done
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(done)
                for n in outs:
                    rows(host_out[n])[sl].copy_(b[n][0], non_blocking=True)
                copied = torch.cuda.Event()
                copied.record(self.s_out)
                self.out_free[c] = copied

    def synchronize(self):
        for s in (self.s_in, self.s_cmp, self.s_out):
            s.synchronize()
