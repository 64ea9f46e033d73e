"""Boundary calls on host-resident (pinned) tensors, overlapping the copies with the
kernels.

`HostPipeline` owns device staging buffers and three CUDA streams (copy in, compute,
copy out).  A call splits its rows into chunks; chunk c's inputs are copied in on the
first stream, its `lb_fold_norm_fp8` runs on the second once they have landed, and
its outputs are copied back on the third, so that copy-in, kernel and copy-out of
different chunks run at the same time.  The first call for a given set of host
buffers captures this fork/join schedule as a CUDA graph; later calls replay it, so
the host issues one launch per call instead of dozens of copies.  All work is the
library's kernel and cudaMemcpyAsync; this module only orders it.
"""
from __future__ import annotations

import torch

from . import lb


class HostPipeline:
    """Pipelined `lb_fold_norm_fp8` over pinned host buffers of one shape.

    K partials [T, H] and a residual [T, H] (bf16 bits as int16), gamma [H] float32 on
    the host; results residual' [T, H] (int16 bits), codes [T, H] uint8 and scales
    [T] float32 on the host.  `chunks` row blocks per call (rows must divide evenly).
    One CUDA graph is kept per distinct set of host buffers.
    """

    def __init__(self, K: int, T: int, H: int, device, chunks: int = 4):
        if T % chunks:
            raise ValueError("T must be a multiple of chunks")
        self.K, self.T, self.H, self.chunks = K, T, H, chunks
        self.dev = torch.device(device)
        self.s_in = torch.cuda.Stream(self.dev)
        self.s_run = torch.cuda.Stream(self.dev)
        self.s_out = torch.cuda.Stream(self.dev)
        d = self.dev
        self.P = [torch.empty((T, H), dtype=torch.int16, device=d) for _ in range(K)]
        self.R = torch.empty((T, H), dtype=torch.int16, device=d)
        self.ro = torch.empty((T, H), dtype=torch.int16, device=d)
        self.q = torch.empty((T, H), dtype=torch.uint8, device=d)
        self.s = torch.empty((T,), dtype=torch.float32, device=d)
        self.gamma = torch.empty(H, dtype=torch.float32, device=d)
        self.graphs = {}

    def _schedule(self, partials_host, residual_host, gamma_host, out_res, out_q, out_scale,
                  eps, origin):
        """Enqueue one call: fork from `origin`, chunked copy-in / kernel / copy-out,
        join back into `origin`."""
        rows = self.T // self.chunks
        fork = torch.cuda.Event()
        fork.record(origin)
        self.s_in.wait_event(fork)
        with torch.cuda.stream(self.s_in):
            self.gamma.copy_(gamma_host, non_blocking=True)
        for c in range(self.chunks):
            sl = slice(c * rows, (c + 1) * rows)
            with torch.cuda.stream(self.s_in):
                for d, h in zip(self.P, partials_host):
                    d[sl].copy_(h[sl], non_blocking=True)
                self.R[sl].copy_(residual_host[sl], non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(self.s_in)
            self.s_run.wait_event(landed)
            with torch.cuda.stream(self.s_run):
                lb.lb_fold_norm_fp8([p[sl] for p in self.P], self.R[sl], self.ro[sl],
                                    self.gamma, self.q[sl], self.s[sl], None, rows, self.H,
                                    eps, stream=self.s_run.cuda_stream)
                done = torch.cuda.Event()
                done.record(self.s_run)
            self.s_out.wait_event(done)
            with torch.cuda.stream(self.s_out):
                out_res[sl].copy_(self.ro[sl], non_blocking=True)
                out_q[sl].copy_(self.q[sl], non_blocking=True)
                out_scale[sl].copy_(self.s[sl], non_blocking=True)
        for st in (self.s_in, self.s_run, self.s_out):
            join = torch.cuda.Event()
            join.record(st)
            origin.wait_event(join)

    def __call__(self, partials_host, residual_host, gamma_host, out_res, out_q, out_scale,
                 eps, stream=None):
        """One boundary call on host tensors, ordered after the work already on
        `stream` (default: the current stream), which it leaves waiting for its
        outputs."""
        origin = stream or torch.cuda.current_stream(self.dev)
        key = (tuple(t.data_ptr() for t in partials_host), residual_host.data_ptr(),
               gamma_host.data_ptr(), out_res.data_ptr(), out_q.data_ptr(),
               out_scale.data_ptr(), float(eps))
        graph = self.graphs.get(key)
        if graph is None:
            cap = torch.cuda.Stream(self.dev)
            cap.wait_stream(origin)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                self._schedule(partials_host, residual_host, gamma_host, out_res, out_q,
                               out_scale, eps, cap)
            origin.wait_stream(cap)
            self.graphs[key] = graph
        with torch.cuda.stream(origin):
            graph.replay()
