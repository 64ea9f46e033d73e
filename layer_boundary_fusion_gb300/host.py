"""Boundary calls on host-resident (pinned) tensors, overlapping the copies with the
kernels and with each other.

`HostPipeline` owns `depth` sets of device staging buffers and three CUDA streams
(copy in, compute, copy out).  A step splits its rows into chunks; chunk c's inputs
are copied in on the first stream, its `lb_fold_norm_fp8` runs on the second once they
have landed, and its outputs are copied back on the third.  Consecutive steps of one
`run()` alternate between the buffer sets, so step i+1's inputs are copied in while
step i's outputs are still being copied out: the two directions of the host link are
busy at the same time.  A step waits only for what it overwrites: its copy-in for the
kernel that last read the same buffer set, its kernel for the copy-out that last read
that set's outputs.

The first call for a given sequence of host buffers captures the whole schedule as a
CUDA graph; later calls replay it, so the host issues one launch per call instead of
dozens of copies.  All work is the library's kernel and
cudaMemcpyAsync; this module only orders it.
"""
from __future__ import annotations

import torch

from . import lb


class _DeviceSet:
    """Device buffers of one step: K partials, residual in / out, gamma, codes, scales."""

    def __init__(self, K, T, H, d):
        self.P = [torch.empty((T, H), dtype=torch.int16, device=d) for _ in range(K)]
        self.R = torch.empty((T, H), dtype=torch.int16, device=d)
        self.gamma = torch.empty(H, dtype=torch.float32, device=d)
        self.ro = torch.empty((T, H), dtype=torch.int16, device=d)
        self.q = torch.empty((T, H), dtype=torch.uint8, device=d)
        self.s = torch.empty((T,), dtype=torch.float32, device=d)


class HostPipeline:
    """Pipelined `lb_fold_norm_fp8` steps over pinned host buffers of one shape.

    K partials [T, H] and a residual [T, H] (bf16 bits as int16), gamma [H] float32 on
    the host; results residual' [T, H] (int16 bits), codes [T, H] uint8 and scales
    [T] float32 on the host.  `chunks` row blocks per step (rows must divide evenly),
    `depth` device buffer sets (consecutive steps overlap when depth >= 2).  One CUDA
    graph is kept per distinct sequence of host buffers (the MAX_GRAPHS most recent).
    """

    MAX_GRAPHS = 8                        # captured schedules kept (oldest dropped first)

    def __init__(self, K: int, T: int, H: int, device, chunks: int = 1, depth: int = 2):
        if T % chunks:
            raise ValueError("T must be a multiple of chunks")
        if depth < 1:
            raise ValueError("depth must be at least 1")
        self.K, self.T, self.H, self.chunks, self.depth = K, T, H, chunks, depth
        self.dev = torch.device(device)
        self.s_in = torch.cuda.Stream(self.dev)
        self.s_run = torch.cuda.Stream(self.dev)
        self.s_out = torch.cuda.Stream(self.dev)
        self.sets = [_DeviceSet(K, T, H, self.dev) for _ in range(depth)]
        self.graphs = {}                  # host-buffer sequence -> graph, oldest first

    def _schedule(self, steps, inputs, gamma_host, outputs, eps, origin):
        """Enqueue `steps` steps: fork from `origin`, pipelined copy-in / kernel /
        copy-out, join back into `origin`.  inputs(i) -> (partials, residual) and
        outputs(i) -> (residual', codes, scales) are step i's host tensors."""
        rows = self.T // self.chunks
        fork = torch.cuda.Event()
        fork.record(origin)
        for st in (self.s_in, self.s_run, self.s_out):
            st.wait_event(fork)
        ran, drained = [], []                 # per step: kernels done, copy-out done
        for i in range(steps):
            partials_host, residual_host = inputs(i)
            out_res, out_q, out_scale = outputs(i)
            d = self.sets[i % self.depth]
            if i >= self.depth:               # the buffer set's previous step
                self.s_in.wait_event(ran[i - self.depth])
                self.s_run.wait_event(drained[i - self.depth])
            with torch.cuda.stream(self.s_in):
                d.gamma.copy_(gamma_host, non_blocking=True)
            for c in range(self.chunks):
                sl = slice(c * rows, (c + 1) * rows)
                with torch.cuda.stream(self.s_in):
                    for dp, hp in zip(d.P, partials_host):
                        dp[sl].copy_(hp[sl], non_blocking=True)
                    d.R[sl].copy_(residual_host[sl], non_blocking=True)
                    landed = torch.cuda.Event()
                    landed.record(self.s_in)
                self.s_run.wait_event(landed)
                with torch.cuda.stream(self.s_run):
                    lb.lb_fold_norm_fp8([p[sl] for p in d.P], d.R[sl], d.ro[sl], d.gamma,
                                        d.q[sl], d.s[sl], None, rows, self.H, eps,
                                        stream=self.s_run.cuda_stream)
                    done = torch.cuda.Event()
                    done.record(self.s_run)
                self.s_out.wait_event(done)
                with torch.cuda.stream(self.s_out):
                    out_res[sl].copy_(d.ro[sl], non_blocking=True)
                    out_q[sl].copy_(d.q[sl], non_blocking=True)
                    out_scale[sl].copy_(d.s[sl], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.s_run)
            ran.append(ev)
            ev = torch.cuda.Event()
            ev.record(self.s_out)
            drained.append(ev)
        for st in (self.s_in, self.s_run, self.s_out):
            join = torch.cuda.Event()
            join.record(st)
            origin.wait_event(join)

    def run_steps(self, inputs, gamma_host, outputs, eps, stream=None):
        """One boundary step per entry of `inputs` ((partials, residual) host tensors)
        into the matching entry of `outputs` ((residual', codes, scales) host tensors),
        ordered after the work already on `stream` (default: the current stream), which
        is left waiting for every step's outputs."""
        if len(inputs) != len(outputs) or not inputs:
            raise ValueError("one output set per input set, at least one step")
        origin = stream or torch.cuda.current_stream(self.dev)
        key = (tuple((tuple(t.data_ptr() for t in P), R.data_ptr()) for P, R in inputs),
               gamma_host.data_ptr(), tuple(tuple(t.data_ptr() for t in o) for o in outputs),
               float(eps))
        graph = self.graphs.get(key)
        if graph is None:
            cap = torch.cuda.Stream(self.dev)
            cap.wait_stream(origin)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                self._schedule(len(inputs), lambda i: inputs[i], gamma_host,
                               lambda i: outputs[i], eps, cap)
            origin.wait_stream(cap)
            if len(self.graphs) >= self.MAX_GRAPHS:
                self.graphs.pop(next(iter(self.graphs)))
            self.graphs[key] = graph
        with torch.cuda.stream(origin):
            graph.replay()

    def run(self, steps, partials_host, residual_host, gamma_host, out_res, out_q, out_scale,
            eps, stream=None):
        """`steps` boundary steps on the same host tensors (each copies its inputs in
        and its results out); see run_steps()."""
        self.run_steps([(partials_host, residual_host)] * steps, gamma_host,
                       [(out_res, out_q, out_scale)] * steps, eps, stream)

    def __call__(self, partials_host, residual_host, gamma_host, out_res, out_q, out_scale,
                 eps, stream=None):
        """One boundary step on host tensors (see run())."""
        self.run(1, partials_host, residual_host, gamma_host, out_res, out_q, out_scale, eps,
                 stream)
