"""Run one boundary workload a few times, for profilers (ncu) and quick timing.

    python -m layer_boundary_fusion_gb300.profile_case prefill_fold_norm_fp8 \
        --launches 4 [--row-scale 3] [--sets 2] [--hidden 12288]
    python -m layer_boundary_fusion_gb300.profile_case ragged_slice [--rsv-rank 1]

Builds the seeded workload (the prefill one optionally at another hidden size; for the
ragged batch, with --rsv-rank, one rank's rows under the variable-size reduce-scatter
instead of slice 3 of 8),
optionally repeats its rows `--row-scale` times (so that a capture's working set
exceeds the L2 cache), and launches the boundary call
`--launches` times, rotating over `--sets` independent buffer sets.  Prints the mean
time per launch measured with CUDA events (not meaningful under a profiler).
"""
import argparse
import sys

import numpy as np
import torch

from . import lb, workloads as wl


def _rep(a, n):
    return a if n == 1 else np.ascontiguousarray(np.concatenate([a] * n, axis=0))


def _bits(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def make_launcher(name, row_scale, dev, stream, hidden=None, rsv_rank=None):
    w = wl.prefill_fold_norm_fp8(H=hidden) if hidden else wl.WORKLOADS[name]()
    sp = stream.cuda_stream
    G = torch.from_numpy(w.gamma).to(dev)
    if name == "moe_finalize":
        T = w.T * row_scale
        n_rows = w.expert_out.shape[0]
        E = _bits(_rep(w.expert_out, row_scale), dev)
        # copy r of the tokens gathers from copy r of the expert rows: no row is read twice
        idx = np.concatenate([w.idx + r * n_rows for r in range(row_scale)]).astype(np.int32)
        idx = torch.from_numpy(idx).to(dev)
        wt = torch.from_numpy(_rep(w.w, row_scale)).to(dev)
        R = _bits(_rep(w.residual, row_scale), dev)
        ro, yo = torch.empty_like(R), torch.empty_like(R)
        return T, lambda: lb.lb_moe_finalize_fold_norm(
            E, n_rows * row_scale, idx, wt, w.topk, R, ro, G, yo, None, None, T, w.H, w.eps,
            None, stream=sp)
    if name == "ragged_slice" and rsv_rank is not None:
        P = [_bits(p, dev) for p in w.partials]
        rows = int(w.set_counts[rsv_rank])
        o = int(w.set_offsets[rsv_rank])
        R = _bits(w.residual_full[o:o + rows], dev)
        ro, yo = torch.empty_like(R), torch.empty_like(R)
        return rows, lambda: lb.lb_slice_fold_norm_v(
            P, w.T_pad, rsv_rank, w.set_offsets, w.set_counts, R, ro, G, yo, None, None,
            w.H, w.eps, stream=sp)
    if name == "ragged_slice":
        P = [_bits(p, dev) for p in w.partials]
        R = _bits(w.residual, dev)
        ro, yo = torch.empty_like(R), torch.empty_like(R)
        return w.T, lambda: lb.lb_slice_fold_norm(
            P, w.T_pad, w.num_slices, w.slice, w.set_offsets, w.set_counts, R, ro, G, yo,
            None, None, w.H, w.eps, stream=sp)
    T = w.T * row_scale
    P = [_bits(_rep(p, row_scale), dev) for p in w.partials]
    R = None if w.residual is None else _bits(_rep(w.residual, row_scale), dev)
    ro = torch.empty((T, w.H), dtype=torch.bfloat16, device=dev)
    if w.fp8:
        q = torch.empty((T, w.H), dtype=torch.uint8, device=dev)
        s = torch.empty((T,), dtype=torch.float32, device=dev)
        return T, lambda: lb.lb_fold_norm_fp8(P, R, ro, G, q, s, None, T, w.H, w.eps, stream=sp)
    yo = torch.empty_like(ro)
    return T, lambda: lb.lb_fold_norm(P, R, ro, G, yo, T, w.H, w.eps, stream=sp)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("workload", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--row-scale", type=int, default=1)
    ap.add_argument("--sets", type=int, default=2)
    ap.add_argument("--hidden", type=int, default=None,
                    help="prefill_fold_norm_fp8 only: hidden size (default 4096)")
    ap.add_argument("--rsv-rank", type=int, default=None, choices=range(4),
                    help="ragged_slice only: this rank's rows under the variable-size "
                         "reduce-scatter instead of slice 3")
    a = ap.parse_args(argv)
    if a.hidden is not None and a.workload != "prefill_fold_norm_fp8":
        ap.error("--hidden applies to prefill_fold_norm_fp8 only")
    if a.rsv_rank is not None and a.workload != "ragged_slice":
        ap.error("--rsv-rank applies to ragged_slice only")
    dev = torch.device("cuda", 0)
    lb.load()
    stream = torch.cuda.Stream(dev)
    runs = [make_launcher(a.workload, a.row_scale, dev, stream, a.hidden, a.rsv_rank)
            for _ in range(a.sets)]
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(a.launches):
        runs[i % len(runs)][1]()
    e1.record(stream)
    torch.cuda.synchronize()
    print(f"{a.workload}: rows {runs[0][0]}, {a.launches} launches, "
          f"{e0.elapsed_time(e1) * 1e3 / a.launches:.2f} us per launch")
    return 0


if __name__ == "__main__":
    sys.exit(main())
