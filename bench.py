"""Benchmark of the layer-boundary hot path on GB300.

A step is one fused boundary call over the prefill workload the headline metric is
quoted on: K=4 bf16 partial buffers [2048, 4096] (1% outlier rows x50) + residual ->
residual' (bf16) and the per-token FP8 E4M3 RMSNorm read (codes + scales), one
lb_fold_norm_fp8 launch.  Inputs are synthetic and seeded.

Timing: W untimed warm-up steps, then exactly K steps replayed from CUDA graphs,
bracketed by a barrier and a device synchronise, timed with CUDA events on the
launching stream; consecutive steps rotate over enough independent buffer sets that
their total exceeds 3x the L2 size, so every step streams from HBM.  GPU clocks are
sampled with nvidia-smi during the timed region.  Under torchrun each rank runs its
own replica of the workload (rows are independent: weak scaling, no collective on
the data path) and the slowest rank's time counts.

Printed: one JSON line (rank 0).  `--impl reference` times the CPU oracle instead,
on a bounded sample of rows per step.
"""
import argparse
import concurrent.futures
import glob
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from layer_boundary_fusion_gb300 import workloads as wl  # noqa: E402

METRIC = "boundary tokens/s and achieved HBM GB/s (% of ~8 TB/s) at T=2048,H=4096"
HEADLINE = "prefill_fold_norm_fp8"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0    # the ~8 TB/s the metric is stated against
# GPU clock cycles of the delay kernel queued before each timed region (~0.2 ms)
DELAY_CYCLES = 400_000
# variants: timed regions of --variant-steps launches each, the median reported
VARIANT_REPEATS = 5


# --------------------------------------------------------------------------------------
# Process group
# --------------------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False

    def init(self, backend):
        if self.world > 1 and not self.pg:
            import torch.distributed as td
            td.init_process_group(backend)
            self.pg = True

    def barrier(self):
        if self.pg:
            import torch.distributed as td
            td.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch.distributed as td
        dev = "cuda" if td.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        td.all_reduce(t, op=td.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            import torch.distributed as td
            td.destroy_process_group()


def aggregate(elapsed_s: float, rows_per_rank: int, steps: int, dist: Dist):
    """Whole-job throughput: every rank's rows over the slowest rank's time."""
    worst = dist.max(elapsed_s)
    return dist.world * rows_per_rank * steps / worst, worst


# --------------------------------------------------------------------------------------
# Algorithmic bytes (every input byte read once, every output byte written once)
# --------------------------------------------------------------------------------------

def bytes_fold(K, rows, H, residual=True, res_out=True, y=True, fp8=False):
    b = (K + (1 if residual else 0)) * rows * H * 2 + H * 4
    b += rows * H * 2 * ((1 if res_out else 0) + (1 if y else 0))
    if fp8:
        b += rows * H + rows * 4
    return b


def bytes_moe(T, H, topk, residual=True, y=True, fp8=False):
    b = T * topk * H * 2 + 2 * T * topk * 4 + (T * H * 2 if residual else 0) + H * 4
    b += T * H * 2 * (1 + (1 if y else 0))
    if fp8:
        b += T * H + T * 4
    return b


# --------------------------------------------------------------------------------------
# Clocks during the timed region
# --------------------------------------------------------------------------------------

_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.samples = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [f.strip() for f in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [(t, f) for t, f in self.samples if len(f) >= 9]
        mine = [(t, f) for t, f in rows if self.uuid and f[0] == self.uuid] or rows
        inside = [f for t, f in mine if t0 <= t <= t1]
        if not inside:                       # the nearest samples around a short window
            inside = [f for t, f in sorted(mine, key=lambda x: abs(x[0] - (t0 + t1) / 2))[:3]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(f[1]) for f in inside if f[1].replace(".", "").isdigit()]
        mx = [float(f[2]) for f in inside if f[2].replace(".", "").isdigit()]
        reasons = sorted({name for f in inside for name, v in zip(_REASONS, f[5:9])
                          if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside)}


# --------------------------------------------------------------------------------------
# Device helpers
# --------------------------------------------------------------------------------------

def dev_bits(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def n_sets(bytes_per_call, dev):
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    return max(2, math.ceil(3 * l2 / bytes_per_call))


def time_graph(launches, steps, warmup, stream, dist, repeats=1):
    """Replays `steps` launches (cycling over the callables in `launches`) from CUDA
    graphs after `warmup` eager launches, `repeats` times; returns the elapsed seconds
    of each timed region (CUDA events on `stream`; a float when repeats == 1) and the
    wall-clock window of the last one.

    Before each start event the stream gets a self-terminating delay kernel (torch's
    clock-bounded sleep, ~0.2 ms) that keeps the GPU busy while the host submits the
    replays, so the timed region holds the launches alone and not the host's graph
    submission latency."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            launches[i % len(launches)]()
    torch.cuda.synchronize()
    chunk = min(steps, 500)
    graphs = []
    done = 0
    while done < steps:
        n = min(chunk, steps - done)
        if graphs and n == graphs[0][1]:
            graphs.append(graphs[0])
        else:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    launches[(done + i) % len(launches)]()
            graphs.append((g, n))
        done += n
    # untimed replays of each distinct graph (at least ~2000 launches in all), so that
    # the timed region starts with clocks, caches and translations settled
    distinct = list({id(g): (g, n) for g, n in graphs}.values())
    for _ in range(max(1, -(-2000 // steps))):
        for g, _ in distinct:
            g.replay()
    torch.cuda.synchronize()
    out = []
    window = (0.0, 0.0)
    for _ in range(repeats):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        dist.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(DELAY_CYCLES)
            start.record(stream)
            for g, _ in graphs:
                g.replay()
            end.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        dist.barrier()
        out.append(start.elapsed_time(end) / 1e3)
        window = (t0, t1)
    return (out[0] if repeats == 1 else out), window


def plan_of(lb, rows, H, n_inputs, props):
    smem = getattr(props, "shared_memory_per_block_optin", 232448)
    return lb.lb_launch_plan(rows, H, n_inputs, props.multi_processor_count, smem).as_dict()


def kernel_name(plan, mode, fp8):
    kind = "stream_kernel" if plan["kernel"] == 1 else "boundary_kernel"
    return (f"{kind}<{mode}, {'fp8' if fp8 else 'bf16'}, "
            f"{plan['vectors_per_thread']} vectors/thread>")


def kernel_source_hash():
    """Hash of the files that define the library's kernels (their device code, the
    parameter block and the launch-shape constants) as the product build sees them:
    host-side launch and API files, blocks that only the test build compiles, comments
    and blank lines are left out."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "layer_boundary_fusion_gb300", "csrc")
    files = [os.path.join(csrc, n) for n in ("lb_internal.h", "lb_kernel.cuh", "lb_stream.cuh")]
    for f in files:
        text = re.sub(rb"#ifdef LB_TEST_HOOKS\n.*?#endif\n", b"", open(f, "rb").read(),
                      flags=re.S)
        text = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)     # comments do not compile
        text = re.sub(rb"//[^\n]*", b"", text)
        text = b"\n".join(line.rstrip() for line in text.split(b"\n") if line.strip())
        h.update(os.path.basename(f).encode())
        h.update(text)
    return h.hexdigest()


def ncu_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != kernel_source_hash():
        return None
    ent = rec.get("workloads", {}).get(workload)
    return None if ent is None else ent.get("dram_bytes_per_launch")


def peak_hbm():
    try:
        p = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(p["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------------------------
# Workload setup
# --------------------------------------------------------------------------------------

class FoldSet:
    """One independent set of device buffers of a fold workload."""

    def __init__(self, base, dev, fp8):
        self.P = [p.clone() for p in base["P"]]
        self.R = None if base["R"] is None else base["R"].clone()
        self.G = base["G"]
        T, H = base["T"], base["H"]
        self.ro = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.yo = None if fp8 else torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.qo = torch.empty((T, H), dtype=torch.uint8, device=dev) if fp8 else None
        self.so = torch.empty((T,), dtype=torch.float32, device=dev) if fp8 else None


def fold_launcher(lb, s, T, H, eps, fp8, stream):
    sp = stream.cuda_stream
    if fp8:
        return lambda: lb.lb_fold_norm_fp8(s.P, s.R, s.ro, s.G, s.qo, s.so, None, T, H, eps,
                                           stream=sp)
    return lambda: lb.lb_fold_norm(s.P, s.R, s.ro, s.G, s.yo, T, H, eps, stream=sp)


def fold_sets(w, dev, nsets, fp8):
    base = {"P": [dev_bits(p, dev) for p in w.partials],
            "R": None if w.residual is None else dev_bits(w.residual, dev),
            "G": torch.from_numpy(w.gamma).to(dev), "T": w.T, "H": w.H}
    return [FoldSet(base, dev, fp8) for _ in range(nsets)]


# --------------------------------------------------------------------------------------
# Native arm
# --------------------------------------------------------------------------------------

def measure_variants(lb, dev, stream, dist, steps):
    """Per-workload kernel timing of the other specified configurations."""
    out = {}
    peak, _ = peak_hbm()

    def record(name, rows, nbytes, elapsed, launches, shape, l2):
        t = elapsed / launches
        out[name] = {"rows": rows, "us_per_call": round(t * 1e6, 3),
                     "tokens_per_s": round(rows / t, 1), "gbs": round(nbytes / t / 1e9, 1),
                     "frac_of_measured_hbm": round(nbytes / t / 1e9 / peak, 4),
                     "frac_of_nominal_hbm": round(nbytes / t / 1e9 / NOMINAL_HBM_GBS, 4),
                     "bytes_per_call": nbytes, "launch": shape, "l2": l2}

    def tg(ls):
        """Median over VARIANT_REPEATS timed regions of `steps` launches each."""
        runs, _ = time_graph(ls, steps, 20, stream, dist, repeats=VARIANT_REPEATS)
        return statistics.median(runs)

    props = torch.cuda.get_device_properties(dev)
    # decode: K=8 T=64, with and without a residual; rotated and hot-L2
    for name, w in (("decode_fold_norm", wl.decode_fold_norm()),
                    ("decode_initial", wl.decode_fold_norm(initial=True))):
        nb = bytes_fold(w.K, w.T, w.H, residual=w.residual is not None)
        ns = n_sets(nb, dev)
        sets = fold_sets(w, dev, ns, False)
        ls = [fold_launcher(lb, s, w.T, w.H, w.eps, False, stream) for s in sets]
        el = tg(ls)
        record(name, w.T, nb, el, steps, plan_of(lb, w.T, w.H, w.K + (w.residual is not None), props),
               f"rotated {ns} sets")
        el = tg(ls[:1])
        record(name + "_hot_l2", w.T, nb, el, steps,
               plan_of(lb, w.T, w.H, w.K + (w.residual is not None), props),
               "hot: one buffer set, L2-resident")
        # with the residual promise (LB_OPT_RESIDUAL_READY: no call here writes a
        # residual or gamma that the next call reads): residual and gamma load while
        # the previous call drains
        ls = [(lambda s=s: lb.lb_fold_norm(s.P, s.R, s.ro, s.G, s.yo, w.T, w.H, w.eps,
                                           stream=stream.cuda_stream, residual_ready=True))
              for s in sets]
        el = tg(ls)
        record(name + "_residual_ready", w.T, nb, el, steps,
               plan_of(lb, w.T, w.H, w.K + (w.residual is not None), props),
               f"rotated {ns} sets")
        del sets, ls
    # ragged row slice r=3 of 8
    w = wl.ragged_slice()
    S = w.T
    v = sum(max(0, min(o + c, (w.slice + 1) * S) - max(o, w.slice * S))
            for o, c in zip(w.set_offsets.tolist(), w.set_counts.tolist()))
    nb = bytes_fold(w.K, v, w.H)
    ns = n_sets(nb, dev)
    P0 = [dev_bits(p, dev) for p in w.partials]
    R0 = dev_bits(w.residual, dev)
    G = torch.from_numpy(w.gamma).to(dev)
    sets = []
    for _ in range(ns):
        sets.append(([p.clone() for p in P0], R0.clone(), torch.empty_like(R0),
                     torch.empty_like(R0)))
    sp = stream.cuda_stream
    ls = [(lambda s=s: lb.lb_slice_fold_norm(s[0], w.T_pad, w.num_slices, w.slice,
                                            w.set_offsets, w.set_counts, s[1], s[2], G, s[3],
                                            None, None, w.H, w.eps, stream=sp)) for s in sets]
    el = tg(ls)
    record("ragged_slice", v, nb, el, steps, plan_of(lb, S, w.H, w.K + 1, props),
           f"rotated {ns} sets")
    # with the residual promise: the first rows' residual copies go out early
    ls = [(lambda s=s: lb.lb_slice_fold_norm(s[0], w.T_pad, w.num_slices, w.slice,
                                            w.set_offsets, w.set_counts, s[1], s[2], G, s[3],
                                            None, None, w.H, w.eps, stream=sp,
                                            residual_ready=True)) for s in sets]
    el = tg(ls)
    record("ragged_slice_residual_ready", v, nb, el, steps,
           plan_of(lb, S, w.H, w.K + 1, props), f"rotated {ns} sets")
    # the same slice with the FP8 read
    nb8 = bytes_fold(w.K, v, w.H, y=False, fp8=True)
    Q = [(torch.empty((S, w.H), dtype=torch.uint8, device=dev),
          torch.empty((S,), dtype=torch.float32, device=dev)) for _ in sets]
    ls = [(lambda s=s, q=q: lb.lb_slice_fold_norm(s[0], w.T_pad, w.num_slices, w.slice,
                                                 w.set_offsets, w.set_counts, s[1], s[2], G,
                                                 None, q[0], q[1], w.H, w.eps, stream=sp))
          for s, q in zip(sets, Q)]
    el = tg(ls)
    record("ragged_slice_fp8", v, nb8, el, steps, plan_of(lb, S, w.H, w.K + 1, props),
           f"rotated {ns} sets")
    del sets, ls, P0, Q
    # variable-size reduce-scatter (rsv): ranks 1 (512 rows) and 3 (1470 rows)
    for rank in (1, 3):
        o, c = int(w.set_offsets[rank]), int(w.set_counts[rank])
        nb = bytes_fold(w.K, c, w.H)
        ns = n_sets(nb, dev)
        P0 = [dev_bits(p, dev) for p in w.partials]
        R0 = dev_bits(w.residual_full[o:o + c], dev)
        sets = [([p.clone() for p in P0], R0.clone(), torch.empty_like(R0),
                 torch.empty_like(R0)) for _ in range(ns)]
        ls = [(lambda s=s, rank=rank: lb.lb_slice_fold_norm_v(
            s[0], w.T_pad, rank, w.set_offsets, w.set_counts, s[1], s[2], G, s[3], None, None,
            w.H, w.eps, stream=sp)) for s in sets]
        el = tg(ls)
        record(f"ragged_rsv_rank{rank}", c, nb, el, steps, plan_of(lb, c, w.H, w.K + 1, props),
               f"rotated {ns} sets")
        del sets, ls, P0
    # MoE finalize T=1024 top-8
    w = wl.moe_finalize()
    nb = bytes_moe(w.T, w.H, w.topk)
    ns = n_sets(nb, dev)
    E0, R0 = dev_bits(w.expert_out, dev), dev_bits(w.residual, dev)
    I = torch.from_numpy(w.idx).to(dev)
    Wt = torch.from_numpy(w.w).to(dev)
    G = torch.from_numpy(w.gamma).to(dev)
    sets = [(E0.clone(), R0.clone(), torch.empty_like(R0), torch.empty_like(R0))
            for _ in range(ns)]
    ls = [(lambda s=s: lb.lb_moe_finalize_fold_norm(s[0], w.expert_out.shape[0], I, Wt, w.topk,
                                                   s[1], s[2], G, s[3], None, None, w.T, w.H,
                                                   w.eps, None, stream=sp)) for s in sets]
    el = tg(ls)
    record("moe_finalize", w.T, nb, el, steps, plan_of(lb, w.T, w.H, w.topk + 1, props),
           f"rotated {ns} sets")
    # the terminal handoff: the same finalize feeding a Gemma final norm (1 + gamma)
    ls = [(lambda s=s: lb.lb_moe_finalize_fold_norm(s[0], w.expert_out.shape[0], I, Wt, w.topk,
                                                   s[1], s[2], G, s[3], None, None, w.T, w.H,
                                                   w.eps, None, stream=sp, gemma=True))
          for s in sets]
    el = tg(ls)
    record("moe_finalize_gemma", w.T, nb, el, steps, plan_of(lb, w.T, w.H, w.topk + 1, props),
           f"rotated {ns} sets")
    # the FP8 read on the finalize (codes + scales instead of the bf16 read)
    nb8 = bytes_moe(w.T, w.H, w.topk, y=False, fp8=True)
    Q = [(torch.empty((w.T, w.H), dtype=torch.uint8, device=dev),
          torch.empty((w.T,), dtype=torch.float32, device=dev)) for _ in sets]
    ls = [(lambda s=s, q=q: lb.lb_moe_finalize_fold_norm(
        s[0], w.expert_out.shape[0], I, Wt, w.topk, s[1], s[2], G, None, q[0], q[1], w.T, w.H,
        w.eps, None, stream=sp)) for s, q in zip(sets, Q)]
    el = tg(ls)
    record("moe_finalize_fp8", w.T, nb8, el, steps, plan_of(lb, w.T, w.H, w.topk + 1, props),
           f"rotated {ns} sets")
    # with the routing promise (LB_OPT_ROUTING_READY: idx and w are never written by the
    # kernel before a call, here the previous finalize): the first tokens' routing is
    # read before the previous launch finishes
    ls = [(lambda s=s: lb.lb_moe_finalize_fold_norm(s[0], w.expert_out.shape[0], I, Wt, w.topk,
                                                   s[1], s[2], G, s[3], None, None, w.T, w.H,
                                                   w.eps, None, stream=sp, routing_ready=True))
          for s in sets]
    el = tg(ls)
    record("moe_finalize_routing_ready", w.T, nb, el, steps,
           plan_of(lb, w.T, w.H, w.topk + 1, props), f"rotated {ns} sets")
    ls = [(lambda s=s: lb.lb_moe_finalize_fold_norm(s[0], w.expert_out.shape[0], I, Wt, w.topk,
                                                   s[1], s[2], G, s[3], None, None, w.T, w.H,
                                                   w.eps, None, stream=sp, routing_ready=True,
                                                   residual_ready=True))
          for s in sets]
    el = tg(ls)
    record("moe_finalize_both_promises", w.T, nb, el, steps,
           plan_of(lb, w.T, w.H, w.topk + 1, props), f"rotated {ns} sets")
    del sets, ls, Q
    # a decode-size finalize (T=64 tokens of the same routing recipe) on the row kernel,
    # without and with the routing promise
    # (each set holds only the 512 expert rows those tokens gather, renumbered)
    T64 = 64
    E64 = E0[I[:T64].reshape(-1).long()]
    I64 = torch.arange(T64 * w.topk, dtype=torch.int32, device=dev).view(T64, w.topk)
    W64 = Wt[:T64].contiguous()
    nb64 = bytes_moe(T64, w.H, w.topk)
    ns64 = n_sets(nb64, dev)
    sets = [(E64.clone(), R0[:T64].clone(), torch.empty_like(R0[:T64]),
             torch.empty_like(R0[:T64])) for _ in range(ns64)]
    for name, ready, res_ready in (("moe_decode_t64", False, False),
                                   ("moe_decode_t64_routing_ready", True, False),
                                   ("moe_decode_t64_both_promises", True, True)):
        ls = [(lambda s=s: lb.lb_moe_finalize_fold_norm(
            s[0], T64 * w.topk, I64, W64, w.topk, s[1], s[2], G, s[3], None, None,
            T64, w.H, w.eps, None, stream=sp, routing_ready=ready,
            residual_ready=res_ready)) for s in sets]
        el = tg(ls)
        record(name, T64, nb64, el, steps, plan_of(lb, T64, w.H, w.topk + 1, props),
               f"rotated {ns64} sets")
    del sets, ls
    # the headline call with the Gemma weight and an owned snapshot of residual'
    w = wl.prefill_fold_norm_fp8()
    nb = bytes_fold(w.K, w.T, w.H, fp8=True, y=False) + w.T * w.H * 2
    ns = n_sets(nb, dev)
    sets = fold_sets(w, dev, ns, True)
    for s in sets:
        s.snap = torch.empty_like(s.ro)
    ls = [(lambda s=s: lb.lb_fold_norm_fp8(s.P, s.R, s.ro, s.G, s.qo, s.so, None, w.T, w.H,
                                          w.eps, stream=sp, gemma=True,
                                          residual_snapshot=s.snap)) for s in sets]
    el = tg(ls)
    record("prefill_fp8_gemma_snapshot", w.T, nb, el, steps,
           plan_of(lb, w.T, w.H, w.K + 1, props), f"rotated {ns} sets")
    # the headline call with the residual promise
    nb = bytes_fold(w.K, w.T, w.H, fp8=True, y=False)
    ls = [(lambda s=s: lb.lb_fold_norm_fp8(s.P, s.R, s.ro, s.G, s.qo, s.so, None, w.T, w.H,
                                          w.eps, stream=sp, residual_ready=True))
          for s in sets]
    el = tg(ls)
    record("prefill_fp8_residual_ready", w.T, nb, el, steps,
           plan_of(lb, w.T, w.H, w.K + 1, props), f"rotated {ns} sets")
    del sets, ls
    # fusion gain: the same fold + bf16 read as one fused call and as the unfused
    # fallback of two calls (the completed sum written to a bf16 buffer, then residual
    # add + RMSNorm of that buffer), both on this library's kernels
    for name, w in (("prefill_bf16", wl.prefill_fold_norm_fp8()),
                    ("decode", wl.decode_fold_norm())):
        nb = bytes_fold(w.K, w.T, w.H)
        moved = nb + 2 * 2 * w.T * w.H                 # + the sum written and read back
        ns = n_sets(moved, dev)
        sets = fold_sets(w, dev, ns, False)
        fused = [fold_launcher(lb, s, w.T, w.H, w.eps, False, stream) for s in sets]
        el = tg(fused)
        record(f"{name}_fused", w.T, nb, el, steps,
               plan_of(lb, w.T, w.H, w.K + 1, props), f"rotated {ns} sets")
        for s in sets:
            s.sum = torch.empty_like(s.ro)

        def unfused(s=None, w=w):
            lb.lb_fold_norm(s.P, None, s.sum, None, None, w.T, w.H, w.eps, stream=sp)
            lb.lb_fold_norm([s.sum], s.R, s.ro, s.G, s.yo, w.T, w.H, w.eps, stream=sp)
        ls = [(lambda s=s: unfused(s)) for s in sets]
        el = tg(ls)
        record(f"{name}_unfused", w.T, nb, el, steps,
               [plan_of(lb, w.T, w.H, w.K, props), plan_of(lb, w.T, w.H, 2, props)],
               f"rotated {ns} sets")
        out[f"{name}_unfused"]["bytes_moved_per_call"] = moved
        out[f"{name}_fusion_speedup"] = round(out[f"{name}_unfused"]["us_per_call"]
                                              / out[f"{name}_fused"]["us_per_call"], 3)
        del sets, ls, fused
    # tiny correctness configuration
    w = wl.tiny_fold_norm()
    nb = bytes_fold(w.K, w.T, w.H)
    sets = fold_sets(w, dev, 1, False)
    ls = [fold_launcher(lb, sets[0], w.T, w.H, w.eps, False, stream)]
    el = tg(ls)
    record("tiny_fold_norm", w.T, nb, el, steps, plan_of(lb, w.T, w.H, w.K + 1, props),
           "hot: one buffer set, L2-resident")
    torch.cuda.empty_cache()
    return out


# The five specified workloads and the bench entries that time them.
CONFIGS = (
    ("cfg1_tiny_K2_T16_H512", "tiny_fold_norm"),
    ("cfg2_decode_K8_T64", "decode_fold_norm"),
    ("cfg2_decode_initial_K8_T64", "decode_initial"),
    ("cfg3_prefill_fp8_K4_T2048", None),               # the headline call itself
    ("cfg4_ragged_slice_r3_K8_S254", "ragged_slice"),
    ("cfg5_moe_finalize_T1024_top8", "moe_finalize"),
)


def config_summary(variants, headline):
    """One compact entry per specified workload: us per call, GB/s, fractions of the
    measured copy peak and of the nominal 8 TB/s, the kernel and the L2 mode."""
    out = {}
    for name, key in CONFIGS:
        v = headline if key is None else variants.get(key)
        if v is None:
            continue
        launch = v["launch"]
        kind = "stream" if launch.get("kernel") == 1 else "row"
        out[name] = {"us": v["us_per_call"], "gbs": v["gbs"],
                     "frac_measured": v["frac_of_measured_hbm"],
                     "frac_8tbs": v["frac_of_nominal_hbm"],
                     "kernel": f"{kind} grid {launch.get('grid')}",
                     "l2": "hot" if v["l2"].startswith("hot") else "rotated"}
    return out


def host_cpu():
    """Host cores this process may use, and the CPU model as /proc/cpuinfo names it."""
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    model = platform.machine()
    try:
        info = open("/proc/cpuinfo").read()
        m = re.search(r"^model name\s*:\s*(.+)$", info, re.M)
        if m:
            model = m.group(1).strip()
        else:
            imp = re.search(r"^CPU implementer\s*:\s*(\S+)$", info, re.M)
            part = re.search(r"^CPU part\s*:\s*(\S+)$", info, re.M)
            if imp and part:
                model = f"{platform.machine()} implementer {imp.group(1)} part {part.group(1)}"
    except OSError:
        pass
    return cores, model


def oracle_rate(w, threads, seconds, rows_per_thread):
    """Tokens/s of the oracle, as it stands, on the headline workload's rows: `threads`
    threads each run oracle calls on their own block of `rows_per_thread` rows until
    `seconds` have passed (the oracle releases the GIL inside its C code)."""
    import oracle
    oracle._load()
    blocks = []
    for i in range(threads):
        lo = (i * rows_per_thread) % w.T
        hi = min(w.T, lo + rows_per_thread)
        blocks.append(([p[lo:hi] for p in w.partials], w.residual[lo:hi]))
    t0 = time.perf_counter()
    stop = t0 + seconds

    def work(block):
        P, R = block
        n = 0
        while time.perf_counter() < stop:
            oracle.fold_norm(P, R, w.gamma, w.eps, want_y=False, want_fp8=True)
            n += R.shape[0]
        return n

    with concurrent.futures.ThreadPoolExecutor(threads) as ex:
        done = sum(ex.map(work, blocks))
    el = time.perf_counter() - t0
    return done / el, done, el


def cpu_baseline(w, seconds=10.0):
    """The oracle, as it stands, on a bounded sample of the headline workload: rows
    partitioned over every host core (the reported value), and on one core."""
    cores, model = host_cpu()
    rows = 16
    v1, n1, e1 = oracle_rate(w, 1, seconds / 3, rows)
    vn, nn, en = oracle_rate(w, cores, seconds, rows)
    return {"value": round(vn, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{nn} rows of the K=4 T=2048 H=4096 prefill workload (FP8 read), "
                      f"{rows}-row blocks, one per thread, over {cores} threads for "
                      f"{en:.1f} s",
            "single_thread": {"value": round(v1, 1), "rows": n1, "seconds": round(e1, 1)},
            "cpu": model}


def run_native(args, dist):
    from layer_boundary_fusion_gb300 import build as lb_build
    from layer_boundary_fusion_gb300 import lb

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the native arm has no CPU path)")
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    if dist.rank == 0:
        lb_build.build()
    dist.barrier()
    lb.load()
    stream = torch.cuda.Stream(dev)

    w = wl.prefill_fold_norm_fp8()
    nbytes = bytes_fold(w.K, w.T, w.H, fp8=True, y=False)
    ns = n_sets(nbytes, dev)
    sets = fold_sets(w, dev, ns, True)
    launches = [fold_launcher(lb, s, w.T, w.H, w.eps, True, stream) for s in sets]
    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(getattr(props, "uuid", None) and f"GPU-{props.uuid}")
    sampler.start()
    time.sleep(0.3)
    elapsed, window = time_graph(launches, args.steps, args.warmup, stream, dist)
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(*window)
    value, worst = aggregate(elapsed, w.T, args.steps, dist)
    per_launch = elapsed / args.steps
    peak, peak_src = peak_hbm()
    achieved = nbytes / per_launch / 1e9

    # end to end through the public API: pinned host inputs -> device -> call -> host,
    # each step copying its inputs in and its results out, overlapped in row chunks
    from layer_boundary_fusion_gb300.host import HostPipeline
    e2e_steps = args.e2e_steps
    hP = [torch.from_numpy(p.view(np.int16)).pin_memory() for p in w.partials]
    hR = torch.from_numpy(w.residual.view(np.int16)).pin_memory()
    hG = torch.from_numpy(w.gamma).pin_memory()
    hro = torch.empty((w.T, w.H), dtype=torch.int16).pin_memory()
    hq = torch.empty((w.T, w.H), dtype=torch.uint8).pin_memory()
    hs = torch.empty((w.T,), dtype=torch.float32).pin_memory()
    h2d = sum(p.numel() * 2 for p in hP) + hR.numel() * 2 + hG.numel() * 4
    d2h = hro.numel() * 2 + hq.numel() + hs.numel() * 4
    del sets, launches
    torch.cuda.empty_cache()
    pipe = HostPipeline(w.K, w.T, w.H, dev, chunks=1, depth=2)
    per_run = min(20, e2e_steps)                   # steps per pipelined run (one graph)
    runs = max(1, -(-e2e_steps // per_run))
    e2e_steps = runs * per_run
    cur = torch.cuda.current_stream(dev)
    for _ in range(2):
        pipe.run(per_run, hP, hR, hG, hro, hq, hs, w.eps, stream=cur)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    ev0.record(cur)
    for _ in range(runs):
        pipe.run(per_run, hP, hR, hG, hro, hq, hs, w.eps, stream=cur)
    ev1.record(cur)
    torch.cuda.synchronize()
    e2e_value, _ = aggregate(ev0.elapsed_time(ev1) / 1e3, w.T, e2e_steps, dist)
    del pipe
    torch.cuda.empty_cache()

    variants = measure_variants(lb, dev, stream, dist, args.variant_steps)
    cpu = cpu_baseline(w) if (dist.rank == 0 and dist.world == 1) else None

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(worst / args.steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded normal bf16 inputs)",
        "config": {"workload": HEADLINE, "K": w.K, "T": w.T, "H": w.H, "eps": w.eps,
                   "outliers": "1% of rows x50 in every partial",
                   "storage": "bf16 partials/residual/residual', fp32 gamma, e4m3 codes + "
                              "fp32 per-token scales",
                   "l2": f"inputs larger than L2: {ns} rotating buffer sets of "
                         f"{nbytes / 1e6:.1f} MB ({ns * nbytes / 1e6:.0f} MB total, L2 "
                         f"{props.L2_cache_size / 1e6:.0f} MB)",
                   "launch": plan_of(lb, w.T, w.H, w.K + 1, props),
                   "timing": "CUDA graphs of up to 500 launches, CUDA events on the "
                             "launching stream, a clock-bounded delay kernel queued before "
                             "the start event; variants: median of "
                             f"{VARIANT_REPEATS} timed regions",
                   "parallelism": f"replica per GPU x{dist.world} (rows independent)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "traffic": ncu_traffic(HEADLINE), "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": nbytes,
                     "kernel": kernel_name(plan_of(lb, w.T, w.H, w.K + 1, props), "fold", True)},
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "how": "pinned host buffers; per step gamma and inputs copied in and "
                       "residual', codes and scales copied out; consecutive steps on two "
                       "device buffer sets so that one step's copy-in overlaps the "
                       "previous step's copy-out; 20 steps per CUDA graph "
                       "(layer_boundary_fusion_gb300.host)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "variants": variants,
    }
    headline = {"us_per_call": round(per_launch * 1e6, 3), "gbs": round(achieved, 1),
                "frac_of_measured_hbm": round(achieved / peak, 4),
                "frac_of_nominal_hbm": round(achieved / NOMINAL_HBM_GBS, 4),
                "launch": plan_of(lb, w.T, w.H, w.K + 1, props),
                "l2": f"rotated {ns} sets"}
    # last key of the line: the five specified workloads at a glance
    line["configs"] = config_summary(variants, headline)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


# --------------------------------------------------------------------------------------
# Reference arm: the CPU oracle, as it stands
# --------------------------------------------------------------------------------------

def run_reference(args, dist):
    if dist.rank != 0:
        return                                # rank 0 alone runs the oracle
    import oracle
    oracle._load()
    w = wl.prefill_fold_norm_fp8()
    cores, model = host_cpu()
    # calibrate, then size each step's sample so the whole run takes ~2 minutes with
    # the step's rows split into one contiguous block per host core
    t0 = time.perf_counter()
    oracle.fold_norm([p[:8] for p in w.partials], w.residual[:8], w.gamma, w.eps,
                     want_y=False, want_fp8=True)
    per_row = (time.perf_counter() - t0) / 8
    budget = 120.0
    rows = int(budget / max(1, args.steps + args.warmup) / per_row * cores)
    rows = max(cores, min(w.T, rows))
    edges = [rows * i // cores for i in range(cores + 1)]
    blocks = [([p[lo:hi] for p in w.partials], w.residual[lo:hi])
              for lo, hi in zip(edges[:-1], edges[1:]) if hi > lo]

    def one(block):
        oracle.fold_norm(block[0], block[1], w.gamma, w.eps, want_y=False, want_fp8=True)

    with concurrent.futures.ThreadPoolExecutor(len(blocks)) as ex:
        def step():
            for _ in ex.map(one, blocks):
                pass
        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        el = time.perf_counter() - t0
    value = rows * args.steps / el
    sample = (f"{rows} rows of the K=4 T=2048 H=4096 prefill workload per step, split "
              f"into {len(blocks)} row blocks run by {len(blocks)} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded normal bf16 inputs)",
        "config": {"workload": HEADLINE, "K": w.K, "T": w.T, "H": w.H, "eps": w.eps,
                   "rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": len(blocks),
                         "kind": "oracle", "sample": sample, "cpu": model},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--variant-steps", type=int, default=5000)
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    dist = Dist()
    if dist.world != args.gpus and dist.world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={dist.world}")
    if args.impl == "reference":
        run_reference(args, dist)
    else:
        run_native(args, dist)


if __name__ == "__main__":
    main()
