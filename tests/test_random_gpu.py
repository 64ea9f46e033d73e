"""Seeded random sweep of the boundary calls against the oracle on the GPU.

Each case draws a shape (K, T, H with H % 8 == 0), a stream mode (Initial or not,
bf16 read, FP8 read, both, none) and the options (Gemma weight, residual snapshot,
in-place residual, the residual and routing promises) from a fixed seed, runs the call through the C ABI with guard rows
around every output, and compares element by element with the oracle under the parity
bar of tests/parity_util.py.  The shapes straddle both kernels (rows below and above
the SM count), 1, 2 and 4 vectors per thread and ragged last vectors of a warp.  MoE
and ragged-slice cases draw their routing and set layouts the same way.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from layer_boundary_fusion_gb300 import workloads as wl
from parity_util import (Guarded, assert_bf16_close, assert_bits_equal, assert_fp8_close,
                         dev_bits, host_bits)

pytestmark = pytest.mark.gpu

MAX_ELEMS = 3_000_000      # rows x H per case: the oracle finishes each in about a second
# cases per sweep (a deeper one-off run: LB_RANDOM_SCALE=10)
SCALE = int(os.environ.get("LB_RANDOM_SCALE", "1"))


@pytest.fixture(scope="module")
def lb():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the parity tests")
    from layer_boundary_fusion_gb300 import build, lb as binding
    build.build()
    binding.load()
    binding.lb_device_error(clear=True)
    yield binding
    assert binding.lb_device_error(clear=True) == 0


def _draw_shape(rng):
    H = int(rng.choice([8, 24, 64, 520, 1024, 2048, 2056, 4096, 6144, 8192, 10240, 12288,
                          16384]))
    T = int(rng.choice([1, 3, 17, 64, 151, 152, 153, 300, 777, 1500]))
    while T * H > MAX_ELEMS and T > 1:
        T //= 2
    return T, H


def _compare(got, want, what, res_exact=True):
    if "residual_out" in got:
        if res_exact:
            assert_bits_equal(got["residual_out"], want["residual_out"], f"{what} residual'")
        assert_bf16_close(got["residual_out"], want["residual_out"], f"{what} residual'")
    if "snapshot" in got:
        assert_bits_equal(got["snapshot"], want["residual_out"], f"{what} snapshot")
    if "y" in got:
        assert_bf16_close(got["y"], want["y"], f"{what} y")
    if "q" in got:
        assert_fp8_close(got["q"], want["q"], got["scale"], want["scale"], f"{what} fp8")


@pytest.mark.parametrize("case", range(40 * SCALE))
def test_random_fold(lb, case):
    rng = np.random.default_rng(1000 + case)
    T, H = _draw_shape(rng)
    residual = bool(rng.random() < 0.8)
    K = int(rng.integers(0 if residual else 1, 17))
    read = str(rng.choice(["bf16", "fp8", "both", "none"]))
    gemma = bool(rng.random() < 0.3)
    snapshot = bool(rng.random() < 0.3)
    in_place = residual and bool(rng.random() < 0.3)
    if read == "none" and not residual and K == 0:
        read = "bf16"
    w = wl.fold_workload("rand", K, T, H, seed=2000 + case, residual=residual,
                         outlier_frac=0.02 if rng.random() < 0.3 else 0.0)
    residual_ready = bool(rng.random() < 0.4)     # the promise changes no result
    fp8 = read in ("fp8", "both")
    want_y = read in ("bf16", "both")
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_y=True,
                            want_fp8=fp8, gemma=gemma)
    P = [dev_bits(p) for p in w.partials]
    R = dev_bits(w.residual) if residual else None
    G = torch.from_numpy(w.gamma).cuda()
    ro = None if in_place else Guarded(T, H, torch.bfloat16)
    yo = Guarded(T, H, torch.bfloat16) if want_y else None
    qo = Guarded(T, H, torch.uint8) if fp8 else None
    so = Guarded(T, 0, torch.float32) if fp8 else None
    sn = Guarded(T, H, torch.bfloat16) if snapshot else None
    res_out = R if in_place else ro.t
    kw = dict(gemma=gemma, residual_snapshot=sn.t if sn else None,
              residual_ready=residual_ready)
    if fp8:
        lb.lb_fold_norm_fp8(P, R, res_out, G, qo.t, so.t, yo.t if yo else None, T, H, w.eps,
                            **kw)
    else:
        lb.lb_fold_norm(P, R, res_out, G if want_y else None, yo.t if yo else None, T, H,
                        w.eps, **kw)
    torch.cuda.synchronize()
    got = {}
    for name, g in (("residual_out", ro), ("y", yo), ("q", qo), ("scale", so),
                    ("snapshot", sn)):
        if g is not None:
            g.check()
            got[name] = g.host()
    if in_place:
        got["residual_out"] = host_bits(R)
    _compare(got, want, f"case {case}: K={K} T={T} H={H} read={read} res={residual} "
                        f"gemma={gemma} snap={snapshot} inplace={in_place} "
                        f"promise={residual_ready}")


@pytest.mark.parametrize("case", range(16 * SCALE))
def test_random_moe(lb, case):
    rng = np.random.default_rng(3000 + case)
    T, H = _draw_shape(rng)
    topk = int(rng.integers(1, 17))
    E = int(rng.integers(topk, 4 * topk + 2))
    while T * topk * H > 4 * MAX_ELEMS and T > 1:
        T //= 2
    residual = bool(rng.random() < 0.8)
    fp8 = bool(rng.random() < 0.4)
    gemma = bool(rng.random() < 0.3)
    w = wl.moe_workload("rand_moe", T, H, E, topk, seed=4000 + case, residual=residual)
    routing_ready, residual_ready = bool(rng.random() < 0.4), bool(rng.random() < 0.4)
    want = oracle.moe_finalize_fold_norm(w.expert_out, w.idx, w.w, w.residual, w.gamma,
                                         w.eps, want_fp8=fp8, gemma=gemma)
    Ex = dev_bits(w.expert_out)
    I = torch.from_numpy(w.idx).cuda()
    Wt = torch.from_numpy(w.w).cuda()
    R = dev_bits(w.residual) if residual else None
    G = torch.from_numpy(w.gamma).cuda()
    ro, yo = Guarded(T, H, torch.bfloat16), Guarded(T, H, torch.bfloat16)
    qo = Guarded(T, H, torch.uint8) if fp8 else None
    so = Guarded(T, 0, torch.float32) if fp8 else None
    lb.lb_moe_finalize_fold_norm(Ex, w.expert_out.shape[0], I, Wt, topk, R, ro.t, G, yo.t,
                                 qo.t if fp8 else None, so.t if fp8 else None, T, H, w.eps,
                                 None, gemma=gemma, routing_ready=routing_ready,
                                 residual_ready=residual_ready)
    torch.cuda.synchronize()
    got = {}
    for name, g in (("residual_out", ro), ("y", yo), ("q", qo), ("scale", so)):
        if g is not None:
            g.check()
            got[name] = g.host()
    _compare(got, want, f"moe case {case}: T={T} H={H} E={E} topk={topk} res={residual} "
                        f"fp8={fp8} gemma={gemma} promises={routing_ready},{residual_ready}")


@pytest.mark.parametrize("case", range(12 * SCALE))
def test_random_slices(lb, case):
    rng = np.random.default_rng(5000 + case)
    H = int(rng.choice([64, 1024, 4096]))
    n_sets = int(rng.integers(1, 7))
    counts = [int(c) for c in rng.integers(0, 400, n_sets)]
    K = int(rng.integers(1, 9))
    _, _, T_pad = wl.ragged_layout(counts)
    if T_pad == 0:
        counts[0], T_pad = 5, 8                 # keep the batch non-empty
    num_slices = int(rng.choice([1, 2, 4, 8]))  # T_pad is a multiple of 8
    fp8 = bool(rng.random() < 0.4)
    w = wl.slice_workload("rand_slice", K, H, counts, num_slices, 0, seed=6000 + case)
    S = T_pad // num_slices
    P = [dev_bits(p) for p in w.partials]
    G = torch.from_numpy(w.gamma).cuda()
    valid = np.zeros(T_pad, bool)
    for o, c in zip(w.set_offsets, w.set_counts):
        valid[o:o + c] = True
    for r in range(num_slices):
        R = dev_bits(w.residual_full[r * S:(r + 1) * S])
        ro, yo = Guarded(S, H, torch.bfloat16), Guarded(S, H, torch.bfloat16)
        qo = Guarded(S, H, torch.uint8) if fp8 else None
        so = Guarded(S, 0, torch.float32) if fp8 else None
        lb.lb_slice_fold_norm(P, T_pad, num_slices, r, w.set_offsets, w.set_counts, R, ro.t,
                              G, yo.t, qo.t if fp8 else None, so.t if fp8 else None, H, w.eps,
                              residual_ready=bool(r % 2))
        torch.cuda.synchronize()
        want = oracle.slice_fold_norm(w.partials, T_pad, num_slices, r, w.set_offsets,
                                      w.set_counts, w.residual_full[r * S:(r + 1) * S],
                                      w.gamma, w.eps, want_fp8=fp8)
        v = valid[r * S:(r + 1) * S]
        for g in (ro, yo, qo, so):
            if g is not None:
                g.check()
        gr, gy = ro.host(), yo.host()
        what = f"slice case {case} r={r}: counts={counts} K={K} H={H} slices={num_slices}"
        assert np.all(gr[~v] == 0x7FC1) and np.all(gy[~v] == 0x7FC1), what + " padding written"
        assert_bits_equal(gr, want["residual_out"], what, rows=v)
        assert_bf16_close(gy, want["y"], what, rows=v)
        if fp8:
            assert_fp8_close(qo.host(), want["q"], so.host(), want["scale"], what, rows=v)
