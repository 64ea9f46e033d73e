"""GPU parity: every entry point of liblb.so, called through the C ABI, against the
CPU oracle on the same seeded bf16 inputs, element by element.

Covered: the five specified workloads at full size (tiny fold+norm; decode K=8
T=64 with and without a residual; prefill K=4 T=2048 with the FP8 read; every slice
of the ragged batch; the MoE finalize), every stream mode (enter, complete_output,
fold, read, fold+read, in place), the launch shapes (cluster split, 1/2/4 vectors
per thread, partly active warps), the maximum K and topk, empty batches, zero rows,
bad expert indices, guard rows around every output and unchanged inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from layer_boundary_fusion_gb300 import workloads as wl
from parity_util import (Guarded, assert_bf16_close, assert_bits_equal, assert_fp8_close,
                         dev_bits, f32, host_bits, SENTINEL16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lb():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the parity tests")
    from layer_boundary_fusion_gb300 import build, lb as binding
    build.build()
    binding.load()
    binding.lb_device_error(clear=True)
    yield binding
    # no bounded wait of the stream kernel may have timed out in any test
    assert binding.lb_device_error(clear=True) == 0


def plan(lb, rows, H, n_in):
    props = torch.cuda.get_device_properties(0)
    return lb.lb_launch_plan(rows, H, n_in, props.multi_processor_count,
                             props.shared_memory_per_block_optin)


def _snapshot(ts):
    return [None if t is None else t.clone() for t in ts]


def _assert_unchanged(before, after):
    for b, a in zip(before, after):
        if b is not None:
            assert torch.equal(b.view(torch.int16) if b.dtype == torch.bfloat16 else b,
                               a.view(torch.int16) if a.dtype == torch.bfloat16 else a), \
                "an input buffer was modified"


def gpu_fold(lb, partials, residual, gamma, eps, *, want_res=True, want_y=True, fp8=False,
             want_y_fp8=False, in_place=False):
    T, H = (partials[0] if partials else residual).shape
    P = [dev_bits(p) for p in partials]
    R = dev_bits(residual) if residual is not None else None
    G = torch.from_numpy(np.ascontiguousarray(gamma)).cuda()
    ro = Guarded(T, H, torch.bfloat16) if want_res and not in_place else None
    yo = Guarded(T, H, torch.bfloat16) if (want_y and not fp8) or want_y_fp8 else None
    qo = Guarded(T, H, torch.uint8) if fp8 else None
    so = Guarded(T, 0, torch.float32) if fp8 else None
    res_out = R if in_place else (ro.t if ro else None)
    before = _snapshot(P + [None if in_place else R, G])
    if fp8:
        lb.lb_fold_norm_fp8(P, R, res_out, G, qo.t, so.t, yo.t if yo else None, T, H, eps)
    else:
        lb.lb_fold_norm(P, R, res_out, G if want_y else None, yo.t if yo else None, T, H, eps)
    torch.cuda.synchronize()
    _assert_unchanged(before, P + [None if in_place else R, G])
    out = {}
    for name, g in (("residual_out", ro), ("y", yo), ("q", qo), ("scale", so)):
        if g is not None:
            g.check()
            out[name] = g.host()
    if in_place:
        out["residual_out"] = host_bits(R)
    return out


def check_fold(got, want, what):
    if "residual_out" in want and want.get("residual_out") is not None and "residual_out" in got:
        assert_bits_equal(got["residual_out"], want["residual_out"], f"{what} residual'")
        assert_bf16_close(got["residual_out"], want["residual_out"], f"{what} residual'")
    if "y" in got:
        assert_bf16_close(got["y"], want["y"], f"{what} y")
    if "q" in got:
        assert_fp8_close(got["q"], want["q"], got["scale"], want["scale"], f"{what} fp8")


# --------------------------------------------------------------------------------------
# The specified workloads
# --------------------------------------------------------------------------------------

def test_tiny_fold_norm(lb):
    w = wl.tiny_fold_norm()
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps)
    check_fold(gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps), want, "tiny")


@pytest.mark.parametrize("initial", [False, True])
def test_decode_fold_norm(lb, initial):
    w = wl.decode_fold_norm(initial=initial)
    assert (w.residual is None) == initial
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps)
    check_fold(gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps), want, w.name)


def test_prefill_fold_norm_fp8_full_size(lb):
    w = wl.prefill_fold_norm_fp8()
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_fp8=True)
    got = gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, fp8=True)
    check_fold(got, want, "prefill fp8")
    # outlier rows: residual' carries the x50 rows, the normalised read does not
    big = np.abs((got["residual_out"].astype(np.uint32) << 16).view(np.float32)).max()
    assert big > 50.0


def test_prefill_fp8_with_bf16_read(lb):
    w = wl.fold_workload("p", 4, 256, 4096, seed=2, outlier_frac=0.01, fp8=True)
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_fp8=True)
    got = gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, fp8=True, want_y_fp8=True)
    check_fold(got, want, "fp8 + y")


def _gpu_slice(lb, w, r, fp8=False):
    S, H = w.T // 1, w.H
    P = [dev_bits(p) for p in w.partials]
    R = dev_bits(w.residual_full[r * S:(r + 1) * S])
    G = torch.from_numpy(w.gamma).cuda()
    ro, yo = Guarded(S, H, torch.bfloat16), Guarded(S, H, torch.bfloat16)
    qo = Guarded(S, H, torch.uint8) if fp8 else None
    so = Guarded(S, 0, torch.float32) if fp8 else None
    before = _snapshot(P + [R, G])
    lb.lb_slice_fold_norm(P, w.T_pad, w.num_slices, r, w.set_offsets, w.set_counts, R,
                          ro.t, G, yo.t, qo.t if fp8 else None, so.t if fp8 else None, H,
                          w.eps)
    torch.cuda.synchronize()
    _assert_unchanged(before, P + [R, G])
    out = {"residual_out": ro, "y": yo}
    if fp8:
        out.update(q=qo, scale=so)
    for g in out.values():
        g.check()
    return {k: g.host() for k, g in out.items()}


@pytest.mark.parametrize("fp8", [False, True])
def test_ragged_slice_every_rank(lb, fp8):
    w = wl.ragged_slice()
    S = w.T
    assert (w.T_pad, S) == (2032, 254)
    valid = np.zeros(w.T_pad, bool)
    for o, c in zip(w.set_offsets, w.set_counts):
        valid[o:o + c] = True
    for r in range(w.num_slices):
        sent = {"residual_out": np.full((S, w.H), SENTINEL16, np.uint16),
                "y": np.full((S, w.H), SENTINEL16, np.uint16)}
        want = oracle.slice_fold_norm(w.partials, w.T_pad, w.num_slices, r, w.set_offsets,
                                      w.set_counts, w.residual_full[r * S:(r + 1) * S],
                                      w.gamma, w.eps, want_fp8=fp8, out=sent)
        got = _gpu_slice(lb, w, r, fp8=fp8)
        v = valid[r * S:(r + 1) * S]
        # placement: padding rows untouched, valid rows written -- bit-exact
        assert_bits_equal(got["residual_out"][~v], want["residual_out"][~v], f"slice {r} pad")
        assert np.all(got["y"][~v] == SENTINEL16)
        assert_bits_equal(got["residual_out"], want["residual_out"], f"slice {r} residual'",
                          rows=v)
        assert_bf16_close(got["y"], want["y"], f"slice {r} y", rows=v)
        if fp8:
            assert np.all(got["q"][~v] == 0x7F)
            assert_fp8_close(got["q"], want["q"], got["scale"], want["scale"],
                             f"slice {r} fp8", rows=v)


def _gpu_moe(lb, w, *, idx=None, residual=True, fp8=False, flag=False, want_y=True,
             routing_ready=False, residual_ready=False):
    T, H = w.T, w.H
    idx = w.idx if idx is None else idx
    E = dev_bits(w.expert_out)
    I = torch.from_numpy(np.ascontiguousarray(idx)).cuda()
    Wt = torch.from_numpy(np.ascontiguousarray(w.w)).cuda()
    R = dev_bits(w.residual) if residual else None
    G = torch.from_numpy(w.gamma).cuda()
    ro = Guarded(T, H, torch.bfloat16)
    yo = Guarded(T, H, torch.bfloat16) if want_y else None
    qo = Guarded(T, H, torch.uint8) if fp8 else None
    so = Guarded(T, 0, torch.float32) if fp8 else None
    F = torch.zeros(1, dtype=torch.int32, device="cuda") if flag else None
    before = _snapshot([E, I, Wt, R, G])
    lb.lb_moe_finalize_fold_norm(E, w.expert_out.shape[0], I, Wt, idx.shape[1], R, ro.t, G,
                                 yo.t if yo else None, qo.t if fp8 else None,
                                 so.t if fp8 else None, T, H, w.eps, F,
                                 routing_ready=routing_ready, residual_ready=residual_ready)
    torch.cuda.synchronize()
    _assert_unchanged(before, [E, I, Wt, R, G])
    out = {"residual_out": ro}
    if want_y:
        out["y"] = yo
    if fp8:
        out.update(q=qo, scale=so)
    for g in out.values():
        g.check()
    res = {k: g.host() for k, g in out.items()}
    if flag:
        res["flag"] = int(F.item())
    return res


def test_moe_finalize_full_size(lb):
    w = wl.moe_finalize()
    want = oracle.moe_finalize_fold_norm(w.expert_out, w.idx, w.w, w.residual, w.gamma, w.eps)
    got = _gpu_moe(lb, w)
    check_fold(got, want, "moe")


def test_moe_finalize_fp8_and_initial(lb):
    w = wl.moe_workload("m", 200, 2048, 32, 6, seed=41)
    want = oracle.moe_finalize_fold_norm(w.expert_out, w.idx, w.w, None, w.gamma, w.eps,
                                         want_fp8=True)
    got = _gpu_moe(lb, w, residual=False, fp8=True)
    check_fold(got, want, "moe fp8 initial")


@pytest.mark.parametrize("T,H,E,topk", [(1, 4096, 16, 16), (37, 520, 8, 3), (64, 8192, 64, 8),
                                        (5, 16384, 8, 1), (200, 1024, 16, 16),
                                        (1, 2048, 128, 8),
                                        (300, 8192, 64, 8),     # row kernel past the SMs
                                        (200, 12288, 16, 4),    # stream kernel, 3 chunks
                                        (160, 10240, 32, 8),    # 3 chunks, the last short
                                        (1200, 12288, 64, 2)])  # chunked, many wraps
def test_moe_shapes(lb, T, H, E, topk):
    w = wl.moe_workload("m", T, H, E, topk, seed=T + H)
    want = oracle.moe_finalize_fold_norm(w.expert_out, w.idx, w.w, w.residual, w.gamma, w.eps)
    check_fold(_gpu_moe(lb, w), want, f"moe {T}x{H} top{topk}")


def test_moe_bad_index_is_skipped_and_flagged(lb):
    w = wl.moe_workload("bad", 16, 256, 4, 4, seed=42)
    idx = w.idx.copy()
    idx[3, 2] = w.expert_out.shape[0]
    idx[9, 0] = -5
    want = oracle.moe_finalize_fold_norm(w.expert_out, idx, w.w, w.residual, w.gamma, w.eps)
    assert want["bad_index"]
    got = _gpu_moe(lb, w, idx=idx, flag=True)
    assert got["flag"] == 1
    check_fold(got, want, "moe bad index")
    clean = _gpu_moe(lb, w, flag=True)
    assert clean["flag"] == 0


# --------------------------------------------------------------------------------------
# Stream modes ("Residual stream" state table)
# --------------------------------------------------------------------------------------

def test_stream_modes(lb):
    w = wl.fold_workload("modes", 3, 50, 1024, seed=51)
    full = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps)
    # enter (Initial): no residual
    init = oracle.fold_norm(w.partials, None, w.gamma, w.eps)
    check_fold(gpu_fold(lb, w.partials, None, w.gamma, w.eps), init, "enter")
    # complete_output: the sum alone, no read
    got = gpu_fold(lb, w.partials, None, w.gamma, w.eps, want_y=False)
    assert set(got) == {"residual_out"}
    assert_bits_equal(got["residual_out"], init["residual_out"], "complete_output")
    # fold: residual updated, no read
    got = gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, want_y=False)
    assert_bits_equal(got["residual_out"], full["residual_out"], "fold")
    # read of a Written stream: K = 0, no residual output
    rd = oracle.fold_norm([], full["residual_out"], w.gamma, w.eps, want_residual=False)
    got = gpu_fold(lb, [], full["residual_out"], w.gamma, w.eps, want_res=False)
    assert set(got) == {"y"}
    assert_bf16_close(got["y"], rd["y"], "read")
    # fold + read in place (residual_out == residual_in)
    got = gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, in_place=True)
    check_fold(got, full, "in place")


@pytest.mark.parametrize("T,H", [(50, 2048), (700, 2048), (300, 12288)])
def test_stream_modes_on_both_kernels(lb, T, H):
    """The same stream modes with enough rows for the persistent TMA kernel (T=700;
    T=300 with rows in column chunks) and few enough for the row kernel (T=50)."""
    w = wl.fold_workload("modes2", 3, T, H, seed=52 + T)
    kernel = lb.LB_KERNEL_STREAM if T > torch.cuda.get_device_properties(0) \
        .multi_processor_count else lb.LB_KERNEL_ROW
    assert plan(lb, T, H, 4).kernel == kernel
    full = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_fp8=True)
    init = oracle.fold_norm(w.partials, None, w.gamma, w.eps, want_fp8=True)
    check_fold(gpu_fold(lb, w.partials, None, w.gamma, w.eps), init, "enter")
    check_fold(gpu_fold(lb, w.partials, None, w.gamma, w.eps, fp8=True), init, "enter fp8")
    got = gpu_fold(lb, w.partials, None, w.gamma, w.eps, want_y=False)
    assert_bits_equal(got["residual_out"], init["residual_out"], "complete_output")
    got = gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, want_y=False)
    assert_bits_equal(got["residual_out"], full["residual_out"], "fold")
    rd = oracle.fold_norm([], full["residual_out"], w.gamma, w.eps, want_residual=False,
                          want_fp8=True)
    check_fold(gpu_fold(lb, [], full["residual_out"], w.gamma, w.eps, want_res=False), rd,
               "read")
    check_fold(gpu_fold(lb, [], full["residual_out"], w.gamma, w.eps, want_res=False,
                        fp8=True), rd, "read fp8")
    check_fold(gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, in_place=True), full,
               "in place")
    check_fold(gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, in_place=True, fp8=True,
                        want_y_fp8=True), full, "in place fp8")


@pytest.mark.parametrize("T", [64, 1024])             # row kernel, stream kernel
@pytest.mark.parametrize("fp8", [False, True])
def test_moe_routing_ready(lb, T, fp8):
    """With the routing promise the MoE call reads its first tokens' routing early and
    computes exactly what it computes without it."""
    w = wl.moe_workload("ready", T, 4096, 64, 8, seed=44 + T)
    want = oracle.moe_finalize_fold_norm(w.expert_out, w.idx, w.w, w.residual, w.gamma,
                                         w.eps, want_fp8=fp8)
    got = _gpu_moe(lb, w, fp8=fp8, routing_ready=True)
    check_fold(got, want, f"moe routing ready T={T}")
    plain = _gpu_moe(lb, w, fp8=fp8)
    for k in got:
        assert_bits_equal(got[k], plain[k], f"routing ready vs default: {k}")


@pytest.mark.parametrize("T,H", [(64, 4096), (300, 4096), (300, 12288)])  # row, stream, chunked
@pytest.mark.parametrize("fp8", [False, True])
def test_residual_ready(lb, T, H, fp8):
    """With the residual promise the call loads residual and gamma early and computes
    exactly what it computes without it (Gemma weight included)."""
    w = wl.fold_workload("res_ready", 4, T, H, seed=45 + T + H)
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_fp8=True,
                            gemma=True)
    got = _options_fold(lb, w, fp8=fp8, gemma=True, snapshot=False, residual_ready=True)
    check_fold(got, want, f"residual ready T={T} H={H}")
    plain = _options_fold(lb, w, fp8=fp8, gemma=True, snapshot=False)
    for k in got:
        assert_bits_equal(got[k], plain[k], f"residual ready vs default: {k}")


def test_promises_on_slices_and_moe(lb):
    """The residual (and, for MoE, routing) promise on the slice and MoE calls of the
    stream kernel, whose first rows' residual copies then go out early: results equal
    the oracle and the default call bit for bit."""
    w = wl.ragged_slice(seed=13, slice_=3)
    P = [dev_bits(p) for p in w.partials]
    R = dev_bits(w.residual)
    G = torch.from_numpy(w.gamma).cuda()
    outs = []
    for ready in (False, True):
        ro, yo = Guarded(w.T, w.H, torch.bfloat16), Guarded(w.T, w.H, torch.bfloat16)
        lb.lb_slice_fold_norm(P, w.T_pad, w.num_slices, w.slice, w.set_offsets, w.set_counts,
                              R, ro.t, G, yo.t, None, None, w.H, w.eps, residual_ready=ready)
        torch.cuda.synchronize()
        ro.check(), yo.check()
        outs.append((ro.host(), yo.host()))
    assert plan(lb, w.T, w.H, w.K + 1).kernel == lb.LB_KERNEL_STREAM
    want = oracle.slice_fold_norm(w.partials, w.T_pad, w.num_slices, w.slice, w.set_offsets,
                                  w.set_counts, w.residual, w.gamma, w.eps)
    assert_bits_equal(outs[1][0], want["residual_out"], "slice, promised: residual'")
    assert_bf16_close(outs[1][1], want["y"], "slice, promised: y")
    assert_bits_equal(outs[1][0], outs[0][0], "slice: promised vs default residual'")
    assert_bits_equal(outs[1][1], outs[0][1], "slice: promised vs default y")
    m = wl.moe_workload("promise_moe", 600, 4096, 64, 8, seed=46)
    want = oracle.moe_finalize_fold_norm(m.expert_out, m.idx, m.w, m.residual, m.gamma, m.eps,
                                         want_fp8=True)
    for fp8 in (False, True):
        got = _gpu_moe(lb, m, fp8=fp8, routing_ready=True, residual_ready=True)
        check_fold(got, want, f"moe, both promises, fp8={fp8}")
        plain = _gpu_moe(lb, m, fp8=fp8)
        for k in got:
            assert_bits_equal(got[k], plain[k], f"moe promised vs default: {k}")


def test_moe_bad_index_on_the_stream_kernel(lb):
    w = wl.moe_workload("bad2", 400, 2048, 16, 4, seed=43)
    assert plan(lb, 400, 2048, 5).kernel == lb.LB_KERNEL_STREAM
    idx = w.idx.copy()
    idx[7, 1] = 1 << 30
    idx[300, 3] = -1
    idx[301, :] = -2                                   # a row with no valid expert
    want = oracle.moe_finalize_fold_norm(w.expert_out, idx, w.w, w.residual, w.gamma, w.eps)
    got = _gpu_moe(lb, w, idx=idx, flag=True)
    assert got["flag"] == 1
    check_fold(got, want, "moe bad index, stream kernel")


@pytest.mark.parametrize("promises", [False, True])
def test_dependent_chain_of_boundaries(lb, promises):
    """Layers back to back on one stream with no host synchronisation: each boundary
    reads the residual the previous one wrote, and a torch kernel writes the next
    partials just before each call (the kernels are programmatic dependents of the
    previous launch, so this checks that every read waits for its producer).  With
    promises the MoE layers' routing is written before their expert rows and every call
    is told that its routing, residual and gamma were complete before the kernel just
    before it began (true here: torch writes the partials after the residual's
    producer has finished): the partials and expert rows, written by that kernel, must
    still be read after it."""
    routing_ready = promises
    rows = (2048, 64, 700, 1024, 2048, 64)       # stream, row, stream, MoE, stream, MoE(row)
    H = 2048
    rng = np.random.default_rng(81)
    gamma = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    res_host = wl.to_bf16_bits(rng.standard_normal((max(rows), H)).astype(np.float32))
    G = torch.from_numpy(gamma).cuda()
    R = dev_bits(res_host)
    want_res = res_host.copy()
    ys = []
    for li, T in enumerate(rows):
        moe = li in (3, 5)                         # MoE finalize layers
        if moe and routing_ready:                  # the router ran before the experts
            idx = torch.arange(T * 3, dtype=torch.int32, device="cuda").view(T, 3)
            wts = torch.full((T, 3), 1.0, dtype=torch.float32, device="cuda")
        seeds = [1000 * li + k for k in range(3)]
        P_host = [wl.to_bf16_bits(np.random.default_rng(sd).standard_normal((T, H))
                                  .astype(np.float32)) for sd in seeds]
        P = [torch.empty((T, H), dtype=torch.bfloat16, device="cuda") for _ in seeds]
        for d, h in zip(P, P_host):               # written by torch right before the call
            d.view(torch.int16).copy_(torch.from_numpy(h.view(np.int16)).cuda() * 1)
        Rn = torch.empty_like(R)
        Y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        if moe:
            if not routing_ready:
                idx = torch.arange(T * 3, dtype=torch.int32, device="cuda").view(T, 3)
            E = torch.cat(P, dim=1).view(T * 3, H)
            if not routing_ready:
                wts = torch.full((T, 3), 1.0, dtype=torch.float32, device="cuda")
            lb.lb_moe_finalize_fold_norm(E, T * 3, idx, wts, 3, R[:T], Rn[:T], G, Y, None,
                                         None, T, H, 1e-6, routing_ready=promises,
                                         residual_ready=promises)
            Eh = np.stack(P_host, axis=1).reshape(T * 3, H)
            o = oracle.moe_finalize_fold_norm(Eh, np.arange(T * 3, dtype=np.int32)
                                              .reshape(T, 3), np.ones((T, 3), np.float32),
                                              want_res[:T], gamma, 1e-6)
        else:
            lb.lb_fold_norm(P, R[:T], Rn[:T], G, Y, T, H, 1e-6, residual_ready=promises)
            o = oracle.fold_norm(P_host, want_res[:T], gamma, 1e-6)
        Rn[T:] = R[T:]
        R = Rn
        want_res[:T] = o["residual_out"]
        ys.append((Y, o["y"]))
    torch.cuda.synchronize()
    assert_bits_equal(host_bits(R), want_res, "chained residual'")
    for li, (Y, want_y) in enumerate(ys):
        assert_bf16_close(host_bits(Y), want_y, f"chained layer {li} y")


def test_specified_workloads_take_the_intended_kernels(lb):
    assert plan(lb, 2048, 4096, 5).kernel == lb.LB_KERNEL_STREAM     # prefill
    assert plan(lb, 1024, 4096, 9).kernel == lb.LB_KERNEL_STREAM     # MoE finalize
    assert plan(lb, 254, 4096, 9).kernel == lb.LB_KERNEL_STREAM      # ragged slice
    p = plan(lb, 64, 4096, 9)                                        # decode
    assert p.kernel == lb.LB_KERNEL_ROW and p.grid == 64
    assert plan(lb, 4, 32768, 2).ctas_per_row == 2                   # long rows: cluster
    p = plan(lb, 2048, 12288, 5)                                     # wide prefill
    assert p.kernel == lb.LB_KERNEL_STREAM and p.chunks == 3


# --------------------------------------------------------------------------------------
# Launch shapes and edge cases
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("K,T,H", [
    (1, 1, 8),          # a single vector per row
    (3, 5, 520),        # 65 vectors: partly active warp
    (16, 3, 4096),      # maximum K, two load chunks
    (2, 33, 8192),      # two vectors per thread, row kernel
    (2, 400, 8192),     # two vectors per thread, no cluster
    (2, 9, 16384),      # four vectors per thread
    (1, 4, 32768),      # four vectors per thread, a row split over a 2-CTA cluster
    (5, 301, 4096),     # K above one load chunk, ragged last wave
    (4, 2048, 1024),    # row kernel past the SM count (rows of <= 1024 elements)
    (8, 152, 2048),     # row kernel: one row per SM
    (8, 153, 2048),     # stream kernel, one vector per thread, a copy per producer lane
    (2, 160, 4096),     # stream kernel, one or two rows per CTA
    (4, 1000, 4096),    # stream kernel
    (16, 300, 1024),    # row kernel at the maximum K, past the SM count
    (16, 300, 2048),    # stream kernel at the maximum K (17 staged rows per stage)
    (1, 2, 131072),     # the largest hidden size: a row split over an 8-CTA cluster
    (3, 151, 4096),     # one row short of the SM count: row kernel
    (3, 153, 8),        # row kernel, one vector per row
    (16, 160, 24),      # row kernel, maximum K, three vectors per row
    (3, 153, 1032),     # stream kernel, 129 vectors: a partly active warp, a ragged wave
    (2, 200, 12288),    # stream kernel, rows in 3 column chunks
    (2, 30000, 256),    # row kernel, 30000 one-warp CTAs
    (2, 30000, 1032),   # stream kernel, ~200 rows per CTA: every stage wraps many times
    (4, 300, 5120),     # stream kernel, two groups of 10 warps
    (4, 300, 6144),     # stream kernel, two groups of 12 warps
    (3, 200, 7168),     # stream kernel, one group of 14 warps
    (4, 300, 12288),    # stream kernel, 3 chunks of 16 warps
    (2, 160, 16384),    # stream kernel, 4 chunks of 16 warps
    (3, 160, 10240),    # stream kernel, 3 chunks of 14 warps, the last one short
    (8, 200, 8192),     # row kernel: whole rows of 9 inputs do not double-buffer
    (16, 153, 8200),    # stream kernel, maximum K, 4 chunks of 10 warps, 65 vectors in the last
    (8, 160, 12288),    # stream kernel, 3 chunks of 16 warps, 2 stages
    (2, 1500, 10240),   # stream kernel, chunked rows: ~10 rows per CTA, the ring wraps often
])
def test_shapes(lb, K, T, H):
    w = wl.fold_workload("shape", K, T, H, seed=K * 1000 + T + H)
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_fp8=True)
    check_fold(gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps), want, f"{K}x{T}x{H}")
    check_fold(gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, fp8=True,
                        want_y_fp8=True), want, f"fp8 {K}x{T}x{H}")


def test_empty_batch_writes_nothing(lb):
    H = 256
    P = [torch.zeros((1, H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ro, yo = Guarded(0, H, torch.bfloat16), Guarded(0, H, torch.bfloat16)
    G = torch.ones(H, device="cuda")
    lb.lb_fold_norm(P, P[0], ro.t, G, yo.t, 0, H, 1e-6)
    torch.cuda.synchronize()
    ro.check(), yo.check()


def test_zero_rows_fp8(lb):
    w = wl.fold_workload("z", 2, 8, 512, seed=61)
    for a in w.partials + [w.residual]:
        a[[1, 5]] = 0
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_fp8=True)
    assert want["scale"][1] == 0 and want["scale"][5] == 0
    got = gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, fp8=True)
    check_fold(got, want, "zero rows")
    assert np.all(got["q"][[1, 5]] == 0) and np.all(got["scale"][[1, 5]] == 0)


def test_repeat_calls_are_bit_identical(lb):
    w = wl.fold_workload("rep", 4, 100, 4096, seed=71, fp8=True)
    a = gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, fp8=True, want_y_fp8=True)
    b = gpu_fold(lb, w.partials, w.residual, w.gamma, w.eps, fp8=True, want_y_fp8=True)
    for k in a:
        assert np.array_equal(a[k], b[k])


def test_runs_on_a_side_stream(lb):
    w = wl.fold_workload("stream", 2, 64, 2048, seed=72)
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps)
    P = [dev_bits(p) for p in w.partials]
    R = dev_bits(w.residual)
    G = torch.from_numpy(w.gamma).cuda()
    s = torch.cuda.Stream()
    ro = torch.empty_like(R)
    yo = torch.empty_like(R)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lb.lb_fold_norm(P, R, ro, G, yo, 64, 2048, w.eps)
    s.synchronize()
    assert_bits_equal(host_bits(ro), want["residual_out"], "side stream residual'")
    assert_bf16_close(host_bits(yo), want["y"], "side stream y")


# --------------------------------------------------------------------------------------
# Gemma weight (1 + gamma), residual snapshot, variable-size reduce-scatter (rsv)
# --------------------------------------------------------------------------------------

def _options_fold(lb, w, *, fp8, gemma, snapshot, residual_ready=False):
    T, H = w.T, w.H
    P = [dev_bits(p) for p in w.partials]
    R = dev_bits(w.residual)
    G = torch.from_numpy(w.gamma).cuda()
    ro, yo = Guarded(T, H, torch.bfloat16), Guarded(T, H, torch.bfloat16)
    sn = Guarded(T, H, torch.bfloat16) if snapshot else None
    qo = Guarded(T, H, torch.uint8) if fp8 else None
    so = Guarded(T, 0, torch.float32) if fp8 else None
    kw = dict(gemma=gemma, residual_snapshot=sn.t if sn else None,
              residual_ready=residual_ready)
    if fp8:
        lb.lb_fold_norm_fp8(P, R, ro.t, G, qo.t, so.t, yo.t, T, H, w.eps, **kw)
    else:
        lb.lb_fold_norm(P, R, ro.t, G, yo.t, T, H, w.eps, **kw)
    torch.cuda.synchronize()
    out = {"residual_out": ro, "y": yo}
    if snapshot:
        out["snapshot"] = sn
    if fp8:
        out.update(q=qo, scale=so)
    for g in out.values():
        g.check()
    return {k: g.host() for k, g in out.items()}


@pytest.mark.parametrize("T,H", [(50, 2048), (700, 2048), (200, 12288)])   # chunked rows last
@pytest.mark.parametrize("fp8", [False, True])
def test_gemma_weight_and_snapshot(lb, T, H, fp8):
    w = wl.fold_workload("gem", 3, T, H, seed=93 + T)
    w.gamma = (0.05 * np.random.default_rng(T).standard_normal(w.H)).astype(np.float32)
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_fp8=True, gemma=True)
    got = _options_fold(lb, w, fp8=fp8, gemma=True, snapshot=True)
    check_fold(got, want, f"gemma T={T}")
    assert_bits_equal(got["snapshot"], want["residual_out"], "snapshot")
    plain = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps)
    assert not np.array_equal(plain["y"], want["y"])


def test_moe_terminal_handoff_with_gemma_norm(lb):
    """The terminal layer's deferred MoE finalize fused with the final (Gemma) norm."""
    w = wl.moe_workload("term", 300, 2048, 32, 8, seed=94)
    w.gamma = (0.05 * np.random.default_rng(9).standard_normal(w.H)).astype(np.float32)
    want = oracle.moe_finalize_fold_norm(w.expert_out, w.idx, w.w, w.residual, w.gamma, w.eps,
                                         gemma=True)
    E, I = dev_bits(w.expert_out), torch.from_numpy(w.idx).cuda()
    Wt, R = torch.from_numpy(w.w).cuda(), dev_bits(w.residual)
    G = torch.from_numpy(w.gamma).cuda()
    ro, yo, sn = (Guarded(w.T, w.H, torch.bfloat16) for _ in range(3))
    lb.lb_moe_finalize_fold_norm(E, w.expert_out.shape[0], I, Wt, w.topk, R, ro.t, G, yo.t,
                                 None, None, w.T, w.H, w.eps, gemma=True,
                                 residual_snapshot=sn.t)
    torch.cuda.synchronize()
    for g in (ro, yo, sn):
        g.check()
    got = {"residual_out": ro.host(), "y": yo.host()}
    check_fold(got, want, "moe + gemma norm")
    assert_bits_equal(sn.host(), want["residual_out"], "moe snapshot")


@pytest.mark.parametrize("fp8", [False, True])
def test_rsv_every_rank(lb, fp8):
    w = wl.ragged_slice()
    P = [dev_bits(p) for p in w.partials]
    G = torch.from_numpy(w.gamma).cuda()
    for s, (o, c) in enumerate(zip(w.set_offsets.tolist(), w.set_counts.tolist())):
        res = w.residual_full[o:o + c]
        want = oracle.set_slice_fold_norm(w.partials, w.T_pad, s, w.set_offsets,
                                          w.set_counts, res, w.gamma, w.eps, want_fp8=fp8,
                                          gemma=(s % 2 == 1))
        R = dev_bits(res)
        ro, yo = Guarded(c, w.H, torch.bfloat16), Guarded(c, w.H, torch.bfloat16)
        qo = Guarded(c, w.H, torch.uint8) if fp8 else None
        so = Guarded(c, 0, torch.float32) if fp8 else None
        before = _snapshot(P + [R, G])
        lb.lb_slice_fold_norm_v(P, w.T_pad, s, w.set_offsets, w.set_counts, R, ro.t, G, yo.t,
                                qo.t if fp8 else None, so.t if fp8 else None, w.H, w.eps,
                                gemma=(s % 2 == 1))
        torch.cuda.synchronize()
        _assert_unchanged(before, P + [R, G])
        outs = {"residual_out": ro, "y": yo}
        if fp8:
            outs.update(q=qo, scale=so)
        for g in outs.values():
            g.check()
        check_fold({k: g.host() for k, g in outs.items()}, want, f"rsv rank {s}")


def test_slice_with_gemma_and_snapshot(lb):
    w = wl.ragged_slice(slice_=2)
    S = w.T
    want = oracle.slice_fold_norm(w.partials, w.T_pad, 8, 2, w.set_offsets, w.set_counts,
                                  w.residual_full[2 * S:3 * S], w.gamma, w.eps, gemma=True,
                                  out={"residual_out": np.full((S, w.H), SENTINEL16, np.uint16),
                                       "y": np.full((S, w.H), SENTINEL16, np.uint16)})
    P = [dev_bits(p) for p in w.partials]
    R = dev_bits(w.residual_full[2 * S:3 * S])
    G = torch.from_numpy(w.gamma).cuda()
    ro, yo, sn = (Guarded(S, w.H, torch.bfloat16) for _ in range(3))
    lb.lb_slice_fold_norm(P, w.T_pad, 8, 2, w.set_offsets, w.set_counts, R, ro.t, G, yo.t,
                          None, None, w.H, w.eps, gemma=True, residual_snapshot=sn.t)
    torch.cuda.synchronize()
    for g in (ro, yo, sn):
        g.check()
    assert_bits_equal(ro.host(), want["residual_out"], "slice residual' (incl. padding)")
    assert_bits_equal(sn.host(), want["residual_out"], "slice snapshot (incl. padding)")
    valid = ~np.all(want["y"] == SENTINEL16, axis=1)
    assert_bf16_close(yo.host(), want["y"], "slice gemma y", rows=valid)


def test_host_pipeline_matches_the_oracle(lb):
    """Pinned host buffers in, pinned host buffers out, chunks overlapped across three
    streams and two device buffer sets; three calls in a row."""
    from layer_boundary_fusion_gb300.host import HostPipeline
    w = wl.fold_workload("host", 3, 512, 2048, seed=95, fp8=True)
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_y=False,
                            want_fp8=True)
    pipe = HostPipeline(w.K, w.T, w.H, "cuda:0", chunks=4)
    hP = [torch.from_numpy(p.view(np.int16)).pin_memory() for p in w.partials]
    hR = torch.from_numpy(w.residual.view(np.int16)).pin_memory()
    hG = torch.from_numpy(w.gamma).pin_memory()
    ro = torch.empty((w.T, w.H), dtype=torch.int16).pin_memory()
    q = torch.empty((w.T, w.H), dtype=torch.uint8).pin_memory()
    sc = torch.empty((w.T,), dtype=torch.float32).pin_memory()
    for call in range(3):                  # the first call captures, the others replay
        ro.fill_(-1), q.fill_(0x7F), sc.fill_(float("nan"))
        pipe(hP, hR, hG, ro, q, sc, w.eps)
        torch.cuda.synchronize()
        assert_bits_equal(ro.numpy().view(np.uint16), want["residual_out"], f"host residual' {call}")
        assert_fp8_close(q.numpy(), want["q"], sc.numpy(), want["scale"], f"host fp8 {call}")


def test_host_pipeline_overlapped_steps_keep_their_own_data(lb):
    """Five steps with different inputs and outputs run as one pipelined schedule on
    two device buffer sets (step i+1 copies in while step i copies out): every step's
    outputs match the oracle on that step's inputs, so no step reads or overwrites
    another's buffers."""
    from layer_boundary_fusion_gb300.host import HostPipeline
    K, T, H = 2, 300, 1024
    ws = [wl.fold_workload("host_steps", K, T, H, seed=200 + i, fp8=True) for i in range(5)]
    gamma = torch.from_numpy(ws[0].gamma).pin_memory()
    inputs, outputs, wants = [], [], []
    for w in ws:
        inputs.append(([torch.from_numpy(p.view(np.int16)).pin_memory() for p in w.partials],
                       torch.from_numpy(w.residual.view(np.int16)).pin_memory()))
        outputs.append((torch.full((T, H), -1, dtype=torch.int16).pin_memory(),
                        torch.full((T, H), 0x7F, dtype=torch.uint8).pin_memory(),
                        torch.full((T,), float("nan"), dtype=torch.float32).pin_memory()))
        wants.append(oracle.fold_norm(w.partials, w.residual, ws[0].gamma, w.eps,
                                      want_y=False, want_fp8=True))
    for chunks in (1, 3):
        pipe = HostPipeline(K, T, H, "cuda:0", chunks=chunks, depth=2)
        for rep in range(2):                    # capture, then replay
            pipe.run_steps(inputs, gamma, outputs, ws[0].eps)
            torch.cuda.synchronize()
            for i, ((ro, q, sc), want) in enumerate(zip(outputs, wants)):
                what = f"chunks {chunks} rep {rep} step {i}"
                assert_bits_equal(ro.numpy().view(np.uint16), want["residual_out"], what)
                assert_fp8_close(q.numpy(), want["q"], sc.numpy(), want["scale"], what)
                ro.fill_(-1), q.fill_(0x7F), sc.fill_(float("nan"))


def test_non_finite_inputs_propagate_like_the_oracle(lb):
    """A NaN or an infinity in a partial makes its row's outputs non-finite where the
    definition says so; other rows are unaffected.  Compared as float values
    (NaN == NaN), since NaN payloads need not match."""
    w = wl.fold_workload("nan", 2, 200, 2048, seed=96)
    P = [p.copy() for p in w.partials]
    P[0][3, 10] = 0x7FC0                      # NaN
    P[1][7, 20] = 0x7F80                      # +inf
    P[1][9, 30] = 0xFF80                      # -inf
    P[0][9, 30] = 0x7F80                      # +inf + -inf = NaN
    want = oracle.fold_norm(P, w.residual, w.gamma, w.eps)
    for T in (200, 100):                      # stream kernel, row kernel
        got = gpu_fold(lb, [p[:T] for p in P], w.residual[:T], w.gamma, w.eps)
        for k in ("residual_out", "y"):
            g = f32(got[k]).astype(np.float64)
            e = f32(want[k][:T]).astype(np.float64)
            assert np.array_equal(np.isnan(g), np.isnan(e)), k
            fin = np.isfinite(e)
            assert np.array_equal(np.isinf(g), np.isinf(e)), k
            assert np.all(g[np.isinf(e)] == e[np.isinf(e)])
            assert np.all(np.abs(g[fin] - e[fin]) <= 1e-2 * np.abs(e[fin]) + 1e-3), k


def test_unfused_two_call_path_matches_the_oracle(lb):
    """The unfused fallback the benchmark compares against (the completed sum written
    to a bf16 buffer, then residual add + RMSNorm of that buffer) computes what the
    oracle computes for the same two calls."""
    w = wl.fold_workload("unfused", 4, 300, 4096, seed=97)
    s_want = oracle.fold_norm(w.partials, None, None, w.eps, want_y=False)["residual_out"]
    want = oracle.fold_norm([s_want], w.residual, w.gamma, w.eps)
    s_got = gpu_fold(lb, w.partials, None, w.gamma, w.eps, want_y=False)["residual_out"]
    assert_bits_equal(s_got, s_want, "unfused sum")
    check_fold(gpu_fold(lb, [s_got], w.residual, w.gamma, w.eps), want, "unfused add+norm")


@pytest.mark.parametrize("T", [40, 300])           # row kernel, stream kernel
def test_residual_stream_through_a_layer_stack(lb, T):
    """A layer stack driven through the residual stream (lb_residual.h): enter, a
    completed and extended contribution with an FP8 read, fold then a plain read, and a
    MoE handoff consumed by a Gemma final norm.  Each read and the residual after each
    step match the oracle evaluating the same sequence of boundary operations."""
    H, eps = 2048, 1e-6
    fw = wl.fold_workload("stack", 4, T, H, seed=98)
    mw = wl.moe_workload("stack_moe", T, H, 16, 4, seed=99)
    E0, P0, P1, X = fw.partials
    P2 = fw.residual
    gamma = fw.gamma
    R = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    buf = torch.empty_like(R)
    y1, y3, y4 = (torch.empty_like(R) for _ in range(3))
    q = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    sc = torch.empty((T,), dtype=torch.float32, device="cuda")
    G = torch.from_numpy(gamma).cuda()
    d = {k: dev_bits(v) for k, v in (("E0", E0), ("P0", P0), ("P1", P1), ("X", X), ("P2", P2),
                                     ("EX", mw.expert_out))}
    I = torch.from_numpy(mw.idx).cuda()
    Wt = torch.from_numpy(mw.w).cuda()
    s = lb.ResidualStream()
    lb.lb_residual_init(s, R, T, H)
    h = lb.lb_residual_start(s)
    # enter: the embedding's contribution becomes the residual, then the first read
    h = lb.lb_residual_leave(s, h, [d["E0"]])
    h = lb.lb_residual_prepare(s, h, G, y1, None, None, eps)
    torch.cuda.synchronize()
    r1 = host_bits(R)
    want1 = oracle.fold_norm([E0], None, gamma, eps)
    check_fold({"residual_out": r1, "y": host_bits(y1)}, want1, "enter")
    # an owed sum completed into a buffer, an extra contribution, then the FP8 read
    h = lb.lb_residual_leave(s, h, [d["P0"], d["P1"]])
    h = lb.lb_residual_complete_output(s, h, buf)
    h = lb.lb_residual_add_to_output(s, h, d["X"])
    h = lb.lb_residual_prepare(s, h, G, None, q, sc, eps)
    torch.cuda.synchronize()
    s_want = oracle.fold_norm([P0, P1], None, None, eps, want_y=False)["residual_out"]
    assert_bits_equal(host_bits(buf), s_want, "complete_output")
    want2 = oracle.fold_norm([s_want, X], r1, gamma, eps, want_y=False, want_fp8=True)
    r2 = host_bits(R)
    check_fold({"residual_out": r2, "q": q.cpu().numpy(), "scale": sc.cpu().numpy()}, want2,
               "add_to_output + fp8 read")
    # fold, then a read of the written stream
    h = lb.lb_residual_leave(s, h, [d["P2"]])
    h = lb.lb_residual_fold(s, h)
    h = lb.lb_residual_prepare(s, h, G, y3, None, None, eps)
    torch.cuda.synchronize()
    r3_want = oracle.fold_norm([P2], r2, None, eps, want_y=False)["residual_out"]
    r3 = host_bits(R)
    assert_bits_equal(r3, r3_want, "fold")
    check_fold({"y": host_bits(y3)}, oracle.fold_norm([], r3_want, gamma, eps), "read")
    # a MoE finalize handoff consumed by a Gemma final norm, which releases the stream
    h = lb.lb_residual_leave_moe(s, h, d["EX"], mw.expert_out.shape[0], I, Wt, mw.topk)
    lb.lb_residual_norm(s, h, G, y4, None, None, eps, gemma=True)
    torch.cuda.synchronize()
    want4 = oracle.moe_finalize_fold_norm(mw.expert_out, mw.idx, mw.w, r3_want, gamma, eps,
                                          gemma=True)
    check_fold({"residual_out": host_bits(R), "y": host_bits(y4)}, want4, "final norm")
    assert s.started == 0
    with pytest.raises(lb.LBError) as e:
        lb.lb_residual_take_output(s, h + 1)
    assert e.value.status == lb.LB_ERR_NOT_STARTED


def test_concurrent_host_threads_and_streams(lb):
    """Two host threads each enqueue a chain of boundaries on their own stream at the
    same time (the library keeps no per-call state: only a cached device description and
    the device error word).  Each thread's results match the oracle."""
    import threading
    cases = []
    for i, (K, T, H) in enumerate([(4, 300, 2048), (8, 64, 4096)]):
        w = wl.fold_workload("threads", K, T, H, seed=400 + i)
        cases.append((w, oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps)))
    results, errors = [None, None], []

    def worker(i):
        try:
            w, _ = cases[i]
            st = torch.cuda.Stream()
            P = [dev_bits(p) for p in w.partials]
            R = dev_bits(w.residual)
            G = torch.from_numpy(w.gamma).cuda()
            outs = [(torch.empty_like(R), torch.empty_like(R)) for _ in range(20)]
            torch.cuda.synchronize()
            with torch.cuda.stream(st):
                for ro, yo in outs:
                    lb.lb_fold_norm(P, R, ro, G, yo, w.T, w.H, w.eps, stream=st)
            st.synchronize()
            results[i] = [(host_bits(ro), host_bits(yo)) for ro, yo in outs]
        except Exception as e:       # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (w, want), res in zip(cases, results):
        for ro, yo in res:
            check_fold({"residual_out": ro, "y": yo}, want, f"thread K={w.K}")


def test_fp8_read_of_near_zero_rows(lb):
    """Rows whose read is tiny (bf16 subnormal inputs: the per-token scale is a binary32
    subnormal, its reciprocal overflows) and rows of ordinary size side by side, on both
    kernels: codes and scales match the oracle, which divides by the scale."""
    for T in (100, 300):                       # row kernel, stream kernel
        w = wl.fold_workload("tiny_rows", 2, T, 2048, seed=97)
        P = [p.copy() for p in w.partials]
        R = w.residual.copy()
        rng = np.random.default_rng(5)
        for t in range(0, T, 3):               # every third row: subnormal bf16 values
            top = 128 if t % 2 else 3           # and every sixth the smallest of them
            for arr in P + [R]:
                mant = rng.integers(1, top, arr.shape[1]).astype(np.uint16)
                sign = (rng.integers(0, 2, arr.shape[1]).astype(np.uint16) << 15)
                arr[t] = sign | mant            # exponent 0: subnormal
        want = oracle.fold_norm(P, R, w.gamma, w.eps, want_y=False, want_fp8=True)
        got = gpu_fold(lb, P, R, w.gamma, w.eps, want_y=False, fp8=True)
        check_fold(got, want, f"near-zero rows T={T}")


@pytest.mark.parametrize("mode", ["global", "thread_local", "relaxed"])
def test_calls_captured_into_a_graph(lb, mode):
    """Every call kind captured into a CUDA graph on a side stream (a capturing stream
    cannot be asked for its device) and replayed twice: the replays write what the
    oracle computes, on the row kernel (T=64), the stream kernel (T=300) and the MoE
    finalize."""
    wr = wl.fold_workload("cap_row", 3, 64, 2048, seed=31)
    ws = wl.fold_workload("cap_stream", 2, 300, 2048, seed=32, fp8=True)
    wm = wl.moe_workload("cap_moe", 200, 2048, 16, 2, seed=33)
    want_r = oracle.fold_norm(wr.partials, wr.residual, wr.gamma, wr.eps)
    want_s = oracle.fold_norm(ws.partials, ws.residual, ws.gamma, ws.eps, want_y=False,
                              want_fp8=True)
    want_m = oracle.moe_finalize_fold_norm(wm.expert_out, wm.idx, wm.w, wm.residual, wm.gamma,
                                            wm.eps)
    Pr = [dev_bits(p) for p in wr.partials]
    Rr = dev_bits(wr.residual)
    Gr = torch.from_numpy(wr.gamma).cuda()
    ror, yor = torch.empty_like(Rr), torch.empty_like(Rr)
    Ps = [dev_bits(p) for p in ws.partials]
    Rs = dev_bits(ws.residual)
    Gs = torch.from_numpy(ws.gamma).cuda()
    ros = torch.empty_like(Rs)
    qs = torch.empty((ws.T, ws.H), dtype=torch.uint8, device="cuda")
    ss = torch.empty((ws.T,), dtype=torch.float32, device="cuda")
    E = dev_bits(wm.expert_out)
    idx = torch.from_numpy(wm.idx).cuda()
    wt = torch.from_numpy(wm.w).cuda()
    Rm = dev_bits(wm.residual)
    Gm = torch.from_numpy(wm.gamma).cuda()
    rom, yom = torch.empty_like(Rm), torch.empty_like(Rm)
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap, capture_error_mode=mode):
        lb.lb_fold_norm(Pr, Rr, ror, Gr, yor, wr.T, wr.H, wr.eps)
        lb.lb_fold_norm_fp8(Ps, Rs, ros, Gs, qs, ss, None, ws.T, ws.H, ws.eps)
        lb.lb_moe_finalize_fold_norm(E, wm.expert_out.shape[0], idx, wt, wm.topk, Rm, rom, Gm, yom,
                                     None, None, wm.T, wm.H, wm.eps)
    for _ in range(2):
        for t in (ror, yor, ros, rom, yom):
            t.view(torch.int16).fill_(SENTINEL16)
        qs.fill_(0x7F)
        ss.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_bits_equal(host_bits(ror), want_r["residual_out"], "captured row residual'")
        assert_bf16_close(host_bits(yor), want_r["y"], "captured row y")
        assert_bits_equal(host_bits(ros), want_s["residual_out"], "captured stream residual'")
        assert_fp8_close(qs.cpu().numpy(), want_s["q"], ss.cpu().numpy(), want_s["scale"],
                         "captured stream fp8")
        assert_bf16_close(host_bits(rom), want_m["residual_out"], "captured moe residual'")
        assert_bf16_close(host_bits(yom), want_m["y"], "captured moe y")
