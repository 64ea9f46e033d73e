"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something it cannot reproduce by retyping its own
formula: hand-worked rows (tests/golden), the FP8/bf16 format definitions checked
exhaustively, library routines (torch's bf16 and float8_e4m3fn casts, torch's float64
RMSNorm), exact sums in binary64, and invariants of the boundary operation (the RMS of
the read, linearity and exactness of the fold, relocation of expert rows, slice
placement).  A dropped term, a wrong sign or index, eps outside the root, a sum in
place of the mean, amax over rounded values or a misplaced slice row fails one of them.
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from layer_boundary_fusion_gb300 import workloads as wl


def bits(values):
    return wl.to_bf16_bits(np.asarray(values, np.float32))


def f32_of_bits(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def close_bf16(got_bits, want, rel=2.0 ** -8, abs_=0.0):
    got = f32_of_bits(got_bits).astype(np.float64)
    want = np.asarray(want, np.float64)
    return np.abs(got - want) <= rel * np.abs(want) + abs_


# --------------------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------------------

def test_bf16_widen_then_round_is_identity(ora):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = ora.bf16_to_f32(allbits)
    assert np.array_equal(f.view(np.uint32) >> 16, allbits.astype(np.uint32))
    assert np.array_equal(f.view(np.uint32) & 0xFFFF, np.zeros(65536, np.uint32))
    back = ora.f32_to_bf16(f)
    finite = ~np.isnan(f)
    assert np.array_equal(back[finite], allbits[finite])
    assert np.all(np.isnan(ora.bf16_to_f32(back[~finite])))


def test_bf16_rounding_matches_torch_including_ties(ora):
    rng = np.random.default_rng(7)
    hi = rng.integers(0, 1 << 16, 200000, dtype=np.uint32)
    lo = rng.integers(0, 1 << 16, 200000, dtype=np.uint32)
    lo[:50000] = 0x8000                                        # exact ties
    lo[50000:60000] = 0x7FFF
    lo[60000:70000] = 0x8001
    u = (hi << 16) | lo
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = ora.f32_to_bf16(x)
    assert np.array_equal(got, want)


def test_e4m3_decode_matches_torch_for_all_codes(ora):
    codes = np.arange(256, dtype=np.uint8)
    got = ora.e4m3_to_f32(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    nan = np.isnan(want)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_e4m3_every_finite_code_round_trips(ora):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(ora.f32_to_e4m3(ora.e4m3_to_f32(codes)), codes)


def test_e4m3_spot_values(ora):
    rows = read_golden("e4m3_spots.txt")[None]
    x = np.array([float(r[0]) for r in rows], np.float32)
    want = np.array([int(r[1], 16) for r in rows], np.uint8)
    got = ora.f32_to_e4m3(x)
    assert [hex(v) for v in got] == [hex(v) for v in want]
    assert ora.f32_to_e4m3(np.array([np.nan], np.float32))[0] == 0x7F


def test_e4m3_encoder_matches_torch_in_range(ora):
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.uniform(-448, 448, 100000),
        rng.standard_normal(100000) * 2.0 ** rng.integers(-12, 8, 100000),
        # every midpoint between neighbouring codes (exact ties)
        (ora.e4m3_to_f32(np.arange(0, 0x7E, dtype=np.uint8)).astype(np.float64)
         + ora.e4m3_to_f32(np.arange(1, 0x7F, dtype=np.uint8))) / 2.0,
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    x = np.concatenate([x, -x])
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ora.f32_to_e4m3(x), want)


def test_e4m3_encoder_monotone_and_symmetric(ora):
    x = np.linspace(0.0, 520.0, 400001, dtype=np.float32)
    c = ora.f32_to_e4m3(x)
    assert np.all(np.diff(c.astype(np.int32)) >= 0)
    assert c[-1] == 0x7E
    assert np.array_equal(ora.f32_to_e4m3(-x[1:]), c[1:] | 0x80)


# --------------------------------------------------------------------------------------
# Fold + RMSNorm: hand-worked rows
# --------------------------------------------------------------------------------------

def _golden_row(name):
    g = read_golden(name)
    return {k: np.array([float(v) for v in vals], np.float32)
            for k, vals in g.items() if k is not None and vals}


def test_fold_norm_hand_row(ora):
    g = _golden_row("fold_norm_h4.txt")
    p = [bits(g["p0"])[None], bits(g["p1"])[None]]
    res = bits(g["res"])[None]
    for eps in (0.0, 1e-6):
        out = ora.fold_norm(p, res, g["gamma"], eps)
        assert np.array_equal(f32_of_bits(out["residual_out"][0]), g["residual_out"])
        assert np.array_equal(f32_of_bits(out["y"][0]), g["y"])
    # Initial state: residual' is the completed sum itself
    out = ora.fold_norm(p, None, g["gamma"], 0.0)
    assert np.array_equal(f32_of_bits(out["residual_out"][0]), g["initial_residual_out"])
    s = g["initial_residual_out"].astype(np.float64)
    want_y = s / math.sqrt(np.mean(s * s)) * g["gamma"]
    assert np.all(close_bf16(out["y"][0], want_y))


def test_complete_fold_read_modes_of_the_stream(ora):
    """complete_output leaves the sum pending; a later K=1 fold of it plus a read of
    the Written stream equals the fused fold+read (up to the bf16 rounding of the
    completed sum, which is exact for these inputs)."""
    g = _golden_row("fold_norm_h4.txt")
    p = [bits(g["p0"])[None], bits(g["p1"])[None]]
    res = bits(g["res"])[None]
    done = ora.fold_norm(p, None, g["gamma"], 0.0, want_y=False)      # complete_output
    assert set(done) == {"residual_out"}
    folded = ora.fold_norm([done["residual_out"]], res, g["gamma"], 0.0, want_y=False)
    read = ora.fold_norm([], folded["residual_out"], g["gamma"], 0.0, want_residual=False)
    fused = ora.fold_norm(p, res, g["gamma"], 0.0)
    assert np.array_equal(folded["residual_out"], fused["residual_out"])
    assert np.array_equal(read["y"], fused["y"])


def test_eps_inside_the_root_and_mean_of_squares(ora):
    g = _golden_row("eps_inside_root.txt")
    p = [bits(g["p0"])[None]]
    assert f32_of_bits(p[0][0]).tolist() == g["p0"].tolist()
    out = ora.fold_norm(p, None, g["gamma"], float(g["eps"][0]))
    assert np.array_equal(f32_of_bits(out["y"][0]), g["y"])
    out0 = ora.fold_norm(p, None, g["gamma"], 0.0)
    assert np.array_equal(f32_of_bits(out0["y"][0]), g["y_eps0"])


# --------------------------------------------------------------------------------------
# Fold + RMSNorm: closed forms and library cross-checks on seeded data
# --------------------------------------------------------------------------------------

def test_read_matches_torch_float64_rmsnorm(ora):
    """K = 1 and no residual: o is the partial itself, so y must be torch's float64
    RMSNorm of it (weight gamma), up to the final bf16 rounding."""
    w = wl.fold_workload("k1", 1, 37, 1000, seed=11, residual=False)
    out = ora.fold_norm(w.partials, None, w.gamma, w.eps)
    x = torch.from_numpy(f32_of_bits(w.partials[0]).astype(np.float64))
    ref = torch.nn.functional.rms_norm(x, (w.H,), weight=torch.from_numpy(
        w.gamma.astype(np.float64)), eps=w.eps).numpy()
    assert np.all(close_bf16(out["y"], ref, rel=2.0 ** -8 + 1e-6))
    # nearly every element is the bf16 rounding of the binary64 value itself
    assert np.mean(out["y"] == wl.to_bf16_bits(ref.astype(np.float32))) > 0.99


def test_fold_equals_exact_binary64_sum(ora):
    """residual' is the bf16 rounding of the exact sum of the inputs (the binary32 sum
    of a few bf16 values is exact unless their exponents are far apart)."""
    w = wl.fold_workload("exact", 8, 24, 512, seed=12, partial_std=0.5)
    out = ora.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_y=False)
    exact = sum(f32_of_bits(p).astype(np.float64) for p in w.partials)
    exact = exact + f32_of_bits(w.residual).astype(np.float64)
    want = torch.from_numpy(exact).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    same = out["residual_out"] == want
    assert np.mean(same) > 0.999
    got = f32_of_bits(out["residual_out"]).astype(np.float64)
    ulp = np.abs(f32_of_bits(want).astype(np.float64)) * 2.0 ** -7
    assert np.all(np.abs(got - exact) <= ulp + 1e-30)


def test_rms_of_the_read_is_one(ora):
    """RMS(yf / gamma) = sqrt(ms / (ms + eps)) for every row."""
    w = wl.fold_workload("rms", 4, 40, 768, seed=13, outlier_frac=0.05)
    out = ora.fold_norm(w.partials, w.residual, w.gamma, w.eps)
    o = sum(f32_of_bits(p).astype(np.float64) for p in w.partials)
    o = o + f32_of_bits(w.residual)
    ms = np.mean(o * o, axis=1)
    want = np.sqrt(ms / (ms + w.eps))
    got = np.sqrt(np.mean((f32_of_bits(out["y"]) / w.gamma) ** 2, axis=1))
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * want)


def test_fold_linearity_and_exactness(ora):
    w = wl.fold_workload("lin", 3, 12, 256, seed=14)
    base = ora.fold_norm(w.partials, w.residual, w.gamma, w.eps)
    # a zero partial changes nothing, bit for bit
    zero = np.zeros_like(w.partials[0])
    z = ora.fold_norm(w.partials[:1] + [zero] + w.partials[1:], w.residual, w.gamma, w.eps)
    assert all(np.array_equal(z[k], base[k]) for k in base)
    # splitting a partial into two exact halves changes nothing, bit for bit
    half = bits(f32_of_bits(w.partials[0]) * np.float32(0.5))
    assert np.array_equal(f32_of_bits(half) * 2, f32_of_bits(w.partials[0]))
    s = ora.fold_norm([half, half] + w.partials[1:], w.residual, w.gamma, w.eps)
    assert all(np.array_equal(s[k], base[k]) for k in base)
    # permuting the partials changes only rounding
    p = ora.fold_norm(w.partials[::-1], w.residual, w.gamma, w.eps)
    for k in base:
        assert np.all(close_bf16(p[k], f32_of_bits(base[k]), rel=1e-2, abs_=1e-3))
    # scaling every input by 2 doubles residual' exactly and leaves y unchanged (eps 0)
    b0 = ora.fold_norm(w.partials, w.residual, w.gamma, 0.0)
    dbl = [bits(f32_of_bits(x) * np.float32(2.0)) for x in w.partials + [w.residual]]
    d = ora.fold_norm(dbl[:-1], dbl[-1], w.gamma, 0.0)
    assert np.array_equal(f32_of_bits(d["residual_out"]), 2 * f32_of_bits(b0["residual_out"]))
    assert np.array_equal(d["y"], b0["y"])


# --------------------------------------------------------------------------------------
# FP8 consumer input
# --------------------------------------------------------------------------------------

def _yf64(w):
    o = sum(f32_of_bits(p).astype(np.float64) for p in w.partials)
    if w.residual is not None:
        o = o + f32_of_bits(w.residual)
    return torch.nn.functional.rms_norm(torch.from_numpy(o), (w.H,), weight=torch.from_numpy(
        w.gamma.astype(np.float64)), eps=w.eps).numpy()


def test_fp8_scale_is_amax_of_unrounded_read(ora):
    w = wl.fold_workload("fp8", 4, 64, 1024, seed=15, outlier_frac=0.05, fp8=True)
    out = ora.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_fp8=True)
    yf = _yf64(w)
    want = np.max(np.abs(yf), axis=1) / 448.0
    assert np.all(np.abs(out["scale"] - want) <= 1e-5 * want)
    # the bf16 y is not what the scale is taken over: it would miss this bound often
    y_rounded = np.max(np.abs(f32_of_bits(out["y"]).astype(np.float64)), axis=1) / 448.0
    assert np.mean(np.abs(y_rounded - want) > 1e-5 * want) > 0.2


def test_fp8_codes_round_trip_bound_and_reach_448(ora):
    w = wl.fold_workload("fp8b", 4, 64, 1024, seed=16, outlier_frac=0.05, fp8=True)
    out = ora.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_fp8=True)
    yf = _yf64(w)
    scale = out["scale"].astype(np.float64)[:, None]
    deq = ora.e4m3_to_f32(out["q"]).astype(np.float64) * scale
    v = np.abs(yf) / scale
    normal = v >= 2.0 ** -6
    err = np.abs(deq - yf)
    assert np.all(err[normal] <= (2.0 ** -4 + 1e-5) * np.abs(yf[normal]))
    sub = ~normal
    assert np.all(err[sub] <= (2.0 ** -10 + 1e-6) * np.broadcast_to(scale, yf.shape)[sub])
    mag = out["q"] & 0x7F
    assert np.all(np.max(mag, axis=1) == 0x7E)
    assert np.array_equal(out["q"] >> 7, (yf < 0).astype(np.uint8))


def test_fp8_zero_row(ora):
    z = np.zeros((3, 64), np.uint16)
    out = ora.fold_norm([z, z], z, np.ones(64, np.float32), 1e-6, want_fp8=True)
    assert np.all(out["scale"] == 0.0)
    assert np.all(out["q"] == 0)


# --------------------------------------------------------------------------------------
# Deferred MoE finalize
# --------------------------------------------------------------------------------------

def test_moe_brute_force_tiny(ora):
    """Three tokens, six expert rows, top-2: the definition evaluated term by term in
    binary64 Python floats."""
    rng = np.random.default_rng(21)
    T, H, n, topk = 3, 16, 6, 2
    E = bits(rng.standard_normal((n, H)))
    idx = np.array([[4, 0], [1, 5], [3, 2]], np.int32)
    w = np.array([[0.75, 0.25], [0.5, 0.5], [0.9, 0.1]], np.float32)
    res = bits(rng.standard_normal((T, H)))
    gamma = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    out = ora.moe_finalize_fold_norm(E, idx, w, res, gamma, 1e-6)
    Ef, rf = f32_of_bits(E), f32_of_bits(res)
    for t in range(T):
        o = [sum(float(w[t, j]) * float(Ef[idx[t, j], h]) for j in range(topk)) + float(rf[t, h])
             for h in range(H)]
        r = 1.0 / math.sqrt(sum(v * v for v in o) / H + 1e-6)
        y = [o[h] * r * float(gamma[h]) for h in range(H)]
        assert np.all(close_bf16(out["residual_out"][t], o, rel=2.0 ** -8))
        assert np.all(close_bf16(out["y"][t], y, rel=2.0 ** -7))
    assert not out["bad_index"]


def test_moe_relocating_expert_rows_is_exact(ora):
    w = wl.moe_workload("moe", 40, 256, 16, 4, seed=22)
    base = ora.moe_finalize_fold_norm(w.expert_out, w.idx, w.w, w.residual, w.gamma, w.eps)
    perm = np.random.default_rng(5).permutation(w.expert_out.shape[0])
    E2 = np.empty_like(w.expert_out)
    E2[perm] = w.expert_out                       # row p moves to perm[p]
    moved = ora.moe_finalize_fold_norm(E2, perm[w.idx].astype(np.int32), w.w, w.residual,
                                       w.gamma, w.eps)
    assert np.array_equal(moved["residual_out"], base["residual_out"])
    assert np.array_equal(moved["y"], base["y"])
    # permuting the slots of each token (index and weight together): rounding only
    sl = np.random.default_rng(6).permutation(4)
    p = ora.moe_finalize_fold_norm(w.expert_out, w.idx[:, sl].copy(), w.w[:, sl].copy(),
                                   w.residual, w.gamma, w.eps)
    for k in ("residual_out", "y"):
        assert np.all(close_bf16(p[k], f32_of_bits(base[k]), rel=1e-2, abs_=1e-3))


def test_moe_single_slot_reduces_to_fold(ora):
    w = wl.moe_workload("moe1", 30, 128, 8, 3, seed=23)
    one = np.zeros_like(w.w)
    one[:, 1] = 1.0
    out = ora.moe_finalize_fold_norm(w.expert_out, w.idx, one, w.residual, w.gamma, w.eps)
    gathered = w.expert_out[w.idx[:, 1]]
    ref = ora.fold_norm([gathered], w.residual, w.gamma, w.eps)
    assert np.array_equal(out["residual_out"], ref["residual_out"])
    assert np.array_equal(out["y"], ref["y"])


def test_moe_generator_layout(ora):
    """Routing weights are a softmax over the chosen k (sum to 1, descending) and the
    index map is a permutation of the expert-sorted rows."""
    w = wl.moe_workload("lay", 64, 32, 16, 4, seed=24)
    assert np.allclose(w.w.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(w.w, axis=1) <= 0)
    assert np.array_equal(np.sort(w.idx.reshape(-1)), np.arange(64 * 4))


def test_moe_bad_index_contributes_nothing(ora):
    w = wl.moe_workload("bad", 4, 64, 4, 2, seed=25)
    idx = w.idx.copy()
    idx[2, 1] = w.expert_out.shape[0]                          # one past the end
    out = ora.moe_finalize_fold_norm(w.expert_out, idx, w.w, w.residual, w.gamma, w.eps)
    assert out["bad_index"]
    w0 = w.w.copy()
    w0[2, 1] = 0.0
    ref = ora.moe_finalize_fold_norm(w.expert_out, w.idx, w0, w.residual, w.gamma, w.eps)
    assert np.array_equal(out["residual_out"], ref["residual_out"])


# --------------------------------------------------------------------------------------
# Row slice of a padded ragged batch
# --------------------------------------------------------------------------------------

SENT = 0x7FC1          # a NaN bit pattern no computed value takes


def test_slice_padding_rows_match_hand_layout(ora):
    g = read_golden("ragged_slice_padding.txt")
    counts = [int(v) for v in g["counts"]]
    offsets, counts_a, T_pad = wl.ragged_layout(counts)
    assert offsets.tolist() == [int(v) for v in g["offsets"]]
    assert T_pad == int(g["t_pad"][0])
    W = int(g["slices"][0])
    H = 16
    w = wl.slice_workload("pad", 2, H, counts, W, 0, seed=31)
    S = T_pad // W
    for r in range(W):
        pad = [int(v) for v in g.get(f"slice{r}", [])]
        out = {"residual_out": np.full((S, H), SENT, np.uint16),
               "y": np.full((S, H), SENT, np.uint16)}
        res = ora.slice_fold_norm(w.partials, T_pad, W, r, offsets, counts_a,
                                  w.residual_full[r * S:(r + 1) * S], w.gamma, w.eps, out=out)
        untouched = np.nonzero(np.all(res["residual_out"] == SENT, axis=1))[0].tolist()
        assert untouched == pad
        assert np.nonzero(np.all(res["y"] == SENT, axis=1))[0].tolist() == pad
        assert res["rows_written"] == S - len(pad)


def test_slices_together_equal_the_full_batch(ora):
    counts = wl.RAGGED_COUNTS
    w = wl.slice_workload("union", 3, 32, counts, 8, 0, seed=32)
    full = ora.fold_norm(w.partials, w.residual_full, w.gamma, w.eps)
    S = w.T_pad // 8
    valid = np.zeros(w.T_pad, bool)
    for o, c in zip(w.set_offsets, w.set_counts):
        valid[o:o + c] = True
    for r in range(8):
        out = {"residual_out": np.full((S, 32), SENT, np.uint16),
               "y": np.full((S, 32), SENT, np.uint16)}
        res = ora.slice_fold_norm(w.partials, w.T_pad, 8, r, w.set_offsets, w.set_counts,
                                  w.residual_full[r * S:(r + 1) * S], w.gamma, w.eps, out=out)
        rows = np.arange(r * S, (r + 1) * S)
        v = valid[rows]
        assert np.array_equal(res["residual_out"][v], full["residual_out"][rows[v]])
        assert np.array_equal(res["y"][v], full["y"][rows[v]])
        assert np.all(res["residual_out"][~v] == SENT)
    # the generator leaves the padding rows of every input at zero
    for p in w.partials + [w.residual_full]:
        assert np.all(p[~valid] == 0)


def test_slice_rejects_unequal_slices(ora):
    w = wl.slice_workload("bad", 1, 16, (3, 5), 2, 0, seed=33)
    with pytest.raises(ValueError):
        ora.slice_fold_norm(w.partials, w.T_pad, 3, 0, w.set_offsets, w.set_counts,
                            w.residual, w.gamma, w.eps)


# --------------------------------------------------------------------------------------
# Gemma weight (1 + gamma) and variable-size reduce-scatter (rsv)
# --------------------------------------------------------------------------------------

def test_gemma_weight_on_the_hand_row(ora):
    """With weight 1 + gamma, passing gamma - 1 must reproduce the plain hand row."""
    g = _golden_row("fold_norm_h4.txt")
    p = [bits(g["p0"])[None], bits(g["p1"])[None]]
    res = bits(g["res"])[None]
    out = ora.fold_norm(p, res, (g["gamma"] - 1).astype(np.float32), 0.0, gemma=True)
    assert np.array_equal(f32_of_bits(out["y"][0]), g["y"])
    assert np.array_equal(f32_of_bits(out["residual_out"][0]), g["residual_out"])


def test_gemma_weight_matches_torch_rmsnorm(ora):
    w = wl.fold_workload("gemma", 2, 30, 640, seed=91, residual=False)
    small = (0.05 * np.random.default_rng(3).standard_normal(w.H)).astype(np.float32)
    out = ora.fold_norm([w.partials[0]], None, small, w.eps, gemma=True)
    x = torch.from_numpy(f32_of_bits(w.partials[0]).astype(np.float64))
    ref = torch.nn.functional.rms_norm(x, (w.H,), weight=torch.from_numpy(
        1.0 + small.astype(np.float64)), eps=w.eps).numpy()
    assert np.all(close_bf16(out["y"], ref, rel=2.0 ** -8 + 1e-6))
    plain = ora.fold_norm([w.partials[0]], None, small, w.eps)
    assert not np.array_equal(plain["y"], out["y"])


def test_rsv_gives_each_rank_exactly_its_token_set(ora):
    counts = wl.RAGGED_COUNTS
    w = wl.slice_workload("rsv", 3, 32, counts, 8, 0, seed=92)
    full = ora.fold_norm(w.partials, w.residual_full, w.gamma, w.eps, want_fp8=True)
    for s, (o, c) in enumerate(zip(w.set_offsets, w.set_counts)):
        res = ora.set_slice_fold_norm(w.partials, w.T_pad, s, w.set_offsets, w.set_counts,
                                      w.residual_full[o:o + c], w.gamma, w.eps,
                                      want_fp8=True)
        assert res["rows_written"] == counts[s] and res["residual_out"].shape[0] == counts[s]
        for k in ("residual_out", "y", "q", "scale"):
            assert np.array_equal(res[k], full[k][o:o + c])
    with pytest.raises(ValueError):
        ora.set_slice_fold_norm(w.partials, w.T_pad, 4, w.set_offsets, w.set_counts,
                                None, w.gamma, w.eps)
