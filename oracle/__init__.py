"""CPU oracle for the layer-boundary hot path (numpy wrappers over ``lb_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline
leg are the only callers.  The CUDA library never imports, links or calls this
package, and this package never touches the CUDA library.

Every array of bf16 values is a ``numpy.uint16`` array of raw bf16 bit patterns; FP8
codes are ``numpy.uint8``.  Each function states the definition it evaluates; the
citations are in ``lb_oracle.c`` (sglang developer guide "Layer boundaries",
sections "Residual stream", "Residual update and input read", "Token layouts and
sums", "Enter and leave the layer stack", "Choose a reduction policy").
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_i32p = ctypes.POINTER(ctypes.c_int32)


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        vp = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        lib.ora_fold_norm.argtypes = [ctypes.POINTER(vp), ci, vp, vp, ci, i64, i64,
                                      ctypes.c_float, vp, vp, vp, vp, vp]
        lib.ora_fold_norm.restype = ctypes.c_int
        lib.ora_moe_finalize_fold_norm.argtypes = [vp, i64, vp, vp, ci, vp, vp, ci,
                                                   i64, i64, ctypes.c_float, vp, vp, vp,
                                                   vp, vp]
        lib.ora_moe_finalize_fold_norm.restype = ctypes.c_int
        lib.ora_slice_fold_norm.argtypes = [ctypes.POINTER(vp), ci, i64, ci, ci, vp, vp,
                                            ci, vp, vp, ci, i64, ctypes.c_float,
                                            vp, vp, vp, vp, vp]
        lib.ora_slice_fold_norm.restype = ctypes.c_int64
        lib.ora_set_slice_fold_norm.argtypes = [ctypes.POINTER(vp), ci, i64, ci, vp, vp, ci,
                                                vp, vp, ci, i64, ctypes.c_float, vp, vp, vp,
                                                vp, vp]
        lib.ora_set_slice_fold_norm.restype = ctypes.c_int64
        for name in ("ora_bf16_to_f32_array", "ora_f32_to_bf16_array",
                     "ora_f32_to_e4m3_array", "ora_e4m3_to_f32_array"):
            getattr(lib, name).argtypes = [vp, vp, i64]
            getattr(lib, name).restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    """Contiguous array of exactly `dtype` (no value conversion for bit arrays)."""
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return np.ascontiguousarray(a)


# --------------------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------------------

def bf16_to_f32(bits):
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float32)
    _load().ora_bf16_to_f32_array(_ptr(bits), _ptr(out), bits.size)
    return out


def f32_to_bf16(x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().ora_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def f32_to_e4m3(x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().ora_f32_to_e4m3_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_to_f32(codes):
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float32)
    _load().ora_e4m3_to_f32_array(_ptr(codes), _ptr(out), codes.size)
    return out


# --------------------------------------------------------------------------------------
# Boundary operations
# --------------------------------------------------------------------------------------

def _outputs(shape_rows, H, want_residual, want_y, want_fp8, out=None):
    out = dict(out or {})
    if want_residual and "residual_out" not in out:
        out["residual_out"] = np.zeros((shape_rows, H), np.uint16)
    if want_y and "y" not in out:
        out["y"] = np.zeros((shape_rows, H), np.uint16)
    if want_fp8:
        out.setdefault("q", np.zeros((shape_rows, H), np.uint8))
        out.setdefault("scale", np.zeros((shape_rows,), np.float32))
    for k, v in out.items():
        if not v.flags.c_contiguous:
            raise ValueError(f"output {k} must be C-contiguous")
    return out


def fold_norm(partials, residual_in, gamma, eps, *, want_residual=True, want_y=True,
              want_fp8=False, out=None, gemma=False):
    """Complete the owed sum of K partials, fold it into the residual, then read.

    o = (sum_k partials[k], k ascending, from +0) + residual_in (absent if None);
    residual_out = bf16(o); y = bf16(RMSNorm(o) * weight) with weight = gamma, or
    1 + gamma when `gemma`; FP8: q, scale per token.
    Returns a dict with the requested outputs ("residual_out", "y", "q", "scale").
    `out` may supply preallocated outputs (rows not written keep their bytes).
    """
    partials = [_c(p, np.uint16) for p in partials]
    if residual_in is not None:
        residual_in = _c(residual_in, np.uint16)
    shape = (partials[0] if partials else residual_in).shape
    T, H = shape
    for p in partials:
        assert p.shape == shape
    gamma = None if gamma is None else _c(gamma, np.float32)
    res = _outputs(T, H, want_residual, want_y, want_fp8, out)
    arr = (ctypes.c_void_p * max(1, len(partials)))(*[p.ctypes.data for p in partials])
    work = np.empty(2 * H, np.float32)
    rc = _load().ora_fold_norm(arr, len(partials), _ptr(residual_in), _ptr(gamma),
                               int(gemma), T, H,
                               ctypes.c_float(eps), _ptr(res.get("residual_out")),
                               _ptr(res.get("y")), _ptr(res.get("q")),
                               _ptr(res.get("scale")), _ptr(work))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return res


def moe_finalize_fold_norm(expert_out, idx, w, residual_in, gamma, eps, *,
                           want_residual=True, want_y=True, want_fp8=False, out=None,
                           gemma=False):
    """Deferred MoE finalize folded into the residual, then read.

    o[t] = sum_j (w[t,j] * expert_out[idx[t,j]]) (j ascending, each product rounded
    to FP32) + residual_in[t].  Returns the outputs dict plus "bad_index" (bool):
    an index outside [0, n_rows) contributes nothing.
    """
    expert_out = _c(expert_out, np.uint16)
    idx = _c(idx, np.int32)
    w = _c(w, np.float32)
    T, topk = idx.shape
    n_rows, H = expert_out.shape
    if residual_in is not None:
        residual_in = _c(residual_in, np.uint16)
    gamma = None if gamma is None else _c(gamma, np.float32)
    res = _outputs(T, H, want_residual, want_y, want_fp8, out)
    work = np.empty(2 * H, np.float32)
    bad = _load().ora_moe_finalize_fold_norm(
        _ptr(expert_out), n_rows, _ptr(idx), _ptr(w), topk, _ptr(residual_in),
        _ptr(gamma), int(gemma), T, H, ctypes.c_float(eps), _ptr(res.get("residual_out")),
        _ptr(res.get("y")), _ptr(res.get("q")), _ptr(res.get("scale")), _ptr(work))
    res["bad_index"] = bool(bad)
    return res


def slice_fold_norm(partials, T_pad, num_slices, slice_, offsets, counts, residual_in,
                    gamma, eps, *, want_residual=True, want_y=True, want_fp8=False,
                    out=None, gemma=False):
    """Slice `slice_` of a padded ragged batch (fixed-size reduce-scatter completion).

    Outputs are compact [S, H] with S = T_pad / num_slices; padding rows are left
    untouched (pass `out` arrays prefilled with a sentinel to observe that).
    Returns the outputs dict plus "rows_written".
    """
    partials = [_c(p, np.uint16) for p in partials]
    H = partials[0].shape[1] if partials else residual_in.shape[1]
    S = T_pad // num_slices
    if residual_in is not None:
        residual_in = _c(residual_in, np.uint16)
    gamma = None if gamma is None else _c(gamma, np.float32)
    offsets = _c(np.asarray(offsets, np.int32), np.int32)
    counts = _c(np.asarray(counts, np.int32), np.int32)
    res = _outputs(S, H, want_residual, want_y, want_fp8, out)
    arr = (ctypes.c_void_p * max(1, len(partials)))(*[p.ctypes.data for p in partials])
    work = np.empty(2 * H, np.float32)
    n = _load().ora_slice_fold_norm(
        arr, len(partials), T_pad, num_slices, slice_, _ptr(offsets), _ptr(counts),
        len(offsets), _ptr(residual_in), _ptr(gamma), int(gemma), H, ctypes.c_float(eps),
        _ptr(res.get("residual_out")), _ptr(res.get("y")), _ptr(res.get("q")),
        _ptr(res.get("scale")), _ptr(work))
    if n < 0:
        raise ValueError("oracle rejected the slice metadata")
    res["rows_written"] = int(n)
    return res


def set_slice_fold_norm(partials, T_pad, set_, offsets, counts, residual_in, gamma, eps, *,
                        want_residual=True, want_y=True, want_fp8=False, out=None,
                        gemma=False):
    """Rank `set_`'s rows under a variable-size reduce-scatter: the valid rows of
    token set `set_`, as compact [counts[set_], H] outputs."""
    partials = [_c(p, np.uint16) for p in partials]
    H = partials[0].shape[1] if partials else residual_in.shape[1]
    offsets = _c(np.asarray(offsets, np.int32), np.int32)
    counts = _c(np.asarray(counts, np.int32), np.int32)
    if not 0 <= set_ < len(counts):
        raise ValueError("set index out of range")
    rows = int(counts[set_])
    if residual_in is not None:
        residual_in = _c(residual_in, np.uint16)
    gamma = None if gamma is None else _c(gamma, np.float32)
    res = _outputs(rows, H, want_residual, want_y, want_fp8, out)
    arr = (ctypes.c_void_p * max(1, len(partials)))(*[p.ctypes.data for p in partials])
    work = np.empty(2 * H, np.float32)
    n = _load().ora_set_slice_fold_norm(
        arr, len(partials), T_pad, set_, _ptr(offsets), _ptr(counts), len(offsets),
        _ptr(residual_in), _ptr(gamma), int(gemma), H, ctypes.c_float(eps),
        _ptr(res.get("residual_out")), _ptr(res.get("y")), _ptr(res.get("q")),
        _ptr(res.get("scale")), _ptr(work))
    if n < 0:
        raise ValueError("oracle rejected the set metadata")
    res["rows_written"] = int(n)
    return res


def library_path() -> str:
    return os.path.abspath(_build.LIB)
