"""Thin ctypes binding of ``liblb.so`` (declared in include/lb.h).

Argument marshalling only: every function has the name and argument order of the C
entry point, turns tensors into device pointers (a ``torch.Tensor``, an integer
address or ``None`` for NULL are accepted wherever the C side takes a pointer),
passes the stream, and raises :class:`LBError` on a non-OK status.  A tensor argument
must be a contiguous CUDA tensor of the element type the C side reads (bf16 data as
``bfloat16`` or its raw ``int16``/``uint16`` bits; gamma, weights and scales
``float32``; indices and the bad-index flag ``int32``; FP8 codes ``uint8``), and all
tensors of one call must be on one device: anything else raises before the call.  All work runs in
the library's kernels; there is no fallback.  If the library has not been built the
first call raises :class:`LibraryMissing`.

The ``lb_options`` argument of the calls is built from keywords:

* ``gemma=True`` -- LB_OPT_GEMMA_WEIGHT, the read's weight is 1 + gamma;
* ``residual_snapshot=t`` -- a second bf16 copy of residual' into ``t``;
* ``residual_ready=True`` -- LB_OPT_RESIDUAL_READY, the caller's promise that the
  residual and gamma were complete before the kernel preceding the call began;
* ``routing_ready=True`` (MoE finalize only) -- LB_OPT_ROUTING_READY, the same promise
  for the routing indices and weights.

Without keywords NULL is passed (the defaults).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblb.so")

LB_OK = 0
LB_ERR_INVALID_ARGUMENT = 1
LB_ERR_MISALIGNED = 2
LB_ERR_UNSUPPORTED = 3
LB_ERR_CUDA = 4
LB_ERR_NOT_STARTED = 5
LB_ERR_FOREIGN_OUTPUT = 6
LB_ERR_UPDATE_PENDING = 7
LB_MAX_K = 16
LB_MAX_TOPK = 16
LB_MAX_SETS = 64
LB_MAX_H = 131072
LB_MAX_ROWS = 1 << 27

LB_KERNEL_ROW = 0
LB_KERNEL_STREAM = 1
LB_DEVICE_ERR_TIMEOUT = 1
LB_DEVICE_ERR_LAUNCH = 2
LB_OPT_GEMMA_WEIGHT = 1
LB_OPT_ROUTING_READY = 2
LB_OPT_RESIDUAL_READY = 4

LB_RESIDUAL_INITIAL = 0
LB_RESIDUAL_WRITTEN = 1
LB_RESIDUAL_PENDING = 2
LB_CONTRIB_PARTIALS = 0
LB_CONTRIB_MOE = 1

EXPORTED = ("lb_status_string", "lb_last_cuda_error", "lb_version", "lb_launch_plan",
            "lb_device_error", "lb_fold_norm", "lb_fold_norm_fp8",
            "lb_moe_finalize_fold_norm", "lb_slice_fold_norm", "lb_slice_fold_norm_v",
            "lb_residual_init", "lb_residual_start", "lb_residual_leave",
            "lb_residual_leave_moe", "lb_residual_prepare", "lb_residual_complete_output",
            "lb_residual_fold", "lb_residual_add_to_output", "lb_residual_written",
            "lb_residual_take_output", "lb_residual_norm")


class Plan(ctypes.Structure):
    """lb_plan: how the library launches a call."""
    _fields_ = [("kernel", ctypes.c_int), ("grid", ctypes.c_int), ("threads", ctypes.c_int),
                ("vectors_per_thread", ctypes.c_int), ("ctas_per_row", ctypes.c_int),
                ("stages", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("groups", ctypes.c_int), ("chunks", ctypes.c_int)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class Options(ctypes.Structure):
    """lb_options: optional behaviour of a call."""
    _fields_ = [("flags", ctypes.c_uint), ("residual_snapshot", ctypes.c_void_p)]


class ResidualStream(ctypes.Structure):
    """lb_residual_stream (include/lb_residual.h): the host-side residual stream.  It
    holds raw device pointers: keep the tensors it refers to alive while it does."""
    _fields_ = [("magic", ctypes.c_uint32), ("started", ctypes.c_int),
                ("state", ctypes.c_int), ("has_residual", ctypes.c_int),
                ("serial", ctypes.c_uint64), ("residual", ctypes.c_void_p),
                ("T", ctypes.c_int64), ("H", ctypes.c_int64), ("kind", ctypes.c_int),
                ("K", ctypes.c_int), ("partials", ctypes.c_void_p * LB_MAX_K),
                ("expert_out", ctypes.c_void_p), ("n_expert_rows", ctypes.c_int64),
                ("idx", ctypes.c_void_p), ("w", ctypes.c_void_p), ("topk", ctypes.c_int)]


class LibraryMissing(RuntimeError):
    pass


class LBError(RuntimeError):
    def __init__(self, status: int, func: str):
        self.status = status
        name = _lib.lb_status_string(status).decode() if _lib else str(status)
        extra = ""
        if status == LB_ERR_CUDA and _lib:
            extra = f" (cudaError {_lib.lb_last_cuda_error()})"
        super().__init__(f"{func} failed: {name}{extra}")


_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_f32 = ctypes.c_float


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load liblb.so (once).  Raises LibraryMissing when it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise LibraryMissing(
            f"{path} is missing: build it with `python -m layer_boundary_fusion_gb300.build`")
    lib = ctypes.CDLL(path)
    lib.lb_status_string.argtypes = [_int]
    lib.lb_status_string.restype = ctypes.c_char_p
    lib.lb_last_cuda_error.argtypes = []
    lib.lb_last_cuda_error.restype = _int
    lib.lb_version.argtypes = []
    lib.lb_version.restype = _int
    lib.lb_launch_plan.argtypes = [_i64, _i64, _int, _int, _int, ctypes.POINTER(Plan)]
    lib.lb_launch_plan.restype = _int
    lib.lb_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), _int]
    lib.lb_device_error.restype = _int
    op = ctypes.POINTER(Options)
    lib.lb_fold_norm.argtypes = [ctypes.POINTER(_vp), _int, _vp, _vp, _vp, _vp, _i64, _i64,
                                 _f32, op, _vp]
    lib.lb_fold_norm.restype = _int
    lib.lb_fold_norm_fp8.argtypes = [ctypes.POINTER(_vp), _int, _vp, _vp, _vp, _vp, _vp, _vp,
                                     _i64, _i64, _f32, op, _vp]
    lib.lb_fold_norm_fp8.restype = _int
    lib.lb_moe_finalize_fold_norm.argtypes = [_vp, _i64, _vp, _vp, _int, _vp, _vp, _vp, _vp,
                                              _vp, _vp, _i64, _i64, _f32, _vp, op, _vp]
    lib.lb_moe_finalize_fold_norm.restype = _int
    lib.lb_slice_fold_norm.argtypes = [ctypes.POINTER(_vp), _int, _i64, _int, _int, _vp, _vp,
                                       _int, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _f32, op, _vp]
    lib.lb_slice_fold_norm.restype = _int
    lib.lb_slice_fold_norm_v.argtypes = [ctypes.POINTER(_vp), _int, _i64, _int, _vp, _vp,
                                         _int, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _f32, op,
                                         _vp]
    lib.lb_slice_fold_norm_v.restype = _int
    rs = ctypes.POINTER(ResidualStream)
    out = ctypes.POINTER(ctypes.c_uint64)
    u64 = ctypes.c_uint64
    for name, args in (
            ("lb_residual_init", [rs, _vp, _i64, _i64]),
            ("lb_residual_start", [rs, out]),
            ("lb_residual_leave", [rs, u64, ctypes.POINTER(_vp), _int, out]),
            ("lb_residual_leave_moe", [rs, u64, _vp, _i64, _vp, _vp, _int, out]),
            ("lb_residual_prepare", [rs, u64, _vp, _vp, _vp, _vp, _f32, op, _vp, out]),
            ("lb_residual_complete_output", [rs, u64, _vp, _vp, out]),
            ("lb_residual_fold", [rs, u64, _vp, out]),
            ("lb_residual_add_to_output", [rs, u64, _vp, _vp, out]),
            ("lb_residual_written", [rs, u64, _vp, out]),
            ("lb_residual_take_output", [rs, u64, ctypes.POINTER(_vp)]),
            ("lb_residual_norm", [rs, u64, _vp, _vp, _vp, _vp, _f32, op, _vp])):
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _int
    _lib = lib
    return lib


# element types accepted per kind of tensor argument (bf16 data may come as raw bits)
_DTYPES = {"bf16": ("bfloat16", "int16", "uint16"), "f32": ("float32",), "i32": ("int32",),
           "u8": ("uint8",)}


class _Marshal:
    """Turns the tensor arguments of one call into device addresses.  A tensor must be
    a contiguous CUDA tensor of the element type the C side expects, and every tensor
    of the call must be on the same device; an ``int`` is passed as a raw address and
    ``None`` as NULL, unchecked."""

    def __init__(self, func: str):
        self.func = func
        self.devices = set()

    def __call__(self, x, kind: str, name: str) -> Optional[int]:
        if x is None:
            return None
        if isinstance(x, int):
            return x
        if not getattr(x, "is_cuda", False):
            raise ValueError(f"{self.func}: {name} must be a CUDA tensor")
        if not x.is_contiguous():
            raise ValueError(f"{self.func}: {name} must be contiguous")
        dt = str(x.dtype).replace("torch.", "")
        if dt not in _DTYPES[kind]:
            raise TypeError(f"{self.func}: {name} has dtype {dt}, expected "
                            f"{' or '.join(_DTYPES[kind])}")
        self.devices.add(x.device)
        if len(self.devices) > 1:
            raise ValueError(f"{self.func}: tensor arguments on different devices "
                             f"{sorted(str(d) for d in self.devices)}")
        return x.data_ptr()

    def array(self, items: Sequence, kind: str, name: str) -> ctypes.Array:
        arr = (_vp * max(1, len(items)))()
        for i, x in enumerate(items):
            arr[i] = self(x, kind, f"{name}[{i}]")
        return arr


def _stream(stream, *tensors) -> Optional[int]:
    """An explicit stream (torch.cuda.Stream or raw handle), else torch's current
    stream on the device of the first CUDA tensor argument, else the default stream."""
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    for t in tensors:
        if t is not None and not isinstance(t, int) and getattr(t, "is_cuda", False):
            import torch
            return torch.cuda.current_stream(t.device).cuda_stream
    return None


def _options(m: _Marshal, gemma: bool, residual_snapshot, routing_ready: bool = False,
             residual_ready: bool = False):
    """lb_options for the keyword arguments, or None (NULL) for the defaults."""
    if not gemma and residual_snapshot is None and not routing_ready and not residual_ready:
        return None
    flags = ((LB_OPT_GEMMA_WEIGHT if gemma else 0) | (LB_OPT_ROUTING_READY if routing_ready else 0)
             | (LB_OPT_RESIDUAL_READY if residual_ready else 0))
    return ctypes.byref(Options(flags, m(residual_snapshot, "bf16", "residual_snapshot")))


def _check(status: int, func: str) -> None:
    if status != LB_OK:
        raise LBError(status, func)


def lb_status_string(status: int) -> str:
    return load().lb_status_string(status).decode()


def lb_version() -> int:
    return load().lb_version()


def lb_launch_plan(rows: int, H: int, n_inputs: int, num_sms: int,
                   smem_per_block: int) -> Plan:
    """The launch the library makes for such a call (pure host function)."""
    plan = Plan()
    _check(load().lb_launch_plan(rows, H, n_inputs, num_sms, smem_per_block,
                                 ctypes.byref(plan)), "lb_launch_plan")
    return plan


def lb_device_error(clear: bool = True) -> int:
    """Synchronise the device; return (and clear) the kernels' device error flags."""
    flags = ctypes.c_uint(0)
    _check(load().lb_device_error(ctypes.byref(flags), int(clear)), "lb_device_error")
    return flags.value


def lb_fold_norm(partials, residual_in, residual_out, gamma, y_out, T, H, eps,
                 stream=None, *, gemma=False, residual_snapshot=None,
                 residual_ready=False) -> None:
    lib = load()
    partials = list(partials)
    m = _Marshal("lb_fold_norm")
    s = _stream(stream, *partials, residual_in, residual_out, y_out)
    _check(lib.lb_fold_norm(m.array(partials, "bf16", "partials"), len(partials),
                            m(residual_in, "bf16", "residual_in"),
                            m(residual_out, "bf16", "residual_out"), m(gamma, "f32", "gamma"),
                            m(y_out, "bf16", "y_out"), T, H, eps,
                            _options(m, gemma, residual_snapshot, False, residual_ready), s),
           "lb_fold_norm")


def lb_fold_norm_fp8(partials, residual_in, residual_out, gamma, q_out, scale_out, y_out,
                     T, H, eps, stream=None, *, gemma=False, residual_snapshot=None,
                     residual_ready=False) -> None:
    lib = load()
    partials = list(partials)
    m = _Marshal("lb_fold_norm_fp8")
    s = _stream(stream, *partials, residual_in, residual_out, q_out)
    _check(lib.lb_fold_norm_fp8(m.array(partials, "bf16", "partials"), len(partials),
                                m(residual_in, "bf16", "residual_in"),
                                m(residual_out, "bf16", "residual_out"),
                                m(gamma, "f32", "gamma"), m(q_out, "u8", "q_out"),
                                m(scale_out, "f32", "scale_out"), m(y_out, "bf16", "y_out"),
                                T, H, eps,
                                _options(m, gemma, residual_snapshot, False, residual_ready), s),
           "lb_fold_norm_fp8")


def lb_moe_finalize_fold_norm(expert_out, n_expert_rows, idx, w, topk, residual_in,
                              residual_out, gamma, y_out, q_out, scale_out, T, H, eps,
                              bad_index_flag=None, stream=None, *, gemma=False,
                              residual_snapshot=None, routing_ready=False,
                              residual_ready=False) -> None:
    lib = load()
    m = _Marshal("lb_moe_finalize_fold_norm")
    s = _stream(stream, expert_out, residual_out, y_out, q_out)
    _check(lib.lb_moe_finalize_fold_norm(
        m(expert_out, "bf16", "expert_out"), n_expert_rows, m(idx, "i32", "idx"),
        m(w, "f32", "w"), topk, m(residual_in, "bf16", "residual_in"),
        m(residual_out, "bf16", "residual_out"), m(gamma, "f32", "gamma"),
        m(y_out, "bf16", "y_out"), m(q_out, "u8", "q_out"), m(scale_out, "f32", "scale_out"),
        T, H, eps, m(bad_index_flag, "i32", "bad_index_flag"),
        _options(m, gemma, residual_snapshot, routing_ready, residual_ready), s),
        "lb_moe_finalize_fold_norm")


def _int32_array(values):
    n = len(values)
    return (ctypes.c_int32 * max(1, n))(*[int(v) for v in values]), n


def lb_slice_fold_norm(partials, T_pad, num_slices, slice_, set_offsets, set_counts,
                       residual_in, residual_out, gamma, y_out, q_out, scale_out, H, eps,
                       stream=None, *, gemma=False, residual_snapshot=None,
                       residual_ready=False) -> None:
    lib = load()
    partials = list(partials)
    if len(set_offsets) != len(set_counts):
        raise ValueError("set_offsets and set_counts differ in length")
    offs, n = _int32_array(set_offsets)
    cnts, _ = _int32_array(set_counts)
    m = _Marshal("lb_slice_fold_norm")
    s = _stream(stream, *partials, residual_out, y_out, q_out)
    _check(lib.lb_slice_fold_norm(m.array(partials, "bf16", "partials"), len(partials), T_pad,
                                  num_slices, slice_, ctypes.cast(offs, _vp),
                                  ctypes.cast(cnts, _vp), n,
                                  m(residual_in, "bf16", "residual_in"),
                                  m(residual_out, "bf16", "residual_out"),
                                  m(gamma, "f32", "gamma"), m(y_out, "bf16", "y_out"),
                                  m(q_out, "u8", "q_out"), m(scale_out, "f32", "scale_out"),
                                  H, eps,
                                  _options(m, gemma, residual_snapshot, False, residual_ready),
                                  s),
           "lb_slice_fold_norm")


def lb_slice_fold_norm_v(partials, T_pad, set_, set_offsets, set_counts, residual_in,
                         residual_out, gamma, y_out, q_out, scale_out, H, eps, stream=None, *,
                         gemma=False, residual_snapshot=None,
                         residual_ready=False) -> None:
    lib = load()
    partials = list(partials)
    if len(set_offsets) != len(set_counts):
        raise ValueError("set_offsets and set_counts differ in length")
    offs, n = _int32_array(set_offsets)
    cnts, _ = _int32_array(set_counts)
    m = _Marshal("lb_slice_fold_norm_v")
    s = _stream(stream, *partials, residual_out, y_out, q_out)
    _check(lib.lb_slice_fold_norm_v(m.array(partials, "bf16", "partials"), len(partials), T_pad,
                                    set_, ctypes.cast(offs, _vp), ctypes.cast(cnts, _vp), n,
                                    m(residual_in, "bf16", "residual_in"),
                                    m(residual_out, "bf16", "residual_out"),
                                    m(gamma, "f32", "gamma"), m(y_out, "bf16", "y_out"),
                                    m(q_out, "u8", "q_out"), m(scale_out, "f32", "scale_out"),
                                    H, eps,
                                    _options(m, gemma, residual_snapshot, False,
                                             residual_ready), s),
           "lb_slice_fold_norm_v")


# --------------------------------------------------------------------------------------
# Residual stream (include/lb_residual.h).  Each function that hands on an output
# returns its handle (an int); pass it to the next call.
# --------------------------------------------------------------------------------------

def _handle(func: str, call) -> int:
    h = ctypes.c_uint64(0)
    _check(call(ctypes.byref(h)), func)
    return h.value


def lb_residual_init(s: ResidualStream, residual, T, H) -> None:
    m = _Marshal("lb_residual_init")
    _check(load().lb_residual_init(ctypes.byref(s), m(residual, "bf16", "residual"), T, H),
           "lb_residual_init")


def lb_residual_start(s: ResidualStream) -> int:
    return _handle("lb_residual_start", lambda o: load().lb_residual_start(ctypes.byref(s), o))


def lb_residual_leave(s: ResidualStream, h: int, partials) -> int:
    partials = list(partials)
    arr = _Marshal("lb_residual_leave").array(partials, "bf16", "partials")
    return _handle("lb_residual_leave", lambda o: load().lb_residual_leave(
        ctypes.byref(s), h, arr, len(partials), o))


def lb_residual_leave_moe(s: ResidualStream, h: int, expert_out, n_expert_rows, idx, w,
                          topk) -> int:
    m = _Marshal("lb_residual_leave_moe")
    e, i, wt = m(expert_out, "bf16", "expert_out"), m(idx, "i32", "idx"), m(w, "f32", "w")
    return _handle("lb_residual_leave_moe", lambda o: load().lb_residual_leave_moe(
        ctypes.byref(s), h, e, n_expert_rows, i, wt, topk, o))


def lb_residual_prepare(s: ResidualStream, h: int, gamma, y_out, q_out, scale_out, eps,
                        stream=None, *, gemma=False, residual_snapshot=None,
                        residual_ready=False) -> int:
    st = _stream(stream, gamma, y_out, q_out)
    m = _Marshal("lb_residual_prepare")
    args = (m(gamma, "f32", "gamma"), m(y_out, "bf16", "y_out"), m(q_out, "u8", "q_out"),
            m(scale_out, "f32", "scale_out"))
    opt = _options(m, gemma, residual_snapshot, False, residual_ready)
    return _handle("lb_residual_prepare", lambda o: load().lb_residual_prepare(
        ctypes.byref(s), h, *args, eps, opt, st, o))


def lb_residual_complete_output(s: ResidualStream, h: int, sum_out, stream=None) -> int:
    st = _stream(stream, sum_out)
    p = _Marshal("lb_residual_complete_output")(sum_out, "bf16", "sum_out")
    return _handle("lb_residual_complete_output", lambda o: load().lb_residual_complete_output(
        ctypes.byref(s), h, p, st, o))


def lb_residual_fold(s: ResidualStream, h: int, stream=None) -> int:
    st = _stream(stream)
    return _handle("lb_residual_fold",
                   lambda o: load().lb_residual_fold(ctypes.byref(s), h, st, o))


def lb_residual_add_to_output(s: ResidualStream, h: int, extra, stream=None) -> int:
    st = _stream(stream, extra)
    p = _Marshal("lb_residual_add_to_output")(extra, "bf16", "extra")
    return _handle("lb_residual_add_to_output", lambda o: load().lb_residual_add_to_output(
        ctypes.byref(s), h, p, st, o))


def lb_residual_written(s: ResidualStream, h: int, hidden) -> int:
    p = _Marshal("lb_residual_written")(hidden, "bf16", "hidden")
    return _handle("lb_residual_written", lambda o: load().lb_residual_written(
        ctypes.byref(s), h, p, o))


def lb_residual_take_output(s: ResidualStream, h: int) -> int:
    """Release the stream; returns the residual buffer's device address."""
    p = ctypes.c_void_p(0)
    _check(load().lb_residual_take_output(ctypes.byref(s), h, ctypes.byref(p)),
           "lb_residual_take_output")
    return p.value or 0


def lb_residual_norm(s: ResidualStream, h: int, gamma, y_out, q_out, scale_out, eps,
                     stream=None, *, gemma=False, residual_snapshot=None,
                     residual_ready=False) -> None:
    st = _stream(stream, gamma, y_out, q_out)
    m = _Marshal("lb_residual_norm")
    _check(load().lb_residual_norm(ctypes.byref(s), h, m(gamma, "f32", "gamma"),
                                   m(y_out, "bf16", "y_out"), m(q_out, "u8", "q_out"),
                                   m(scale_out, "f32", "scale_out"), eps,
                                   _options(m, gemma, residual_snapshot, False, residual_ready),
                                   st), "lb_residual_norm")
