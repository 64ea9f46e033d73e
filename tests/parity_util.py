"""Helpers shared by the GPU parity tests: device buffers with guard rows, and the
comparisons the parity bar is stated in.

Tolerances (binary32 accumulation on both sides, bf16 outputs):
  * bf16 outputs: |gpu - oracle| <= 1e-2 * |oracle| + 1e-3, element by element;
  * residual' of the fold variants: bit-identical (same binary32 order of additions);
  * FP8 codes: at most 1 code apart, on at most 0.1% of the elements;
  * FP8 scales: within 1e-5 relative;
  * placement (which rows are written, guard and padding bytes): bit-exact.
"""
import numpy as np
import torch

SENTINEL16 = 0x7FC1       # a NaN bf16 pattern no computed value takes
SENTINEL8 = 0x7F          # the E4M3 NaN code, never produced (saturating conversion)
GUARD = 2                 # guard rows before and after every output


def dev_bits(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits -> a CUDA bfloat16 tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class Guarded:
    """An output of `rows` x `cols` elements inside a buffer with GUARD sentinel rows on
    each side; `.t` is the view to pass, `.check()` verifies the guards."""

    def __init__(self, rows, cols, dtype):
        self.rows, self.cols, self.dtype = rows, cols, dtype
        shape = (rows + 2 * GUARD, cols) if cols else (rows + 2 * GUARD * 4,)
        if dtype == torch.bfloat16:
            self.buf = torch.full(shape, SENTINEL16, dtype=torch.int16, device="cuda")
            self.buf = self.buf.view(torch.bfloat16)
        elif dtype == torch.uint8:
            self.buf = torch.full(shape, SENTINEL8, dtype=torch.uint8, device="cuda")
        else:
            self.buf = torch.full(shape, float("nan"), dtype=dtype, device="cuda")
        g = GUARD if cols else GUARD * 4
        self.g = g
        self.t = self.buf[g:g + rows]

    def host(self):
        if self.dtype == torch.bfloat16:
            return host_bits(self.t)
        return self.t.cpu().numpy()

    def check(self):
        whole = self.buf.view(torch.int16) if self.dtype == torch.bfloat16 else self.buf
        head = whole[:self.g].cpu().numpy()
        tail = whole[self.g + self.rows:].cpu().numpy()
        for part in (head, tail):
            if self.dtype == torch.bfloat16:
                assert np.all(part.view(np.uint16) == SENTINEL16), "guard row overwritten"
            elif self.dtype == torch.uint8:
                assert np.all(part == SENTINEL8), "guard row overwritten"
            else:
                assert np.all(np.isnan(part)), "guard row overwritten"


def f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def assert_bf16_close(got, want, what, rows=None):
    g, w = f32(got).astype(np.float64), f32(want).astype(np.float64)
    if rows is not None:
        g, w = g[rows], w[rows]
    bad = ~(np.abs(g - w) <= 1e-2 * np.abs(w) + 1e-3)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, first at "
                             f"{tuple(i)}: gpu {g[tuple(i)]} oracle {w[tuple(i)]}")


def assert_bits_equal(got, want, what, rows=None):
    g, w = np.asarray(got), np.asarray(want)
    if rows is not None:
        g, w = g[rows], w[rows]
    if not np.array_equal(g, w):
        n = int((g != w).sum())
        i = np.argwhere(g != w)[0]
        raise AssertionError(f"{what}: {n} elements differ, first at {tuple(i)}: "
                             f"gpu {g[tuple(i)]:#x} oracle {w[tuple(i)]:#x}")


def e4m3_ordinal(c):
    c = np.asarray(c, np.int32)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def assert_fp8_close(q_got, q_want, s_got, s_want, what, rows=None):
    qg, qw = np.asarray(q_got), np.asarray(q_want)
    sg, sw = np.asarray(s_got, np.float64), np.asarray(s_want, np.float64)
    if rows is not None:
        qg, qw, sg, sw = qg[rows], qw[rows], sg[rows], sw[rows]
    rel = np.abs(sg - sw) / np.maximum(np.abs(sw), 1e-30)
    assert np.all((rel <= 1e-5) | (sw == sg)), f"{what}: scale rel err {rel.max():.3g}"
    d = np.abs(e4m3_ordinal(qg) - e4m3_ordinal(qw))
    assert d.max(initial=0) <= 1, f"{what}: codes {int(d.max())} apart"
    frac = float(np.mean(d > 0)) if d.size else 0.0
    assert frac <= 1e-3, f"{what}: {frac:.4%} of codes differ"
