"""Host-side tests of the C ABI: the library builds and loads, exports exactly what
include/lb.h declares, chooses launch shapes as documented, and rejects every invalid
argument before launching anything.

No kernel runs here.  The argument-validation cases use fake device addresses, so
they execute in a child process that sees no GPU at all: a case that wrongly passed
validation would get a CUDA "no device" error, never a launch on a bad address.
"""
import glob
import json
import os
import re
import subprocess
import sys

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from layer_boundary_fusion_gb300 import build, lb
    build.build()
    return lb


def declared_functions():
    names = set()
    for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(lb_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_four_boundary_calls():
    names = declared_functions()
    for f in ("lb_fold_norm", "lb_fold_norm_fp8", "lb_moe_finalize_fold_norm",
              "lb_slice_fold_norm", "lb_slice_fold_norm_v"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b[TW] (lb_[a-z0-9_]+)$", out, flags=re.M))
    assert set(names) <= exported, set(names) - exported
    assert exported == set(lib.EXPORTED), exported ^ set(lib.EXPORTED)
    L = lib.load()
    for n in names:
        assert hasattr(L, n)


def test_status_strings_and_version(lib):
    assert lib.lb_status_string(0) == "LB_OK"
    assert lib.lb_status_string(4) == "LB_ERR_CUDA"
    assert lib.lb_status_string(5) == "LB_ERR_NOT_STARTED"
    assert lib.lb_status_string(6) == "LB_ERR_FOREIGN_OUTPUT"
    assert lib.lb_status_string(7) == "LB_ERR_UPDATE_PENDING"
    assert lib.lb_version() >= 100


def test_header_constants_match_binding(lib):
    text = open(os.path.join(ROOT, "include", "lb.h")).read()
    for name in ("LB_MAX_K", "LB_MAX_TOPK", "LB_MAX_SETS", "LB_MAX_H", "LB_MAX_ROWS"):
        m = re.search(rf"#define {name} (\d+)", text)
        assert int(m.group(1)) == getattr(lib, name)


SMEM = 232448          # opt-in shared memory per CTA on GB300


@pytest.mark.parametrize("rows,H,n_in,plan", [
    # (kernel, grid, threads, vectors/thread, ctas/row, stages, smem)
    (2048, 4096, 5, (1, 152, 800, 2, 1, 3, 123792)),    # prefill K=4 + residual: stream
    (1024, 4096, 9, (1, 152, 800, 2, 1, 3, 222096)),    # MoE top-8 + residual: stream
    (254, 4096, 9, (1, 152, 800, 2, 1, 3, 222096)),     # one ragged slice: stream
    (64, 4096, 9, (0, 64, 512, 1, 1, 0, 0)),            # decode: row kernel, a CTA per row
    (1, 4096, 2, (0, 1, 512, 1, 1, 0, 0)),
    (16, 512, 3, (0, 16, 64, 1, 1, 0, 0)),              # tiny: one CTA per row
    (4096, 8192, 5, (1, 152, 544, 2, 1, 2, 164448)),    # one group of 16 warps
    (4096, 6144, 2, (1, 152, 800, 2, 1, 8, 199040)),    # two groups of 12 warps
    (4096, 8192, 9, (0, 4096, 512, 2, 1, 0, 0)),        # no double-buffered stage fits
    (4096, 4096, 17, (0, 4096, 512, 1, 1, 0, 0)),
    (4096, 8200, 17, (1, 152, 352, 4, 1, 2, 207488)),   # 4 chunks of 10 warps
    (4096, 12288, 5, (1, 152, 544, 4, 1, 4, 214208)),   # 3 chunks of 16 warps
    (4096, 16384, 3, (1, 152, 544, 4, 1, 6, 214816)),   # 4 chunks
    (4096, 16384, 17, (0, 4096, 512, 4, 1, 0, 0)),      # no chunked stage fits twice
    (4096, 32768, 2, (0, 8192, 512, 4, 2, 0, 0)),
    (4096, 520, 2, (0, 4096, 96, 1, 1, 0, 0)),          # short rows: row kernel at any T
    (4096, 8, 2, (0, 4096, 32, 1, 1, 0, 0)),
    (4096, 1032, 2, (1, 152, 608, 1, 1, 6, 26592)),     # 129 vectors: partly active warp
])
def test_launch_plan(lib, rows, H, n_in, plan):
    p = lib.lb_launch_plan(rows, H, n_in, 152, SMEM)
    got = (p.kernel, p.grid, p.threads, p.vectors_per_thread, p.ctas_per_row, p.stages,
           p.smem_bytes)
    assert got == plan


def test_launch_plan_covers_every_row_vector(lib):
    for H in list(range(8, 4096, 8)) + [8192, 12288, 16384, 24576, 65536, 131072]:
        for rows in (1, 7, 64, 300, 5000):
            for n_in in (1, 2, 5, 9, 17):
                p = lib.lb_launch_plan(rows, H, n_in, 152, SMEM)
                nvec = H // 8
                if p.kernel == lib.LB_KERNEL_ROW:
                    per_cta = -(-nvec // p.ctas_per_row)
                    assert p.threads % 32 == 0 and 32 <= p.threads <= 512
                    assert p.threads * p.vectors_per_thread >= per_cta
                    assert p.ctas_per_row * per_cta >= nvec and 1 <= p.ctas_per_row <= 8
                    assert p.grid == rows * p.ctas_per_row
                else:
                    assert nvec > 128              # short rows never stream
                    groups = p.groups
                    assert 1 <= groups <= min(3, p.stages) and p.threads <= 800
                    consumers = (p.threads - 32) // groups
                    assert consumers * groups + 32 == p.threads
                    assert consumers % 64 == 0 and 64 <= consumers <= 512
                    assert 2 <= p.stages <= 8 and p.grid == 152 and rows > 152
                    # every stage belongs to one consumer group
                    assert p.stages % groups == 0
                    if p.chunks == 1:            # whole rows: 1 or 2 vectors a thread
                        assert p.vectors_per_thread in (1, 2)
                        assert consumers * p.vectors_per_thread >= nvec
                        width, weight = H, 0
                    else:                        # chunks of one vector per thread
                        assert p.vectors_per_thread == 4 and groups == 1
                        assert 2 <= p.chunks <= 4
                        assert (p.chunks - 1) * consumers < nvec <= p.chunks * consumers
                        width, weight = consumers * 8, H * 4
                    assert p.smem_bytes == (p.stages * (n_in * width * 2 + 16 + 2 * 144)
                                            + weight)
                    assert p.smem_bytes + 1024 <= SMEM
                assert p.vectors_per_thread in (1, 2, 4)


def test_launch_plan_rejects(lib):
    for args in ((10, 12, 2, 152, SMEM), (10, 0, 2, 152, SMEM),
                 (10, lib.LB_MAX_H + 8, 2, 152, SMEM), (10, 4096, 2, 0, SMEM),
                 (10, 4096, 0, 152, SMEM), (10, 4096, 18, 152, SMEM)):
        with pytest.raises(lib.LBError):
            lib.lb_launch_plan(*args)


_VALIDATION_SCRIPT = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
from layer_boundary_fusion_gb300 import lb
L = lb.load()
A = 1 << 32          # fake, 16-byte aligned "device" addresses; nothing dereferences them
def a(i): return A + i * (1 << 28)
T, H = 4, 64
P = [a(0), a(1)]
results = {}
def run(name, fn, *args):
    try:
        fn(*args); results[name] = 0
    except lb.LBError as e:
        results[name] = e.status
f = lb.lb_fold_norm
run("ok_empty", f, P, a(2), a(3), a(4), a(5), 0, H, 1e-6, 0)
results["K_negative"] = L.lb_fold_norm(None, -1, a(2), a(3), a(4), a(5), T, H, 1e-6, None, None)
opts = lb.Options(7, None)
results["unknown_flag"] = L.lb_fold_norm((lb._vp * 2)(a(0), a(1)), 2, a(2), a(3), a(4), a(5), T, H, 1e-6, lb.ctypes.byref(opts), None)
run("snapshot_misaligned", lambda: f(P, a(2), a(3), a(4), a(5), T, H, 1e-6, 0, residual_snapshot=a(9) + 8))
run("snapshot_overlaps_y", lambda: f(P, a(2), a(3), a(4), a(5), T, H, 1e-6, 0, residual_snapshot=a(5) + 16))
run("snapshot_empty_ok", lambda: f(P, a(2), a(3), a(4), a(5), 0, H, 1e-6, 0, gemma=True, residual_snapshot=a(9)))
run("K_too_big", f, [a(i) for i in range(17)], a(20), a(21), a(22), a(23), T, H, 1e-6, 0)
run("partial_null", f, [a(0), None], a(2), a(3), a(4), a(5), T, H, 1e-6, 0)
run("partial_misaligned", f, [a(0), a(1) + 8], a(2), a(3), a(4), a(5), T, H, 1e-6, 0)
run("K0_no_residual", f, [], None, a(3), a(4), a(5), T, H, 1e-6, 0)
run("nothing_to_write", f, P, a(2), None, a(4), None, T, H, 1e-6, 0)
run("y_without_gamma", f, P, a(2), a(3), None, a(5), T, H, 1e-6, 0)
run("H_not_multiple_of_8", f, P, a(2), a(3), a(4), a(5), T, 60, 1e-6, 0)
run("H_zero", f, P, a(2), a(3), a(4), a(5), T, 0, 1e-6, 0)
run("H_too_big", f, P, a(2), a(3), a(4), a(5), T, lb.LB_MAX_H + 8, 1e-6, 0)
run("T_negative", f, P, a(2), a(3), a(4), a(5), -1, H, 1e-6, 0)
run("T_too_big", f, P, a(2), a(3), a(4), a(5), lb.LB_MAX_ROWS + 1, H, 1e-6, 0)
run("eps_negative", f, P, a(2), a(3), a(4), a(5), T, H, -1e-6, 0)
run("eps_nan", f, P, a(2), a(3), a(4), a(5), T, H, float("nan"), 0)
run("y_misaligned", f, P, a(2), a(3), a(4), a(5) + 2, T, H, 1e-6, 0)
run("gamma_misaligned", f, P, a(2), a(3), a(4) + 4, a(5), T, H, 1e-6, 0)
run("y_overlaps_partial", f, P, a(2), a(3), a(4), a(0) + 16, T, H, 1e-6, 0)
run("y_overlaps_residual_out", f, P, a(2), a(3), a(4), a(3) + 16, T, H, 1e-6, 0)
run("residual_out_shifted_over_in", f, P, a(2), a(2) + 16, a(4), a(5), T, H, 1e-6, 0)
run("in_place_empty_ok", f, P, a(2), a(2), a(4), a(5), 0, H, 1e-6, 0)
run("empty_null_buffers_ok", f, [], None, None, None, None, 0, H, 1e-6, 0)
run("empty_bad_H", f, [], None, None, None, None, 0, 12, 1e-6, 0)
run("empty_K_too_big", f, [None] * 17, None, None, None, None, 0, H, 1e-6, 0)
g = lb.lb_fold_norm_fp8
run("fp8_empty_ok", g, P, a(2), a(3), a(4), a(6), a(7), a(5), 0, H, 1e-6, 0)
run("fp8_no_q", g, P, a(2), a(3), a(4), None, a(7), a(5), T, H, 1e-6, 0)
run("fp8_no_scale", g, P, a(2), a(3), a(4), a(6), None, a(5), T, H, 1e-6, 0)
run("fp8_no_gamma", g, P, a(2), a(3), None, a(6), a(7), None, T, H, 1e-6, 0)
run("fp8_scale_misaligned", g, P, a(2), a(3), a(4), a(6), a(7) + 2, None, T, H, 1e-6, 0)
run("fp8_q_overlaps_y", g, P, a(2), a(3), a(4), a(6), a(7), a(6), T, H, 1e-6, 0)
m = lb.lb_moe_finalize_fold_norm
run("moe_empty_ok", m, a(0), 32, a(1), a(8), 8, a(2), a(3), a(4), a(5), None, None, 0, H, 1e-6, None, 0)
run("moe_topk0", m, a(0), 32, a(1), a(8), 0, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, None, 0)
run("moe_topk_big", m, a(0), 32, a(1), a(8), 17, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, None, 0)
run("moe_no_idx", m, a(0), 32, None, a(8), 8, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, None, 0)
run("moe_no_w", m, a(0), 32, a(1), None, 8, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, None, 0)
run("moe_no_experts", m, None, 32, a(1), a(8), 8, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, None, 0)
run("moe_rows_negative", m, a(0), -1, a(1), a(8), 8, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, None, 0)
run("moe_idx_misaligned", m, a(0), 32, a(1) + 2, a(8), 8, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, None, 0)
run("moe_half_fp8", m, a(0), 32, a(1), a(8), 8, a(2), a(3), a(4), a(5), a(6), None, T, H, 1e-6, None, 0)
run("moe_flag_in_experts", m, a(0), 32, a(1), a(8), 8, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, a(0) + 64, 0)
# the routing promise: accepted by the MoE call (which then fails only for want of a
# device), refused by the others
run("moe_routing_ready_valid", lambda: m(a(0), 32, a(1), a(8), 8, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, None, 0, routing_ready=True))
mo = lb.Options(8, None)
results["moe_unknown_flag"] = L.lb_moe_finalize_fold_norm(a(0), 32, a(1), a(8), 8, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, None, lb.ctypes.byref(mo), None)
ro = lb.Options(lb.LB_OPT_ROUTING_READY, None)
results["fold_routing_ready"] = L.lb_fold_norm((lb._vp * 2)(a(0), a(1)), 2, a(2), a(3), a(4), a(5), T, H, 1e-6, lb.ctypes.byref(ro), None)
# the residual promise: accepted by every call
run("fold_residual_ready_valid", lambda: f(P, a(2), a(3), a(4), a(5), T, H, 1e-6, 0, residual_ready=True))
run("moe_both_promises_valid", lambda: m(a(0), 32, a(1), a(8), 8, a(2), a(3), a(4), a(5), None, None, T, H, 1e-6, None, 0, routing_ready=True, residual_ready=True))
s = lb.lb_slice_fold_norm
off, cnt = [0, 40, 552, 560], [37, 512, 5, 1470]
run("slice_empty_ok", s, P, 0, 8, 0, off[:0], cnt[:0], a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("slice_uneven", s, P, 2031, 8, 3, off, cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("slice_index_high", s, P, 2032, 8, 8, off, cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("slice_index_negative", s, P, 2032, 8, -1, off, cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("slice_zero_slices", s, P, 2032, 0, 0, off, cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("slice_sets_overlap", s, P, 2032, 8, 3, [0, 30, 552, 560], cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("slice_sets_descending", s, P, 2032, 8, 3, [560, 552, 40, 0], cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("slice_set_past_end", s, P, 2032, 8, 3, [0, 40, 552, 570], cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("slice_count_negative", s, P, 2032, 8, 3, off, [37, -1, 5, 1470], a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("slice_too_many_sets", s, P, 2032, 8, 3, list(range(65)), [0] * 65, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("slice_padding_only_ok", s, P, 2032, 8, 7, [0], [8], a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
v = lb.lb_slice_fold_norm_v
run("rsv_empty_set_ok", v, P, 2032, 1, [0, 40], [37, 0], a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("rsv_set_high", v, P, 2032, 4, off, cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("rsv_set_negative", v, P, 2032, -1, off, cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("rsv_no_sets", v, P, 2032, 0, [], [], a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("rsv_sets_overlap", v, P, 2032, 1, [0, 30, 552, 560], cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("rsv_set_past_end", v, P, 2000, 3, off, cnt, a(2), a(3), a(4), a(5), None, None, H, 1e-6, 0)
run("rsv_nothing_to_write", v, P, 2032, 3, off, cnt, a(2), None, a(4), None, None, None, H, 1e-6, 0)
print(json.dumps(results))
"""

EXPECTED = {
    "ok_empty": 0, "K_negative": 1, "K_too_big": 3, "partial_null": 1,
    "partial_misaligned": 2, "K0_no_residual": 1, "nothing_to_write": 1,
    "y_without_gamma": 1, "H_not_multiple_of_8": 3, "H_zero": 1, "H_too_big": 3,
    "T_negative": 1, "T_too_big": 3, "eps_negative": 1, "eps_nan": 1, "y_misaligned": 2,
    "gamma_misaligned": 2, "y_overlaps_partial": 1, "y_overlaps_residual_out": 1,
    "residual_out_shifted_over_in": 1, "in_place_empty_ok": 0,
    "empty_null_buffers_ok": 0, "empty_bad_H": 3, "empty_K_too_big": 3,
    "fp8_empty_ok": 0, "fp8_no_q": 1, "fp8_no_scale": 1, "fp8_no_gamma": 1,
    "fp8_scale_misaligned": 2, "fp8_q_overlaps_y": 1,
    "moe_empty_ok": 0, "moe_topk0": 1, "moe_topk_big": 3, "moe_no_idx": 1, "moe_no_w": 1,
    "moe_no_experts": 1, "moe_rows_negative": 1, "moe_idx_misaligned": 2,
    "moe_half_fp8": 1, "moe_flag_in_experts": 1,
    "moe_routing_ready_valid": 4, "moe_unknown_flag": 3, "fold_routing_ready": 3,
    "fold_residual_ready_valid": 4, "moe_both_promises_valid": 4,
    "slice_empty_ok": 0, "slice_uneven": 1, "slice_index_high": 1,
    "slice_index_negative": 1, "slice_zero_slices": 1, "slice_sets_overlap": 1,
    "slice_sets_descending": 1, "slice_set_past_end": 1, "slice_count_negative": 1,
    "slice_too_many_sets": 3, "slice_padding_only_ok": 0,
    "unknown_flag": 3, "snapshot_misaligned": 2, "snapshot_overlaps_y": 1,
    "snapshot_empty_ok": 0,
    "rsv_empty_set_ok": 0, "rsv_set_high": 1, "rsv_set_negative": 1, "rsv_no_sets": 1,
    "rsv_sets_overlap": 1, "rsv_set_past_end": 1, "rsv_nothing_to_write": 1,
}


def test_invalid_arguments_are_rejected_before_any_launch(lib):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _VALIDATION_SCRIPT, ROOT], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    assert got == EXPECTED


def test_binding_fails_loudly_without_the_library(tmp_path):
    code = ("import sys; sys.path.insert(0, sys.argv[1]);"
            "from layer_boundary_fusion_gb300 import lb\n"
            "try:\n    lb.load(sys.argv[2])\nexcept lb.LibraryMissing:\n    print('missing')\n")
    r = subprocess.run([sys.executable, "-c", code, ROOT, str(tmp_path / "none.so")],
                       capture_output=True, text=True, timeout=120)
    assert r.stdout.strip() == "missing"


class _FakeTensor:
    """Stands in for a torch tensor in the binding's argument checks (no GPU needed)."""

    def __init__(self, dtype="bfloat16", cuda=True, contiguous=True, device="cuda:0"):
        self.dtype = f"torch.{dtype}"
        self.is_cuda = cuda
        self._contiguous = contiguous
        self.device = device

    def is_contiguous(self):
        return self._contiguous

    def data_ptr(self):
        return 0x10000


def test_binding_rejects_bad_tensor_arguments(lib):
    m = lib._Marshal("lb_fold_norm")
    assert m(None, "bf16", "y_out") is None
    assert m(0x1234, "bf16", "y_out") == 0x1234            # raw addresses pass unchecked
    assert m(_FakeTensor("int16"), "bf16", "residual_in") == 0x10000
    with pytest.raises(ValueError, match="CUDA tensor"):
        m(_FakeTensor(cuda=False), "bf16", "residual_in")
    with pytest.raises(ValueError, match="contiguous"):
        m(_FakeTensor(contiguous=False), "bf16", "residual_in")
    with pytest.raises(TypeError, match="float32"):
        m(_FakeTensor("bfloat16"), "f32", "gamma")
    with pytest.raises(TypeError, match="uint8"):
        m(_FakeTensor("int8"), "u8", "q_out")
    with pytest.raises(ValueError, match="different devices"):
        m(_FakeTensor(device="cuda:1"), "bf16", "y_out")
