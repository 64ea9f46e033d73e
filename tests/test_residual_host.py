"""Residual stream (include/lb_residual.h) on the host: the states, handles and errors of
"Layer boundaries", sections "Residual stream", "Enter and leave the layer stack",
"Auxiliary capture and extra contributions" and "Integration checklist and common
errors".  No GPU: state errors are decided before any launch, and an empty batch (T = 0)
runs every transition without launching anything.  The ctypes struct is checked against
the C header's layout with gcc."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from layer_boundary_fusion_gb300 import build, lb
    build.build()
    return lb


def test_struct_layout_matches_the_header(lib, tmp_path):
    fields = [name for name, _ in lib.ResidualStream._fields_]
    src = tmp_path / "layout.c"
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "lb_residual.h"',
             'int main(void) {', '  printf("%zu\\n", sizeof(lb_residual_stream));']
    lines += [f'  printf("%zu\\n", offsetof(lb_residual_stream, {f}));' for f in fields]
    lines += ['  return 0;', '}']
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", f"-I{os.path.join(ROOT, 'include')}", str(src), "-o",
                    str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    import ctypes
    want = [ctypes.sizeof(lib.ResidualStream)] + [getattr(lib.ResidualStream, f).offset
                                                 for f in fields]
    assert got == want


_SCRIPT = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
from layer_boundary_fusion_gb300 import lb
lb.load()
A = 1 << 32
def a(i): return A + i * (1 << 28)
out = {}
def status(fn, *args, **kw):
    try:
        return fn(*args, **kw)
    except lb.LBError as e:
        return -e.status
H = 64

# -- errors on a stream of 4 rows, decided before any launch ------------------------
s = lb.ResidualStream()
lb.lb_residual_init(s, a(0), 4, H)
out["leave_before_start"] = status(lb.lb_residual_leave, s, 0, [a(1)])
out["take_before_start"] = status(lb.lb_residual_take_output, s, 0)
h0 = lb.lb_residual_start(s)
out["initial_state"] = s.state
out["prepare_initial"] = status(lb.lb_residual_prepare, s, h0, a(5), a(6), None, None, 1e-6)
out["take_initial"] = status(lb.lb_residual_take_output, s, h0)
out["foreign_handle"] = status(lb.lb_residual_leave, s, h0 + 7, [a(1)])
out["leave_K0"] = status(lb.lb_residual_leave, s, h0, [])
out["leave_K17"] = status(lb.lb_residual_leave, s, h0, [a(i) for i in range(1, 18)])
h1 = lb.lb_residual_leave(s, h0, [a(1), a(2)])
out["pending_state"] = (s.state, s.K, s.kind)
out["stale_handle"] = status(lb.lb_residual_fold, s, h0)
out["leave_while_pending"] = status(lb.lb_residual_leave, s, h1, [a(3)])
out["take_while_pending"] = status(lb.lb_residual_take_output, s, h1)
h2 = lb.lb_residual_add_to_output(s, h1, a(3))
out["after_add_to_output"] = (s.state, s.K)
for i in range(13):
    h2 = lb.lb_residual_add_to_output(s, h2, a(4))
out["add_to_output_full"] = status(lb.lb_residual_add_to_output, s, h2, a(4))
h3 = lb.lb_residual_written(s, h2, a(9))
out["written"] = (s.state, s.K, s.has_residual, s.residual == a(9))
out["leave_moe_topk17"] = status(lb.lb_residual_leave_moe, s, h3, a(10), 32, a(11), a(12), 17)
h4 = lb.lb_residual_leave_moe(s, h3, a(10), 32, a(11), a(12), 8)
out["moe_pending"] = (s.state, s.kind, s.topk)
out["add_to_moe_handoff"] = status(lb.lb_residual_add_to_output, s, h4, a(4))
out["prepare_no_output"] = status(lb.lb_residual_prepare, s, h4, a(5), None, None, None, 1e-6)
h5 = lb.lb_residual_written(s, h4, a(9))
out["take_output"] = lb.lb_residual_take_output(s, h5) == a(9)
out["released"] = (s.started, status(lb.lb_residual_leave, s, h5 + 1, [a(1)]))

# -- every transition on an empty batch (T = 0: the boundary calls launch nothing) ----
e = lb.ResidualStream()
lb.lb_residual_init(e, None, 0, H)
g = lb.lb_residual_start(e)
trace = []
g = lb.lb_residual_leave(e, g, [None]); trace.append((e.state, e.has_residual, e.K))
g = lb.lb_residual_fold(e, g); trace.append((e.state, e.has_residual, e.K))
g = lb.lb_residual_prepare(e, g, a(5), a(6), None, None, 1e-6); trace.append((e.state, e.has_residual, e.K))
g = lb.lb_residual_leave(e, g, [None, None]); trace.append((e.state, e.has_residual, e.K))
g = lb.lb_residual_complete_output(e, g, None); trace.append((e.state, e.has_residual, e.K))
g = lb.lb_residual_add_to_output(e, g, None); trace.append((e.state, e.has_residual, e.K))
g = lb.lb_residual_prepare(e, g, a(5), None, a(7), a(8), 1e-6); trace.append((e.state, e.has_residual, e.K))
g = lb.lb_residual_leave_moe(e, g, None, 0, None, None, 8); trace.append((e.state, e.has_residual, e.kind))
lb.lb_residual_norm(e, g, a(5), a(6), None, None, 1e-6, gemma=True); trace.append((e.state, e.started))
out["empty_trace"] = trace
print(json.dumps(out))
"""

_PENDING, _WRITTEN, _INITIAL = 2, 1, 0


def test_residual_stream_states_and_errors(lib):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _SCRIPT, ROOT], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    NS, FO, UP, IA, UN = -lib.LB_ERR_NOT_STARTED, -lib.LB_ERR_FOREIGN_OUTPUT, \
        -lib.LB_ERR_UPDATE_PENDING, -lib.LB_ERR_INVALID_ARGUMENT, -lib.LB_ERR_UNSUPPORTED
    # "start the layer stack before entering a stage"
    assert got["leave_before_start"] == NS and got["take_before_start"] == NS
    assert got["initial_state"] == _INITIAL
    assert got["prepare_initial"] == IA and got["take_initial"] == IA
    # "output does not belong to this residual stream": any other handle is refused
    assert got["foreign_handle"] == FO and got["stale_handle"] == FO
    assert got["leave_K0"] == IA and got["leave_K17"] == UN
    assert got["pending_state"] == [_PENDING, 2, lib.LB_CONTRIB_PARTIALS]
    # a second contribution may not overwrite an owed one
    assert got["leave_while_pending"] == UP
    # "write the residual update before taking the final output"
    assert got["take_while_pending"] == UP
    # add_to_output: the extra buffer joins the owed sum once; the update stays pending
    assert got["after_add_to_output"] == [_PENDING, 3]
    assert got["add_to_output_full"] == UN
    # written(): a written stream on the given residual; the contribution is discarded
    assert got["written"] == [_WRITTEN, 0, 1, True]
    assert got["moe_pending"] == [_PENDING, lib.LB_CONTRIB_MOE, 8]
    assert got["add_to_moe_handoff"] == UN and got["leave_moe_topk17"] == UN
    assert got["prepare_no_output"] == IA
    # take_output releases the stream; the stack must start again
    assert got["take_output"] is True
    assert got["released"] == [0, NS]
    assert got["empty_trace"] == [
        [_PENDING, 0, 1],          # leave: owed sum, no residual yet
        [_WRITTEN, 1, 0],          # fold: the sum becomes the residual (enter)
        [_WRITTEN, 1, 0],          # prepare on a written stream: read only
        [_PENDING, 1, 2],          # leave
        [_PENDING, 1, 1],          # complete_output: owed as one completed buffer
        [_PENDING, 1, 2],          # add_to_output: one more owed buffer
        [_WRITTEN, 1, 0],          # prepare (FP8 read): update and read
        [_PENDING, 1, lib.LB_CONTRIB_MOE],   # a MoE finalize handoff
        [_WRITTEN, 0],             # final norm: finalize + fold + Gemma norm, released
    ]
