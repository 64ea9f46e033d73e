"""The stream kernel's bounded waits, run out on purpose on the GPU.

A test-only build of the library (liblb_test.so, LB_TEST_HOOKS) can make the stream
kernel post one row's bytes on its stage barrier without issuing the row's copies.  The
consumers of that row then wait until their bounded wait gives up (about a second):
the kernel must record LB_DEVICE_ERR_TIMEOUT, leave that CTA's unfinished rows
unwritten, finish every other CTA's rows correctly, return, and leave the context
usable, so that the next call completes and matches the oracle.  No fault, trap or hang
is involved: every wait in the kernel has an iteration and a time limit.

Runs in a child process, which loads the test build instead of liblb.so.
"""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu

_SCRIPT = r"""
import ctypes, json, sys, time
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np, torch
import oracle
from layer_boundary_fusion_gb300 import build, lb, workloads as wl
from parity_util import Guarded, dev_bits, f32
L = lb.load(build.build(test_hooks=True))
L.lb_test_withhold_row.argtypes = [ctypes.c_int64]
L.lb_test_withhold_row.restype = None
K, T, H, eps, ROW = 2, 300, int(sys.argv[2]), 1e-6, 5
PROMISE = sys.argv[3] == "1"      # residual promise: the rows' residual copies go out early
w = wl.fold_workload("timeout", K, T, H, seed=77)
want = oracle.fold_norm(w.partials, w.residual, w.gamma, eps)
P = [dev_bits(p) for p in w.partials]
R = dev_bits(w.residual)
G = torch.from_numpy(w.gamma).cuda()
plan = lb.lb_launch_plan(T, H, K + 1, torch.cuda.get_device_properties(0).multi_processor_count,
                         torch.cuda.get_device_properties(0).shared_memory_per_block_optin)

def call():
    ro, yo = Guarded(T, H, torch.bfloat16), Guarded(T, H, torch.bfloat16)
    lb.lb_fold_norm(P, R, ro.t, G, yo.t, T, H, eps, residual_ready=PROMISE)
    return ro, yo

def rows_state(ro, yo):
    # per row: "ok" (equal to the oracle), "untouched" (all sentinel), else "bad"
    r, y = ro.host(), yo.host()
    out = []
    for t in range(T):
        if np.array_equal(r[t], want["residual_out"][t]):
            g, e = f32(y[t]).astype(np.float64), f32(want["y"][t]).astype(np.float64)
            out.append("ok" if np.all(np.abs(g - e) <= 1e-2 * np.abs(e) + 1e-3) else "bad")
        elif np.all(np.isnan(f32(r[t]))) and np.all(np.isnan(f32(y[t]))):
            out.append("untouched")
        else:
            out.append("bad")
    return out

lb.lb_device_error(clear=True)
L.lb_test_withhold_row(ROW)
t0 = time.time()
ro, yo = call()
err = lb.lb_device_error(clear=True)          # synchronises
elapsed = time.time() - t0
L.lb_test_withhold_row(-1)
ro.check(); yo.check()                       # guard rows around the outputs untouched
state = rows_state(ro, yo)
cta = ROW % plan.grid
own = [t for t in range(T) if t % plan.grid == cta]
ro2, yo2 = call()
err2 = lb.lb_device_error(clear=True)
state2 = rows_state(ro2, yo2)
print(json.dumps({"kernel": plan.kernel, "chunks": plan.chunks, "err": err, "elapsed": elapsed,
                  "row": state[ROW], "others_ok": all(state[t] == "ok" for t in range(T) if t not in own),
                  "own": [state[t] for t in own], "err2": err2,
                  "after_ok": all(s == "ok" for s in state2)}))
"""


@pytest.mark.parametrize("H,chunks,promise", [(2048, 1, False), (4096, 1, False),
                                              (12288, 3, False), (4096, 1, True)])
# whole rows with a copy per producer lane, whole rows with lane 0 issuing, chunked rows,
# and whole rows whose residual copies went out before the rest (the withheld row's
# residual lands, its stage must still wait for the bytes that never come)
def test_a_withheld_row_times_out_and_the_context_survives(H, chunks, promise):
    r = subprocess.run([sys.executable, "-c", _SCRIPT, ROOT, str(H), "1" if promise else "0"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-4000:]
    got = json.loads(r.stdout.strip().splitlines()[-1])
    from layer_boundary_fusion_gb300 import lb
    assert got["kernel"] == lb.LB_KERNEL_STREAM and got["chunks"] == chunks
    assert got["err"] & lb.LB_DEVICE_ERR_TIMEOUT
    assert 0.5 < got["elapsed"] < 60.0               # the wait ran out after about a second
    assert got["row"] == "untouched"                 # the withheld row was never written
    assert got["others_ok"]                          # every other CTA finished its rows
    assert all(s in ("ok", "untouched") for s in got["own"])   # nothing half-written
    assert got["err2"] == 0 and got["after_ok"]      # the next call is complete and correct
