"""The library from plain C: a C program (tests/c/abi_fold_fp8.c) that includes only
include/lb.h and the CUDA runtime API, allocates device memory, calls lb_fold_norm_fp8
on its own stream and writes the outputs to files.  Its results must match the CPU
oracle like the binding's do (residual' bit-exact, FP8 codes and scales within the
parity bar).
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from conftest import ROOT
from layer_boundary_fusion_gb300 import workloads as wl
from parity_util import assert_bits_equal, assert_fp8_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def c_program(tmp_path_factory):
    from layer_boundary_fusion_gb300 import build
    lib = build.build()
    nvcc = build.nvcc()
    cuda_include = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))),
                                "include")
    out = tmp_path_factory.mktemp("c_abi")
    obj, exe = str(out / "abi_fold_fp8.o"), str(out / "abi_fold_fp8")
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-c", "-std=c11", "-Wall", "-Werror",
                    f"-I{os.path.join(ROOT, 'include')}", f"-I{cuda_include}",
                    os.path.join(ROOT, "tests", "c", "abi_fold_fp8.c"), "-o", obj], check=True)
    subprocess.run([nvcc, obj, f"-L{libdir}", "-llb", "-Xlinker", f"-rpath,{libdir}", "-o",
                    exe], check=True)
    return exe


@pytest.mark.parametrize("K,T,H", [(4, 2048, 4096), (3, 40, 1024)])   # stream, row kernel
def test_c_caller_matches_the_oracle(c_program, tmp_path, K, T, H):
    w = wl.fold_workload("c_abi", K, T, H, seed=300 + K, fp8=True, outlier_frac=0.01)
    for k, p in enumerate(w.partials):
        p.tofile(tmp_path / f"p{k}.bin")
    w.residual.tofile(tmp_path / "res.bin")
    w.gamma.tofile(tmp_path / "gamma.bin")
    r = subprocess.run([c_program, str(tmp_path), str(K), str(T), str(H), repr(w.eps)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr + r.stdout
    got_res = np.fromfile(tmp_path / "res_out.bin", np.uint16).reshape(T, H)
    got_q = np.fromfile(tmp_path / "q.bin", np.uint8).reshape(T, H)
    got_s = np.fromfile(tmp_path / "scale.bin", np.float32)
    want = oracle.fold_norm(w.partials, w.residual, w.gamma, w.eps, want_y=False,
                            want_fp8=True)
    assert_bits_equal(got_res, want["residual_out"], "C caller residual'")
    assert_fp8_close(got_q, want["q"], got_s, want["scale"], "C caller fp8")
