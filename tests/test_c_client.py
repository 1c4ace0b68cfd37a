"""The C ABI from a plain C11 program (tests/c/abi_client.c): it compiles
against include/memory_bound.h alone and links libmemory_bound.so.  Without a
GPU it checks the host-side argument paths; on a GPU it runs two chains on
seeded inputs and the outputs are compared with the CPU oracle."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    from memory_bound_gb300 import build as lib_build
    lib = lib_build.build()
    exe = str(tmp_path / "abi_client")
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c11", "-O1", "-Wall", "-Wextra", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c", "abi_client.c"),
           "-o", exe, "-L", libdir, "-lmemory_bound", "-Wl,-rpath," + libdir,
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def test_c_client_argument_checks(tmp_path):
    exe = _build(tmp_path)
    res = subprocess.run([exe, "args"], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr
    assert "args ok" in res.stdout


@pytest.mark.gpu
def test_c_client_runs_chains(tmp_path):
    exe = _build(tmp_path)
    n, rows, hidden = 100003, 37, 4096
    t = {"x": synth.normal(1301, 0, (n,)), "b1": synth.normal(1301, 1, (n,)),
         "b2": synth.normal(1301, 2, (n,)), "lx": synth.normal(1302, 0, (rows, hidden)),
         "lr": synth.normal(1302, 1, (rows, hidden)),
         "lw": synth.uniform(1302, 2, (hidden,), 0.5, 1.5),
         "lb": synth.normal(1302, 3, (hidden,), 0.0, 0.1)}
    for k, v in t.items():
        v.astype(np.float32).tofile(tmp_path / f"{k}.f32")
    res = subprocess.run([exe, "run", str(tmp_path), str(n), str(rows), str(hidden)],
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    y = np.fromfile(tmp_path / "y.f32", np.float32)
    assert np.array_equal(y.view(np.uint32),
                          oracle.add_relu_scale(t["x"], t["b1"], t["b2"], 0.5).view(np.uint32))
    lo = np.fromfile(tmp_path / "lout.f32", np.float32).reshape(rows, hidden)
    want = oracle.residual_layernorm_gelu(t["lx"], t["lr"], t["lw"], t["lb"], 1e-5)
    err = np.abs(lo.astype(np.float64) - want)
    assert np.all(err <= 1e-5 * np.maximum(np.abs(want), 1.0))
