"""Calls from several host threads at once, each on its own stream.

Runs in a fresh process, so the first calls also race on the library's
per-device set-up.  Four threads start together at a barrier and each calls
one chain repeatedly on its own CUDA stream; every result is then checked
against the CPU oracle.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys, threading
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import numpy as np, torch
import memory_bound_gb300 as mb, oracle, synth
from gpu_util import to_dev, to_host, assert_close
torch.cuda.set_device(0)
mb.load_library()
start = threading.Barrier(4)
errors = []

def run(fn):
    try:
        fn()
    except BaseException as e:      # reported by the main thread
        errors.append(repr(e))

def pointwise():
    x, b1, b2 = (synth.normal(1101, k, (1 << 20,)) for k in range(3))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = [to_dev(a) for a in (x, b1, b2)]
        start.wait()
        for _ in range(30):
            y = mb.fused_add_relu_scale(*d, 0.5)
    s.synchronize()
    assert np.array_equal(to_host(y).view(np.uint32), oracle.add_relu_scale(x, b1, b2, 0.5).view(np.uint32))

def layernorm():
    x, r = synth.normal(1102, 0, (512, 4096)), synth.normal(1102, 1, (512, 4096))
    w, b = synth.uniform(1102, 2, (4096,), 0.5, 1.5), synth.normal(1102, 3, (4096,), 0, 0.1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = [to_dev(a) for a in (x, r, w, b)]
        start.wait()
        for _ in range(30):
            out = mb.fused_residual_layernorm_gelu(*d, 1e-5)
    s.synchronize()
    assert_close(to_host(out), oracle.residual_layernorm_gelu(x, r, w, b, 1e-5))

def softmax():
    x = synth.normal(1103, 0, (300, 2048), 0.0, 2.0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = to_dev(x)
        start.wait()
        for _ in range(30):
            y = mb.fused_row_softmax(d)
    s.synchronize()
    g, w = to_host(y).astype(np.float64), oracle.row_softmax(x).astype(np.float64)
    assert np.all(np.abs(g - w) <= 1e-5 * w + 2.0 ** -126)

def inductor():
    x = synth.normal(1104, 0, (1024, 1024))
    bias, gamma, beta = (synth.normal(1104, 1, (1024,), 0, 0.1), synth.uniform(1104, 2, (1024,), 0.5, 1.5),
                         synth.normal(1104, 3, (1024,), 0, 0.1))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = [to_dev(a) for a in (x, bias, gamma, beta)]
        start.wait()
        for _ in range(30):
            y = mb.fused_bias_relu_branch_mean_epilogue(*d, 1.1, 0.1)
    s.synchronize()
    assert_close(to_host(y), oracle.bias_relu_branch_mean_epilogue(x, bias, gamma, beta))

ts = [threading.Thread(target=run, args=(f,)) for f in (pointwise, layernorm, softmax, inductor)]
for t in ts: t.start()
for t in ts: t.join()
torch.cuda.synchronize()
assert mb.device_error() == 0
if errors:
    print("\n".join(errors)); sys.exit(1)
print("concurrent ok")
'''


def test_threads_on_separate_streams():
    from memory_bound_gb300 import build as lib_build
    lib_build.build()
    code = "ROOT = %r\n" % ROOT + SCRIPT
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-3000:] + res.stderr[-3000:]
    assert "concurrent ok" in res.stdout


def test_path_setter_racing_calls():
    """One thread keeps switching the process-wide row path and launch shape
    while another calls the LayerNorm chain on fixed inputs: every call reads
    the setting whole (it is copied under the library's lock), so every
    result matches the oracle whichever engine ran it."""
    import threading

    import numpy as np
    import torch

    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import memory_bound_gb300 as mb
    import oracle
    import synth
    from gpu_util import assert_close, to_dev, to_host

    torch.cuda.set_device(0)
    x, r = synth.normal(1201, 0, (64, 4096)), synth.normal(1201, 1, (64, 4096))
    w, b = synth.uniform(1201, 2, (4096,), 0.5, 1.5), synth.normal(1201, 3, (4096,), 0, 0.1)
    want = oracle.residual_layernorm_gelu(x, r, w, b, 1e-5)
    d = [to_dev(a) for a in (x, r, w, b)]
    stop = threading.Event()
    shapes = [("auto", 0, 0, 0), ("direct", 2, 0, 1), ("staged", 3, 2, 2), ("warp", 0, 0, 0),
              ("cluster", 0, 2, 0), ("direct", 0, 0, 8)]

    def flip():
        k = 0
        while not stop.is_set():
            mb.set_row_path(*shapes[k % len(shapes)])
            k += 1

    t = threading.Thread(target=flip)
    t.start()
    try:
        outs = []
        for _ in range(200):
            outs.append(mb.fused_residual_layernorm_gelu(*d, 1e-5))
        torch.cuda.synchronize()
    finally:
        stop.set()
        t.join()
        mb.set_row_path("auto")
    for o in outs:
        assert_close(to_host(o), want)
    assert mb.device_error() == 0
