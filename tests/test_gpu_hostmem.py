"""Zero-copy calls: tensors in pinned (page-locked) host memory, read and
written by the kernels over the host link, checked against the CPU oracle.

Row inputs held in host memory must never reach the bulk-async staged path
(it copies device memory only): the library checks where the rows live when
it plans that path and falls back to a plain-load path, also when the staged
path is forced.  Outputs get canaries on both sides, in host memory too.
"""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth
from synth import workloads as W

from gpu_util import (assert_bitexact, assert_close, bf16_to_f64, check_guard, report, to_dev,
                      to_host)
from row_blocks import map_row_blocks, worst

pytestmark = pytest.mark.gpu

# where each tensor of a call lives: row tensors (inputs and outputs) and
# per-column vectors
PLACEMENTS = {
    "all_host": dict(rows="host", cols="host", out="host"),
    "rows_host": dict(rows="host", cols="dev", out="host"),
    "in_host_out_dev": dict(rows="host", cols="dev", out="dev"),
    "in_dev_out_host": dict(rows="dev", cols="dev", out="host"),
}


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from memory_bound_gb300 import build as lib_build
    lib_build.build()
    torch.cuda.set_device(0)
    mb.set_row_path("auto")
    yield
    mb.set_row_path("auto")
    torch.cuda.synchronize()
    assert mb.device_error() == 0


@pytest.fixture
def row_path():
    yield mb.set_row_path
    mb.set_row_path("auto")


def to_pinned(a, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16
                         else np.ascontiguousarray(a)).pin_memory()
    return t.view(torch.bfloat16) if bf16 else t


def place(a, where, bf16=False):
    return to_pinned(a, bf16) if where == "host" else to_dev(a, bf16)


def guarded(shape, dtype, where, guard=64):
    """An output in pinned host or device memory with canaries on both sides."""
    n = int(np.prod(shape))
    if where == "host":
        buf = torch.empty(n + 2 * guard, dtype=dtype, pin_memory=True)
    else:
        buf = torch.empty(n + 2 * guard, dtype=dtype, device="cuda")
    if dtype == torch.bfloat16:
        buf.view(torch.int16).fill_(0x7FA5)
    else:
        buf.view(torch.int32).fill_(0x7FA5A5A5)
    return buf, buf[guard:guard + n].view(shape)


def assert_rel(got, want, bf16, what=""):
    if bf16:
        g, w, rtol = bf16_to_f64(got), bf16_to_f64(want), 1e-2
    else:
        g, w, rtol = np.asarray(got, np.float64), np.asarray(want, np.float64), 1e-5
    bad = np.abs(g - w) > rtol * np.abs(w) + 2.0 ** -126
    assert not bad.any(), f"{what}: {int(bad.sum())} out of tolerance"


@pytest.mark.parametrize("placement", sorted(PLACEMENTS))
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 4099, 3 * (1 << 20) + 5])
def test_pointwise(placement, bf16, n):
    pl = PLACEMENTS[placement]
    dt = "bf16" if bf16 else "f32"
    x, b1, b2 = (synth.normal(1201, k, (n,), dtype=dt) for k in range(3))
    buf, y = guarded((n,), torch.bfloat16 if bf16 else torch.float32, pl["out"])
    mb.fused_add_relu_scale(place(x, pl["rows"], bf16), place(b1, pl["cols"], bf16),
                            place(b2, pl["rows"], bf16), 0.5, out=y)
    torch.cuda.synchronize()
    assert_bitexact(to_host(y), oracle.add_relu_scale(x, b1, b2, 0.5), f"{placement} n={n}")
    check_guard(buf)


LN_SHAPES = [(1, 1), (5, 33), (300, 4096), (257, 4099), (3, 8192), (2, 32768), (4, 131072)]


@pytest.mark.parametrize("shape", LN_SHAPES)
@pytest.mark.parametrize("path", ["auto", "staged"])
@pytest.mark.parametrize("placement", ["all_host", "rows_host", "in_host_out_dev"])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_residual_layernorm_gelu(shape, path, placement, bf16, row_path):
    """Forcing the staged path with rows in host memory still takes a
    plain-load path (and stays correct)."""
    pl = PLACEMENTS[placement]
    rows, hidden = shape
    row_path(path)
    dt = "bf16" if bf16 else "f32"
    seed = 1300 + rows + hidden
    x, r = synth.normal(seed, 0, shape, dtype=dt), synth.normal(seed, 1, shape, dtype=dt)
    w = synth.uniform(seed, 2, (hidden,), 0.5, 1.5, dtype=dt)
    b = synth.normal(seed, 3, (hidden,), 0.0, 0.1, dtype=dt)
    buf, out = guarded(shape, torch.bfloat16 if bf16 else torch.float32, pl["out"])
    mb.fused_residual_layernorm_gelu(place(x, pl["rows"], bf16), place(r, pl["rows"], bf16),
                                     place(w, pl["cols"], bf16), place(b, pl["cols"], bf16),
                                     1e-5, out=out)
    torch.cuda.synchronize()
    assert_close(to_host(out), oracle.residual_layernorm_gelu(x, r, w, b, 1e-5), bf16=bf16,
                 what=f"{shape} {path} {placement}")
    check_guard(buf)


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_layernorm_act_with_residual_stream(bf16, row_path):
    row_path("staged")
    shape = (129, 4096)
    dt = "bf16" if bf16 else "f32"
    tdt = torch.bfloat16 if bf16 else torch.float32
    x, r = synth.normal(1401, 0, shape, dtype=dt), synth.normal(1401, 1, shape, dtype=dt)
    w = synth.uniform(1401, 2, (4096,), 0.5, 1.5, dtype=dt)
    b = synth.normal(1401, 3, (4096,), 0.0, 0.1, dtype=dt)
    obuf, out = guarded(shape, tdt, "host")
    hbuf, h = guarded(shape, tdt, "host")
    mb.fused_layernorm_act(to_pinned(x, bf16), to_pinned(r, bf16), to_dev(w, bf16),
                           to_dev(b, bf16), eps=1e-5, act="relu", out=out, h_out=h)
    torch.cuda.synchronize()
    want, want_h = oracle.layernorm_act(x, r, w, b, 1e-5, oracle.ACT_RELU, want_h=True)
    assert_close(to_host(out), want, bf16=bf16)
    assert_bitexact(to_host(h), want_h, "h")
    check_guard(obuf)
    check_guard(hbuf)


@pytest.mark.parametrize("path", ["auto", "staged"])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_softmax(path, bf16, row_path):
    row_path(path)
    shape = (300, 4096)
    x = synth.normal(1501, 0, shape, 0.0, 3.0, dtype="bf16" if bf16 else "f32")
    buf, y = guarded(shape, torch.bfloat16 if bf16 else torch.float32, "host")
    mb.fused_row_softmax(to_pinned(x, bf16), out=y)
    torch.cuda.synchronize()
    assert_rel(to_host(y), oracle.row_softmax(x), bf16, f"softmax {path}")
    check_guard(buf)


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_inductor_chain(bf16):
    dt = "bf16" if bf16 else "f32"
    x = synth.normal(1601, 0, (1024, 1024), dtype=dt)
    bias = synth.normal(1601, 1, (1024,), 0.0, 0.1, dtype=dt)
    gamma = synth.uniform(1601, 2, (1024,), 0.5, 1.5, dtype=dt)
    beta = synth.normal(1601, 3, (1024,), 0.0, 0.1, dtype=dt)
    buf, y = guarded((1024, 1024), torch.bfloat16 if bf16 else torch.float32, "host")
    mb.fused_bias_relu_branch_mean_epilogue(to_pinned(x, bf16), to_dev(bias, bf16),
                                            to_dev(gamma, bf16), to_dev(beta, bf16), 1.1, 0.1,
                                            out=y)
    torch.cuda.synchronize()
    fn = oracle.bias_relu_branch_mean_epilogue_bf16 if bf16 else oracle.bias_relu_branch_mean_epilogue
    assert_close(to_host(y), fn(x, bias, gamma, beta, 1.1, 0.1), bf16=bf16)
    check_guard(buf)


def test_graph_capture_of_host_and_staged_calls():
    """The residence check runs while a graph is being captured (global
    capture mode): a staged call on device rows and a call on host rows."""
    shape = (512, 4096)
    x, r = synth.normal(1701, 0, shape), synth.normal(1701, 1, shape)
    w, b = synth.uniform(1701, 2, (4096,), 0.5, 1.5), synth.normal(1701, 3, (4096,), 0.0, 0.1)
    dx, dr, dw, db = (to_dev(a) for a in (x, r, w, b))
    hx, hr = to_pinned(x), to_pinned(r)
    dout = torch.empty(shape, device="cuda")
    hout = torch.empty(shape, pin_memory=True)
    assert mb.row_plan("ln", "f32", *shape)["path"] == "staged"
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                   # warm-up outside the capture
        mb.fused_residual_layernorm_gelu(dx, dr, dw, db, out=dout)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mb.fused_residual_layernorm_gelu(dx, dr, dw, db, out=dout)
        mb.fused_residual_layernorm_gelu(hx, hr, dw, db, out=hout)
    dout.zero_()
    hout.zero_()
    g.replay()
    torch.cuda.synchronize()
    want = oracle.residual_layernorm_gelu(x, r, w, b, 1e-5)
    assert_close(to_host(dout), want)
    assert_close(to_host(hout), want)


def test_full_size_ln_bf16_from_host():
    """The 32768 x 8192 bf16 workload with its rows in pinned host memory
    (1.5 GB over the host link), every row against the oracle."""
    w = W.LN_BF16
    t = w.generate_all()
    out = mb.fused_residual_layernorm_gelu(to_pinned(t["x"], True), to_pinned(t["r"], True),
                                           to_dev(t["w"], True), to_dev(t["b"], True), 1e-5)
    assert out.device.type == "cpu" and out.is_pinned()
    torch.cuda.synchronize()
    got = to_host(out)

    def block(r0, r1):
        want = oracle.residual_layernorm_gelu(t["x"][r0:r1], t["r"][r0:r1], t["w"], t["b"], 1e-5)
        return assert_close(got[r0:r1], want, bf16=True, what=f"{w.name} rows {r0}:{r1}")

    err, ratio = worst(map_row_blocks(w.rows, block))
    report(w.name + " (host memory)", max_abs_err=err, max_err_over_bar=ratio)
