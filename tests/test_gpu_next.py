"""Parity of the further chains built on the row engines (the scope table's
"next" rows) with the CPU oracle: the LayerNorm family (optional residual,
residual-stream output, activation none / relu / gelu-tanh), row softmax,
and the TorchInductor chain with bf16 I/O."""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth
from synth import workloads as W

from gpu_util import (assert_bitexact, assert_close, bf16_to_f64, check_guard, guarded_empty,
                      report, to_dev, to_host)
from row_blocks import map_row_blocks, worst

pytestmark = pytest.mark.gpu

PATHS = ["auto", "warp", "direct", "staged"]
ACTS = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU}


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


def assert_rel(got, want, bf16, what=""):
    """Softmax outputs are probabilities, small but never near a cancellation:
    a pure relative bound (fp32: 1e-5, bf16: 1e-2) with a floor only at the
    fp32 underflow threshold."""
    if bf16:
        g, w, rtol = bf16_to_f64(got), bf16_to_f64(want), 1e-2
    else:
        g, w, rtol = np.asarray(got, np.float64), np.asarray(want, np.float64), 1e-5
    err = np.abs(g - w)
    lim = rtol * np.abs(w) + 2.0 ** -126
    bad = err > lim
    assert not bad.any(), (f"{what}: {int(bad.sum())} out of tolerance, worst rel "
                           f"{float((err / np.maximum(np.abs(w), 1e-38)).max()):.3e}")
    big = np.abs(w) >= 2.0 ** -100
    return float((err[big] / np.abs(w[big])).max()) if big.any() else 0.0


def _ln_inputs(rows, hidden, seed, bf16):
    dt = "bf16" if bf16 else "f32"
    return (synth.normal(seed, 0, (rows, hidden), dtype=dt),
            synth.normal(seed, 1, (rows, hidden), dtype=dt),
            synth.uniform(seed, 2, (hidden,), 0.5, 1.5, dtype=dt),
            synth.normal(seed, 3, (hidden,), 0.0, 0.1, dtype=dt))


# --------------------------------------------------------------------------
# LayerNorm family
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(1, 1), (3, 2), (5, 33), (4, 1000), (9, 4096), (6, 4099),
                                   (3, 8192), (2, 32768), (300, 4096)])
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("res", [True, False], ids=["res", "nores"])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_layernorm_act(shape, path, res, bf16, row_path):
    rows, hidden = shape
    row_path(path)
    x, r, w, b = _ln_inputs(rows, hidden, 500 + hidden + rows, bf16)
    dt = torch.bfloat16 if bf16 else torch.float32
    for act in ("none", "relu", "gelu_tanh"):
        obuf, out = guarded_empty(shape, dt)
        hbuf, h = guarded_empty(shape, dt)
        mb.fused_layernorm_act(to_dev(x, bf16), to_dev(r, bf16) if res else None,
                               to_dev(w, bf16), to_dev(b, bf16), eps=1e-5, act=act,
                               out=out, h_out=h)
        want, want_h = oracle.layernorm_act(x, r if res else None, w, b, 1e-5, ACTS[act],
                                            want_h=True)
        assert_close(to_host(out), want, bf16=bf16, what=f"{shape} {path} {act}")
        assert_bitexact(to_host(h), want_h, f"h {shape} {path}")
        check_guard(obuf)
        check_guard(hbuf)


def test_layernorm_act_without_h_matches_the_gelu_entry_point():
    """fused_layernorm_act(r, gelu) is the same chain as
    fused_residual_layernorm_gelu: both within the bar of one oracle."""
    x, r, w, b = _ln_inputs(64, 4096, 77, False)
    out = mb.fused_layernorm_act(to_dev(x), to_dev(r), to_dev(w), to_dev(b))
    ref = mb.fused_residual_layernorm_gelu(to_dev(x), to_dev(r), to_dev(w), to_dev(b))
    want = oracle.residual_layernorm_gelu(x, r, w, b, 1e-5)
    assert_close(to_host(out), want)
    assert_close(to_host(ref), want)


@pytest.mark.parametrize("w", [W.LNACT_RES_BF16, W.LNACT_RELU_F32], ids=lambda w: w.name)
def test_layernorm_act_workload_full_size(w):
    bf16 = w.dtype == "bf16"
    t = w.generate_all()
    res = w.params["residual"]
    d = {k: to_dev(v, bf16) for k, v in t.items()}
    out, h = mb.fused_layernorm_act(d["x"], d.get("r"), d["w"], d["b"], eps=1e-5,
                                    act=w.params["act"], want_h=True)
    torch.cuda.synchronize()
    got, got_h = to_host(out), to_host(h)

    def block(r0, r1):
        want, want_h = oracle.layernorm_act(t["x"][r0:r1], t["r"][r0:r1] if res else None,
                                            t["w"], t["b"], 1e-5, ACTS[w.params["act"]],
                                            want_h=True)
        assert_bitexact(got_h[r0:r1], want_h, f"h rows {r0}:{r1}")
        return assert_close(got[r0:r1], want, bf16=bf16, what=f"{w.name} rows {r0}:{r1}")

    err, ratio = worst(map_row_blocks(w.rows, block))
    report(w.name, max_abs_err=err, max_err_over_bar=ratio)


# --------------------------------------------------------------------------
# row softmax
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(1, 1), (3, 2), (5, 33), (4, 1000), (9, 4096), (6, 4099),
                                   (3, 8192), (2, 32768), (300, 1024)])
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_softmax(shape, path, bf16, row_path):
    rows, cols = shape
    row_path(path)
    x = synth.normal(700 + cols, 0, shape, 0.0, 3.0, dtype="bf16" if bf16 else "f32")
    buf, y = guarded_empty(shape, torch.bfloat16 if bf16 else torch.float32)
    mb.fused_row_softmax(to_dev(x, bf16), out=y)
    assert_rel(to_host(y), oracle.row_softmax(x), bf16, f"{shape} {path}")
    check_guard(buf)


def test_softmax_extreme_rows():
    """Shifts by 1000, a row spanning +-1000 and constant rows."""
    q = np.round(synth.normal(71, 0, (4, 512)) * 1024) / 1024
    x = np.concatenate([q, q + 1000.0, np.full((1, 512), 2.5), np.zeros((1, 512))]).astype(np.float32)
    x[-1, 7], x[-1, 8] = 1000.0, -1000.0
    y = to_host(mb.fused_row_softmax(to_dev(x)))
    want = oracle.row_softmax(x)
    assert_rel(y, want, False, "extreme rows")
    assert np.all(np.isfinite(y))


def test_softmax_workload_full_size():
    """[P1] §4.1's score matrix (32 heads x 4096 queries, 4096 keys): every
    row against the oracle at the pure relative bar."""
    w = W.SOFTMAX_F32
    x = synth.normal(w.seed, 0, (w.rows, w.cols))
    y = mb.fused_row_softmax(to_dev(x))
    torch.cuda.synchronize()
    got = to_host(y)

    def block(r0, r1):
        return assert_rel(got[r0:r1], oracle.row_softmax(x[r0:r1]), False,
                          f"{w.name} rows {r0}:{r1}")

    rel = max(map_row_blocks(w.rows, block))
    report(w.name, max_rel_err=rel)
    sums = got.astype(np.float64).sum(axis=1)
    assert np.all(np.abs(sums - 1.0) <= 1e-4)


# --------------------------------------------------------------------------
# TorchInductor chain, bf16 I/O
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(1, 1), (3, 5), (7, 1000), (5, 1027), (1024, 1024),
                                   (33, 4096), (4, 32768)])
@pytest.mark.parametrize("path", PATHS)
def test_inductor_bf16(shape, path, row_path):
    rows, cols = shape
    row_path(path)
    x = synth.normal(800 + cols, 0, shape, dtype="bf16")
    bias = synth.normal(800 + cols, 1, (cols,), 0.0, 0.1, dtype="bf16")
    gamma = synth.uniform(800 + cols, 2, (cols,), 0.5, 1.5, dtype="bf16")
    beta = synth.normal(800 + cols, 3, (cols,), 0.0, 0.1, dtype="bf16")
    buf, y = guarded_empty(shape, torch.bfloat16)
    mb.fused_bias_relu_branch_mean_epilogue(to_dev(x, True), to_dev(bias, True),
                                            to_dev(gamma, True), to_dev(beta, True),
                                            1.1, 0.1, out=y)
    want = oracle.bias_relu_branch_mean_epilogue_bf16(x, bias, gamma, beta)
    assert_close(to_host(y), want, bf16=True, what=f"{shape} {path}")
    check_guard(buf)


def test_inductor_bf16_workload_full_size():
    """The benchmark's bf16 Inductor workload (its own seed), every element
    against the oracle."""
    w = W.INDUCTOR_BF16
    t = w.generate_all()
    y = mb.fused_bias_relu_branch_mean_epilogue(to_dev(t["x"], True), to_dev(t["bias"], True),
                                                to_dev(t["gamma"], True), to_dev(t["beta"], True),
                                                w.params["x_scale"], w.params["branch_scale"])
    want = oracle.bias_relu_branch_mean_epilogue_bf16(t["x"], t["bias"], t["gamma"], t["beta"],
                                                      w.params["x_scale"],
                                                      w.params["branch_scale"])
    err, ratio = assert_close(to_host(y), want, bf16=True, what=w.name)
    report(w.name, max_abs_err=err, max_err_over_bar=ratio)
