"""Rows that are not whole 16-byte vectors (the scalar path of every row
engine): lengths from a few thousand to past one CTA's reach, where the
one-CTA engine's 16- and 32-slot forms (bounded at 512 threads, so they hold
their values in registers) and then the cluster engine serve them; plain and
offset views; every chain against the oracle.  The full ragged workload
(8192 x 4099 fp32, the benchmark's row) is checked on every element."""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth
from synth import workloads as W

from gpu_util import assert_close, report, to_dev, to_host
from row_blocks import map_row_blocks, worst

pytestmark = pytest.mark.gpu

LENGTHS = [4099, 8195, 12291, 16383, 16385, 24579, 32767]


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


def _dev(a, bf16, offset):
    """A device copy of a, starting `offset` elements into its allocation."""
    d = to_dev(a, bf16)
    if not offset:
        return d
    flat = torch.empty(d.numel() + offset, dtype=d.dtype, device=d.device)
    v = flat[offset:].view(d.shape)
    v.copy_(d)
    return v


def _rows(rows, cols, seed, bf16, n):
    dt = "bf16" if bf16 else "f32"
    return [synth.normal(seed, k, (rows, cols), dtype=dt) for k in range(n)]


def _vecs(cols, seed, bf16):
    dt = "bf16" if bf16 else "f32"
    return (synth.uniform(seed, 2, (cols,), 0.5, 1.5, dtype=dt),
            synth.normal(seed, 3, (cols,), 0.0, 0.1, dtype=dt))


@pytest.mark.parametrize("cols", LENGTHS)
@pytest.mark.parametrize("path", ["auto", "direct", "cluster"])
@pytest.mark.parametrize("offset", [0, 1], ids=["base", "offset"])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_ln_gelu_unaligned(cols, path, offset, bf16):
    mb.set_row_path(path)
    try:
        rows = 37
        x, r = _rows(rows, cols, cols + 1, bf16, 2)
        w, b = _vecs(cols, cols + 1, bf16)
        out = mb.fused_residual_layernorm_gelu(_dev(x, bf16, offset), _dev(r, bf16, offset),
                                               to_dev(w, bf16), to_dev(b, bf16), 1e-5)
        assert_close(to_host(out), oracle.residual_layernorm_gelu(x, r, w, b, 1e-5), bf16=bf16,
                     what=f"{cols} {path} offset={offset}")
    finally:
        mb.set_row_path("auto")


@pytest.mark.parametrize("cols", LENGTHS)
@pytest.mark.parametrize("chain", ["inductor", "lnact_relu", "lnact_dropout", "softmax"])
def test_chains_unaligned(cols, chain):
    rows = 29
    if chain == "inductor":
        x = synth.normal(cols, 0, (rows, cols))
        bias = synth.normal(cols, 1, (cols,), 0.0, 0.1)
        gamma = synth.uniform(cols, 2, (cols,), 0.5, 1.5)
        beta = synth.normal(cols, 3, (cols,), 0.0, 0.1)
        y = mb.fused_bias_relu_branch_mean_epilogue(_dev(x, False, 1), to_dev(bias),
                                                    to_dev(gamma), to_dev(beta), 1.1, 0.1)
        assert_close(to_host(y), oracle.bias_relu_branch_mean_epilogue(x, bias, gamma, beta),
                     what=f"inductor {cols}")
    elif chain.startswith("lnact"):
        x = synth.normal(cols + 5, 0, (rows, cols))
        w, b = _vecs(cols, cols + 5, False)
        p = 0.1 if chain == "lnact_dropout" else 0.0
        out = mb.fused_layernorm_act(_dev(x, False, 1), None, to_dev(w), to_dev(b), act="relu",
                                     p=p, seed=99)
        want, _, _, _ = oracle.layernorm_act_ex(x, None, w, b, 1e-5, oracle.ACT_RELU, p=p, seed=99)
        got = to_host(out)
        if p:
            keep = oracle.dropout_mask(99, 0, 0, x.size, p).reshape(x.shape)
            assert np.all(got[~keep] == 0)
        assert_close(got, want, what=f"{chain} {cols}")
    else:
        x = synth.normal(cols + 9, 0, (rows, cols), 0.0, 2.0)
        y = mb.fused_row_softmax(_dev(x, False, 1))
        g, w = to_host(y).astype(np.float64), oracle.row_softmax(x).astype(np.float64)
        assert np.all(np.abs(g - w) <= 1e-5 * w + 2.0 ** -126), f"softmax {cols}"


def test_ragged_workload_full_size():
    """ln_gelu_f32_8192x4099 (the benchmark's unaligned row): every element."""
    w = W.LN_F32_RAGGED
    t = w.generate_all()
    assert mb.row_plan("ln", "f32", w.rows, w.cols)["vec"] == 1
    out = mb.fused_residual_layernorm_gelu(to_dev(t["x"]), to_dev(t["r"]), to_dev(t["w"]),
                                           to_dev(t["b"]), 1e-5)
    torch.cuda.synchronize()
    got = to_host(out)

    def block(r0, r1):
        want = oracle.residual_layernorm_gelu(t["x"][r0:r1], t["r"][r0:r1], t["w"], t["b"], 1e-5)
        return assert_close(got[r0:r1], want, what=f"{w.name} rows {r0}:{r1}")

    err, ratio = worst(map_row_blocks(w.rows, block))
    report(w.name, max_abs_err=err, max_err_over_bar=ratio)
