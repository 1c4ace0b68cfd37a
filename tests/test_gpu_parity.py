"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every input comes from the seeded generator (synth) or is hand-built here;
every expected value comes from the oracle.  Full workloads run at their real
sizes in the launch configuration the benchmark uses, and every element is
compared with the oracle (row blocks on the host's cores, tests/row_blocks.py);
an fp32 torch eager run on the same GPU is a further opinion, never the check.
"""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
from synth import workloads as W
import synth

from gpu_util import (assert_bitexact, assert_close, check_guard, guarded_empty,
                      max_rel_above, max_ulp_f32, report, to_dev, to_host)
from row_blocks import map_row_blocks, worst

pytestmark = pytest.mark.gpu

PATHS = ["auto", "warp", "direct", "staged"]


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


def rng_f32(seed, shape, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


# --------------------------------------------------------------------------
# pointwise chain
# --------------------------------------------------------------------------

@pytest.mark.parametrize("w", [W.POINTWISE_TINY, W.POINTWISE_4M], ids=lambda w: w.name)
def test_pointwise_workload(w):
    t = w.generate_all()
    buf, y = guarded_empty((w.cols,), torch.float32)
    mb.fused_add_relu_scale(to_dev(t["x"]), to_dev(t["b1"]), to_dev(t["b2"]), 0.5, out=y)
    want = oracle.add_relu_scale(t["x"], t["b1"], t["b2"], 0.5)
    got = to_host(y)
    assert_bitexact(got, want, w.name)
    assert max_ulp_f32(got, want) == 0
    report(w.name, max_ulp=max_ulp_f32(got, want))
    check_guard(buf)


def test_pointwise_bf16():
    n = (1 << 20) + 13
    x, b1, b2 = (synth.normal(21, k, (n,), dtype="bf16") for k in range(3))
    buf, y = guarded_empty((n,), torch.bfloat16)
    mb.fused_add_relu_scale(to_dev(x, True), to_dev(b1, True), to_dev(b2, True), 0.5, out=y)
    assert_bitexact(to_host(y), oracle.add_relu_scale(x, b1, b2, 0.5), "bf16")
    check_guard(buf)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 33, 255, 1023, 1025,
                               4099, 100003, 1 << 20])
@pytest.mark.parametrize("bf16", [False, True])
def test_pointwise_ragged(n, bf16):
    x, b1, b2 = (rng_f32(n * 3 + k, (n,)) for k in range(3))
    if bf16:
        x, b1, b2 = (synth.f32_to_bf16_bits(a) for a in (x, b1, b2))
    dt = torch.bfloat16 if bf16 else torch.float32
    buf, y = guarded_empty((n,), dt)
    mb.fused_add_relu_scale(to_dev(x, bf16), to_dev(b1, bf16), to_dev(b2, bf16), 0.5, out=y)
    assert_bitexact(to_host(y), oracle.add_relu_scale(x, b1, b2, 0.5), f"n={n}")
    check_guard(buf)


@pytest.mark.parametrize("offsets", [(1, 1, 1, 1), (3, 3, 3, 3), (2, 2, 2, 2), (0, 1, 2, 3),
                                     (1, 0, 0, 0), (0, 0, 0, 1)])
@pytest.mark.parametrize("bf16", [False, True])
def test_pointwise_unaligned(offsets, bf16):
    """Element offsets from 16-byte boundaries: one shared offset takes the
    vector path with a scalar head; mixed offsets take the scalar path."""
    n = 10007
    dt = torch.bfloat16 if bf16 else torch.float32
    host = []
    dev = []
    for k, off in enumerate(offsets[:3]):
        a = rng_f32(500 + k, (n,))
        if bf16:
            a = synth.f32_to_bf16_bits(a)
        host.append(a)
        big = torch.zeros(n + 8, dtype=dt, device="cuda")
        big[off:off + n] = to_dev(a, bf16)
        dev.append(big[off:off + n])
    ybig = torch.zeros(n + 8, dtype=dt, device="cuda")
    y = ybig[offsets[3]:offsets[3] + n]
    mb.fused_add_relu_scale(*dev, 0.5, out=y)
    assert_bitexact(to_host(y), oracle.add_relu_scale(*host, 0.5), str(offsets))
    assert not bool(ybig[:offsets[3]].any()) and not bool(ybig[offsets[3] + n:].any())


@pytest.mark.parametrize("blocks,unroll", [(1, 1), (2, 2), (0, 8), (3, 4), (0, 1)])
@pytest.mark.parametrize("n", [1 << 20, 4 * 1024 * 1024 + 5, 777777])
def test_pointwise_launch_shapes(blocks, unroll, n):
    """Other launch shapes: several fragments per thread and per block, and
    ragged block shares."""
    x, b1, b2 = (rng_f32(n + k, (n,)) for k in range(3))
    mb.set_pointwise_shape(blocks, unroll)
    try:
        buf, y = guarded_empty((n,), torch.float32)
        mb.fused_add_relu_scale(to_dev(x), to_dev(b1), to_dev(b2), 0.5, out=y)
        assert_bitexact(to_host(y), oracle.add_relu_scale(x, b1, b2, 0.5), f"{blocks},{unroll}")
        check_guard(buf)
    finally:
        mb.set_pointwise_shape(0, 0)


@pytest.mark.parametrize("scale", [0.3, 1.0, -2.0, 0.0, 1e-30, 3.0])
def test_pointwise_scales(scale):
    n = 65537
    x, b1, b2 = (rng_f32(900 + k, (n,)) for k in range(3))
    y = mb.fused_add_relu_scale(to_dev(x), to_dev(b1), to_dev(b2), scale)
    assert_bitexact(to_host(y), oracle.add_relu_scale(x, b1, b2, scale), f"scale={scale}")


def test_pointwise_special_values():
    vals = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 3.4e38,
                     -3.4e38, 1.17549435e-38], np.float32)
    xx, bb = np.meshgrid(vals, vals)
    x, b1 = xx.reshape(-1).copy(), bb.reshape(-1).copy()
    b2 = np.tile(np.array([0.5, -0.0, 2.0], np.float32), x.size // 3 + 1)[:x.size]
    y = to_host(mb.fused_add_relu_scale(to_dev(x), to_dev(b1), to_dev(b2), 0.5))
    want = oracle.add_relu_scale(x, b1, b2, 0.5)
    both_nan = np.isnan(y) & np.isnan(want)
    assert np.array_equal(y.view(np.uint32)[~both_nan], want.view(np.uint32)[~both_nan])
    assert np.array_equal(np.isnan(y), np.isnan(want))


def test_pointwise_empty_and_side_stream():
    e = torch.empty(0, device="cuda")
    mb.fused_add_relu_scale(e, e, e, 0.5, out=torch.empty(0, device="cuda"))
    n = 300001
    x, b1, b2 = (rng_f32(77 + k, (n,)) for k in range(3))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dx, d1, d2 = to_dev(x), to_dev(b1), to_dev(b2)
        y = mb.fused_add_relu_scale(dx, d1, d2, 0.5)
    s.synchronize()
    assert_bitexact(to_host(y), oracle.add_relu_scale(x, b1, b2, 0.5), "side stream")


# --------------------------------------------------------------------------
# TorchInductor chain
# --------------------------------------------------------------------------

def _inductor_inputs(rows, cols, seed):
    x = rng_f32(seed, (rows, cols))
    bias = rng_f32(seed + 1, (cols,), 0.1)
    gamma = np.random.default_rng(seed + 2).uniform(0.5, 1.5, cols).astype(np.float32)
    beta = rng_f32(seed + 3, (cols,), 0.1)
    return x, bias, gamma, beta


def test_inductor_workload():
    w = W.INDUCTOR_1024
    t = w.generate_all()
    buf, y = guarded_empty((w.rows, w.cols), torch.float32)
    mb.fused_bias_relu_branch_mean_epilogue(to_dev(t["x"]), to_dev(t["bias"]),
                                            to_dev(t["gamma"]), to_dev(t["beta"]),
                                            1.1, 0.1, out=y)
    want = oracle.bias_relu_branch_mean_epilogue(t["x"], t["bias"], t["gamma"], t["beta"])
    err, ratio = assert_close(to_host(y), want, what=w.name)
    assert ratio < 0.5       # well inside the bar
    report(w.name, max_abs_err=err, max_err_over_bar=ratio,
           max_rel_err_where_abs_ge_1e_3=max_rel_above(to_host(y), want))
    check_guard(buf)


@pytest.mark.parametrize("shape", [(1, 1), (3, 5), (2, 31), (7, 1000), (5, 1027), (1024, 1024),
                                   (33, 4096), (6, 4099), (4, 32768), (3, 20001)])
@pytest.mark.parametrize("path", PATHS)
def test_inductor_shapes_and_paths(shape, path, row_path):
    rows, cols = shape
    row_path(path)
    x, bias, gamma, beta = _inductor_inputs(rows, cols, rows * 7 + cols)
    buf, y = guarded_empty(shape, torch.float32)
    mb.fused_bias_relu_branch_mean_epilogue(to_dev(x), to_dev(bias), to_dev(gamma),
                                            to_dev(beta), 1.1, 0.1, out=y)
    want = oracle.bias_relu_branch_mean_epilogue(x, bias, gamma, beta)
    assert_close(to_host(y), want, what=f"{shape} {path}")
    check_guard(buf)


def test_inductor_degenerate_rows():
    """Rows whose t is never positive give s = 0, m = 0 and y = beta exactly.
    A constant row (bias 0) gives s constant; its fp32 tree-sum mean equals s
    only to rounding (3s is not exact in fp32), so y = beta to tolerance."""
    cols = 1024
    x = np.stack([-np.abs(rng_f32(1, (cols,))) - 0.5, np.full(cols, 0.75, np.float32)])
    bias = np.zeros(cols, np.float32)
    gamma = np.random.default_rng(2).uniform(0.5, 1.5, cols).astype(np.float32)
    beta = rng_f32(3, (cols,))
    y = to_host(mb.fused_bias_relu_branch_mean_epilogue(
        to_dev(x), to_dev(bias), to_dev(gamma), to_dev(beta), 1.1, 0.1))
    assert_bitexact(y[0], beta, "all-negative row")
    want = oracle.bias_relu_branch_mean_epilogue(x, bias, gamma, beta)
    assert_bitexact(want[1], beta, "oracle constant row")
    assert_close(y[1], want[1], what="constant row")


def test_inductor_offset_pointers():
    rows, cols = 9, 1024
    x, bias, gamma, beta = _inductor_inputs(rows, cols, 5)
    big = torch.zeros(rows * cols + 1, device="cuda")
    big[1:] = to_dev(x).reshape(-1)
    ybig = torch.zeros(rows * cols + 3, device="cuda")
    y = ybig[3:].view(rows, cols)
    mb.fused_bias_relu_branch_mean_epilogue(big[1:].view(rows, cols), to_dev(bias),
                                            to_dev(gamma), to_dev(beta), 1.1, 0.1, out=y)
    assert_close(to_host(y), oracle.bias_relu_branch_mean_epilogue(x, bias, gamma, beta))


# --------------------------------------------------------------------------
# residual + LayerNorm + GeLU
# --------------------------------------------------------------------------

def _ln_inputs(rows, hidden, seed, bf16):
    dt = "bf16" if bf16 else "f32"
    return (synth.normal(seed, 0, (rows, hidden), dtype=dt),
            synth.normal(seed, 1, (rows, hidden), dtype=dt),
            synth.uniform(seed, 2, (hidden,), 0.5, 1.5, dtype=dt),
            synth.normal(seed, 3, (hidden,), 0.0, 0.1, dtype=dt))


def _run_ln(x, r, w, b, bf16, eps=1e-5, out=None):
    return mb.fused_residual_layernorm_gelu(to_dev(x, bf16), to_dev(r, bf16), to_dev(w, bf16),
                                            to_dev(b, bf16), eps, out=out)


@pytest.mark.parametrize("w", [W.LN_F32, W.LN_BF16], ids=lambda w: w.name)
def test_ln_workload_full_size(w):
    """The full workload on the GPU in the benchmark's launch, every element
    against the oracle at the stated bar (row blocks on the host's cores);
    fp32 eager torch on the same GPU is a further opinion over every row."""
    bf16 = w.dtype == "bf16"
    t = w.generate_all()
    dx, dr, dw, db = (to_dev(t[k], bf16) for k in ("x", "r", "w", "b"))
    out = mb.fused_residual_layernorm_gelu(dx, dr, dw, db, 1e-5)
    torch.cuda.synchronize()
    got = to_host(out)

    def block(r0, r1):
        want = oracle.residual_layernorm_gelu(t["x"][r0:r1], t["r"][r0:r1], t["w"], t["b"], 1e-5)
        e = assert_close(got[r0:r1], want, bf16=bf16, what=f"{w.name} rows {r0}:{r1}")
        return e + (max_rel_above(got[r0:r1], want, bf16),)

    stats = map_row_blocks(w.rows, block)
    err, ratio = worst(stats)
    report(w.name, max_abs_err=err, max_err_over_bar=ratio,
           max_rel_err_where_abs_ge_1e_3=max(s[2] for s in stats))
    # third opinion over every row: fp32 eager torch (its own rounding of
    # x + r for bf16 inputs is avoided by widening first)
    ref = torch.nn.functional.gelu(torch.nn.functional.layer_norm(
        dx.float() + dr.float(), (w.cols,), dw.float(), db.float(), 1e-5), approximate="tanh")
    g = out.float()
    tol = (2e-2 * torch.clamp(ref.abs(), min=1e-2)) if bf16 else (2e-5 * torch.clamp(ref.abs(), min=1.0))
    assert bool(torch.isfinite(g).all())
    assert bool(((g - ref).abs() <= tol).all())


LN_SHAPES = [(1, 1), (3, 2), (5, 33), (4, 1000), (2, 1024), (9, 4096), (6, 4099), (3, 8192),
             (2, 32768), (16, 2048), (1, 12288), (300, 4096)]


@pytest.mark.parametrize("shape", LN_SHAPES)
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_ln_shapes_and_paths(shape, path, bf16, row_path):
    rows, hidden = shape
    row_path(path)
    x, r, w, b = _ln_inputs(rows, hidden, 100 + hidden, bf16)
    buf, out = guarded_empty(shape, torch.bfloat16 if bf16 else torch.float32)
    _run_ln(x, r, w, b, bf16, out=out)
    want = oracle.residual_layernorm_gelu(x, r, w, b, 1e-5)
    assert_close(to_host(out), want, bf16=bf16, what=f"{shape} {path}")
    check_guard(buf)


@pytest.mark.parametrize("ctas,stages,vpt", [(1, 1, 0), (1, 2, 0), (2, 2, 0), (1, 5, 0),
                                             (2, 3, 0), (1, 0, 0), (3, 0, 0), (4, 1, 0),
                                             (0, 0, 1), (0, 0, 2), (0, 0, 4), (2, 2, 4)])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_ln_staged_ring_shapes(ctas, stages, vpt, bf16, row_path):
    """The staged ring at several depths, CTAs per SM and vectors per thread
    (row counts that are not multiples of the grid, so CTAs end at different
    ring phases)."""
    row_path("staged", ctas, stages, vpt)
    rows, hidden = 1111, 4096 if not bf16 else 8192
    x, r, w, b = _ln_inputs(rows, hidden, 7 + ctas * 10 + stages, bf16)
    got = to_host(_run_ln(x, r, w, b, bf16))

    def block(r0, r1):
        want = oracle.residual_layernorm_gelu(x[r0:r1], r[r0:r1], w, b, 1e-5)
        return assert_close(got[r0:r1], want, bf16=bf16,
                            what=f"ctas={ctas} stages={stages} rows {r0}:{r1}")

    map_row_blocks(rows, block)


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_ln_degenerate_rows(bf16):
    """Constant rows and H = 1: v - mean = 0, so out = GeLU(b) (the oracle's
    value); eps = 0 on a constant row gives 0 * inf, which both sides leave
    alone only when eps > 0, so eps stays 1e-5 here."""
    for hidden in (1, 4096):
        x = np.full((3, hidden), 0.75, np.float32)
        r = np.full((3, hidden), -0.25, np.float32)
        w = np.random.default_rng(1).uniform(0.5, 1.5, hidden).astype(np.float32)
        b = rng_f32(2, (hidden,))
        if bf16:
            x, r, w, b = (synth.f32_to_bf16_bits(a) for a in (x, r, w, b))
        out = to_host(_run_ln(x, r, w, b, bf16))
        want = oracle.residual_layernorm_gelu(x, r, w, b, 1e-5)
        assert_close(out, want, bf16=bf16, what=f"constant rows H={hidden}")


def test_ln_eps_values():
    x, r, w, b = _ln_inputs(4, 4096, 55, False)
    for eps in (0.0, 1e-5, 1e-2, 1.0):
        out = to_host(_run_ln(x, r, w, b, False, eps=eps))
        assert_close(out, oracle.residual_layernorm_gelu(x, r, w, b, eps), what=f"eps={eps}")


def test_ln_deterministic():
    x, r, w, b = _ln_inputs(512, 4096, 9, False)
    a = to_host(_run_ln(x, r, w, b, False))
    c = to_host(_run_ln(x, r, w, b, False))
    assert_bitexact(a, c, "two runs")


def test_ln_empty_rows():
    z = torch.empty((0, 64), device="cuda")
    v = torch.ones(64, device="cuda")
    mb.fused_residual_layernorm_gelu(z, z, v, v, 1e-5, out=torch.empty((0, 64), device="cuda"))


def test_row_plan_reports_paths():
    p = mb.row_plan("ln", "bf16", 32768, 8192)
    assert p["path"] == "staged" and p["stages"] >= 1 and p["vec"] == 8
    p = mb.row_plan("ln", "f32", 8192, 4096)
    assert p["path"] == "staged" and p["vec"] == 4
    p = mb.row_plan("inductor", "f32", 1024, 1024)
    assert p["path"] == "warp"
    p = mb.row_plan("ln", "f32", 8, 4099, aligned=False)
    assert p["path"] == "direct" and p["vec"] == 1
