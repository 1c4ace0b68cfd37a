"""The fused chains inside a captured CUDA graph.

The library neither allocates nor synchronises, so its calls can be captured
once and replayed (the way the pages remove per-launch overhead for small,
launch-bound calls: capture a sequence of kernels, then launch the graph).
Each test captures the calls, replays the graph on two different input sets
copied into the captured buffers, and checks every replay against the CPU
oracle.
"""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
from synth import workloads as W

from gpu_util import assert_bitexact, assert_close, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from memory_bound_gb300 import build as lib_build
    lib_build.build()
    torch.cuda.set_device(0)
    mb.set_row_path("auto")
    yield
    torch.cuda.synchronize()
    assert mb.device_error() == 0


def _capture(fn):
    """The package's graph harness (one call outside the capture first)."""
    return mb.graph.ChainGraph(fn)


def _inputs(w, seed):
    """The workload's tensors drawn with another seed (same distributions)."""
    import dataclasses
    return dataclasses.replace(w, seed=seed).generate_all(
        rows=min(w.rows, 256) if w.chain != "add_relu_scale" else None)


@pytest.mark.parametrize("w", [W.POINTWISE_TINY, W.POINTWISE_4M], ids=lambda w: w.name)
def test_graph_pointwise(w):
    t0 = w.generate_all()
    dev = {k: to_dev(v) for k, v in t0.items()}
    out = torch.empty_like(dev["x"])
    g = _capture(lambda: mb.fused_add_relu_scale(dev["x"], dev["b1"], dev["b2"], 0.5, out=out))
    for seed in (100, 101):
        t = _inputs(w, seed)
        for k in dev:
            dev[k].copy_(to_dev(t[k]))
        g.replay()
        torch.cuda.synchronize()
        assert_bitexact(to_host(out), oracle.add_relu_scale(t["x"], t["b1"], t["b2"], 0.5),
                        f"replay seed {seed}")


def test_graph_inductor_sequence():
    """Ten captured calls on ten buffer sets, replayed twice."""
    w = W.INDUCTOR_1024
    sets = []
    for k in range(10):
        t = _inputs(w, 200 + k)
        sets.append(({n: to_dev(v) for n, v in t.items()}, torch.empty((256, 1024), device="cuda")))

    def calls():
        for d, y in sets:
            mb.fused_bias_relu_branch_mean_epilogue(d["x"], d["bias"], d["gamma"], d["beta"],
                                                    1.1, 0.1, out=y)

    g = _capture(calls)
    for rep in range(2):
        for d, _ in sets:
            d["x"].mul_(-1.0 if rep else 1.0)
        g.replay()
        torch.cuda.synchronize()
        for d, y in sets:
            h = {n: to_host(v) for n, v in d.items()}
            want = oracle.bias_relu_branch_mean_epilogue(h["x"], h["bias"], h["gamma"], h["beta"])
            assert_close(to_host(y), want, what=f"replay {rep}")


@pytest.mark.parametrize("w", [W.LN_F32, W.LN_BF16], ids=lambda w: w.name)
def test_graph_layernorm(w):
    bf16 = w.dtype == "bf16"
    t0 = _inputs(w, 300)
    dev = {k: to_dev(v, bf16) for k, v in t0.items()}
    out = torch.empty_like(dev["x"])
    g = _capture(lambda: mb.fused_residual_layernorm_gelu(dev["x"], dev["r"], dev["w"], dev["b"],
                                                          1e-5, out=out))
    for seed in (301, 302):
        t = _inputs(w, seed)
        for k in dev:
            dev[k].copy_(to_dev(t[k], bf16))
        g.replay()
        torch.cuda.synchronize()
        want = oracle.residual_layernorm_gelu(t["x"], t["r"], t["w"], t["b"], 1e-5)
        assert_close(to_host(out), want, bf16=bf16, what=f"replay seed {seed}")
    assert np.all(np.isfinite(to_host(out).astype(np.float32) if not bf16 else 1.0))


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_graph_long_rows_cluster_path(bf16):
    """Rows of 65536 elements (one cluster per row: staged for bf16, direct
    for fp32) and LayerNorm -> ReLU -> Dropout, captured and replayed on new
    inputs copied into the captured buffers."""
    import synth
    rows, cols = 12, 65536
    dt = "bf16" if bf16 else "f32"
    tdt = torch.bfloat16 if bf16 else torch.float32
    assert mb.row_plan("ln", dt, rows, cols)["path"] == "cluster"
    dx = torch.empty(rows, cols, dtype=tdt, device="cuda")
    dr = torch.empty_like(dx)
    w = to_dev(synth.uniform(77, 2, (cols,), 0.5, 1.5, dtype=dt), bf16)
    b = to_dev(synth.normal(77, 3, (cols,), 0.0, 0.1, dtype=dt), bf16)
    out = torch.empty_like(dx)
    dout = torch.empty_like(dx)
    def calls():
        mb.fused_residual_layernorm_gelu(dx, dr, w, b, 1e-5, out=out)
        mb.fused_layernorm_act(dx, None, w, b, act="relu", out=dout, p=0.1, seed=5, offset=3)
    x0 = synth.normal(78, 0, (rows, cols), dtype=dt)
    r0 = synth.normal(78, 1, (rows, cols), dtype=dt)
    dx.copy_(to_dev(x0, bf16)); dr.copy_(to_dev(r0, bf16))
    g = _capture(calls)
    for seed in (79, 80):
        x = synth.normal(seed, 0, (rows, cols), dtype=dt)
        r = synth.normal(seed, 1, (rows, cols), dtype=dt)
        dx.copy_(to_dev(x, bf16)); dr.copy_(to_dev(r, bf16))
        g.replay()
        torch.cuda.synchronize()
        wh, bh = to_host(w), to_host(b)
        assert_close(to_host(out), oracle.residual_layernorm_gelu(x, r, wh, bh, 1e-5), bf16=bf16)
        want, _, _, _ = oracle.layernorm_act_ex(x, None, wh, bh, 1e-5, oracle.ACT_RELU, p=0.1,
                                                seed=5, offset=3)
        assert_close(to_host(dout), want, bf16=bf16)
