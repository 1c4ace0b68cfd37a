"""Back-to-back dependent calls with launch overlap (programmatic stream
serialisation) on and off: each call consumes the previous call's output with
no synchronisation in between, in a stream and inside a captured graph, and
the end result must equal the oracle composition.  A torch kernel writing an
input right before a call is covered as well."""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth

from gpu_util import assert_close, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from memory_bound_gb300 import build as lib_build
    lib_build.build()
    torch.cuda.set_device(0)
    yield
    mb.set_launch_overlap(True)
    torch.cuda.synchronize()
    assert mb.device_error() == 0


ROWS, COLS = 2048, 4096


def _inputs():
    x = synth.normal(901, 0, (ROWS, COLS))
    b1 = synth.normal(901, 1, (ROWS, COLS))
    b2 = synth.normal(901, 2, (ROWS, COLS))
    r = synth.normal(901, 3, (ROWS, COLS))
    w = synth.uniform(901, 4, (COLS,), 0.5, 1.5)
    b = synth.normal(901, 5, (COLS,), 0.0, 0.1)
    return x, b1, b2, r, w, b


def _oracle_chain(x, b1, b2, r, w, b):
    y1 = oracle.add_relu_scale(x, b1, b2, 0.5)
    y2 = oracle.residual_layernorm_gelu(y1, r, w, b, 1e-5)
    return oracle.row_softmax(y2)


def _device_chain(d, y1, y2, y3):
    mb.fused_add_relu_scale(d["x"], d["b1"], d["b2"], 0.5, out=y1)
    mb.fused_residual_layernorm_gelu(y1, d["r"], d["w"], d["b"], 1e-5, out=y2)
    mb.fused_row_softmax(y2, out=y3)


@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("graph", [False, True])
def test_dependent_chain(overlap, graph):
    mb.set_launch_overlap(overlap)
    x, b1, b2, r, w, b = _inputs()
    d = {k: to_dev(v) for k, v in zip(("x", "b1", "b2", "r", "w", "b"), (x, b1, b2, r, w, b))}
    y1, y2, y3 = (torch.empty((ROWS, COLS), device="cuda") for _ in range(3))
    if graph:
        _device_chain(d, y1, y2, y3)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            _device_chain(d, y1, y2, y3)
        for t in (y1, y2, y3):
            t.zero_()
        g.replay()
    else:
        _device_chain(d, y1, y2, y3)
    torch.cuda.synchronize()
    want = _oracle_chain(x, b1, b2, r, w, b)
    got = to_host(y3)
    err = np.abs(got.astype(np.float64) - want) / np.maximum(np.abs(want), 1e-30)
    # softmax of LN outputs: each stage within its bar, the composition within 1e-4 relative
    assert float(err.max()) < 1e-4, float(err.max())
    assert np.allclose(got.sum(axis=1), 1.0, atol=1e-4)


@pytest.mark.parametrize("overlap", [True, False])
def test_torch_writer_then_call(overlap):
    """A torch kernel writes x immediately before the fused call reads it."""
    mb.set_launch_overlap(overlap)
    n = 1 << 22
    a = synth.normal(902, 0, (n,))
    b1 = synth.normal(902, 1, (n,))
    b2 = synth.normal(902, 2, (n,))
    da, d1, d2 = to_dev(a), to_dev(b1), to_dev(b2)
    for k in range(5):
        x = da * float(k + 1)                  # torch kernel, then ours at once
        y = mb.fused_add_relu_scale(x, d1, d2, 0.5)
        want = oracle.add_relu_scale((a * np.float32(k + 1)).astype(np.float32), b1, b2, 0.5)
        assert np.array_equal(to_host(y).view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("graph", [False, True])
def test_dependent_chain_off_grid_rows(overlap, graph):
    """The same composition on rows off the 16-byte grid (4099 columns: the
    shifted-vector engine for the LayerNorm and softmax calls): pointwise ->
    residual + LayerNorm + GeLU -> softmax, each call reading the previous
    call's output at once."""
    mb.set_launch_overlap(overlap)
    rows, cols = 1031, 4099
    x, b1, b2, r = (synth.normal(903, k, (rows, cols)) for k in range(4))
    w = synth.uniform(903, 4, (cols,), 0.5, 1.5)
    b = synth.normal(903, 5, (cols,), 0.0, 0.1)
    assert mb.row_plan("ln", "f32", rows, cols)["vec"] == 4        # shifted vectors
    d = {k: to_dev(v) for k, v in zip(("x", "b1", "b2", "r", "w", "b"), (x, b1, b2, r, w, b))}
    y1, y2, y3 = (torch.empty((rows, cols), device="cuda") for _ in range(3))
    if graph:
        _device_chain(d, y1, y2, y3)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            _device_chain(d, y1, y2, y3)
        for t in (y1, y2, y3):
            t.zero_()
        g.replay()
    else:
        _device_chain(d, y1, y2, y3)
    torch.cuda.synchronize()
    want = _oracle_chain(x, b1, b2, r, w, b)
    got = to_host(y3)
    err = np.abs(got.astype(np.float64) - want) / np.maximum(np.abs(want), 1e-30)
    assert float(err.max()) < 1e-4, float(err.max())
