"""Parity of the pointwise chain with per-column (broadcast) b1 / b2 with the
CPU oracle: bit-exact for every flag combination, both dtypes, the vector and
scalar paths, short and long rows, and the full-size workload."""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth
from synth import workloads as W

from gpu_util import assert_bitexact, check_guard, guarded_empty, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from memory_bound_gb300 import build as lib_build
    lib_build.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()
    assert mb.device_error() == 0


SHAPES = [(1, 1), (3, 5), (5, 8), (1000, 3), (7, 1000), (64, 4096), (33, 4099), (1024, 1024),
          (2, 300000), (4097, 16)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("flags", [(1, 1), (1, 0), (0, 1), (0, 0)], ids=lambda f: f"c{f[0]}{f[1]}")
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_bcast(shape, flags, bf16):
    rows, cols = shape
    dt = "bf16" if bf16 else "f32"
    seed = 1800 + rows + cols
    x = synth.normal(seed, 0, shape, dtype=dt)
    b1 = synth.normal(seed, 1, (cols,) if flags[0] else shape, dtype=dt)
    b2 = synth.normal(seed, 2, (cols,) if flags[1] else shape, dtype=dt)
    buf, y = guarded_empty(shape, torch.bfloat16 if bf16 else torch.float32)
    mb.fused_add_relu_scale(to_dev(x, bf16), to_dev(b1, bf16), to_dev(b2, bf16), 0.5, out=y)
    assert_bitexact(to_host(y), oracle.add_relu_scale_bcast(x, b1, b2, 0.5),
                    f"{shape} {flags}")
    check_guard(buf)


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_unaligned_views_take_the_scalar_path(bf16):
    """Operands one element off a 16-byte boundary."""
    rows, cols = 37, 1024
    dt = "bf16" if bf16 else "f32"
    tdt = torch.bfloat16 if bf16 else torch.float32
    x = synth.normal(1900, 0, (rows, cols), dtype=dt)
    b1 = synth.normal(1900, 1, (cols,), dtype=dt)
    b2 = synth.normal(1900, 2, (cols,), dtype=dt)
    xs = torch.empty(rows * cols + 1, dtype=tdt, device="cuda")[1:].view(rows, cols)
    xs.copy_(to_dev(x, bf16))
    b1s = torch.empty(cols + 1, dtype=tdt, device="cuda")[1:]
    b1s.copy_(to_dev(b1, bf16))
    ys = torch.empty(rows * cols + 1, dtype=tdt, device="cuda")[1:].view(rows, cols)
    mb.fused_add_relu_scale(xs, b1s, to_dev(b2, bf16), 0.5, out=ys)
    assert_bitexact(to_host(ys), oracle.add_relu_scale_bcast(x, b1, b2, 0.5), "unaligned")


def test_other_scales_and_3d_input():
    """The leading dimensions of x are flattened into rows."""
    x = synth.normal(1901, 0, (4, 6, 256))
    b1 = synth.normal(1901, 1, (256,))
    b2 = synth.normal(1901, 2, (4, 6, 256))
    y = mb.fused_add_relu_scale(to_dev(x), to_dev(b1), to_dev(b2), 1.25)
    want = oracle.add_relu_scale_bcast(x.reshape(24, 256), b1, b2.reshape(24, 256), 1.25)
    assert_bitexact(to_host(y).reshape(24, 256), want, "3-d")


def test_full_size_workload():
    w = W.POINTWISE_BCAST_F32
    t = w.generate_all()
    y = mb.fused_add_relu_scale(to_dev(t["x"]), to_dev(t["b1"]), to_dev(t["b2"]),
                                w.params["scale"])
    want = oracle.add_relu_scale_bcast(t["x"], t["b1"], t["b2"], w.params["scale"])
    assert_bitexact(to_host(y), want, w.name)
    # torch eager with broadcasting gives the same bits
    d = {k: to_dev(v) for k, v in t.items()}
    eager = torch.relu(d["x"] + d["b1"]) * w.params["scale"] + d["b2"]
    assert torch.equal(eager.view(torch.int32), y.view(torch.int32))


def test_graph_capture():
    rows, cols = 2048, 1024
    x = synth.normal(1902, 0, (rows, cols))
    b1, b2 = synth.normal(1902, 1, (cols,)), synth.normal(1902, 2, (cols,))
    d = [to_dev(a) for a in (x, b1, b2)]
    y = torch.empty(rows, cols, device="cuda")
    mb.fused_add_relu_scale(*d, 0.5, out=y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        for _ in range(3):
            mb.fused_add_relu_scale(*d, 0.5, out=y)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_bitexact(to_host(y), oracle.add_relu_scale_bcast(x, b1, b2, 0.5), "graph")
