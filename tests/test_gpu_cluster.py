"""Rows longer than one CTA holds (more than 32768 elements), spread over a
thread-block cluster whose CTAs combine their partial statistics through
distributed shared memory; and the cluster path forced on ordinary rows with
explicit cluster sizes.  Every chain, against the CPU oracle."""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth

from gpu_util import assert_bitexact, assert_close, check_guard, guarded_empty, to_dev, to_host

pytestmark = pytest.mark.gpu


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


def _ln(rows, cols, seed, bf16):
    dt = "bf16" if bf16 else "f32"
    return (synth.normal(seed, 0, (rows, cols), dtype=dt), synth.normal(seed, 1, (rows, cols), dtype=dt),
            synth.uniform(seed, 2, (cols,), 0.5, 1.5, dtype=dt),
            synth.normal(seed, 3, (cols,), 0.0, 0.1, dtype=dt))


def _check_chains(rows, cols, seed, bf16):
    dt = torch.bfloat16 if bf16 else torch.float32
    x, r, w, b = _ln(rows, cols, seed, bf16)
    buf, out = guarded_empty((rows, cols), dt)
    mb.fused_residual_layernorm_gelu(to_dev(x, bf16), to_dev(r, bf16), to_dev(w, bf16),
                                     to_dev(b, bf16), 1e-5, out=out)
    assert_close(to_host(out), oracle.residual_layernorm_gelu(x, r, w, b, 1e-5), bf16=bf16,
                 what=f"LN {rows}x{cols}")
    check_guard(buf)
    out, h = mb.fused_layernorm_act(to_dev(x, bf16), to_dev(r, bf16), to_dev(w, bf16),
                                    to_dev(b, bf16), act="relu", want_h=True)
    want, want_h = oracle.layernorm_act(x, r, w, b, 1e-5, oracle.ACT_RELU, want_h=True)
    assert_close(to_host(out), want, bf16=bf16, what="LN relu")
    assert_bitexact(to_host(h), want_h, "h")
    y = to_host(mb.fused_row_softmax(to_dev(x, bf16)))
    ws = oracle.row_softmax(x)
    g = (y.astype(np.uint32) << 16).view(np.float32) if bf16 else y
    wf = (ws.astype(np.uint32) << 16).view(np.float32) if bf16 else ws
    rtol = 1e-2 if bf16 else 1e-5
    assert np.all(np.abs(g.astype(np.float64) - wf) <= rtol * np.abs(wf) + 2.0 ** -126), "softmax"
    bias = synth.normal(seed, 4, (cols,), 0.0, 0.1, dtype="bf16" if bf16 else "f32")
    yi = mb.fused_bias_relu_branch_mean_epilogue(to_dev(x, bf16), to_dev(bias, bf16), to_dev(w, bf16),
                                                 to_dev(b, bf16), 1.1, 0.1)
    want = (oracle.bias_relu_branch_mean_epilogue_bf16 if bf16 else
            oracle.bias_relu_branch_mean_epilogue)(x, bias, w, b, 1.1, 0.1)
    assert_close(to_host(yi), want, bf16=bf16, what="inductor")


@pytest.mark.parametrize("cols", [32769, 40000, 65536, 131072, 262144, 524288])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_long_rows(cols, bf16):
    rows = 3 if cols > 131072 else 5
    assert mb.row_plan("ln", "bf16" if bf16 else "f32", rows, cols)["path"] == "cluster"
    _check_chains(rows, cols, 3000 + cols % 997, bf16)


@pytest.mark.parametrize("cs", [2, 3, 5, 8, 16])
@pytest.mark.parametrize("shape", [(7, 4096), (4, 1000), (9, 33), (300, 2048)])
def test_forced_cluster_sizes(cs, shape, row_path):
    row_path("cluster", 0, cs)
    rows, cols = shape
    _check_chains(rows, cols, 4000 + cs * 31 + cols, False)


@pytest.mark.parametrize("ring", [0, 1], ids=["direct", "staged"])
@pytest.mark.parametrize("cs", [2, 4])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_32_value_kernel_forms(cs, ring, bf16, row_path):
    """32 values per thread on 65536 columns: four CTAs of 512 threads take
    the kernel form bounded at 512 threads (up to 128 registers), two CTAs
    of 1024 threads the 1024-thread form; directly loaded and staged."""
    vpt = 4 if bf16 else 8
    row_path("cluster", ring, cs, vpt)
    p = mb.row_plan("ln", "bf16" if bf16 else "f32", 5, 65536)
    assert p["path"] == "cluster" and p["vpt"] == vpt and p["stages"] == cs
    assert p["threads"] == 65536 // cs // 32
    _check_chains(5, 65536, 7000 + 10 * cs + ring, bf16)


def _bf16_to_f64(a):
    return (np.asarray(a).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("cols", [65536, 65544, 131072, 262152])
def test_bf16_softmax_slices_in_shared_memory(cols):
    """bf16 softmax rows whose CTA slices reach 64 KB keep the slice in the
    shared-memory ring (1024 threads a CTA, every pass reading the stage):
    plain and scaled, causally masked rows, more rows than resident
    clusters, ragged row lengths."""
    rows = 200
    p = mb.row_plan("softmax", "bf16", rows, cols)
    assert p["path"] == "cluster" and p["threads"] == 1024 and p["smem"] >= 65536, p
    x = synth.normal(8000 + cols % 101, 0, (rows, cols), 0.0, 2.0, dtype="bf16")
    buf, y = guarded_empty((rows, cols), torch.bfloat16)
    mb.fused_row_softmax(to_dev(x, True), out=y)
    want = _bf16_to_f64(oracle.row_softmax(x))
    got = _bf16_to_f64(to_host(y))
    assert np.all(np.abs(got - want) <= 1e-2 * np.abs(want) + 2.0 ** -126), "softmax"
    check_guard(buf)
    period, offset = 7, cols // 3
    ym = to_host(mb.fused_row_softmax(to_dev(x, True), scale=0.125, causal=True, period=period,
                                      offset=offset))
    wm = _bf16_to_f64(oracle.scale_mask_softmax(x, 0.125, True, period, offset))
    gm = _bf16_to_f64(ym)
    masked = np.arange(cols)[None, :] > (np.arange(rows)[:, None] % period + offset)
    assert np.all(gm[masked] == 0), "a masked output is not 0"
    assert np.all(np.abs(gm - wm) <= 1e-2 * np.abs(wm) + 2.0 ** -126), "masked softmax"


def test_long_rows_many_rows_and_unaligned():
    """More rows than clusters fit at once (each cluster loops over rows), and
    an unaligned scalar row length."""
    _check_chains(700, 40000, 5001, True)
    _check_chains(6, 33333, 5002, False)


@pytest.mark.parametrize("ring", [1, 2, 3])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("shape", [(11, 65536), (5, 40000), (9, 4096)])
def test_staged_cluster_ring_depths(ring, bf16, shape, row_path):
    """The bulk-copy ring of the cluster path at every depth, both dtypes
    (auto stages bf16 only), more rows than stages."""
    rows, cols = shape
    row_path("cluster", ring, 0)
    p = mb.row_plan("ln", "bf16" if bf16 else "f32", rows, cols)
    assert p["path"] == "cluster" and p["smem"] > 0
    _check_chains(rows, cols, 6000 + ring * 7 + cols % 101, bf16)


def test_direct_cluster_when_rows_are_unaligned_or_fp32():
    assert mb.row_plan("ln", "f32", 4, 65536)["smem"] == 0
    assert mb.row_plan("ln", "bf16", 4, 65536)["smem"] > 0
    assert mb.row_plan("ln", "bf16", 4, 65536, aligned=False)["smem"] == 0
