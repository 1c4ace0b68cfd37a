"""Parity of the scaled, causally masked softmax of attention-score rows
("PyTorch operator fusion in practice" §4.1-4.2) with the CPU oracle, on
every row engine: masked outputs exactly 0, the rest within the softmax bar
(pure relative: fp32 1e-5, bf16 1e-2)."""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth
from synth import workloads as W

from gpu_util import bf16_to_f64, check_guard, guarded_empty, report, to_dev, to_host
from row_blocks import map_row_blocks

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


def masked(rows, cols, period, offset):
    i = np.arange(rows)[:, None] % period + offset
    return np.arange(cols)[None, :] > i


def check(got, want, bf16, mask, what):
    g = bf16_to_f64(got) if bf16 else np.asarray(got, np.float64)
    w = bf16_to_f64(want) if bf16 else np.asarray(want, np.float64)
    if mask is not None:
        assert np.all(g[mask] == 0), f"{what}: a masked output is not 0"
    rtol = 1e-2 if bf16 else 1e-5
    err = np.abs(g - w)
    bad = err > rtol * np.abs(w) + 2.0 ** -126
    assert not bad.any(), f"{what}: {int(bad.sum())} out of tolerance"
    big = np.abs(w) >= 2.0 ** -100
    return float((err[big] / np.abs(w[big])).max()) if big.any() else 0.0


SHAPES = [(1, 1), (5, 33), (9, 4096), (6, 4099), (300, 1024), (3, 8192), (2, 32768), (3, 65536)]
CONFIGS = {"causal_square": (0.125, True, None, 0), "causal_p4_o2": (0.3, True, 4, 2),
           "scaled_only": (1.5, False, 1, 0), "offset_past_row": (0.125, True, 3, 100000)}


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("path", ["auto", "warp", "direct", "staged", "cluster"])
@pytest.mark.parametrize("cfg", sorted(CONFIGS))
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_scale_mask_softmax(shape, path, cfg, bf16, row_path):
    rows, cols = shape
    scale, causal, period, offset = CONFIGS[cfg]
    period = rows if period is None else period
    row_path(path)
    dt = "bf16" if bf16 else "f32"
    x = synth.normal(2100 + cols % 97 + rows, 0, shape, 0.0, 3.0, dtype=dt)
    buf, y = guarded_empty(shape, torch.bfloat16 if bf16 else torch.float32)
    mb.fused_row_softmax(to_dev(x, bf16), out=y, scale=scale, causal=causal, period=period,
                         offset=offset)
    want = oracle.scale_mask_softmax(x, scale, causal, period, offset)
    check(to_host(y), want, bf16, masked(rows, cols, period, offset) if causal else None,
          f"{shape} {path} {cfg}")
    check_guard(buf)


@pytest.mark.parametrize("path", ["auto", "direct", "staged"])
def test_masked_values_take_no_part(path, row_path):
    """NaN, inf and huge values in the masked region change nothing (on the
    staged path that region is not even read)."""
    row_path(path)
    rows, cols = 64, 4096
    x = synth.normal(2200, 0, (rows, cols), 0.0, 2.0)
    m = masked(rows, cols, rows, 0)
    dirty = x.copy()
    dirty[m] = np.where(np.arange(m.sum()) % 3 == 0, np.nan,
                        np.where(np.arange(m.sum()) % 3 == 1, np.inf, 1e30)).astype(np.float32)
    y = mb.fused_row_softmax(to_dev(dirty), scale=0.125, causal=True)
    check(to_host(y), oracle.scale_mask_softmax(x, 0.125, True), False, m, path)


@pytest.mark.parametrize("cols", [4096, 40000])
def test_masked_values_in_host_memory(cols):
    """Score rows in pinned host memory take the direct paths, which skip
    the slots past each row's unmasked prefix; NaN and inf there change
    nothing (one-CTA rows and rows on a cluster)."""
    rows = 48
    x = synth.normal(2204, 0, (rows, cols), 0.0, 2.0)
    m = masked(rows, cols, rows, 3)
    dirty = x.copy()
    dirty[m] = np.where(np.arange(m.sum()) % 2 == 0, np.nan, np.inf).astype(np.float32)
    y = mb.fused_row_softmax(torch.from_numpy(dirty).pin_memory(), scale=0.125, causal=True,
                             period=rows, offset=3)
    torch.cuda.synchronize()
    check(y.numpy(), oracle.scale_mask_softmax(x, 0.125, True, rows, 3), False, m, f"host {cols}")


def test_multi_head_periods_and_host_memory():
    """Rows of several heads (period 512 queries, keys offset by 256), the
    score rows in pinned host memory."""
    rows, cols, period, offset = 2048, 768, 512, 256
    x = synth.normal(2201, 0, (rows, cols), 0.0, 2.0)
    hx = torch.from_numpy(x).pin_memory()
    y = mb.fused_row_softmax(hx, scale=0.0884, causal=True, period=period, offset=offset)
    torch.cuda.synchronize()
    assert y.device.type == "cpu"
    check(y.numpy(), oracle.scale_mask_softmax(x, 0.0884, True, period, offset), False,
          masked(rows, cols, period, offset), "host")


def test_graph_capture_replays_new_scores():
    rows, cols = 1024, 4096
    dx = torch.empty(rows, cols, device="cuda")
    y = torch.empty_like(dx)
    x0 = synth.normal(2202, 0, (rows, cols))
    dx.copy_(to_dev(x0))
    mb.fused_row_softmax(dx, out=y, scale=0.125, causal=True)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        mb.fused_row_softmax(dx, out=y, scale=0.125, causal=True)
    x1 = synth.normal(2203, 0, (rows, cols))
    dx.copy_(to_dev(x1))
    g.replay()
    torch.cuda.synchronize()
    check(to_host(y), oracle.scale_mask_softmax(x1, 0.125, True), False,
          masked(rows, cols, rows, 0), "graph")


def test_workload_full_size_and_eager():
    """[P1] §4.1's 32 x 4096 x 4096 score matrix, scaled by 1/8 and causally
    masked: every row against the oracle (blocks of one head each, so the
    mask's row modulo the period starts at 0 in every block), and every row
    against the eager chain (scale, masked_fill(-inf), softmax) on the GPU."""
    w = W.SOFTMAX_CAUSAL_F32
    p = w.params
    x = w.generate(w.tensors[0])
    dx = to_dev(x)
    y = mb.fused_row_softmax(dx, scale=p["scale"], causal=True, period=p["period"],
                             offset=p["offset"])
    torch.cuda.synchronize()
    got = to_host(y)
    head_mask = masked(p["period"], w.cols, p["period"], p["offset"])

    def block(r0, r1):
        assert r0 % p["period"] == 0 and (r1 - r0) == p["period"]
        want = oracle.scale_mask_softmax(x[r0:r1], p["scale"], True, p["period"], p["offset"])
        return check(got[r0:r1], want, False, head_mask, f"{w.name} rows {r0}:{r1}")

    rel = max(map_row_blocks(w.rows, block, block=p["period"], align=p["period"]))
    report(w.name, max_rel_err=rel)
    q = torch.arange(w.rows, device="cuda")[:, None] % p["period"]
    mask = torch.arange(w.cols, device="cuda")[None, :] > q + p["offset"]
    eager = torch.softmax((dx * p["scale"]).masked_fill(mask, float("-inf")), dim=1)
    assert torch.equal(y == 0, eager == 0)
    assert float(((y - eager).abs() / eager.abs().clamp_min(1e-30)).max()) < 1e-5


def test_planner_counts_the_unmasked_share():
    """A causal score row under a square mask copies half its keys on
    average, so the planner keeps more of them in flight per SM than it does
    full softmax rows of the same length (the per-SM byte budget counts the
    reads over the share of the row that is copied)."""
    mb.set_row_path("auto")
    for dt in ("f32", "bf16"):
        causal = mb.row_plan("softmax_mask", dt, 131072, 4096)
        full = mb.row_plan("softmax", dt, 131072, 4096)
        assert causal["path"] == full["path"] == "staged"
        assert causal["ctas"] >= full["ctas"], (dt, causal, full)
    f32 = mb.row_plan("softmax_mask", "f32", 131072, 4096)
    assert f32["ctas"] > mb.row_plan("softmax", "f32", 131072, 4096)["ctas"]
