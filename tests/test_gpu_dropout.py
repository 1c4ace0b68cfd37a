"""Parity of the LayerNorm family's extras with the CPU oracle: dropout on the
activation output ("Operator fusion and kernel optimisation" §2.1:
LayerNorm -> ReLU -> Dropout in one kernel) and the per-row statistics.

Dropout decisions are integer work (16-bit halves of Philox-4x32-10 words
against an exact threshold), so the kept/dropped pattern must match the
oracle's element for element, dropped elements must be exact (signed) zeros,
and kept ones are within the fp32 / bf16 bar of the oracle's act / (1 - p)."""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth
from synth import workloads as W

from gpu_util import (assert_bitexact, assert_close, bf16_to_f64, check_guard, guarded_empty,
                      to_dev, to_host)
from row_blocks import dropout_block_offset, map_row_blocks

pytestmark = pytest.mark.gpu

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


def _inputs(rows, hidden, seed, bf16):
    dt = "bf16" if bf16 else "f32"
    return (synth.normal(seed, 0, (rows, hidden), dtype=dt),
            synth.normal(seed, 1, (rows, hidden), dtype=dt),
            synth.uniform(seed, 2, (hidden,), 0.5, 1.5, dtype=dt),
            synth.normal(seed, 3, (hidden,), 0.0, 0.1, dtype=dt))


def _as_f64(a, bf16):
    return bf16_to_f64(a) if bf16 else np.asarray(a, np.float64)


def check_dropout(got, want, keep, bf16, what):
    """Same kept/dropped pattern, exact signed zeros where dropped, the
    tolerance elsewhere."""
    g, w = _as_f64(got, bf16), _as_f64(want, bf16)
    assert np.all(g[~keep] == 0), f"{what}: a dropped element is not zero"
    assert np.array_equal(np.signbit(g[~keep]), np.signbit(w[~keep])), f"{what}: sign of zero"
    nz = keep & (w != 0)
    assert np.all(g[nz] != 0), f"{what}: a kept element was dropped"
    assert_close(got, want, bf16=bf16, what=what)


def check_stats(mean, rstd, want_mean, want_rstd, what):
    """mean within 1e-5 of the row's standard deviation (what the normalised
    output sees), rstd within 1e-5 relative."""
    m = (to_host(mean) if torch.is_tensor(mean) else np.asarray(mean)).astype(np.float64)
    r = (to_host(rstd) if torch.is_tensor(rstd) else np.asarray(rstd)).astype(np.float64)
    assert np.all(np.abs(m - want_mean) <= 1e-5 / want_rstd + 1e-7 * np.abs(want_mean)), what
    assert np.all(np.abs(r - want_rstd) <= 1e-5 * want_rstd), what


SHAPES = [(1, 1), (3, 2), (5, 33), (4, 1000), (9, 4096), (6, 4099), (3, 8192), (2, 32768),
          (300, 4096), (3, 65536)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("path", ["auto", "warp", "direct", "staged", "cluster"])
@pytest.mark.parametrize("res", [True, False], ids=["res", "nores"])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_dropout_and_stats(shape, path, res, bf16, row_path):
    rows, hidden = shape
    row_path(path)
    x, r, w, b = _inputs(rows, hidden, 900 + rows + hidden, bf16)
    dt = torch.bfloat16 if bf16 else torch.float32
    seed, offset, p = 0xC0FFEE + hidden, 17 * rows, 0.1 if hidden % 2 else 0.5
    obuf, out = guarded_empty(shape, dt)
    hbuf, h = guarded_empty(shape, dt)
    mbuf, mean = guarded_empty((rows,), torch.float32)
    rbuf, rstd = guarded_empty((rows,), torch.float32)
    mb.fused_layernorm_act(to_dev(x, bf16), to_dev(r, bf16) if res else None, to_dev(w, bf16),
                           to_dev(b, bf16), eps=1e-5, act="relu", out=out, h_out=h, p=p,
                           seed=seed, offset=offset, mean_out=mean, rstd_out=rstd)
    want, want_h, want_mean, want_rstd = oracle.layernorm_act_ex(
        x, r if res else None, w, b, 1e-5, oracle.ACT_RELU, p=p, seed=seed, offset=offset,
        want_h=True, want_stats=True)
    keep = oracle.dropout_mask(seed, offset, 0, rows * hidden, p).reshape(shape)
    what = f"{shape} {path} res={res}"
    check_dropout(to_host(out), want, keep, bf16, what)
    assert_bitexact(to_host(h), want_h, f"h {what}")
    check_stats(mean, rstd, want_mean, want_rstd, what)
    for buf in (obuf, hbuf, mbuf, rbuf):
        check_guard(buf)


@pytest.mark.parametrize("act", sorted(ACTS))
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_dropout_activations(act, bf16):
    """Every activation; with none, dropped negative values are -0."""
    shape = (64, 4096)
    x, r, w, b = _inputs(*shape, 950, bf16)
    out = mb.fused_layernorm_act(to_dev(x, bf16), to_dev(r, bf16), to_dev(w, bf16),
                                 to_dev(b, bf16), eps=1e-5, act=act, p=0.3, seed=5, offset=0)
    want, _, _, _ = oracle.layernorm_act_ex(x, r, w, b, 1e-5, ACTS[act], p=0.3, seed=5)
    keep = oracle.dropout_mask(5, 0, 0, x.size, 0.3).reshape(shape)
    check_dropout(to_host(out), want, keep, bf16, act)


def test_offset_crosses_the_32_bit_counter_word():
    """g = offset + i / 8 carries into the counter's high word inside the call."""
    shape = (8, 1024)
    x, r, w, b = _inputs(*shape, 951, False)
    offset = (1 << 32) - 1000
    out = mb.fused_layernorm_act(to_dev(x), to_dev(r), to_dev(w), to_dev(b), act="relu",
                                 p=0.25, seed=(1 << 64) - 5, offset=offset)
    want, _, _, _ = oracle.layernorm_act_ex(x, r, w, b, 1e-5, oracle.ACT_RELU, p=0.25,
                                            seed=(1 << 64) - 5, offset=offset)
    keep = oracle.dropout_mask((1 << 64) - 5, offset, 0, x.size, 0.25).reshape(shape)
    check_dropout(to_host(out), want, keep, False, "carry")


def test_p_zero_is_the_plain_chain_and_p_tiny_drops_almost_nothing():
    shape = (33, 4096)
    x, r, w, b = _inputs(*shape, 952, False)
    d = [to_dev(a) for a in (x, r, w, b)]
    plain = mb.fused_layernorm_act(*d, act="relu")
    zero, _, _, _ = mb.fused_layernorm_act(*d, act="relu", p=0.0, seed=3, want_stats=True)
    assert torch.equal(plain.view(torch.int32), zero.view(torch.int32))
    tiny = mb.fused_layernorm_act(*d, act="relu", p=2.0 ** -24, seed=3)
    keep = oracle.dropout_mask(3, 0, 0, x.size, 2.0 ** -24).reshape(shape)
    want, _, _, _ = oracle.layernorm_act_ex(x, r, w, b, 1e-5, oracle.ACT_RELU, p=2.0 ** -24,
                                            seed=3)
    check_dropout(to_host(tiny), want, keep, False, "tiny p")


def test_successive_offsets_give_fresh_masks():
    shape = (128, 4096)
    x, r, w, b = _inputs(*shape, 953, False)
    d = [to_dev(a) for a in (x, r, w, b)]
    n8 = x.size // 8
    a = mb.fused_layernorm_act(*d, act="none", p=0.5, seed=9, offset=0)
    c = mb.fused_layernorm_act(*d, act="none", p=0.5, seed=9, offset=n8)
    ka, kc = (a != 0), (c != 0)
    agree = (ka == kc).float().mean().item()
    assert 0.45 < agree < 0.55
    again = mb.fused_layernorm_act(*d, act="none", p=0.5, seed=9, offset=0)
    assert torch.equal(a.view(torch.int32), again.view(torch.int32))


def test_graph_replay_is_deterministic():
    shape = (256, 4096)
    x, r, w, b = _inputs(*shape, 954, True)
    d = [to_dev(a, True) for a in (x, r, w, b)]
    out = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    mb.fused_layernorm_act(*d, act="relu", out=out, p=0.1, seed=77)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        mb.fused_layernorm_act(*d, act="relu", out=out, p=0.1, seed=77)
    first = out.clone()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), out.view(torch.int16))
    want, _, _, _ = oracle.layernorm_act_ex(x, r, w, b, 1e-5, oracle.ACT_RELU, p=0.1, seed=77)
    keep = oracle.dropout_mask(77, 0, 0, x.size, 0.1).reshape(shape)
    check_dropout(to_host(out), want, keep, True, "graph")


def test_pages_chain_full_size():
    """LayerNorm -> ReLU -> Dropout(p = 0.1) on the fp32 8192 x 4096 rows: every
    row against the oracle (keep mask exact, values, statistics), and the keep
    rate over the whole tensor within 5 sigma of 0.9."""
    wl = W.LNACT_RELU_DROP_F32
    t = wl.generate_all()
    p, seed, offset = wl.params["p"], wl.params["seed"], wl.params["offset"]
    d = {k: to_dev(v) for k, v in t.items()}
    out, _, mean, rstd = mb.fused_layernorm_act(d["x"], None, d["w"], d["b"], eps=1e-5,
                                                act="relu", p=p, seed=seed, offset=offset,
                                                want_stats=True)
    torch.cuda.synchronize()
    got, got_mean, got_rstd = to_host(out), to_host(mean), to_host(rstd)
    cols = wl.cols

    def block(r0, r1):
        want, _, wm, wr = oracle.layernorm_act_ex(
            t["x"][r0:r1], None, t["w"], t["b"], 1e-5, oracle.ACT_RELU, p=p, seed=seed,
            offset=dropout_block_offset(offset, r0, cols), want_stats=True)
        keep = oracle.dropout_mask(seed, offset, r0 * cols, (r1 - r0) * cols, p)
        what = f"{wl.name} rows {r0}:{r1}"
        check_dropout(got[r0:r1], want, keep.reshape(r1 - r0, cols), False, what)
        check_stats(got_mean[r0:r1], got_rstd[r0:r1], wm, wr, what)
        return int(keep.sum())

    kept = sum(map_row_blocks(wl.rows, block, align=8))
    n = wl.rows * cols
    sigma = (n * p * (1 - p)) ** 0.5
    assert abs(kept - n * (1 - p)) <= 5 * sigma
    # every element: nonzero iff kept and relu gave a nonzero value
    nonzero = int((out != 0).sum().item())
    positive = int((mb.fused_layernorm_act(d["x"], None, d["w"], d["b"], act="relu") > 0)
                   .sum().item())
    sigma = (positive * p * (1 - p)) ** 0.5
    assert abs(nonzero - positive * (1 - p)) <= 5 * sigma
    assert n > positive > n // 4


def test_host_memory_rows():
    """Zero copy: rows in pinned host memory, dropout and statistics."""
    shape = (96, 4096)
    x, r, w, b = _inputs(*shape, 955, False)
    hx = torch.from_numpy(x).pin_memory()
    hr = torch.from_numpy(r).pin_memory()
    out, _, mean, rstd = mb.fused_layernorm_act(hx, hr, to_dev(w), to_dev(b), act="relu", p=0.2,
                                                seed=4, want_stats=True)
    torch.cuda.synchronize()
    assert out.device.type == "cpu" and mean.device.type == "cpu"
    want, _, wm, wr = oracle.layernorm_act_ex(x, r, w, b, 1e-5, oracle.ACT_RELU, p=0.2, seed=4,
                                              want_stats=True)
    keep = oracle.dropout_mask(4, 0, 0, x.size, 0.2).reshape(shape)
    check_dropout(out.numpy(), want, keep, False, "host")
    check_stats(mean, rstd, wm, wr, "host")
