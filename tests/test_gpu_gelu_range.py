"""The GeLU-tanh epilogue ("Operator fusion and kernel optimisation" §2.3:
0.5 n (1 + tanh(sqrt(2/pi) (n + 0.044715 n^3)))) over its whole argument
range on the GPU, against the oracle.

A constant row (x = c, r = 0, with c and the row length such that the row
sum is exact) has v - mean = 0 on both sides, so the normalised, affine value
is n = b[j] exactly and the chain's output is GeLU(b[j]).  The per-column b
then sets every argument: a dense fp32 grid over [-40, 40], the region where
the exponential of the sigmoid form leaves the fp32 range (|n| about 10),
values near 0, subnormals, signed zeros and huge magnitudes; in bf16, every
finite bf16 value.  Both GeLU entry points, on every row engine, in fp32 and
bf16, at the stated bars.  For n < 0 the result must be negative or a
negative zero (the oracle's values there are tiny negatives)."""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth

from gpu_util import assert_close, bf16_to_f64, max_rel_above, report, to_dev, to_host

pytestmark = pytest.mark.gpu

H = 1024                 # fits every engine, the one-warp engine included


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


def f32_grid():
    """GeLU arguments for the fp32 chains."""
    dense = np.linspace(-40.0, 40.0, 8001)                     # step 0.01
    edge = np.concatenate([np.linspace(-10.6, -9.4, 1201),     # 2^t overflow edge (n < 0)
                           np.linspace(9.4, 10.6, 1201)])      # 2^t underflow edge (n > 0)
    small = np.concatenate([s * np.logspace(-45, 0, 226) for s in (1.0, -1.0)])
    special = np.array([0.0, -0.0, 1e-3, -1e-3, 10.05, -10.05, 10.0, -10.0, 88.0, -88.0,
                        1e5, -1e5, 1e20, -1e20, 3.0e38, -3.0e38, 1.17549435e-38,
                        -1.17549435e-38, 1e-40, -1e-40])
    g = np.concatenate([dense, edge, small, special]).astype(np.float32)
    return g[np.isfinite(g)]


def bf16_grid():
    """Every finite bf16 value, as bit patterns."""
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    return h[(h & 0x7F80) != 0x7F80]          # exponent field not all ones


def _pad(vals, bf16, hidden=H):
    """Split into rows of `hidden` arguments (the last row padded with zeros)."""
    n = -(-vals.size // hidden) * hidden
    out = np.zeros(n, np.uint16 if bf16 else np.float32)
    out[:vals.size] = vals
    return out.reshape(-1, hidden)


def _run(entry, b, bf16):
    """One call on a constant row block: 4 rows of x = 0.75, r = 0 (or no
    residual), w from the generator, the given b (its length is the row
    length, a power of two, so the row sum and mean are exact)."""
    rows, hidden = 4, b.size
    x = np.full((rows, hidden), 0.75, np.float32)
    r = np.zeros((rows, hidden), np.float32)
    w = synth.uniform(4242, 2, (hidden,), 0.5, 1.5)
    if bf16:
        x, r, w = (synth.f32_to_bf16_bits(a) for a in (x, r, w))
    dx, dr, dw, db = (to_dev(a, bf16) for a in (x, r, w, b))
    if entry == "residual_layernorm_gelu":
        out = mb.fused_residual_layernorm_gelu(dx, dr, dw, db, 1e-5)
        want = oracle.residual_layernorm_gelu(x, r, w, b, 1e-5)
    elif entry == "layernorm_act_res":
        out = mb.fused_layernorm_act(dx, dr, dw, db, eps=1e-5, act="gelu_tanh")
        want = oracle.layernorm_act(x, r, w, b, 1e-5, oracle.ACT_GELU)
    else:
        out = mb.fused_layernorm_act(dx, None, dw, db, eps=1e-5, act="gelu_tanh")
        want = oracle.layernorm_act(x, None, w, b, 1e-5, oracle.ACT_GELU)
    torch.cuda.synchronize()
    return to_host(out), want


ENTRIES = ["residual_layernorm_gelu", "layernorm_act_res", "layernorm_act"]


@pytest.mark.parametrize("path", ["auto", "warp", "direct", "staged", "cluster"])
@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_gelu_whole_range(bf16, entry, path):
    mb.set_row_path(path)
    try:
        chunks = _pad(bf16_grid() if bf16 else f32_grid(), bf16)
        worst_ratio, worst_rel = 0.0, 0.0
        for k, b in enumerate(chunks):
            got, want = _run(entry, b, bf16)
            what = f"{entry} {path} {'bf16' if bf16 else 'f32'} chunk {k}"
            _, ratio = assert_close(got, want, bf16=bf16, what=what)
            worst_ratio = max(worst_ratio, ratio)
            worst_rel = max(worst_rel, max_rel_above(got, want, bf16))
            g = bf16_to_f64(got) if bf16 else got.astype(np.float64)
            n = bf16_to_f64(b) if bf16 else b.astype(np.float64)
            neg = n < 0
            assert np.all(g[:, neg] <= 0), f"{what}: a positive GeLU of a negative argument"
            zero_neg = neg[None, :] & (g == 0)
            assert np.all(np.signbit(g[zero_neg])), f"{what}: +0 for a negative argument"
            pos = n > 0
            assert np.all(g[:, pos] >= 0) and not np.any(np.signbit(g[:, pos])), \
                f"{what}: GeLU of a positive argument below +0"
        assert worst_ratio <= 1.0
        report(f"gelu range {entry} {path} {'bf16' if bf16 else 'f32'}",
               args=int(chunks.size), max_err_over_bar=worst_ratio,
               max_rel_err_where_abs_ge_1e_3=worst_rel)
    finally:
        mb.set_row_path("auto")


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_gelu_range_one_call_workload_row_length(bf16):
    """The same arguments in one call with the workload's row length (8192
    values a row), so the benchmark's launch shape runs them."""
    worst_ratio = 0.0
    for b in _pad(bf16_grid() if bf16 else f32_grid(), bf16, 8192):
        got, want = _run("residual_layernorm_gelu", b, bf16)
        worst_ratio = max(worst_ratio, assert_close(got, want, bf16=bf16, what="8192")[1])
    assert worst_ratio <= 1.0
