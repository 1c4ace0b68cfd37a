"""A seeded random sweep over every chain: row counts, row lengths (short,
ragged, just past a vector or a CTA, long enough for the cluster path, off
the 16-byte grid at every length),
dtypes, 16-byte-aligned or offset views, forced row engines, host or device
memory for the rows, and the chains' options; each case against the CPU
oracle.  Rows of 65544 and 131080 elements reach the cluster kernels that
stage or hold slices of 64 KB and more.  The cases are drawn once from a fixed seed, so a failure names a
reproducible case."""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth

from gpu_util import assert_bitexact, assert_close, bf16_to_f64, to_dev
from gpu_util import to_host as _to_host

pytestmark = pytest.mark.gpu

CHAINS = ["pointwise", "bcast", "inductor", "ln_gelu", "lnact", "softmax", "softmax_mask"]
PATHS = ["auto", "warp", "direct", "staged", "cluster"]


def _cases(n=300, seed=20240601):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        chain = CHAINS[i % len(CHAINS)]
        cols = int(rng.choice([1, 2, 3, 7, 8, 31, 64, 255, 256, 257, 1000, 1024, 2049, 4096, 4099,
                               4100, 8192, 12291, 16384, 32769, 40000, 50257, 65537, 65544,
                               131080]))
        rows = int(rng.integers(1, 40 if cols > 16384 else 200))
        out.append(dict(i=i, chain=chain, rows=rows, cols=cols,
                        bf16=bool(rng.integers(0, 2)) and chain != "inductor",
                        offset_view=bool(rng.integers(0, 4) == 0),
                        host=bool(rng.integers(0, 6) == 0),
                        path=PATHS[int(rng.integers(0, len(PATHS)))],
                        opt=int(rng.integers(0, 1 << 30))))
    return out


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from memory_bound_gb300 import build as lib_build
    lib_build.build()
    torch.cuda.set_device(0)
    yield
    mb.set_row_path("auto")
    torch.cuda.synchronize()
    assert mb.device_error() == 0


def to_host(t):
    """Outputs in pinned host memory are written asynchronously by the
    kernels: synchronise before reading them (a device tensor's copy to the
    host synchronises by itself)."""
    torch.cuda.synchronize()
    return _to_host(t)


def _place(a, bf16, offset_view, host):
    """A contiguous tensor holding a (one element past a 16-byte boundary when
    offset_view), on the device or in pinned host memory."""
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else np.ascontiguousarray(a))
    if bf16:
        t = t.view(torch.bfloat16)
    n = t.numel()
    if host:
        buf = torch.empty(n + 1, dtype=t.dtype, pin_memory=True)
    else:
        buf = torch.empty(n + 1, dtype=t.dtype, device="cuda")
    v = buf[1:] if offset_view else buf[:n]
    v.copy_(t.reshape(-1))
    return v.view(a.shape)


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"{c['i']}-{c['chain']}")
def test_random_case(case):
    c = case
    rows, cols, bf16 = c["rows"], c["cols"], c["bf16"]
    dt = "bf16" if bf16 else "f32"
    rng = np.random.default_rng(c["opt"])
    mb.set_row_path(c["path"])
    try:
        put = lambda a, host=c["host"]: _place(a, bf16, c["offset_view"], host)
        seed = 3000 + c["i"]
        if c["chain"] == "pointwise":
            n = rows * cols
            x, b1, b2 = (synth.normal(seed, k, (n,), dtype=dt) for k in range(3))
            y = to_host(mb.fused_add_relu_scale(put(x), put(b1), put(b2), 0.75))
            want = oracle.add_relu_scale(x, b1, b2, 0.75)
            assert_bitexact(y, want, str(c))
            return
        x = synth.normal(seed, 0, (rows, cols), 0.0, 2.0, dtype=dt)
        if c["chain"] == "bcast":
            b1 = synth.normal(seed, 1, (cols,), dtype=dt)
            b2 = synth.normal(seed, 2, (rows, cols) if rng.integers(0, 2) else (cols,), dtype=dt)
            y = to_host(mb.fused_add_relu_scale(put(x), to_dev(b1, bf16), put(b2) if b2.ndim == 2
                                                else to_dev(b2, bf16), 0.5))
            assert_bitexact(y, oracle.add_relu_scale_bcast(x, b1, b2, 0.5), str(c))
            return
        w = synth.uniform(seed, 2, (cols,), 0.5, 1.5, dtype=dt)
        b = synth.normal(seed, 3, (cols,), 0.0, 0.1, dtype=dt)
        if c["chain"] == "inductor":
            y = to_host(mb.fused_bias_relu_branch_mean_epilogue(put(x), to_dev(b), to_dev(w),
                                                                to_dev(b), 1.1, 0.1))
            assert_close(y, oracle.bias_relu_branch_mean_epilogue(x, b, w, b), what=str(c))
            return
        if c["chain"] == "ln_gelu":
            r = synth.normal(seed, 1, (rows, cols), dtype=dt)
            y = to_host(mb.fused_residual_layernorm_gelu(put(x), put(r), to_dev(w, bf16),
                                                         to_dev(b, bf16), 1e-5))
            assert_close(y, oracle.residual_layernorm_gelu(x, r, w, b, 1e-5), bf16=bf16,
                         what=str(c))
            return
        if c["chain"] == "lnact":
            res = bool(rng.integers(0, 2))
            act = ["none", "relu", "gelu_tanh"][int(rng.integers(0, 3))]
            p = [0.0, 0.1, 0.5][int(rng.integers(0, 3))]
            r = synth.normal(seed, 1, (rows, cols), dtype=dt) if res else None
            out, h, mean, rstd = mb.fused_layernorm_act(
                put(x), put(r) if res else None, to_dev(w, bf16), to_dev(b, bf16), 1e-5, act=act,
                want_h=True, p=p, seed=seed, offset=c["opt"] % 1000, want_stats=True)
            want, want_h, wm, wr = oracle.layernorm_act_ex(
                x, r, w, b, 1e-5, {"none": 0, "relu": 1, "gelu_tanh": 2}[act], p=p, seed=seed,
                offset=c["opt"] % 1000, want_h=True, want_stats=True)
            got = to_host(out)
            if p > 0:
                keep = oracle.dropout_mask(seed, c["opt"] % 1000, 0, rows * cols, p)
                g = (bf16_to_f64(got) if bf16 else got.astype(np.float64)).reshape(-1)
                assert np.all(g[~keep] == 0), str(c)
            assert_close(got, want, bf16=bf16, what=str(c))
            assert_bitexact(to_host(h), want_h, str(c))
            m, s = to_host(mean).astype(np.float64), to_host(rstd).astype(np.float64)
            assert np.all(np.abs(m - wm) <= 1e-5 / wr + 1e-7 * np.abs(wm)), str(c)
            assert np.all(np.abs(s - wr) <= 1e-5 * wr), str(c)
            return
        if c["chain"] == "softmax":
            y = to_host(mb.fused_row_softmax(put(x)))
            want = oracle.row_softmax(x)
            causal_mask = None
        else:
            period = int(rng.integers(1, rows + 1))
            off = int(rng.integers(0, cols + 2))
            scale = float(rng.choice([0.125, 0.3, 1.0]))
            y = to_host(mb.fused_row_softmax(put(x), scale=scale, causal=True, period=period,
                                             offset=off))
            want = oracle.scale_mask_softmax(x, scale, True, period, off)
            causal_mask = np.arange(cols)[None, :] > (np.arange(rows)[:, None] % period + off)
        g = bf16_to_f64(y) if bf16 else y.astype(np.float64)
        wv = bf16_to_f64(want) if bf16 else want.astype(np.float64)
        if causal_mask is not None:
            assert np.all(g[causal_mask] == 0), str(c)
        rtol = 1e-2 if bf16 else 1e-5
        assert np.all(np.abs(g - wv) <= rtol * np.abs(wv) + 2.0 ** -126), str(c)
    finally:
        mb.set_row_path("auto")
