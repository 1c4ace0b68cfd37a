"""Maximum sizes: tensors of more than 2^31 elements, so that every engine's
64-bit indexing is exercised past the 32-bit boundary (pointwise, the staged
and direct CTA row engines, the warp row engine).

Inputs are a seeded block from synth tiled on the device (row or element i
takes block entry i mod B, B chosen coprime to powers of two).  Every element
is checked: the first period against the oracle, and every later period bit
for bit against the first on the device (the chains are row- or
element-local, so equal inputs give equal outputs wherever they sit); the
elements around index 2^31 and the last ones are also compared with the
oracle directly.  Dropout keys its decisions by the element's index, so that
test runs the oracle over every row in blocks on the host's cores.  About
35 GB of device memory per test.
"""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth

from gpu_util import assert_bitexact, assert_close, to_dev, to_host
from row_blocks import dropout_block_offset, map_row_blocks

pytestmark = pytest.mark.gpu

TWO31 = 1 << 31


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


@pytest.fixture(autouse=True)
def free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _tile(block, n_lead):
    """Device tensor whose leading dimension is n_lead, entry i = block[i % B]."""
    d = to_dev(block)
    reps = -(-n_lead // block.shape[0])
    return d.repeat((reps,) + (1,) * (block.ndim - 1))[:n_lead].contiguous()


def _assert_periodic(t, B, what):
    """Each period of B entries along t's leading dimension equals the first,
    bit for bit (the ragged last period against the first's prefix)."""
    bits = t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)
    first = bits[:B]
    for k0 in range(B, t.shape[0], B):
        seg = bits[k0:k0 + B]
        assert torch.equal(seg, first[:seg.shape[0]]), f"{what}: period at {k0} differs"


def _sample(n, count=64, seed=5):
    rng = np.random.default_rng(seed)
    pick = {0, n - 1, TWO31 - 1, TWO31, TWO31 + 1} | set(rng.integers(0, n, count).tolist())
    return np.array(sorted(i for i in pick if 0 <= i < n), np.int64)


def test_pointwise_beyond_2_31():
    n = TWO31 + (1 << 20) + 3
    B = (1 << 20) + 7
    blk = [synth.normal(1001, k, (B,)) for k in range(3)]
    x, b1, b2 = (_tile(b, n) for b in blk)
    y = mb.fused_add_relu_scale(x, b1, b2, 0.5)
    idx = _sample(n)
    got = to_host(y[torch.from_numpy(idx).cuda()])
    j = idx % B
    want = oracle.add_relu_scale(blk[0][j], blk[1][j], blk[2][j], 0.5)
    assert_bitexact(got, want, "pointwise > 2^31")
    assert_bitexact(to_host(y[:B]), oracle.add_relu_scale(*blk, 0.5), "pointwise first period")
    _assert_periodic(y, B, "pointwise > 2^31")


@pytest.mark.parametrize("path", ["auto", "direct"])
def test_layernorm_rows_beyond_2_31(path):
    mb.set_row_path(path)
    cols = 4096
    rows = TWO31 // cols + 3                     # rows * cols > 2^31
    B = 997
    x_b, r_b = synth.normal(1002, 0, (B, cols)), synth.normal(1002, 1, (B, cols))
    w = synth.uniform(1002, 2, (cols,), 0.5, 1.5)
    b = synth.normal(1002, 3, (cols,), 0.0, 0.1)
    x, r = _tile(x_b, rows), _tile(r_b, rows)
    out = mb.fused_residual_layernorm_gelu(x, r, to_dev(w), to_dev(b), 1e-5)
    rows_s = np.unique(np.r_[_sample(rows, 24) , [TWO31 // cols - 1, TWO31 // cols]])
    got = to_host(out[torch.from_numpy(rows_s).cuda()])
    j = rows_s % B
    want = oracle.residual_layernorm_gelu(x_b[j], r_b[j], w, b, 1e-5)
    assert_close(got, want, what=f"LN rows > 2^31 elements ({path})")
    assert_close(to_host(out[:B]), oracle.residual_layernorm_gelu(x_b, r_b, w, b, 1e-5),
                 what=f"LN first period ({path})")
    _assert_periodic(out, B, f"LN rows > 2^31 elements ({path})")


def test_warp_rows_beyond_2_31():
    """The Inductor chain's warp-per-row engine on 2^21 + 5 rows of 1024."""
    cols = 1024
    rows = TWO31 // cols + 5
    B = 1009
    x_b = synth.normal(1003, 0, (B, cols))
    bias = synth.normal(1003, 1, (cols,), 0.0, 0.1)
    gamma = synth.uniform(1003, 2, (cols,), 0.5, 1.5)
    beta = synth.normal(1003, 3, (cols,), 0.0, 0.1)
    x = _tile(x_b, rows)
    y = mb.fused_bias_relu_branch_mean_epilogue(x, to_dev(bias), to_dev(gamma), to_dev(beta))
    rows_s = np.unique(np.r_[_sample(rows, 24), [TWO31 // cols - 1, TWO31 // cols]])
    got = to_host(y[torch.from_numpy(rows_s).cuda()])
    want = oracle.bias_relu_branch_mean_epilogue(x_b[rows_s % B], bias, gamma, beta)
    assert_close(got, want, what="Inductor rows > 2^31 elements")
    assert_close(to_host(y[:B]), oracle.bias_relu_branch_mean_epilogue(x_b, bias, gamma, beta),
                 what="Inductor first period")
    _assert_periodic(y, B, "Inductor rows > 2^31 elements")


def test_softmax_rows_beyond_2_31():
    cols = 8192
    rows = TWO31 // cols + 2
    B = 499
    x_b = synth.normal(1004, 0, (B, cols), 0.0, 2.0)
    x = _tile(x_b, rows)
    y = mb.fused_row_softmax(x)
    rows_s = np.unique(np.r_[_sample(rows, 16), [TWO31 // cols - 1, TWO31 // cols]])
    got = to_host(y[torch.from_numpy(rows_s).cuda()]).astype(np.float64)
    want = oracle.row_softmax(x_b[rows_s % B]).astype(np.float64)
    assert np.all(np.abs(got - want) <= 1e-5 * want + 2.0 ** -126)
    got = to_host(y[:B]).astype(np.float64)
    want = oracle.row_softmax(x_b).astype(np.float64)
    assert np.all(np.abs(got - want) <= 1e-5 * want + 2.0 ** -126)
    _assert_periodic(y, B, "softmax rows > 2^31 elements")


def test_layernorm_dropout_rows_beyond_2_31():
    """Dropout decisions keyed by element indices past 2^31 (the Philox
    counter takes the 64-bit index): sampled rows' masks and values."""
    cols = 4096
    rows = TWO31 // cols + 3
    B = 991
    x_b = synth.normal(1005, 0, (B, cols))
    w = synth.uniform(1005, 2, (cols,), 0.5, 1.5)
    b = synth.normal(1005, 3, (cols,), 0.0, 0.1)
    x = _tile(x_b, rows)
    p, seed, offset = 0.1, 31337, 12
    out = mb.fused_layernorm_act(x, None, to_dev(w), to_dev(b), act="relu", p=p, seed=seed,
                                 offset=offset)
    torch.cuda.synchronize()
    got = to_host(out)
    assert got.shape == (rows, cols)

    def block(r0, r1):
        want, _, _, _ = oracle.layernorm_act_ex(
            x_b[np.arange(r0, r1) % B], None, w, b, 1e-5, oracle.ACT_RELU, p=p, seed=seed,
            offset=dropout_block_offset(offset, r0, cols))
        keep = oracle.dropout_mask(seed, offset, r0 * cols, (r1 - r0) * cols, p)
        g, k = got[r0:r1].reshape(-1), keep
        what = f"dropout rows {r0}:{r1} (> 2^31 elements)"
        assert np.all(g[~k] == 0), what
        assert np.all(g[k & (want.reshape(-1) != 0)] != 0), what
        return assert_close(got[r0:r1], want, what=what)

    map_row_blocks(rows, block, align=8)
