"""Rows off the 16-byte grid: lengths that are not whole 16-byte vectors, and
tensors that start off a 16-byte boundary.  When every row tensor of a call
starts at the same offset within 16 bytes, rows up to one CTA's reach take
the shifted-vector engine (a short head, whole 16-byte vectors, a short
tail); otherwise the scalar forms of the one-CTA engine (16 and 32 slots
bounded at 512 threads where the 1024-thread form spills) and past one CTA
the cluster engine.  Every chain against the oracle, with the placements
that select each path; the full ragged workload (8192 x 4099 fp32, the
benchmark's row) on every element."""
import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth
from synth import workloads as W

from gpu_util import assert_bitexact, assert_close, bf16_to_f64, report, to_dev, to_host
from row_blocks import map_row_blocks, worst

pytestmark = pytest.mark.gpu

LENGTHS = [4099, 8195, 12291, 16383, 16385, 24579, 32767]


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


def _dev(a, bf16, offset):
    """A device copy of a, starting `offset` elements into its allocation."""
    d = to_dev(a, bf16)
    if not offset:
        return d
    flat = torch.empty(d.numel() + offset, dtype=d.dtype, device=d.device)
    v = flat[offset:].view(d.shape)
    v.copy_(d)
    return v


def _rows(rows, cols, seed, bf16, n):
    dt = "bf16" if bf16 else "f32"
    return [synth.normal(seed, k, (rows, cols), dtype=dt) for k in range(n)]


def _vecs(cols, seed, bf16):
    dt = "bf16" if bf16 else "f32"
    return (synth.uniform(seed, 2, (cols,), 0.5, 1.5, dtype=dt),
            synth.normal(seed, 3, (cols,), 0.0, 0.1, dtype=dt))


def _out_like(x, bf16, offset):
    """An output tensor like x, starting `offset` elements into its allocation."""
    dt = torch.bfloat16 if bf16 else torch.float32
    flat = torch.empty(x.size + offset, dtype=dt, device="cuda")
    return flat[offset:].view(x.shape)


# placements: every tensor 16-byte aligned; the row inputs one element off
# (the output aligned: no common offset, the scalar path); inputs and output
# one element off (a common offset: the shifted-vector path)
PLACES = {"base": (0, 0), "inputs_off": (1, 0), "all_off": (1, 1)}


@pytest.mark.parametrize("cols", LENGTHS + [1031, 2053])
@pytest.mark.parametrize("path", ["auto", "direct", "cluster"])
@pytest.mark.parametrize("place", sorted(PLACES))
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_ln_gelu_unaligned(cols, path, place, bf16):
    mb.set_row_path(path)
    try:
        rows = 37
        xo, oo = PLACES[place]
        x, r = _rows(rows, cols, cols + 1, bf16, 2)
        w, b = _vecs(cols, cols + 1, bf16)
        out = _out_like(x, bf16, oo)
        mb.fused_residual_layernorm_gelu(_dev(x, bf16, xo), _dev(r, bf16, xo), to_dev(w, bf16),
                                         to_dev(b, bf16), 1e-5, out=out)
        assert_close(to_host(out), oracle.residual_layernorm_gelu(x, r, w, b, 1e-5), bf16=bf16,
                     what=f"{cols} {path} {place}")
    finally:
        mb.set_row_path("auto")


@pytest.mark.parametrize("cols", [4096 + 3, 8192 + 5, 1024 + 1])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_shifted_path_is_planned(cols, bf16):
    """Rows off the 16-byte grid with a common offset plan on 16-byte
    vectors (path direct, or staged with the per-column copies and a ring;
    the vector width), not on the scalar path; the dropout chains too (their
    slots are 8 elements)."""
    dt = "bf16" if bf16 else "f32"
    vec = 8 if bf16 else 4
    for chain in ("ln", "inductor", "lnact", "lnact_res", "softmax", "softmax_mask"):
        if chain == "inductor" and bf16:
            continue
        for al in (1, 2):
            p = mb.row_plan(chain, dt, 512, cols, aligned=al)
            assert p["path"] in ("direct", "staged") and p["vec"] == vec, (chain, al, p)
        assert mb.row_plan(chain, dt, 512, cols, aligned=0)["vec"] == 1
    for chain in ("lnact_dropout", "lnact_res_dropout"):
        p = mb.row_plan(chain, dt, 512, cols, aligned=1)
        assert p["path"] in ("direct", "staged") and p["vec"] == 8, (chain, p)


@pytest.mark.parametrize("cols", [1031, 4099, 12291])
@pytest.mark.parametrize("chain", ["inductor", "lnact_h", "softmax", "softmax_mask"])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_shifted_chains(cols, chain, bf16):
    """Every chain on the shifted-vector path with a non-zero common offset:
    inputs and outputs two elements into their allocations."""
    if chain == "inductor" and bf16:
        pytest.skip("the bf16 Inductor entry point is tested by test_gpu_next")
    rows, off = 23, 2
    dt = "bf16" if bf16 else "f32"
    x = synth.normal(cols + 3, 0, (rows, cols), dtype=dt)
    if chain == "inductor":
        bias = synth.normal(cols + 3, 1, (cols,), 0.0, 0.1)
        gamma = synth.uniform(cols + 3, 2, (cols,), 0.5, 1.5)
        beta = synth.normal(cols + 3, 3, (cols,), 0.0, 0.1)
        y = _out_like(x, False, off)
        mb.fused_bias_relu_branch_mean_epilogue(_dev(x, False, off), to_dev(bias), to_dev(gamma),
                                                to_dev(beta), 1.1, 0.1, out=y)
        assert_close(to_host(y), oracle.bias_relu_branch_mean_epilogue(x, bias, gamma, beta),
                     what=f"inductor {cols}")
    elif chain == "lnact_h":
        r = synth.normal(cols + 3, 1, (rows, cols), dtype=dt)
        w, b = _vecs(cols, cols + 3, bf16)
        out, h = _out_like(x, bf16, off), _out_like(x, bf16, off)
        mb.fused_layernorm_act(_dev(x, bf16, off), _dev(r, bf16, off), to_dev(w, bf16),
                               to_dev(b, bf16), act="gelu_tanh", out=out, h_out=h)
        want, want_h = oracle.layernorm_act(x, r, w, b, 1e-5, oracle.ACT_GELU, want_h=True)
        assert_close(to_host(out), want, bf16=bf16, what=f"lnact {cols}")
        assert_bitexact(to_host(h), want_h, f"h {cols}")
    else:
        y = _out_like(x, bf16, off)
        if chain == "softmax":
            mb.fused_row_softmax(_dev(x, bf16, off), out=y)
            want = oracle.row_softmax(x)
        else:
            mb.fused_row_softmax(_dev(x, bf16, off), out=y, scale=0.25, causal=True, period=rows,
                                 offset=cols // 3)
            want = oracle.scale_mask_softmax(x, 0.25, True, rows, cols // 3)
        g = bf16_to_f64(to_host(y)) if bf16 else to_host(y).astype(np.float64)
        w_ = bf16_to_f64(want) if bf16 else want.astype(np.float64)
        rtol = 1e-2 if bf16 else 1e-5
        assert np.all(np.abs(g - w_) <= rtol * np.abs(w_) + 2.0 ** -126), f"{chain} {cols}"
        if chain == "softmax_mask":
            masked = np.arange(cols)[None, :] > (np.arange(rows)[:, None] % rows + cols // 3)
            assert np.all(g[masked] == 0)


@pytest.mark.parametrize("cols", LENGTHS)
@pytest.mark.parametrize("chain", ["inductor", "lnact_relu", "lnact_dropout", "softmax"])
def test_chains_unaligned(cols, chain):
    rows = 29
    if chain == "inductor":
        x = synth.normal(cols, 0, (rows, cols))
        bias = synth.normal(cols, 1, (cols,), 0.0, 0.1)
        gamma = synth.uniform(cols, 2, (cols,), 0.5, 1.5)
        beta = synth.normal(cols, 3, (cols,), 0.0, 0.1)
        y = mb.fused_bias_relu_branch_mean_epilogue(_dev(x, False, 1), to_dev(bias),
                                                    to_dev(gamma), to_dev(beta), 1.1, 0.1)
        assert_close(to_host(y), oracle.bias_relu_branch_mean_epilogue(x, bias, gamma, beta),
                     what=f"inductor {cols}")
    elif chain.startswith("lnact"):
        x = synth.normal(cols + 5, 0, (rows, cols))
        w, b = _vecs(cols, cols + 5, False)
        p = 0.1 if chain == "lnact_dropout" else 0.0
        out = mb.fused_layernorm_act(_dev(x, False, 1), None, to_dev(w), to_dev(b), act="relu",
                                     p=p, seed=99)
        want, _, _, _ = oracle.layernorm_act_ex(x, None, w, b, 1e-5, oracle.ACT_RELU, p=p, seed=99)
        got = to_host(out)
        if p:
            keep = oracle.dropout_mask(99, 0, 0, x.size, p).reshape(x.shape)
            assert np.all(got[~keep] == 0)
        assert_close(got, want, what=f"{chain} {cols}")
    else:
        x = synth.normal(cols + 9, 0, (rows, cols), 0.0, 2.0)
        y = mb.fused_row_softmax(_dev(x, False, 1))
        g, w = to_host(y).astype(np.float64), oracle.row_softmax(x).astype(np.float64)
        assert np.all(np.abs(g - w) <= 1e-5 * w + 2.0 ** -126), f"softmax {cols}"


def test_ragged_workload_full_size():
    """ln_gelu_f32_8192x4099 (the benchmark's unaligned row): every element."""
    w = W.LN_F32_RAGGED
    t = w.generate_all()
    assert mb.row_plan("ln", "f32", w.rows, w.cols)["vec"] == 4      # shifted vectors
    out = mb.fused_residual_layernorm_gelu(to_dev(t["x"]), to_dev(t["r"]), to_dev(t["w"]),
                                           to_dev(t["b"]), 1e-5)
    torch.cuda.synchronize()
    got = to_host(out)

    def block(r0, r1):
        want = oracle.residual_layernorm_gelu(t["x"][r0:r1], t["r"][r0:r1], t["w"], t["b"], 1e-5)
        return assert_close(got[r0:r1], want, what=f"{w.name} rows {r0}:{r1}")

    err, ratio = worst(map_row_blocks(w.rows, block))
    report(w.name, max_abs_err=err, max_err_over_bar=ratio)


@pytest.mark.parametrize("cols", [1031, 4099, 4100, 12291])
@pytest.mark.parametrize("res", [False, True], ids=["nores", "res"])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_shifted_dropout(cols, res, bf16):
    """LayerNorm -> ReLU -> Dropout on the shifted-vector path (slots that
    start anywhere within a Philox block of eight): the keep mask exact on
    every element, values at the bar, row statistics; inputs and outputs at a
    common offset of three elements, and a generator offset that is not a
    multiple of the row's blocks."""
    rows, off, p, seed, goff = 19, 3, 0.3, 4321, 7
    dt = "bf16" if bf16 else "f32"
    x = synth.normal(cols + 11, 0, (rows, cols), dtype=dt)
    r = synth.normal(cols + 11, 1, (rows, cols), dtype=dt) if res else None
    w, b = _vecs(cols, cols + 11, bf16)
    out = _out_like(x, bf16, off)
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    mb.fused_layernorm_act(_dev(x, bf16, off), _dev(r, bf16, off) if res else None,
                           to_dev(w, bf16), to_dev(b, bf16), act="relu", out=out, p=p, seed=seed,
                           offset=goff, mean_out=mean, rstd_out=rstd)
    want, _, wm, wr = oracle.layernorm_act_ex(x, r, w, b, 1e-5, oracle.ACT_RELU, p=p, seed=seed,
                                              offset=goff, want_stats=True)
    keep = oracle.dropout_mask(seed, goff, 0, x.size, p).reshape(x.shape)
    got = to_host(out)
    g = bf16_to_f64(got) if bf16 else got.astype(np.float64)
    wv = bf16_to_f64(want) if bf16 else want.astype(np.float64)
    assert np.all(g[~keep] == 0), "a dropped element is not zero"
    assert np.all(g[keep & (wv != 0)] != 0), "a kept element was dropped"
    assert_close(got, want, bf16=bf16, what=f"dropout {cols} res={res}")
    m, rs = to_host(mean).astype(np.float64), to_host(rstd).astype(np.float64)
    assert np.all(np.abs(m - wm) <= 1e-5 / wr + 1e-7 * np.abs(wm))
    assert np.all(np.abs(rs - wr) <= 1e-5 * wr)


def test_scalar_reach_and_cluster_boundary():
    """Rows with no common offset take the scalar one-CTA forms up to 16384
    elements (the reach of the 32-slot form, bounded at 512 threads so it
    holds its values in registers), the cluster engine past that; with a
    common offset the same rows take shifted vectors up to one CTA's vector
    reach (32768 elements)."""
    for cols in (16383, 16384):
        p = mb.row_plan("ln", "f32", 64, cols, aligned=0)
        assert p["path"] == "direct" and p["vec"] == 1, p
    p = mb.row_plan("ln", "f32", 64, 16385, aligned=0)
    assert p["path"] == "cluster" and p["vec"] == 1, p
    for cols in (16385, 32767):
        p = mb.row_plan("ln", "f32", 64, cols, aligned=2)
        assert p["path"] == "direct" and p["vec"] == 4, p
    assert mb.row_plan("ln", "f32", 64, 32769, aligned=2)["path"] == "cluster"


def _multi_round_rows(chain, dt, cols):
    """A row count that gives every CTA of the shifted launch two or three
    rows (the per-column copies are planned from two rows a CTA on)."""
    cap = mb.row_plan(chain, dt, 1 << 22, cols, aligned=2)["ctas"]
    return 2 * cap + 5


def _copy_shape(pchain, dt, staged):
    """The first of a few row lengths off the 16-byte grid (with a row count
    of several rows a CTA) that the planner serves with the per-column
    copies, on the staged path (staged; the automatic choice) or the direct
    one (the path asked for); every chain with per-column arrays has both."""
    for cols in (4099, 1031, 2051, 8195):
        rows = _multi_round_rows(pchain, dt, cols)
        plan = mb.row_plan(pchain, dt, rows, cols, aligned=2)
        if plan["smem"] > 1024 and (plan["path"] == "staged") == staged:
            return cols, rows, plan
    pytest.fail(f"no length takes the {'staged' if staged else 'direct'} per-column copies "
                f"for {pchain} {dt}")


@pytest.mark.parametrize("form,chain", [("staged", "ln"), ("staged", "inductor"),
                                        ("staged", "lnact_h"), ("copies", "ln"),
                                        ("copies", "inductor"), ("copies", "lnact_h"),
                                        ("copies", "lnact_dropout")])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("col_off", [0, 1], ids=["cols16", "cols_off"])
def test_shifted_column_copies(form, chain, bf16, col_off):
    """The shifted kernel with its per-column arrays copied to shared memory
    (several rows a CTA), with and without its bulk-copy ring for the rows'
    vectors (the dropout chains have no staged form): every chain that has
    such arrays, inputs and outputs at a common offset of one element, the
    per-column arrays 16-byte aligned or one element off (bf16: copied
    element by element where column h is not 4-byte aligned), every element
    against the oracle."""
    dt = "bf16" if bf16 else "f32"
    pchain = {"ln": "ln", "inductor": "inductor", "lnact_h": "lnact_res_h",
              "lnact_dropout": "lnact_res_dropout"}[chain]
    mb.set_row_path("auto" if form == "staged" else "direct")
    try:
        _shifted_column_copies(pchain, chain, dt, bf16, col_off, form == "staged")
    finally:
        mb.set_row_path("auto")


def _shifted_column_copies(pchain, chain, dt, bf16, col_off, staged):
    cols, rows, plan = _copy_shape(pchain, dt, staged)
    off = 1
    es = 2 if bf16 else 4
    narr = 3 if chain == "inductor" else 2
    nin = 1 if chain == "inductor" else 2
    assert plan["path"] == ("staged" if staged else "direct"), plan
    assert plan["vec"] in (8, 16 // es) and (plan["stages"] > 0) == staged, plan
    padded = (cols + 15) // 16 * 16
    # the copies, and the staged form's ring of plan["stages"] stages
    assert plan["smem"] == 1024 + (narr + plan["stages"] * nin) * padded * es, plan
    seed = cols + 17
    x = synth.normal(seed, 0, (rows, cols), dtype=dt)
    if chain == "inductor":
        bias = synth.normal(seed, 1, (cols,), 0.0, 0.1, dtype=dt)
        gamma = synth.uniform(seed, 2, (cols,), 0.5, 1.5, dtype=dt)
        beta = synth.normal(seed, 3, (cols,), 0.0, 0.1, dtype=dt)
        y = _out_like(x, bf16, off)
        mb.fused_bias_relu_branch_mean_epilogue(
            _dev(x, bf16, off), _dev(bias, bf16, col_off), _dev(gamma, bf16, col_off),
            _dev(beta, bf16, col_off), 1.1, 0.1, out=y)
        want = (oracle.bias_relu_branch_mean_epilogue_bf16(x, bias, gamma, beta) if bf16
                else oracle.bias_relu_branch_mean_epilogue(x, bias, gamma, beta))
        assert_close(to_host(y), want, bf16=bf16, what=f"inductor {cols}")
        return
    w, b = _vecs(cols, seed, bf16)
    wd, bd = _dev(w, bf16, col_off), _dev(b, bf16, col_off)
    if chain == "ln":
        r = synth.normal(seed, 1, (rows, cols), dtype=dt)
        out = _out_like(x, bf16, off)
        mb.fused_residual_layernorm_gelu(_dev(x, bf16, off), _dev(r, bf16, off), wd, bd, 1e-5,
                                         out=out)
        assert_close(to_host(out), oracle.residual_layernorm_gelu(x, r, w, b, 1e-5), bf16=bf16,
                     what=f"ln {cols}")
    elif chain == "lnact_h":
        r = synth.normal(seed, 1, (rows, cols), dtype=dt)
        out, h = _out_like(x, bf16, off), _out_like(x, bf16, off)
        mb.fused_layernorm_act(_dev(x, bf16, off), _dev(r, bf16, off), wd, bd, act="gelu_tanh",
                               out=out, h_out=h)
        want, want_h = oracle.layernorm_act(x, r, w, b, 1e-5, oracle.ACT_GELU, want_h=True)
        assert_close(to_host(out), want, bf16=bf16, what=f"lnact {cols}")
        assert_bitexact(to_host(h), want_h, f"h {cols}")
    else:
        r = synth.normal(seed, 1, (rows, cols), dtype=dt)
        p, dseed, goff = 0.2, 77, 5
        out = _out_like(x, bf16, off)
        mean = torch.empty(rows, device="cuda")
        rstd = torch.empty(rows, device="cuda")
        mb.fused_layernorm_act(_dev(x, bf16, off), _dev(r, bf16, off), wd, bd, act="relu",
                               out=out, p=p, seed=dseed, offset=goff, mean_out=mean,
                               rstd_out=rstd)
        want, _, wm, wr = oracle.layernorm_act_ex(x, r, w, b, 1e-5, oracle.ACT_RELU, p=p,
                                                  seed=dseed, offset=goff, want_stats=True)
        keep = oracle.dropout_mask(dseed, goff, 0, x.size, p).reshape(x.shape)
        got = to_host(out)
        g = bf16_to_f64(got) if bf16 else got.astype(np.float64)
        assert np.all(g[~keep] == 0), "a dropped element is not zero"
        assert_close(got, want, bf16=bf16, what=f"dropout {cols}")
        m, rs = to_host(mean).astype(np.float64), to_host(rstd).astype(np.float64)
        assert np.all(np.abs(m - wm) <= 1e-5 / wr + 1e-7 * np.abs(wm))
        assert np.all(np.abs(rs - wr) <= 1e-5 * wr)


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_shifted_column_copies_planning(bf16):
    """The copies are planned for launches of several rows a CTA, not for one
    row a CTA (there a copy costs as much as reading the values once), not
    for chains without per-column arrays, and not where they would not fit
    one CTA's shared memory (fp32 rows of 32767: 256 KB for w and b); the
    staged form with them, except for the dropout chains, and the staged
    ring alone for the row softmax."""
    dt = "bf16" if bf16 else "f32"
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for chain in ("ln", "inductor", "lnact", "lnact_res_dropout"):
        cap = mb.row_plan(chain, dt, 1 << 22, 4099, aligned=2)["ctas"]
        assert mb.row_plan(chain, dt, sms, 4099, aligned=2)["smem"] == 1024
        assert mb.row_plan(chain, dt, cap + 1, 4099, aligned=2)["smem"] > 1024
        # aligned rows keep their engines
        assert mb.row_plan(chain, dt, 4 * cap, 4096, aligned=1)["vec"] in (4, 8)
    # softmax has no per-column arrays: the ring alone, for bf16 rows
    p = mb.row_plan("softmax", dt, 1 << 20, 4099, aligned=2)
    if bf16:
        assert p["path"] == "staged" and p["smem"] == 1024 + p["stages"] * 4112 * 2, p
    else:
        assert p["path"] == "direct" and p["smem"] == 1024, p
    # the dropout chains keep the unstaged form; the others stage their rows
    for chain in ("lnact_dropout", "lnact_res_dropout"):
        p = mb.row_plan(chain, dt, 1 << 20, 4099, aligned=2)
        assert p["path"] == "direct" and p["stages"] == 0 and p["smem"] > 1024, p
    p = mb.row_plan("ln", dt, 1 << 20, 4099, aligned=2)
    assert p["path"] == "staged" and p["stages"] >= 1, p
    big = mb.row_plan("ln", dt, 1 << 20, 32767, aligned=2)
    assert big["path"] == "direct" and (big["smem"] == 1024) == (not bf16), big


def test_shifted_column_copies_host_vectors():
    """Per-column arrays in pinned host memory: the launch takes the kernel
    without copies (asynchronous copies are planned for device memory only)
    and still matches the oracle."""
    cols = 4099
    rows = _multi_round_rows("ln", "f32", cols)
    x, r = _rows(rows, cols, 5, False, 2)
    w, b = _vecs(cols, 5, False)
    hw, hb = (torch.from_numpy(v.copy()).pin_memory() for v in (w, b))
    out = _out_like(x, False, 1)
    mb.fused_residual_layernorm_gelu(_dev(x, False, 1), _dev(r, False, 1), hw, hb, 1e-5, out=out)
    torch.cuda.synchronize()
    assert_close(to_host(out), oracle.residual_layernorm_gelu(x, r, w, b, 1e-5),
                 what="host w, b")


@pytest.mark.parametrize("cols", [1031, 4099, 8195])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_shifted_softmax_staged(cols, bf16):
    """Row softmax on shifted rows of several rows a CTA: bf16 rows on the
    staged ring alone (the chain has no per-column arrays), fp32 rows
    unstaged; inputs and outputs one element into their allocations, every
    element against the oracle, and the unstaged form the direct path
    keeps."""
    dt = "bf16" if bf16 else "f32"
    rows = _multi_round_rows("softmax", dt, cols)
    plan = mb.row_plan("softmax", dt, rows, cols, aligned=2)
    es = 2 if bf16 else 4
    if bf16:
        assert plan["path"] == "staged" and plan["stages"] >= 1, plan
        assert plan["smem"] == 1024 + plan["stages"] * ((cols + 15) // 16 * 16) * es, plan
    else:
        assert plan["path"] == "direct" and plan["smem"] == 1024, plan
    x = synth.normal(cols + 29, 0, (rows, cols), 0.0, 2.0, dtype=dt)
    want = oracle.row_softmax(x)
    w_ = bf16_to_f64(want) if bf16 else want.astype(np.float64)
    rtol = 1e-2 if bf16 else 1e-5
    for path in ("auto", "direct"):
        mb.set_row_path(path)
        try:
            y = _out_like(x, bf16, 1)
            mb.fused_row_softmax(_dev(x, bf16, 1), out=y)
            g = to_host(y)
        finally:
            mb.set_row_path("auto")
        gv = bf16_to_f64(g) if bf16 else g.astype(np.float64)
        assert np.all(np.abs(gv - w_) <= rtol * np.abs(w_) + 2.0 ** -126), f"softmax {cols} {path}"


@pytest.mark.parametrize("cols", [32769, 50257, 65537])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("ring", [0, 1, 2], ids=["auto", "ring1", "ring2"])
def test_shifted_cluster_rows(cols, bf16, ring):
    """Rows longer than a CTA and off the 16-byte grid, whose tensors share an
    offset (here three elements): the cluster kernel's shifted form, each
    CTA's whole vectors loaded directly or staged through a ring of one or
    two stages, head and tail on rank 0.  LayerNorm + GeLU, the LayerNorm
    family with the residual stream and statistics, dropout (keep mask exact),
    softmax and the Inductor chain, every element against the oracle."""
    dt = "bf16" if bf16 else "f32"
    rows, off = 7, 3
    mb.set_row_path("cluster", ring, 0) if ring else mb.set_row_path("auto")
    try:
        p = mb.row_plan("ln", dt, rows, cols, aligned=2)
        assert p["path"] == "cluster" and p["vec"] == (8 if bf16 else 4), p
        assert (p["smem"] > 0) == (bool(ring) or bf16), p
        seed = cols % 1013
        x, r = _rows(rows, cols, seed, bf16, 2)
        w, b = _vecs(cols, seed, bf16)
        xd, rd, wd, bd = _dev(x, bf16, off), _dev(r, bf16, off), to_dev(w, bf16), to_dev(b, bf16)
        out = _out_like(x, bf16, off)
        mb.fused_residual_layernorm_gelu(xd, rd, wd, bd, 1e-5, out=out)
        assert_close(to_host(out), oracle.residual_layernorm_gelu(x, r, w, b, 1e-5), bf16=bf16,
                     what=f"ln {cols}")
        out, h = _out_like(x, bf16, off), _out_like(x, bf16, off)
        mean = torch.empty(rows, device="cuda")
        rstd = torch.empty(rows, device="cuda")
        mb.fused_layernorm_act(xd, rd, wd, bd, act="gelu_tanh", out=out, h_out=h,
                               mean_out=mean, rstd_out=rstd)
        want, want_h, wm, wr = oracle.layernorm_act_ex(x, r, w, b, 1e-5, oracle.ACT_GELU,
                                                       want_h=True, want_stats=True)
        assert_close(to_host(out), want, bf16=bf16, what=f"lnact {cols}")
        assert_bitexact(to_host(h), want_h, f"h {cols}")
        m, rs = to_host(mean).astype(np.float64), to_host(rstd).astype(np.float64)
        assert np.all(np.abs(m - wm) <= 1e-5 / wr + 1e-7 * np.abs(wm))
        assert np.all(np.abs(rs - wr) <= 1e-5 * wr)
        pd, seed_d, goff = 0.25, 99, 5
        out = _out_like(x, bf16, off)
        mb.fused_layernorm_act(xd, None, wd, bd, act="relu", out=out, p=pd, seed=seed_d,
                               offset=goff)
        want, _, _, _ = oracle.layernorm_act_ex(x, None, w, b, 1e-5, oracle.ACT_RELU, p=pd,
                                                seed=seed_d, offset=goff)
        keep = oracle.dropout_mask(seed_d, goff, 0, x.size, pd).reshape(x.shape)
        got = to_host(out)
        g = bf16_to_f64(got) if bf16 else got.astype(np.float64)
        assert np.all(g[~keep] == 0), "a dropped element is not zero"
        assert_close(got, want, bf16=bf16, what=f"dropout {cols}")
        y = _out_like(x, bf16, off)
        mb.fused_row_softmax(xd, out=y)
        ws = oracle.row_softmax(x)
        gv = bf16_to_f64(to_host(y)) if bf16 else to_host(y).astype(np.float64)
        wv = bf16_to_f64(ws) if bf16 else ws.astype(np.float64)
        rtol = 1e-2 if bf16 else 1e-5
        assert np.all(np.abs(gv - wv) <= rtol * np.abs(wv) + 2.0 ** -126), f"softmax {cols}"
        y = _out_like(x, bf16, off)
        mb.fused_bias_relu_branch_mean_epilogue(xd, bd, wd, bd, 1.1, 0.1, out=y)
        want = (oracle.bias_relu_branch_mean_epilogue_bf16(x, b, w, b) if bf16
                else oracle.bias_relu_branch_mean_epilogue(x, b, w, b))
        assert_close(to_host(y), want, bf16=bf16, what=f"inductor {cols}")
    finally:
        mb.set_row_path("auto")


def test_shifted_cluster_rows_many():
    """More shifted long rows than clusters fit at once (each cluster loops
    over rows whose heads differ), bf16 on the staged ring."""
    rows, cols, off = 300, 40001, 1
    x, r = _rows(rows, cols, 77, True, 2)
    w, b = _vecs(cols, 77, True)
    out = _out_like(x, True, off)
    assert mb.row_plan("ln", "bf16", rows, cols, aligned=2)["vec"] == 8
    mb.fused_residual_layernorm_gelu(_dev(x, True, off), _dev(r, True, off), to_dev(w, True),
                                     to_dev(b, True), 1e-5, out=out)
    assert_close(to_host(out), oracle.residual_layernorm_gelu(x, r, w, b, 1e-5), bf16=True,
                 what="ln 300 x 40001")
