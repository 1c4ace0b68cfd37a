"""Pins of the CPU oracle against things other than itself.

Each ``pin_*`` takes a loaded oracle library (the real one, or a mutant built
by ``test_oracle_mutants.py``) and raises ``AssertionError`` when the oracle
disagrees with what the pages and the mathematics fix:

* hand-computed fixtures from ``tests/golden/`` (exact dyadic arithmetic,
  each citing the page whose formula it instantiates);
* closed forms and invariants (row mean of s - m is 0, the LayerNorm output
  before the affine step has mean 0 and variance var/(var+eps), GeLU's odd
  part is z/2, ...);
* special cases that reduce to library routines (torch CPU eager fp32 for
  the fp32 op sequences, torch float64 ``layer_norm`` / ``gelu``, torch's
  fp32 -> bf16 conversion).

Pages: [P1] "PyTorch operator fusion in practice" (0539edu.com), [P2]
"Operator fusion and kernel optimisation" (plumephp.com), [P3] course chapter
4 "Kernel fusion" (5688vip.com), [P4] "TorchInductor Pipeline and operator
fusion" (blog.kkkzoz.top).
"""
import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U32 = 2.0 ** -24   # unit roundoff of fp32


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


# --------------------------------------------------------------------------
# scalar helpers
# --------------------------------------------------------------------------

def pin_relu_cases(lib):
    """[P1] §3.2 writes relu as fmaxf(v, 0); the two cases fmaxf leaves open
    are fixed to +0 (see the readings)."""
    for v, want in ((1.5, 1.5), (-1.0, 0.0), (0.0, 0.0), (2.0 ** -149, 2.0 ** -149),
                    (-(2.0 ** -149), 0.0), (float("inf"), float("inf")),
                    (float("-inf"), 0.0)):
        got = oracle.relu_f32(v, lib=lib)
        assert got == want, (v, got, want)
    assert math.copysign(1.0, oracle.relu_f32(-0.0, lib=lib)) == 1.0
    got = oracle.relu_f32(float("nan"), lib=lib)
    assert got == 0.0 and math.copysign(1.0, got) == 1.0


def pin_gelu_library(lib):
    """GeLU tanh form ([P2] §2.3) against torch's float64
    gelu(approximate='tanh') over [-12, 12]."""
    z = np.linspace(-12.0, 12.0, 4801)
    want = F.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    got = np.array([oracle.gelu_tanh(v, lib=lib) for v in z])
    err = np.abs(got - want)
    # 1 + tanh(u) cancels for z << 0: absolute error ~ |z|/2 * 2^-52 there
    assert np.all(err <= 1e-14 * np.abs(want) + 1e-15 * np.abs(z)), err.max()


def pin_gelu_whole_range(lib):
    """GeLU tanh form against torch's float64 gelu(approximate='tanh') over
    the arguments the GPU range test feeds the kernels: a dense grid on
    [-40, 40], both 2^t overflow edges (|z| in [9.4, 10.6]), magnitudes from
    1e-45 to 1, signed zeros, subnormals, |z| up to 3e38, and every finite
    bf16 value.  Negative arguments give a result <= 0, positive ones >= 0."""
    grid = np.concatenate([
        np.linspace(-40.0, 40.0, 8001), np.linspace(-10.6, -9.4, 1201),
        np.linspace(9.4, 10.6, 1201), np.logspace(-45, 0, 226), -np.logspace(-45, 0, 226),
        np.array([0.0, -0.0, 1e-3, -1e-3, 88.0, -88.0, 1e5, -1e5, 1e20, -1e20, 3.0e38,
                  -3.0e38, 1e-40, -1e-40])]).astype(np.float32).astype(np.float64)
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    h = h[(h & 0x7F80) != 0x7F80]
    bf = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    z = np.concatenate([grid, bf])
    want = F.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    got = np.array([oracle.gelu_tanh(v, lib=lib) for v in z])
    err = np.abs(got - want)
    assert np.all(err <= 1e-14 * np.abs(want) + 1e-15 * np.abs(z)), float(err.max())
    assert np.all(got[z < 0] <= 0) and np.all(got[z > 0] >= 0)
    assert np.all(got[np.abs(z) >= 30] == np.where(z[np.abs(z) >= 30] > 0, z[np.abs(z) >= 30], 0))


def pin_gelu_invariants(lib):
    """GeLU(0) = 0; GeLU(z) - GeLU(-z) = z (the tanh term is odd);
    GeLU(z) -> z for large z and -> 0 for very negative z."""
    assert oracle.gelu_tanh(0.0, lib=lib) == 0.0
    for z in (1e-3, 0.25, 0.5, 1.0, 1.7, 3.0, 5.5, 9.0):
        d = oracle.gelu_tanh(z, lib=lib) - oracle.gelu_tanh(-z, lib=lib)
        assert abs(d - z) <= 4e-16 * max(z, 1.0), (z, d)
    assert abs(oracle.gelu_tanh(12.0, lib=lib) - 12.0) < 1e-12
    assert abs(oracle.gelu_tanh(-12.0, lib=lib)) < 1e-12
    # Near 0: GeLU(z) = z/2 + sqrt(2/pi) z^2 / 2 + O(z^4)
    z = 1e-4
    want = z / 2 + math.sqrt(2 / math.pi) * z * z / 2
    assert abs(oracle.gelu_tanh(z, lib=lib) - want) < 1e-15


def pin_bf16_roundtrip(lib):
    """Every finite bf16 value widens and rounds back to itself."""
    for h in list(range(0, 0x7F80, 97)) + [0x0001, 0x007F, 0x0080, 0x3F80,
                                           0x7F7F, 0x8001, 0xBF80, 0xFF7F]:
        d = oracle.bf16_to_double(h, lib=lib)
        assert oracle.bf16_from_double(d, lib=lib) == h, hex(h)


def pin_bf16_rounding(lib):
    """Nearest, ties to even: hand cases at 1.0 (quantum 2^-7), the overflow
    edge and the subnormal range; then torch's fp32 -> bf16 on random fp32
    values (a double holding an fp32 value rounds like that fp32)."""
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0 ** -8, 0x3F80),                  # tie -> even (down)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),              # tie -> even (up)
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),     # just above the tie
        (1.0 + 2.0 ** -8 - 2.0 ** -30, 0x3F80),     # just below the tie
        (-1.0 - 2.0 ** -7, 0xBF81),
        (2.0 ** -133, 0x0001),                      # smallest subnormal
        (1.5 * 2.0 ** -133, 0x0002),                # tie -> even (up)
        (2.0 ** -134, 0x0000),                      # tie -> even (zero)
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),     # largest finite
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),     # rounds up to inf
        (float("inf"), 0x7F80),
        (-0.0, 0x8000),
    ]
    for v, want in cases:
        got = oracle.bf16_from_double(v, lib=lib)
        assert got == want, (v, hex(got), hex(want))
    rng = np.random.default_rng(7)
    f = (rng.standard_normal(2000) * np.exp(rng.uniform(-30, 30, 2000))).astype(np.float32)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(v), lib=lib) for v in f], np.uint16)
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------
# o1: y = relu(x + b1) * scale + b2     [P1] §1.1, §3.1
# --------------------------------------------------------------------------

def pin_pointwise_golden(lib):
    """Hand-computed dyadic cases: every step is exact in fp32."""
    g = _golden("pointwise_f32.json")
    for case in g["cases"]:
        x, b1, b2 = (np.array(case[k], np.float32) for k in ("x", "b1", "b2"))
        y = oracle.add_relu_scale(x, b1, b2, case["scale"], lib=lib)
        assert np.array_equal(y, np.array(case["y"], np.float32)), (case, y)


def pin_pointwise_library(lib):
    """torch CPU eager fp32, the [P1] §3.1 baseline (add, relu, mul, add:
    four separately rounded ops), bit for bit, at scale 0.5 and 0.3."""
    w = __import__("synth.workloads", fromlist=["x"]).POINTWISE_TINY
    t = w.generate_all()
    x, b1, b2 = (torch.from_numpy(t[k]) for k in ("x", "b1", "b2"))
    for scale in (0.5, 0.3):
        want = (torch.relu(x + b1) * scale + b2).numpy()
        got = oracle.add_relu_scale(t["x"], t["b1"], t["b2"], scale, lib=lib)
        assert np.array_equal(_bits(got), _bits(want)), scale


def pin_pointwise_special(lib):
    """x + b1 <= 0 gives y = b2 exactly; scale 1, b2 = 0 gives relu(x + b1)."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal(512).astype(np.float32)
    b1 = (-x - np.abs(rng.standard_normal(512)).astype(np.float32))
    b2 = rng.standard_normal(512).astype(np.float32)
    y = oracle.add_relu_scale(x, b1, b2, 0.5, lib=lib)
    assert np.array_equal(_bits(y), _bits(b2))
    b1 = rng.standard_normal(512).astype(np.float32)
    y = oracle.add_relu_scale(x, b1, np.zeros(512, np.float32), 1.0, lib=lib)
    assert np.array_equal(_bits(y), _bits(np.maximum(x + b1, np.float32(0))))


def pin_pointwise_bf16_library(lib):
    """bf16 I/O: widen, fp32 chain (torch eager fp32), one bf16 rounding
    (torch fp32 -> bf16)."""
    n = 3000
    x = synth.normal(11, 0, (n,), dtype="bf16")
    b1 = synth.normal(11, 1, (n,), dtype="bf16")
    b2 = synth.normal(11, 2, (n,), dtype="bf16")
    xf, b1f, b2f = (torch.from_numpy(synth.bf16_bits_to_f32(a)) for a in (x, b1, b2))
    want = (torch.relu(xf + b1f) * 0.5 + b2f).to(torch.bfloat16)
    want = want.view(torch.int16).numpy().view(np.uint16)
    got = oracle.add_relu_scale(x, b1, b2, 0.5, lib=lib)
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------
# o2: TorchInductor example chain       [P4] "model", Figure 1
# --------------------------------------------------------------------------

def pin_inductor_golden(lib):
    """Hand-computed dyadic 1x4 and 2x3 cases (x_scale, branch_scale chosen
    dyadic so every step is exact)."""
    g = _golden("inductor_f32.json")
    for case in g["cases"]:
        x = np.array(case["x"], np.float32)
        vecs = [np.array(case[k], np.float32) for k in ("bias", "gamma", "beta")]
        y = oracle.bias_relu_branch_mean_epilogue(
            x, *vecs, case["x_scale"], case["branch_scale"], lib=lib)
        assert np.array_equal(y, np.array(case["y"], np.float32)), (case["name"], y)


def pin_inductor_library_s(lib):
    """s (t = x*1.1 + bias; a = relu(t); p = a*a; q = a*0.1; s = p + q) against
    torch CPU eager fp32 running the page's model() steps, bit for bit; the
    mean against the float64 mean of that s to one fp32 rounding."""
    w = __import__("synth.workloads", fromlist=["x"]).INDUCTOR_1024
    t = w.generate_all(rows=64)
    x, bias = torch.from_numpy(t["x"]), torch.from_numpy(t["bias"])
    tt = x * 1.1 + bias
    a = torch.relu(tt)
    s_want = (a * a + a * 0.1).numpy()
    y, s, m = oracle.bias_relu_branch_mean_epilogue(
        t["x"], t["bias"], t["gamma"], t["beta"], 1.1, 0.1, intermediates=True,
        lib=lib)
    assert np.array_equal(_bits(s), _bits(s_want))
    m_want = s_want.astype(np.float64).mean(axis=1)
    assert np.all(np.abs(m - m_want) <= U32 * np.abs(m_want) * 1.01)


def pin_inductor_closed_form(lib):
    """Per row, sum_j (y - beta)/gamma = sum_j (s - m) = cols*(mean(s) - m),
    which is zero up to the rounding of m and of the three epilogue ops."""
    w = __import__("synth.workloads", fromlist=["x"]).INDUCTOR_1024
    t = w.generate_all(rows=32)
    y, s, m = oracle.bias_relu_branch_mean_epilogue(
        t["x"], t["bias"], t["gamma"], t["beta"], 1.1, 0.1, intermediates=True,
        lib=lib)
    y64 = y.astype(np.float64)
    g64 = t["gamma"].astype(np.float64)
    b64 = t["beta"].astype(np.float64)
    lhs = ((y64 - b64) / g64).sum(axis=1)
    s64 = s.astype(np.float64)
    m64 = m.astype(np.float64)[:, None]
    bound = (s.shape[1] * U32 * np.abs(m64[:, 0])
             + (2 * U32 * np.abs(s64 - m64) + U32 * np.abs(y64) / g64).sum(axis=1))
    assert np.all(np.abs(lhs) <= 2 * bound), (np.abs(lhs) / bound).max()
    # and m is the row mean of s
    assert np.all(np.abs(m64[:, 0] - s64.mean(axis=1)) <= 1.01 * U32 * np.abs(m64[:, 0]))


def pin_inductor_special(lib):
    """A row with every t <= 0 gives s = 0, m = 0, y = beta exactly; a row of
    one repeated x (bias 0) gives s constant, m = s, y = beta exactly."""
    cols = 37
    rng = np.random.default_rng(5)
    gamma = rng.uniform(0.5, 1.5, cols).astype(np.float32)
    beta = rng.standard_normal(cols).astype(np.float32)
    x = np.stack([-np.abs(rng.standard_normal(cols)).astype(np.float32) - 0.5,
                  np.full(cols, 0.75, np.float32)])
    bias = np.zeros(cols, np.float32)
    y = oracle.bias_relu_branch_mean_epilogue(x, bias, gamma, beta, 1.1, 0.1, lib=lib)
    assert np.array_equal(_bits(y[0]), _bits(beta))
    assert np.array_equal(_bits(y[1]), _bits(beta))


# --------------------------------------------------------------------------
# o3: residual + LayerNorm + GeLU-tanh  [P2] §2.2-2.3, [P3] §4.3
# --------------------------------------------------------------------------

def _ln_inputs(rows, hidden, seed, dtype="f32"):
    x = synth.normal(seed, 0, (rows, hidden), dtype=dtype)
    r = synth.normal(seed, 1, (rows, hidden), dtype=dtype)
    w = synth.uniform(seed, 2, (hidden,), 0.5, 1.5, dtype=dtype)
    b = synth.normal(seed, 3, (hidden,), 0.0, 0.1, dtype=dtype)
    return x, r, w, b


def pin_ln_closed_forms(lib):
    """Before the affine step each row has mean 0 and variance
    var/(var + eps) ([P3] §4.3: (x - mean)/sqrt(var + eps))."""
    x, r, w, b = _ln_inputs(16, 1000, 21)
    eps = 1e-5
    out, mean, rstd, xhat = oracle.residual_layernorm_gelu(
        x, r, w, b, eps, intermediates=True, lib=lib)
    v = (x + r).astype(np.float64)            # fp32 add, exact widening
    var = ((v - v.mean(axis=1, keepdims=True)) ** 2).mean(axis=1)
    assert np.all(np.abs(xhat.mean(axis=1)) <= 1e-12)
    want_var = var / (var + np.float64(np.float32(eps)))
    assert np.all(np.abs((xhat ** 2).mean(axis=1) - want_var) <= 1e-12)
    assert np.all(np.abs(mean - v.mean(axis=1)) <= 1e-12)


def pin_ln_library(lib):
    """torch float64 layer_norm + gelu(tanh) on v = x + r (fp32 add),
    rounded to fp32: equal to within one fp32 rounding."""
    for rows, hidden in ((8, 4096), (5, 33), (3, 1)):
        x, r, w, b = _ln_inputs(rows, hidden, 22 + hidden)
        v = torch.from_numpy(x) + torch.from_numpy(r)
        n = F.layer_norm(v.double(), (hidden,), torch.from_numpy(w).double(),
                         torch.from_numpy(b).double(), eps=float(np.float32(1e-5)))
        want = F.gelu(n, approximate="tanh").numpy()
        got = oracle.residual_layernorm_gelu(x, r, w, b, 1e-5, lib=lib)
        err = np.abs(got.astype(np.float64) - want)
        assert np.all(err <= 1.0001 * U32 * np.abs(want) + 1e-12), err.max()


def pin_ln_special(lib):
    """H = 1: v - mean = 0, so out = GeLU(b).  A row [a, -a]: mean 0,
    var a^2, so n = +-a/sqrt(a^2 + eps) * w + b."""
    b = np.array([0.375], np.float32)
    out = oracle.residual_layernorm_gelu(
        np.array([[1.25]], np.float32), np.array([[-4.0]], np.float32),
        np.array([1.5], np.float32), b, 1e-5, lib=lib)
    want = F.gelu(torch.tensor([0.375], dtype=torch.float64), approximate="tanh")
    assert out[0, 0] == np.float32(want.item())
    a, eps = 3.0, float(np.float32(1e-5))
    w = np.array([1.0, 2.0], np.float32)
    bb = np.array([0.5, -0.25], np.float32)
    out, mean, rstd, xhat = oracle.residual_layernorm_gelu(
        np.array([[a, -a]], np.float32), np.zeros((1, 2), np.float32), w, bb,
        1e-5, intermediates=True, lib=lib)
    k = a / math.sqrt(a * a + eps)
    assert abs(mean[0]) == 0.0
    assert abs(rstd[0] - 1 / math.sqrt(a * a + eps)) <= 1e-16
    n = torch.tensor([k * 1.0 + 0.5, -k * 2.0 - 0.25], dtype=torch.float64)
    want = F.gelu(n, approximate="tanh").numpy().astype(np.float32)
    assert np.array_equal(out[0], want)


def pin_ln_bf16_library(lib):
    """bf16 I/O: widen x, r, w, b exactly, fp32 add, float64 layer_norm +
    gelu, round once to bf16.  torch rounds float64 -> bf16 through fp32, so
    the two may differ by one bf16 step where that double rounding bites."""
    x, r, w, b = _ln_inputs(6, 520, 31, dtype="bf16")
    xf, rf, wf, bf = (torch.from_numpy(synth.bf16_bits_to_f32(a)) for a in (x, r, w, b))
    v = xf + rf
    n = F.layer_norm(v.double(), (520,), wf.double(), bf.double(),
                     eps=float(np.float32(1e-5)))
    g = F.gelu(n, approximate="tanh")
    got = oracle.residual_layernorm_gelu(x, r, w, b, 1e-5, lib=lib)
    gw = synth.bf16_bits_to_f32(got).astype(np.float64)
    gd = g.numpy()
    # within half a bf16 step of the float64 value: the step is 2^-7 of the
    # binade's lower end, so at most 2^-8 of the value
    assert np.all(np.abs(gw - gd) <= 2.0 ** -8 * np.abs(gd) * 1.0001 + 1e-30)
    want = g.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.mean(got == want) > 0.999


# --------------------------------------------------------------------------
# o2 with bf16 I/O
# --------------------------------------------------------------------------

def pin_inductor_bf16_library(lib):
    """bf16 inputs widened, the page's model() steps in torch eager fp32, one
    rounding to bf16: equal except where the mean's summation order moves a
    value across a bf16 rounding boundary (then one bf16 step apart)."""
    x = synth.normal(41, 0, (48, 1024), dtype="bf16")
    bias = synth.normal(41, 1, (1024,), 0.0, 0.1, dtype="bf16")
    gamma = synth.uniform(41, 2, (1024,), 0.5, 1.5, dtype="bf16")
    beta = synth.normal(41, 3, (1024,), 0.0, 0.1, dtype="bf16")
    xf, bf, gf, btf = (torch.from_numpy(synth.bf16_bits_to_f32(a)) for a in (x, bias, gamma, beta))
    a = torch.relu(xf * 1.1 + bf)
    s = a * a + a * 0.1
    m = s.double().mean(dim=1, keepdim=True).float()
    want = ((s - m) * gf + btf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bias_relu_branch_mean_epilogue_bf16(x, bias, gamma, beta, lib=lib)
    g, w = synth.bf16_bits_to_f32(got).astype(np.float64), synth.bf16_bits_to_f32(want).astype(np.float64)
    assert np.all(np.abs(g - w) <= 2.0 ** -7 * np.abs(w) + 1e-30)
    assert np.mean(got == want) > 0.999
    # all-negative row: y = beta exactly
    xn = synth.f32_to_bf16_bits(-np.abs(synth.bf16_bits_to_f32(x[:1])) - 1.0)
    yn = oracle.bias_relu_branch_mean_epilogue_bf16(xn, np.zeros(1024, np.uint16), gamma, beta, lib=lib)
    assert np.array_equal(yn[0], beta)


# --------------------------------------------------------------------------
# o4: LayerNorm family
# --------------------------------------------------------------------------

def pin_layernorm_act_library(lib):
    """Every (residual, activation) combination against torch float64
    layer_norm followed by relu / gelu(tanh), on v = x + r in fp32: within one
    fp32 rounding; h equals the fp32 sum bit for bit."""
    x, r, w, b = _ln_inputs(7, 515, 51)
    eps = float(np.float32(1e-5))
    for res in (False, True):
        v = torch.from_numpy(x) + torch.from_numpy(r) if res else torch.from_numpy(x)
        n = F.layer_norm(v.double(), (515,), torch.from_numpy(w).double(),
                         torch.from_numpy(b).double(), eps=eps)
        for act, f in ((0, lambda t: t), (1, torch.relu),
                       (2, lambda t: F.gelu(t, approximate="tanh"))):
            want = f(n).numpy()
            got, h = oracle.layernorm_act(x, r if res else None, w, b, 1e-5, act,
                                          want_h=True, lib=lib)
            err = np.abs(got.astype(np.float64) - want)
            assert np.all(err <= 1.0001 * U32 * np.abs(want) + 1e-30), (res, act, err.max())
            assert np.array_equal(_bits(h), _bits(v.numpy())), (res, act)


def pin_layernorm_plain_closed_form(lib):
    """act none, w = 1, b = 0: each row has mean 0 and variance
    var/(var + eps) up to the final fp32 rounding ([P3] §4.3)."""
    x, _, _, _ = _ln_inputs(9, 800, 52)
    ones, zeros = np.ones(800, np.float32), np.zeros(800, np.float32)
    y = oracle.layernorm_act(x, None, ones, zeros, 1e-5, 0, lib=lib).astype(np.float64)
    v = x.astype(np.float64)
    var = v.var(axis=1)
    assert np.all(np.abs(y.mean(axis=1)) <= 4 * U32)
    want = var / (var + np.float64(np.float32(1e-5)))
    assert np.all(np.abs((y * y).mean(axis=1) - want) <= 8 * U32)
    # relu of the same: exactly max(y, 0) with -0 mapped to +0
    yr = oracle.layernorm_act(x, None, ones, zeros, 1e-5, 1, lib=lib)
    assert np.array_equal(_bits(yr), _bits(np.where(y > 0, y, 0.0).astype(np.float32)))


def pin_layernorm_act_bf16(lib):
    """bf16: out within half a bf16 step of float64; h is the fp32 sum
    rounded to bf16 (torch's fp32 -> bf16)."""
    x, r, w, b = _ln_inputs(5, 264, 53, dtype="bf16")
    xf, rf, wf, bf = (torch.from_numpy(synth.bf16_bits_to_f32(a)) for a in (x, r, w, b))
    v = xf + rf
    n = F.layer_norm(v.double(), (264,), wf.double(), bf.double(), eps=float(np.float32(1e-5)))
    got, h = oracle.layernorm_act(x, r, w, b, 1e-5, 1, want_h=True, lib=lib)
    want = torch.relu(n).numpy()
    g = synth.bf16_bits_to_f32(got).astype(np.float64)
    assert np.all(np.abs(g - want) <= 2.0 ** -8 * np.abs(want) * 1.0001 + 1e-30)
    assert np.array_equal(h, v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


# --------------------------------------------------------------------------
# o5: row softmax
# --------------------------------------------------------------------------

def pin_softmax_library(lib):
    """torch float64 softmax of the fp32 rows: within one fp32 rounding."""
    x = synth.normal(61, 0, (12, 1000), 0.0, 3.0)
    want = torch.softmax(torch.from_numpy(x).double(), dim=1).numpy()
    got = oracle.row_softmax(x, lib=lib)
    assert np.all(np.abs(got.astype(np.float64) - want) <= 1.0001 * U32 * want + 1e-45)


def pin_softmax_closed_forms(lib):
    """Rows sum to 1; a constant row gives 1/cols; [a, b] gives
    (sigmoid(a - b), sigmoid(b - a)); a shift by 1000 changes nothing (and
    must not overflow); a row spanning +-1000 puts all mass on its maximum."""
    x = synth.normal(62, 0, (6, 333))
    y = oracle.row_softmax(x, lib=lib).astype(np.float64)
    assert np.all(np.abs(y.sum(axis=1) - 1.0) <= 333 * U32)
    c = oracle.row_softmax(np.full((2, 7), 3.25, np.float32), lib=lib)
    assert np.all(c == np.float32(1.0 / 7.0))
    ab = np.array([[1.5, -0.75], [-2.0, 4.0]], np.float32)
    want = torch.sigmoid(torch.tensor([[2.25, -2.25], [-6.0, 6.0]], dtype=torch.float64))
    got = oracle.row_softmax(ab, lib=lib).astype(np.float64)
    assert np.all(np.abs(got - want.numpy()) <= U32 * want.numpy() * 1.0001)
    q = np.round(synth.normal(63, 0, (3, 50)) * 1024) / 1024           # exact + 1000
    s0 = oracle.row_softmax(q.astype(np.float32), lib=lib)
    s1 = oracle.row_softmax((q + 1000.0).astype(np.float32), lib=lib)
    assert np.all(np.isfinite(s1)) and np.array_equal(s0, s1)
    wide = oracle.row_softmax(np.array([[0.0, 1000.0, -1000.0]], np.float32), lib=lib)
    assert np.array_equal(wide, np.array([[0.0, 1.0, 0.0]], np.float32))


def pin_softmax_bf16(lib):
    """bf16 rows: within half a bf16 step of the float64 softmax."""
    x = synth.normal(64, 0, (4, 640), 0.0, 2.0, dtype="bf16")
    want = torch.softmax(torch.from_numpy(synth.bf16_bits_to_f32(x)).double(), dim=1).numpy()
    g = synth.bf16_bits_to_f32(oracle.row_softmax(x, lib=lib)).astype(np.float64)
    assert np.all(np.abs(g - want) <= 2.0 ** -8 * want * 1.0001 + 1e-40)


def pin_pointwise_bcast_library(lib):
    """Per-column b1 / b2 ([P1]'s chain with bias-like operands): torch CPU
    eager fp32 with broadcasting, bit for bit, for every flag combination;
    bf16 against torch's widen / fp32 ops / round-to-nearest-even."""
    rows, cols = 37, 129
    x = synth.normal(81, 0, (rows, cols))
    full = [synth.normal(81, 1, (rows, cols)), synth.normal(81, 2, (rows, cols))]
    vec = [synth.normal(81, 3, (cols,)), synth.normal(81, 4, (cols,))]
    for f1 in (0, 1):
        for f2 in (0, 1):
            b1 = vec[0] if f1 else full[0]
            b2 = vec[1] if f2 else full[1]
            t = torch.relu(torch.from_numpy(x) + torch.from_numpy(b1)) * 0.75 + torch.from_numpy(b2)
            got = oracle.add_relu_scale_bcast(x, b1, b2, 0.75, lib=lib)
            assert np.array_equal(_bits(got), _bits(t.numpy())), (f1, f2)
    xb, v1, v2 = (synth.f32_to_bf16_bits(a) for a in (x, vec[0], vec[1]))
    wide = [torch.from_numpy(synth.bf16_bits_to_f32(a)) for a in (xb, v1, v2)]
    t = (torch.relu(wide[0] + wide[1]) * 0.5 + wide[2]).to(torch.bfloat16)
    got = oracle.add_relu_scale_bcast(xb, v1, v2, 0.5, lib=lib)
    assert np.array_equal(got, t.view(torch.int16).numpy().view(np.uint16))


# --------------------------------------------------------------------------
# o4 extras and o6: row statistics, the Philox generator, dropout
# --------------------------------------------------------------------------

def pin_layernorm_stats_library(lib):
    """The per-row statistics o4 writes out: torch float64 mean and
    1/sqrt(biased variance + eps) of v = x + r ([P3] §4.3)."""
    x, r, w, b = _ln_inputs(7, 300, 71)
    _, _, mean, rstd = oracle.layernorm_act_ex(x, r, w, b, 1e-5, oracle.ACT_RELU,
                                               want_stats=True, lib=lib)
    v = torch.from_numpy(x).double() + torch.from_numpy(r).double()
    v = v.float().double()                              # v = x + r in fp32
    want_mean = v.mean(dim=1).numpy()
    want_rstd = (1.0 / torch.sqrt(v.var(dim=1, unbiased=False) + 1e-5)).numpy()
    assert np.all(np.abs(mean - want_mean) <= 1e-13)
    assert np.all(np.abs(rstd - want_rstd) <= 1e-13 * want_rstd)


def _numpy_philox64(ctr, key, blocks=1):
    """numpy's Philox (4x64-10) bit generator: it advances its counter before
    each block, so a generator set to ctr - 1 yields the block at ctr."""
    prev = np.array(ctr, np.uint64)
    assert prev[0] >= 1
    prev[0] -= np.uint64(1)
    bg = np.random.Philox(key=np.array(key, np.uint64), counter=prev)
    return bg.random_raw(4 * blocks).astype(np.uint64)


def pin_philox64_numpy(lib):
    """Philox-4x64-10 against numpy's Philox bit generator (a library routine)
    on counters and keys with every word in play: the round structure (which
    words are multiplied, what each new word is, the key schedule) that the
    32-bit generator shares."""
    rng = np.random.default_rng(2024)
    cases = [([1, 0, 0, 0], [0, 0]), ([1, 2, 3, 4], [5, 6]),
             ([2 ** 64 - 1, 2 ** 64 - 1, 2 ** 64 - 1, 2 ** 64 - 1], [2 ** 64 - 1, 2 ** 64 - 1])]
    for _ in range(6):
        cases.append((list(rng.integers(1, 2 ** 63, 4, dtype=np.uint64) * np.uint64(2) - np.uint64(1)),
                      list(rng.integers(0, 2 ** 63, 2, dtype=np.uint64) * np.uint64(2))))
    for ctr, key in cases:
        got = oracle.philox4x64_10(ctr, key, lib=lib)
        want = _numpy_philox64(ctr, key)
        assert np.array_equal(got, want), (ctr, key)


def _curand():
    """cuRAND's host-side generator API (runs on the CPU), or None."""
    import ctypes
    import ctypes.util
    cands = [ctypes.util.find_library("curand"), "libcurand.so", "libcurand.so.10"]
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cands += [os.path.join(home, d, "libcurand.so") for d in ("lib64", "lib")]
    for c in cands:
        if not c:
            continue
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    return None


def _curand_philox_words(seed, n, offset=0):
    """n raw 32-bit outputs of cuRAND's host Philox4_32_10 generator."""
    import ctypes
    lib = _curand()
    if lib is None:
        import pytest
        pytest.skip("libcurand not found")
    g = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(g), 161) == 0  # PHILOX4_32_10
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(g, ctypes.c_ulonglong(seed)) == 0
        if offset:
            assert lib.curandSetGeneratorOffset(g, ctypes.c_ulonglong(offset)) == 0
        buf = (ctypes.c_uint32 * n)()
        assert lib.curandGenerate(g, buf, ctypes.c_size_t(n)) == 0
        return np.frombuffer(buf, np.uint32).copy()
    finally:
        lib.curandDestroyGenerator(g)


def pin_philox32_curand(lib):
    """Philox-4x32-10 against cuRAND's Philox4_32_10 host generator (a library
    routine): with seed s its output block b is the generator at counter
    (0, 0, b, 0) under key (lo(s), hi(s)), and a generator offset of 4k starts
    at counter (0, 0, k, 0)."""
    for seed in (0, 1, 0x0123456789ABCDEF, 2 ** 64 - 1):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        words = _curand_philox_words(seed, 4 * 64)
        for blk in range(64):
            got = oracle.philox4x32_10([0, 0, blk, 0], key, lib=lib)
            assert np.array_equal(got, words[4 * blk:4 * blk + 4]), (seed, blk)
        k = 3 * 4096 + 5
        words = _curand_philox_words(seed, 4, offset=4 * k)
        assert np.array_equal(oracle.philox4x32_10([0, 0, k, 0], key, lib=lib), words)


def pin_dropout_decision(lib):
    """Element i of a call (seed, offset 0) takes half i mod 2 (low, high) of
    word (i mod 8) / 2 of block i // 8, which is cuRAND's output word i // 2;
    kept iff half * 2^-16 >= p.  p is also set to the exact u of chosen
    elements (u >= p keeps them), p = 0 keeps everything, and masks nest as p
    grows."""
    seed = 0x5EED0F0D
    words = _curand_philox_words(seed, 4 * 256)
    halves = np.stack([words & np.uint32(0xFFFF), words >> np.uint32(16)], axis=1).reshape(-1)
    u = halves.astype(np.float32) * np.float32(2.0 ** -16)
    for p in (0.1, 0.5, 0.9, float(u[17]), float(u[300])):
        keep = oracle.dropout_mask(seed, 0, 0, u.size, p, lib=lib)
        assert np.array_equal(keep, u >= np.float32(p)), p
    assert oracle.dropout_mask(seed, 0, 0, 1000, 0.0, lib=lib).all()
    lo = oracle.dropout_mask(seed, 9, 40, 4000, 0.2, lib=lib)
    hi = oracle.dropout_mask(seed, 9, 40, 4000, 0.6, lib=lib)
    assert np.all(hi <= lo)


def pin_dropout_counter_and_rate(lib):
    """Counter arithmetic: offset + 1 is the same stream as element index + 8;
    the keep rate over 2^20 elements is within 5 sigma of 1 - p; another seed
    gives another mask."""
    a = oracle.dropout_mask(11, 5, 8, 4096, 0.3, lib=lib)
    b = oracle.dropout_mask(11, 4, 16, 4096, 0.3, lib=lib)
    assert np.array_equal(a, b)
    n = 1 << 20
    for p in (0.1, 0.5):
        keep = oracle.dropout_mask(12345, 0, 0, n, p, lib=lib)
        sigma = math.sqrt(n * p * (1 - p))
        assert abs(keep.sum() - n * (1 - p)) <= 5 * sigma, p
    other = oracle.dropout_mask(12346, 0, 0, n, 0.5, lib=lib)
    same = np.mean(other == oracle.dropout_mask(12345, 0, 0, n, 0.5, lib=lib))
    assert abs(same - 0.5) < 0.01


def pin_layernorm_dropout(lib):
    """[P2] §2.1's LayerNorm -> ReLU -> Dropout: kept elements are the
    undropped output / (1 - p) (within a rounding of each), dropped ones are
    the product with 0 (+0 after a ReLU), by the mask of element index
    row * hidden + col; p = 0 is the undropped chain bit for bit."""
    x, r, w, b = _ln_inputs(9, 257, 72)
    for dt in ("f32", "bf16"):
        if dt == "bf16":
            x, r, w, b = (synth.f32_to_bf16_bits(a) for a in (x, r, w, b))
        base = oracle.layernorm_act(x, None, w, b, 1e-5, oracle.ACT_RELU, lib=lib)
        same, _, _, _ = oracle.layernorm_act_ex(x, None, w, b, 1e-5, oracle.ACT_RELU, p=0.0,
                                                lib=lib)
        assert np.array_equal(base, same)
        p = 0.25
        out, _, _, _ = oracle.layernorm_act_ex(x, None, w, b, 1e-5, oracle.ACT_RELU, p=p,
                                               seed=99, offset=3, lib=lib)
        keep = oracle.dropout_mask(99, 3, 0, x.size, p, lib=lib).reshape(x.shape)
        if dt == "bf16":
            g, o, tol = synth.bf16_bits_to_f32(base), synth.bf16_bits_to_f32(out), 2.0 ** -7
        else:
            g, o, tol = base, out, 2.0 ** -22
        g64, o64 = g.astype(np.float64), o.astype(np.float64)
        assert np.all(np.abs(o64[keep] - g64[keep] / (1 - p)) <= tol * np.abs(g64[keep]) / (1 - p))
        assert np.all(o[~keep] == 0) and not np.any(np.signbit(o[~keep]))
        assert 0.6 < keep.mean() < 0.9


def pin_scale_mask_softmax_library(lib):
    """[P1] §4.1-4.2's scaled, causally masked score rows: torch float64
    softmax of the fp32 product x * scale with the masked keys filled with
    -inf, within one fp32 rounding; masked outputs exactly 0; with period p
    and offset k, row i keeps keys 0 .. (i mod p) + k; bf16 within half a step."""
    rows, cols, period, offset = 12, 9, 4, 2
    x = synth.normal(65, 0, (rows, cols), 0.0, 3.0)
    scale = np.float32(0.3)
    y = oracle.scale_mask_softmax(x, scale, True, period, offset, lib=lib).astype(np.float64)
    v = torch.from_numpy((x * scale).astype(np.float32)).double()      # the fp32 product
    i = torch.arange(rows)[:, None] % period + offset
    j = torch.arange(cols)[None, :]
    masked = j > i
    want = torch.softmax(v.masked_fill(masked, float("-inf")), dim=1).numpy()
    assert np.all(y[masked.numpy()] == 0.0)
    assert np.all(np.abs(y - want) <= U32 * want * 1.0001)
    assert np.all(np.abs(y.sum(axis=1) - 1.0) <= cols * U32)
    y0 = oracle.scale_mask_softmax(x, 1.0, True, period, 0, lib=lib)
    assert np.array_equal(y0[0], np.eye(cols, dtype=np.float32)[0])       # query 0 sees key 0
    xb = synth.normal(66, 0, (8, 40), 0.0, 2.0, dtype="bf16")
    vb = torch.from_numpy(synth.bf16_bits_to_f32(xb) * np.float32(0.25)).double()
    mb_ = torch.arange(40)[None, :] > (torch.arange(8)[:, None] % 8 + 30)
    wb = torch.softmax(vb.masked_fill(mb_, float("-inf")), dim=1).numpy()
    gb = synth.bf16_bits_to_f32(oracle.scale_mask_softmax(xb, 0.25, True, 8, 30, lib=lib))
    assert np.all(np.abs(gb.astype(np.float64) - wb) <= 2.0 ** -8 * wb * 1.0001 + 1e-40)


def pin_scale_mask_softmax_special_cases(lib):
    """No mask and scale 1: the plain row softmax bit for bit; an offset past
    the row length masks nothing; scale 2^-3 is exact, so scaling the input
    by hand gives the same bits."""
    x = synth.normal(67, 0, (5, 33), 0.0, 2.0)
    plain = oracle.row_softmax(x, lib=lib)
    assert np.array_equal(oracle.scale_mask_softmax(x, 1.0, False, lib=lib), plain)
    assert np.array_equal(oracle.scale_mask_softmax(x, 1.0, True, 5, 40, lib=lib), plain)
    a = oracle.scale_mask_softmax(x, 0.125, True, 5, 3, lib=lib)
    b = oracle.scale_mask_softmax((x * np.float32(0.125)).astype(np.float32), 1.0, True, 5, 3,
                                  lib=lib)
    assert np.array_equal(a, b)
    # masked elements take no part, however large: a masked +1000 changes nothing
    big = x.copy()
    big[1, 20] = 1000.0                     # row 1 keeps keys 0 .. 4
    m1 = oracle.scale_mask_softmax(big, 1.0, True, 5, 3, lib=lib)
    m0 = oracle.scale_mask_softmax(x, 1.0, True, 5, 3, lib=lib)
    assert np.all(np.isfinite(m1)) and np.array_equal(m1, m0)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
