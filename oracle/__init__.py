"""CPU oracle for the three fused memory-bound chains (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  The oracle is plain C (``oracle.c``) evaluating the
pages' formulas one operation at a time; this module only marshals numpy
arrays into it.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the product package never does.

Every function takes and returns host numpy arrays: fp32 as ``float32``,
bf16 as raw ``uint16`` bit patterns.

Sources: see ``oracle.h`` for the four pages ([P1]..[P4]) and the section each
function follows.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _f32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _u16p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _f64p(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f32p_opt(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_float)()
    return _f32p(a)


def load(path=None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    so = path or _build.DEFAULT_SO
    if path is None and not os.path.exists(so):
        _build.build()
    lib = ctypes.CDLL(so)
    F32P = ctypes.POINTER(ctypes.c_float)
    U16P = ctypes.POINTER(ctypes.c_uint16)
    F64P = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    f32 = ctypes.c_float
    lib.oracle_relu_f32.argtypes = [f32]
    lib.oracle_relu_f32.restype = f32
    lib.oracle_gelu_tanh.argtypes = [ctypes.c_double]
    lib.oracle_gelu_tanh.restype = ctypes.c_double
    lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
    lib.oracle_bf16_from_double.restype = ctypes.c_uint16
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_add_relu_scale_f32.argtypes = [F32P, F32P, F32P, F32P, i64, f32]
    lib.oracle_add_relu_scale_f32.restype = None
    lib.oracle_add_relu_scale_bf16.argtypes = [U16P, U16P, U16P, U16P, i64, f32]
    lib.oracle_add_relu_scale_bf16.restype = None
    lib.oracle_bias_relu_branch_mean_epilogue.argtypes = [
        F32P, F32P, F32P, F32P, F32P, i64, i64, f32, f32, F32P, F32P]
    lib.oracle_bias_relu_branch_mean_epilogue.restype = None
    lib.oracle_residual_layernorm_gelu_f32.argtypes = [
        F32P, F32P, F32P, F32P, F32P, i64, i64, f32, F64P, F64P, F64P]
    lib.oracle_residual_layernorm_gelu_f32.restype = None
    lib.oracle_residual_layernorm_gelu_bf16.argtypes = [
        U16P, U16P, U16P, U16P, U16P, i64, i64, f32, F64P, F64P, F64P]
    lib.oracle_residual_layernorm_gelu_bf16.restype = None
    lib.oracle_bias_relu_branch_mean_epilogue_bf16.argtypes = [
        U16P, U16P, U16P, U16P, U16P, i64, i64, f32, f32]
    lib.oracle_bias_relu_branch_mean_epilogue_bf16.restype = None
    lib.oracle_layernorm_act_f32.argtypes = [
        F32P, F32P, F32P, F32P, F32P, F32P, i64, i64, f32, ctypes.c_int]
    lib.oracle_layernorm_act_f32.restype = None
    lib.oracle_layernorm_act_bf16.argtypes = [
        U16P, U16P, U16P, U16P, U16P, U16P, i64, i64, f32, ctypes.c_int]
    lib.oracle_layernorm_act_bf16.restype = None
    lib.oracle_add_relu_scale_bcast_f32.argtypes = [
        F32P, F32P, F32P, F32P, i64, i64, ctypes.c_int, ctypes.c_int, f32]
    lib.oracle_add_relu_scale_bcast_f32.restype = None
    lib.oracle_add_relu_scale_bcast_bf16.argtypes = [
        U16P, U16P, U16P, U16P, i64, i64, ctypes.c_int, ctypes.c_int, f32]
    lib.oracle_add_relu_scale_bcast_bf16.restype = None
    u64 = ctypes.c_uint64
    lib.oracle_layernorm_act_ex_f32.argtypes = [
        F32P, F32P, F32P, F32P, F32P, F32P, F64P, F64P, i64, i64, f32, ctypes.c_int, f32,
        u64, u64]
    lib.oracle_layernorm_act_ex_f32.restype = None
    lib.oracle_layernorm_act_ex_bf16.argtypes = [
        U16P, U16P, U16P, U16P, U16P, U16P, F64P, F64P, i64, i64, f32, ctypes.c_int, f32,
        u64, u64]
    lib.oracle_layernorm_act_ex_bf16.restype = None
    U32P = ctypes.POINTER(ctypes.c_uint32)
    U64P = ctypes.POINTER(ctypes.c_uint64)
    lib.oracle_philox4x32_10.argtypes = [U32P, U32P, U32P]
    lib.oracle_philox4x32_10.restype = None
    lib.oracle_philox4x64_10.argtypes = [U64P, U64P, U64P]
    lib.oracle_philox4x64_10.restype = None
    lib.oracle_dropout_keep.argtypes = [u64, u64, i64, f32]
    lib.oracle_dropout_keep.restype = ctypes.c_int
    lib.oracle_dropout_mask.argtypes = [u64, u64, i64, i64, f32, ctypes.POINTER(ctypes.c_uint8)]
    lib.oracle_dropout_mask.restype = None
    lib.oracle_scale_mask_softmax_f32.argtypes = [F32P, F32P, i64, i64, f32, ctypes.c_int, i64, i64]
    lib.oracle_scale_mask_softmax_f32.restype = None
    lib.oracle_scale_mask_softmax_bf16.argtypes = [U16P, U16P, i64, i64, f32, ctypes.c_int, i64, i64]
    lib.oracle_scale_mask_softmax_bf16.restype = None
    lib.oracle_row_softmax_f32.argtypes = [F32P, F32P, i64, i64]
    lib.oracle_row_softmax_f32.restype = None
    lib.oracle_row_softmax_bf16.argtypes = [U16P, U16P, i64, i64]
    lib.oracle_row_softmax_bf16.restype = None
    if path is None:
        _lib = lib
    return lib


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


# --------------------------------------------------------------------------
# scalar helpers
# --------------------------------------------------------------------------

def relu_f32(v, lib=None):
    return (lib or load()).oracle_relu_f32(float(v))


def gelu_tanh(z, lib=None):
    return (lib or load()).oracle_gelu_tanh(float(z))


def bf16_from_double(v, lib=None):
    return (lib or load()).oracle_bf16_from_double(float(v))


def bf16_to_double(h, lib=None):
    return (lib or load()).oracle_bf16_to_double(int(h))


# --------------------------------------------------------------------------
# o1: y = relu(x + b1) * scale + b2   ([P1] §1.1, §3.1)
# --------------------------------------------------------------------------

def add_relu_scale(x, b1, b2, scale=0.5, lib=None):
    """fp32 (float32 arrays) or bf16 (uint16 bit patterns) pointwise chain."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    if not (x.shape == np.shape(b1) == np.shape(b2)):
        raise ValueError("x, b1, b2 must have one shape")
    dt = x.dtype
    if dt == np.float32:
        x, b1, b2 = (_c(a, np.float32) for a in (x, b1, b2))
        y = np.empty_like(x)
        lib.oracle_add_relu_scale_f32(_f32p(x), _f32p(b1), _f32p(b2), _f32p(y),
                                      x.size, scale)
    elif dt == np.uint16:
        x, b1, b2 = (_c(a, np.uint16) for a in (x, b1, b2))
        y = np.empty_like(x)
        lib.oracle_add_relu_scale_bf16(_u16p(x), _u16p(b1), _u16p(b2), _u16p(y),
                                       x.size, scale)
    else:
        raise TypeError(f"unsupported dtype {dt}")
    return y


# --------------------------------------------------------------------------
# o2: TorchInductor example chain   ([P4] "model", Figure 1)
# --------------------------------------------------------------------------

def add_relu_scale_bcast(x, b1, b2, scale=0.5, lib=None):
    """The pointwise chain on a 2-D x (rows, cols); b1 and b2 each either the
    shape of x or a length-cols vector broadcast over the rows."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    if x.dtype == np.float32:
        cv, fn, ptr = np.float32, lib.oracle_add_relu_scale_bcast_f32, _f32p
    elif x.dtype == np.uint16:
        cv, fn, ptr = np.uint16, lib.oracle_add_relu_scale_bcast_bf16, _u16p
    else:
        raise TypeError(f"unsupported dtype {x.dtype}")
    b1, b2 = _c(b1, cv), _c(b2, cv)
    flags = []
    for v in (b1, b2):
        if v.shape == x.shape:
            flags.append(0)
        elif v.shape == (cols,):
            flags.append(1)
        else:
            raise ValueError("b1 / b2 must have x's shape or (cols,)")
    y = np.empty_like(x)
    fn(ptr(x), ptr(b1), ptr(b2), ptr(y), rows, cols, flags[0], flags[1], scale)
    return y


def bias_relu_branch_mean_epilogue(x, bias, gamma, beta, x_scale=1.1,
                                   branch_scale=0.1, intermediates=False,
                                   lib=None):
    """y = (s - mean(s, 1)) * gamma + beta with s = relu(x*x_scale + bias)^2
    + relu(...)*branch_scale.  With ``intermediates`` also returns (s, m)."""
    lib = lib or load()
    x = _c(x, np.float32)
    rows, cols = x.shape
    bias, gamma, beta = (_c(a, np.float32) for a in (bias, gamma, beta))
    for v in (bias, gamma, beta):
        if v.shape != (cols,):
            raise ValueError("per-column vectors must have length cols")
    y = np.empty_like(x)
    s = np.empty_like(x) if intermediates else None
    m = np.empty(rows, np.float32) if intermediates else None
    lib.oracle_bias_relu_branch_mean_epilogue(
        _f32p(x), _f32p(bias), _f32p(gamma), _f32p(beta), _f32p(y), rows, cols,
        x_scale, branch_scale, _f32p_opt(s), _f32p_opt(m))
    if intermediates:
        return y, s, m
    return y


def bias_relu_branch_mean_epilogue_bf16(x, bias, gamma, beta, x_scale=1.1,
                                        branch_scale=0.1, lib=None):
    """o2 with bf16 I/O (uint16 bit patterns): widen, fp32 steps, round y once."""
    lib = lib or load()
    x = _c(x, np.uint16)
    rows, cols = x.shape
    bias, gamma, beta = (_c(a, np.uint16) for a in (bias, gamma, beta))
    for v in (bias, gamma, beta):
        if v.shape != (cols,):
            raise ValueError("per-column vectors must have length cols")
    y = np.empty_like(x)
    lib.oracle_bias_relu_branch_mean_epilogue_bf16(
        _u16p(x), _u16p(bias), _u16p(gamma), _u16p(beta), _u16p(y), rows, cols,
        x_scale, branch_scale)
    return y


# --------------------------------------------------------------------------
# o3: residual + LayerNorm + affine + GeLU-tanh   ([P2] §2.3, [P3] §4.3)
# --------------------------------------------------------------------------

def residual_layernorm_gelu(x, r, w, b, eps=1e-5, intermediates=False, lib=None):
    """out = gelu_tanh(LayerNorm(x + r) * w + b).  float32 or uint16 (bf16)
    inputs; the output has the input dtype.  With ``intermediates`` also
    returns (mean, rstd, xhat) in float64."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    rows, hidden = x.shape
    dt = x.dtype
    out = np.empty_like(x)
    mean = np.empty(rows, np.float64) if intermediates else None
    rstd = np.empty(rows, np.float64) if intermediates else None
    xhat = np.empty((rows, hidden), np.float64) if intermediates else None
    if dt == np.float32:
        r, w, b = (_c(a, np.float32) for a in (r, w, b))
        fn, p = lib.oracle_residual_layernorm_gelu_f32, _f32p
    elif dt == np.uint16:
        r, w, b = (_c(a, np.uint16) for a in (r, w, b))
        fn, p = lib.oracle_residual_layernorm_gelu_bf16, _u16p
    else:
        raise TypeError(f"unsupported dtype {dt}")
    if r.shape != x.shape or w.shape != (hidden,) or b.shape != (hidden,):
        raise ValueError("shape mismatch")
    fn(p(x), p(r), p(w), p(b), p(out), rows, hidden, eps, _f64p(mean),
       _f64p(rstd), _f64p(xhat))
    if intermediates:
        return out, mean, rstd, xhat
    return out


# --------------------------------------------------------------------------
# o4: LayerNorm family   ([P3] §4.3, [P2] §2.1-2.3)
# --------------------------------------------------------------------------

ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2


def layernorm_act(x, r, w, b, eps=1e-5, act=ACT_GELU, want_h=False, lib=None):
    """out = act(LayerNorm(x (+ r)) * w + b); r may be None.  With ``want_h``
    also returns h = x + r (or x) rounded to the I/O type."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    rows, hidden = x.shape
    dt = x.dtype
    if dt == np.float32:
        cv, fn, p, nullp = np.float32, lib.oracle_layernorm_act_f32, _f32p, ctypes.POINTER(ctypes.c_float)()
    elif dt == np.uint16:
        cv, fn, p, nullp = np.uint16, lib.oracle_layernorm_act_bf16, _u16p, ctypes.POINTER(ctypes.c_uint16)()
    else:
        raise TypeError(f"unsupported dtype {dt}")
    w, b = _c(w, cv), _c(b, cv)
    if r is not None:
        r = _c(r, cv)
        if r.shape != x.shape:
            raise ValueError("shape mismatch")
    if w.shape != (hidden,) or b.shape != (hidden,):
        raise ValueError("shape mismatch")
    out = np.empty_like(x)
    h = np.empty_like(x) if want_h else None
    fn(p(x), p(r) if r is not None else nullp, p(w), p(b), p(out),
       p(h) if h is not None else nullp, rows, hidden, eps, int(act))
    return (out, h) if want_h else out


def layernorm_act_ex(x, r, w, b, eps=1e-5, act=ACT_GELU, p=0.0, seed=0, offset=0,
                     want_h=False, want_stats=False, lib=None):
    """o4 with its extras: dropout with probability ``p`` keyed by (seed,
    offset) on the activation output, and the per-row statistics.  Returns
    (out, h, mean, rstd); h is None without ``want_h``, mean and rstd (float64
    per row) None without ``want_stats``."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    rows, hidden = x.shape
    if x.dtype == np.float32:
        cv, fn, ptr, nullp = np.float32, lib.oracle_layernorm_act_ex_f32, _f32p, ctypes.POINTER(ctypes.c_float)()
    elif x.dtype == np.uint16:
        cv, fn, ptr, nullp = np.uint16, lib.oracle_layernorm_act_ex_bf16, _u16p, ctypes.POINTER(ctypes.c_uint16)()
    else:
        raise TypeError(f"unsupported dtype {x.dtype}")
    w, b = _c(w, cv), _c(b, cv)
    if r is not None:
        r = _c(r, cv)
        if r.shape != x.shape:
            raise ValueError("shape mismatch")
    if w.shape != (hidden,) or b.shape != (hidden,):
        raise ValueError("shape mismatch")
    out = np.empty_like(x)
    h = np.empty_like(x) if want_h else None
    mean = np.empty(rows, np.float64) if want_stats else None
    rstd = np.empty(rows, np.float64) if want_stats else None
    fn(ptr(x), ptr(r) if r is not None else nullp, ptr(w), ptr(b), ptr(out),
       ptr(h) if h is not None else nullp, _f64p(mean), _f64p(rstd), rows, hidden, eps,
       int(act), float(p), int(seed), int(offset))
    return out, h, mean, rstd


# --------------------------------------------------------------------------
# o6: Philox counter-based generator and the dropout decision
# --------------------------------------------------------------------------

def philox4x32_10(ctr, key, lib=None):
    """Philox-4x32-10 of a 4-word counter and a 2-word key (uint32 words)."""
    lib = lib or load()
    c = np.ascontiguousarray(ctr, np.uint32)
    k = np.ascontiguousarray(key, np.uint32)
    o = np.empty(4, np.uint32)
    P = ctypes.POINTER(ctypes.c_uint32)
    lib.oracle_philox4x32_10(c.ctypes.data_as(P), k.ctypes.data_as(P), o.ctypes.data_as(P))
    return o


def philox4x64_10(ctr, key, lib=None):
    """Philox-4x64-10 (uint64 words): the same rounds with 64-bit words."""
    lib = lib or load()
    c = np.ascontiguousarray(ctr, np.uint64)
    k = np.ascontiguousarray(key, np.uint64)
    o = np.empty(4, np.uint64)
    P = ctypes.POINTER(ctypes.c_uint64)
    lib.oracle_philox4x64_10(c.ctypes.data_as(P), k.ctypes.data_as(P), o.ctypes.data_as(P))
    return o


def dropout_mask(seed, offset, start, n, p, lib=None):
    """Keep decisions (bool) of elements start .. start + n - 1."""
    lib = lib or load()
    keep = np.empty(n, np.uint8)
    lib.oracle_dropout_mask(int(seed), int(offset), int(start), int(n), float(p),
                            keep.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    return keep.astype(bool)


# --------------------------------------------------------------------------
# o5: row softmax   ([P1] §4.1-4.2, [P2] §3.2)
# --------------------------------------------------------------------------

def row_softmax(x, lib=None):
    """Softmax of each row (float32, or uint16 bf16 bit patterns)."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    y = np.empty_like(x)
    if x.dtype == np.float32:
        lib.oracle_row_softmax_f32(_f32p(x), _f32p(y), rows, cols)
    elif x.dtype == np.uint16:
        lib.oracle_row_softmax_bf16(_u16p(x), _u16p(y), rows, cols)
    else:
        raise TypeError(f"unsupported dtype {x.dtype}")
    return y


def scale_mask_softmax(x, scale=1.0, causal=False, period=None, offset=0, lib=None):
    """Softmax of each row of x * scale, with an optional causal mask: element
    j of row i is masked when j > (i mod period) + offset (period defaults to
    the row count); masked outputs are 0."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    period = rows if period is None else period
    y = np.empty_like(x)
    if x.dtype == np.float32:
        lib.oracle_scale_mask_softmax_f32(_f32p(x), _f32p(y), rows, cols, float(scale),
                                          int(bool(causal)), int(period), int(offset))
    elif x.dtype == np.uint16:
        lib.oracle_scale_mask_softmax_bf16(_u16p(x), _u16p(y), rows, cols, float(scale),
                                           int(bool(causal)), int(period), int(offset))
    else:
        raise TypeError(f"unsupported dtype {x.dtype}")
    return y
