"""ctypes binding of libmemory_bound.so (argument marshalling only)."""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "libmemory_bound.so")

MB_F32, MB_BF16 = 0, 1
MB_MAX_COLS = 524288
ROW_PATHS = {"auto": 0, "warp": 1, "direct": 2, "staged": 3, "cluster": 4}
ACTIVATIONS = {"none": 0, "relu": 1, "gelu_tanh": 2}

STATUS_NAMES = {0: "MB_OK", 1: "MB_ERR_NULL", 2: "MB_ERR_SHAPE", 3: "MB_ERR_DTYPE",
                4: "MB_ERR_OVERLAP", 5: "MB_ERR_ALIGN", 6: "MB_ERR_VALUE",
                7: "MB_ERR_CUDA", 8: "MB_ERR_DEVICE"}

# Entry points declared in include/memory_bound.h: name -> (restype, argtypes)
_P, _I64, _F, _I, _U32P, _I32P = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_float,
                                  ctypes.c_int, ctypes.POINTER(ctypes.c_uint32),
                                  ctypes.POINTER(ctypes.c_int32))
SIGNATURES = {
    "fused_add_relu_scale": (_I, [_P, _P, _P, _P, _I64, _F, _I, _P]),
    "fused_add_relu_scale_bcast": (_I, [_P, _P, _P, _P, _I64, _I64, _I, _I, _F, _I, _P]),
    "fused_bias_relu_branch_mean_epilogue": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _F, _F, _P]),
    "fused_residual_layernorm_gelu": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _F, _I, _P]),
    "fused_bias_relu_branch_mean_epilogue_bf16": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _F, _F, _P]),
    "fused_layernorm_act": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I, _I, _P]),
    "fused_layernorm_act_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I, _F,
                                    ctypes.c_uint64, ctypes.c_uint64, _I, _P]),
    "fused_row_softmax": (_I, [_P, _P, _I64, _I64, _I, _P]),
    "fused_scale_mask_softmax": (_I, [_P, _P, _I64, _I64, _F, _I, _I64, _I64, _I, _P]),
    "mb_status_string": (ctypes.c_char_p, [_I]),
    "mb_abi_version": (_I, []),
    "mb_last_cuda_error": (_I, []),
    "mb_device_error": (_I, [_U32P]),
    "mb_set_row_path": (_I, [_I, _I, _I, _I]),
    "mb_set_pointwise_shape": (_I, [_I, _I]),
    "mb_set_launch_overlap": (_I, [_I]),
    "mb_selftest_wait_timeout": (_I, [ctypes.c_uint32, _P]),
    "mb_selftest_exchange_timeout": (_I, [ctypes.c_uint32, _P]),
    "mb_row_plan": (_I, [_I, _I, _I64, _I64, _I, _I32P]),
}

_lib = None


class MBError(RuntimeError):
    """A non-MB_OK status from the library."""

    def __init__(self, fn, status, detail=""):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        msg = f"{fn}: {name} ({status_string(status)})"
        if detail:
            msg += f"; {detail}"
        super().__init__(msg)


def library_path():
    return _LIB_PATH


def load_library(path=None):
    """Load libmemory_bound.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build it with memory_bound_gb300.build.build() "
            "(the fused chains have no other implementation)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib


class _Raw:
    """The C entry points, loaded on first use."""

    def __getattr__(self, name):
        if name not in SIGNATURES:
            raise AttributeError(name)
        return getattr(load_library(), name)


raw = _Raw()


def status_string(status):
    return load_library().mb_status_string(int(status)).decode()


def _check(fn, status, detail=""):
    if status != 0:
        if status == 7:
            detail = (detail + f" cudaError={load_library().mb_last_cuda_error()}").strip()
        raise MBError(fn, status, detail)


# --------------------------------------------------------------------------
# torch tensor front end
# --------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return MB_F32
    if t.dtype == torch.bfloat16:
        return MB_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _call_device(tensors):
    """The CUDA device a call runs on: that of its CUDA tensors, else (all
    tensors in pinned host memory) the current device."""
    torch = _torch()
    for t in tensors:
        if t is not None and t.is_cuda:
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def _stream_handle(dev):
    torch = _torch()
    return torch.cuda.current_stream(dev).cuda_stream


def _empty_like(x):
    """An output like x: on x's device, or in pinned host memory when x is
    there (the kernels then write it over the host link, asynchronously:
    synchronise the stream before reading it on the host)."""
    torch = _torch()
    if x.is_cuda:
        return torch.empty_like(x)
    if not (x.device.type == "cpu" and x.is_pinned()):
        raise ValueError("tensors must be CUDA tensors or pinned host tensors")
    return torch.empty(x.shape, dtype=x.dtype, pin_memory=True)


class _NoSwitch:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


_NO_SWITCH = _NoSwitch()


def _on_device(dev):
    """Make dev current for the call (a no-op when it already is)."""
    torch = _torch()
    if dev.index == torch.cuda.current_device():
        return _NO_SWITCH
    return torch.cuda.device(dev)


def _require(tensors, dtype):
    """Contiguous tensors of one dtype, each either on one CUDA device or in
    pinned (page-locked) host memory; returns the device the call runs on."""
    for t in tensors:
        if not (t.is_cuda or (t.device.type == "cpu" and t.is_pinned())):
            raise ValueError("tensors must be CUDA tensors or pinned host tensors")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous (row-major)")
        if t.dtype != dtype:
            raise TypeError("all tensors of a call must share one dtype")
    dev = _call_device(tensors)
    if any(t.is_cuda and t.device != dev for t in tensors):
        raise ValueError("all CUDA tensors of a call must be on one device")
    return dev


def fused_add_relu_scale(x, b1, b2, scale=0.5, out=None):
    """y = relu(x + b1) * scale + b2, elementwise (float32 or bfloat16).

    b1 and b2 each have x's size, or (bias-like) the size of x's last
    dimension, broadcast over the leading ones."""
    if out is None:
        out = _empty_like(x)
    dev = _require([x, b1, b2, out], x.dtype)
    n = x.numel()
    if out.numel() != n:
        raise ValueError("out must have x's size")
    if b1.numel() == n and b2.numel() == n:
        with _on_device(dev):
            st = load_library().fused_add_relu_scale(
                x.data_ptr(), b1.data_ptr(), b2.data_ptr(), out.data_ptr(), n,
                float(scale), _dtype_code(x), _stream_handle(dev))
        _check("fused_add_relu_scale", st)
        return out
    cols = x.shape[-1] if x.dim() > 0 else 1
    flags = []
    for v in (b1, b2):
        if v.numel() == n:
            flags.append(0)
        elif v.numel() == cols:
            flags.append(1)
        else:
            raise ValueError("b1 / b2 must have x's size or its last dimension's")
    rows = n // cols if cols else 0
    with _on_device(dev):
        st = load_library().fused_add_relu_scale_bcast(
            x.data_ptr(), b1.data_ptr(), b2.data_ptr(), out.data_ptr(), rows, cols, flags[0],
            flags[1], float(scale), _dtype_code(x), _stream_handle(dev))
    _check("fused_add_relu_scale_bcast", st)
    return out


def fused_bias_relu_branch_mean_epilogue(x, bias, gamma, beta, x_scale=1.1,
                                         branch_scale=0.1, out=None):
    """The TorchInductor example chain on a 2-D x (rows x cols), float32 or
    bfloat16 (all tensors one dtype)."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D (rows, cols)")
    if out is None:
        out = _empty_like(x)
    dev = _require([x, bias, gamma, beta, out], x.dtype)
    fn_name = ("fused_bias_relu_branch_mean_epilogue" if _dtype_code(x) == MB_F32
               else "fused_bias_relu_branch_mean_epilogue_bf16")
    rows, cols = x.shape
    for v in (bias, gamma, beta):
        if v.numel() != cols:
            raise ValueError("per-column vectors must have cols elements")
    if out.numel() != x.numel():
        raise ValueError("out must match x")
    with _on_device(dev):
        st = getattr(load_library(), fn_name)(
            x.data_ptr(), bias.data_ptr(), gamma.data_ptr(), beta.data_ptr(),
            out.data_ptr(), rows, cols, float(x_scale), float(branch_scale),
            _stream_handle(dev))
    _check(fn_name, st)
    return out


def fused_residual_layernorm_gelu(x, r, w, b, eps=1e-5, out=None):
    """GeLU_tanh(LayerNorm(x + r) * w + b) over the last dim of a 2-D x."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D (rows, hidden)")
    if out is None:
        out = _empty_like(x)
    dev = _require([x, r, w, b, out], x.dtype)
    rows, hidden = x.shape
    if r.shape != x.shape or w.numel() != hidden or b.numel() != hidden:
        raise ValueError("shape mismatch")
    if out.numel() != x.numel():
        raise ValueError("out must match x")
    with _on_device(dev):
        st = load_library().fused_residual_layernorm_gelu(
            x.data_ptr(), r.data_ptr(), w.data_ptr(), b.data_ptr(), out.data_ptr(),
            rows, hidden, float(eps), _dtype_code(x), _stream_handle(dev))
    _check("fused_residual_layernorm_gelu", st)
    return out


def fused_layernorm_act(x, r, w, b, eps=1e-5, act="gelu_tanh", out=None, h_out=None,
                        want_h=False, p=0.0, seed=0, offset=0, mean_out=None, rstd_out=None,
                        want_stats=False):
    """act(LayerNorm(x (+ r)) * w + b) over the last dim of a 2-D x; r may be
    None (no residual).

    With ``want_h`` (or an ``h_out`` tensor) also writes h = x + r (or x), the
    residual stream.  With ``p`` > 0, dropout on the output keyed by
    (``seed``, ``offset``) (Philox-4x32-10; see fused_layernorm_act_ex in the
    C header).  With ``want_stats`` (or ``mean_out`` / ``rstd_out`` float32
    tensors of ``rows`` values) also writes each row's mean and rstd.

    Returns out; (out, h) when h is written; (out, h or None, mean, rstd) when
    the statistics are."""
    torch = _torch()
    if x.dim() != 2:
        raise ValueError("x must be 2-D (rows, hidden)")
    rows, hidden = x.shape
    if out is None:
        out = _empty_like(x)
    if want_h and h_out is None:
        h_out = _empty_like(x)
    stats = want_stats or mean_out is not None or rstd_out is not None
    if stats:
        like = x if x.is_cuda else None
        for name, t in (("mean_out", mean_out), ("rstd_out", rstd_out)):
            if t is None:
                t = (torch.empty(rows, dtype=torch.float32, device=like.device) if like is not None
                     else torch.empty(rows, dtype=torch.float32, pin_memory=True))
            elif t.dtype != torch.float32 or t.numel() != rows:
                raise ValueError(f"{name} must be float32 with rows elements")
            if name == "mean_out":
                mean_out = t
            else:
                rstd_out = t
    ts = [x, w, b, out] + [t for t in (r, h_out) if t is not None]
    dev = _require(ts, x.dtype)
    if stats:
        _require([mean_out, rstd_out], torch.float32)
    if (r is not None and r.shape != x.shape) or w.numel() != hidden or b.numel() != hidden:
        raise ValueError("shape mismatch")
    for t in (out, h_out):
        if t is not None and t.numel() != x.numel():
            raise ValueError("outputs must match x")
    code = ACTIVATIONS[act] if isinstance(act, str) else int(act)
    ptr = (lambda t: t.data_ptr() if t is not None else None)
    with _on_device(dev):
        if p == 0.0 and not stats:
            st = load_library().fused_layernorm_act(
                x.data_ptr(), ptr(r), w.data_ptr(), b.data_ptr(), out.data_ptr(), ptr(h_out),
                rows, hidden, float(eps), code, _dtype_code(x), _stream_handle(dev))
        else:
            st = load_library().fused_layernorm_act_ex(
                x.data_ptr(), ptr(r), w.data_ptr(), b.data_ptr(), out.data_ptr(), ptr(h_out),
                ptr(mean_out), ptr(rstd_out), rows, hidden, float(eps), code, float(p),
                int(seed), int(offset), _dtype_code(x), _stream_handle(dev))
    _check("fused_layernorm_act", st)
    if stats:
        return out, h_out, mean_out, rstd_out
    return (out, h_out) if h_out is not None else out


def fused_row_softmax(x, out=None, scale=1.0, causal=False, period=None, offset=0):
    """Softmax over the last dim of a 2-D x (float32 or bfloat16).

    With ``scale`` != 1 or ``causal``: the softmax of attention-score rows
    x * scale, key j of row i masked when j > (i mod period) + offset
    (period defaults to the row count); masked outputs are 0."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D (rows, cols)")
    if out is None:
        out = _empty_like(x)
    dev = _require([x, out], x.dtype)
    if out.numel() != x.numel():
        raise ValueError("out must match x")
    rows, cols = x.shape
    if scale == 1.0 and not causal:
        with _on_device(dev):
            st = load_library().fused_row_softmax(x.data_ptr(), out.data_ptr(), rows, cols,
                                                  _dtype_code(x), _stream_handle(dev))
        _check("fused_row_softmax", st)
        return out
    per = rows if period is None else int(period)
    with _on_device(dev):
        st = load_library().fused_scale_mask_softmax(
            x.data_ptr(), out.data_ptr(), rows, cols, float(scale), int(bool(causal)),
            max(per, 1), int(offset), _dtype_code(x), _stream_handle(dev))
    _check("fused_scale_mask_softmax", st)
    return out


def device_error():
    """Read and clear the current device's failure flags (synchronises)."""
    flags = ctypes.c_uint32(0)
    st = load_library().mb_device_error(ctypes.byref(flags))
    if st not in (0, 8):
        _check("mb_device_error", st)
    return flags.value


def set_row_path(path="auto", ctas_per_sm=0, stages=0, vec_per_thread=0):
    """Process-wide override of the row-chain path ("auto", "warp",
    "direct", "staged") and launch shape (0 = automatic)."""
    code = ROW_PATHS[path] if isinstance(path, str) else int(path)
    _check("mb_set_row_path", load_library().mb_set_row_path(code, ctas_per_sm, stages,
                                                             vec_per_thread))


def set_launch_overlap(enable=True):
    """Process-wide: launch with programmatic stream serialisation (default)."""
    _check("mb_set_launch_overlap", load_library().mb_set_launch_overlap(int(bool(enable))))


def set_pointwise_shape(blocks_per_sm=0, unroll=0):
    """Process-wide override of the pointwise launch shape (0 = automatic)."""
    _check("mb_set_pointwise_shape",
           load_library().mb_set_pointwise_shape(blocks_per_sm, unroll))


def row_plan(chain, dtype, rows, cols, aligned=True):
    """The launch a row chain would use: dict(path, threads, ctas, vpt, vec,
    stages, smem).  chain: "ln", "inductor", "lnact_res", "lnact", "softmax",
    "lnact_res_dropout", "lnact_dropout", "lnact_res_h" (with the
    residual-stream output) or "softmax_mask" (the scaled softmax under a square
    causal mask: period = cols, offset 0); dtype: "f32" or "bf16"; aligned:
    True / 1 every pointer 16-byte aligned, 2 the row tensors at one common
    offset within 16 bytes, False / 0 neither."""
    out = (ctypes.c_int32 * 7)()
    code = {"ln": 0, "inductor": 1, "lnact_res": 2, "lnact": 3, "softmax": 4,
            "lnact_res_dropout": 5, "lnact_dropout": 6, "lnact_res_h": 7,
            "softmax_mask": 8}[chain]
    dt = {"f32": MB_F32, "bf16": MB_BF16}[dtype]
    al = int(aligned)
    st = load_library().mb_row_plan(code, dt, rows, cols, al, out)
    _check("mb_row_plan", st)
    keys = ("path", "threads", "ctas", "vpt", "vec", "stages", "smem")
    d = dict(zip(keys, list(out)))
    d["path"] = {v: k for k, v in ROW_PATHS.items()}[d["path"]]
    return d
