"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import memory_bound_gb300 as mb
from memory_bound_gb300 import build as lib_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "memory_bound.h")

MB_OK, MB_ERR_NULL, MB_ERR_SHAPE, MB_ERR_DTYPE, MB_ERR_OVERLAP = 0, 1, 2, 3, 4
MB_ERR_ALIGN, MB_ERR_VALUE = 5, 6

# Fake but 16-byte aligned, non-overlapping "device" addresses: none of the
# calls below gets as far as using them.
A, B, C, D, E = (0x10000000 * k for k in range(1, 6))


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return mb.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if not n.startswith("defined")))


def test_header_declares_the_three_chains():
    names = declared_functions()
    for n in ("fused_add_relu_scale", "fused_residual_layernorm_gelu",
              "fused_bias_relu_branch_mean_epilogue"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    # and the binding knows each of them
    assert set(names) <= set(mb._binding.SIGNATURES)


def test_version_and_status_strings(lib):
    assert lib.mb_abi_version() == 1
    for s in range(9):
        assert len(mb.status_string(s)) > 0
    assert mb.status_string(99) == "unknown status"


def test_pointwise_argument_checks(lib):
    f = lib.fused_add_relu_scale
    assert f(A, B, C, D, 0, 0.5, 0, None) == MB_OK          # empty: no-op
    assert f(A, B, C, D, 10, 0.5, 2, None) == MB_ERR_DTYPE
    assert f(A, B, C, D, -1, 0.5, 0, None) == MB_ERR_SHAPE
    assert f(A, B, C, D, 10, float("nan"), 0, None) == MB_ERR_VALUE
    assert f(A, B, C, D, 10, float("inf"), 0, None) == MB_ERR_VALUE
    assert f(None, B, C, D, 10, 0.5, 0, None) == MB_ERR_NULL
    assert f(A, B, C, None, 10, 0.5, 0, None) == MB_ERR_NULL
    assert f(A + 2, B, C, D, 10, 0.5, 0, None) == MB_ERR_ALIGN   # f32 needs 4
    assert f(A + 1, B, C, D, 10, 0.5, 1, None) == MB_ERR_ALIGN   # bf16 needs 2
    assert f(A, B, C, A + 36, 10, 0.5, 0, None) == MB_ERR_OVERLAP
    assert f(A, B, C, C - 4, 10, 0.5, 0, None) == MB_ERR_OVERLAP  # y ends inside b2


def test_layernorm_argument_checks(lib):
    f = lib.fused_residual_layernorm_gelu
    assert f(A, B, C, D, E, 0, 64, 1e-5, 0, None) == MB_OK
    assert f(A, B, C, D, E, 4, 0, 1e-5, 0, None) == MB_ERR_SHAPE
    assert f(A, B, C, D, E, 4, mb.MB_MAX_COLS + 1, 1e-5, 0, None) == MB_ERR_SHAPE
    assert f(A, B, C, D, E, -1, 64, 1e-5, 0, None) == MB_ERR_SHAPE
    assert f(A, B, C, D, E, 4, 64, -1e-5, 0, None) == MB_ERR_VALUE
    assert f(A, B, C, D, E, 4, 64, float("nan"), 1, None) == MB_ERR_VALUE
    assert f(A, B, C, D, E, 4, 64, 1e-5, 5, None) == MB_ERR_DTYPE
    assert f(A, B, None, D, E, 4, 64, 1e-5, 0, None) == MB_ERR_NULL
    assert f(A, B, C, D, A + 64, 4, 64, 1e-5, 0, None) == MB_ERR_OVERLAP
    assert f(A, B, C, D, C - 16, 4, 64, 1e-5, 0, None) == MB_ERR_OVERLAP  # over w
    assert f(A, B, C + 2, D, E, 4, 64, 1e-5, 0, None) == MB_ERR_ALIGN


def test_inductor_argument_checks(lib):
    f = lib.fused_bias_relu_branch_mean_epilogue
    assert f(A, B, C, D, E, 0, 1024, 1.1, 0.1, None) == MB_OK
    assert f(A, B, C, D, E, 8, 0, 1.1, 0.1, None) == MB_ERR_SHAPE
    assert f(A, B, C, D, E, 8, 1024, float("nan"), 0.1, None) == MB_ERR_VALUE
    assert f(A, None, C, D, E, 8, 1024, 1.1, 0.1, None) == MB_ERR_NULL
    assert f(A, B, C, D, A + 4096, 8, 1024, 1.1, 0.1, None) == MB_ERR_OVERLAP
    assert f(A + 1, B, C, D, E, 8, 1024, 1.1, 0.1, None) == MB_ERR_ALIGN


def test_row_path_setter_validates(lib):
    assert lib.mb_set_row_path(9, 0, 0, 0) == MB_ERR_VALUE
    assert lib.mb_set_row_path(5, 0, 0, 0) == MB_ERR_VALUE
    assert lib.mb_set_row_path(4, 0, 8, 0) == MB_OK          # cluster path
    assert lib.mb_set_row_path(0, -1, 0, 0) == MB_ERR_VALUE
    assert lib.mb_set_row_path(0, 0, 0, -2) == MB_ERR_VALUE
    assert lib.mb_set_row_path(3, 2, 4, 1) == MB_OK
    assert lib.mb_set_row_path(0, 0, 0, 0) == MB_OK


def test_row_plan_validates_its_arguments(lib):
    """mb_row_plan refuses a NULL output, an unknown chain and an alignment
    class other than 0, 1 or 2 before it queries the device."""
    out = (ctypes.c_int32 * 7)()
    assert lib.mb_row_plan(0, 0, 8, 4096, 1, None) == MB_ERR_NULL
    assert lib.mb_row_plan(9, 0, 8, 4096, 1, out) == MB_ERR_VALUE
    assert lib.mb_row_plan(0, 0, 8, 4096, 3, out) == MB_ERR_VALUE
    assert lib.mb_row_plan(0, 0, 8, 4096, -1, out) == MB_ERR_VALUE


def test_launch_overlap_setter_validates(lib):
    assert lib.mb_set_launch_overlap(2) == MB_ERR_VALUE
    assert lib.mb_set_launch_overlap(0) == MB_OK
    assert lib.mb_set_launch_overlap(1) == MB_OK


def test_pointwise_shape_setter_validates(lib):
    assert lib.mb_set_pointwise_shape(-1, 0) == MB_ERR_VALUE
    assert lib.mb_set_pointwise_shape(0, 3) == MB_ERR_VALUE
    assert lib.mb_set_pointwise_shape(2, 8) == MB_OK
    assert lib.mb_set_pointwise_shape(0, 0) == MB_OK


def test_null_out_pointers(lib):
    assert lib.mb_device_error(None) == MB_ERR_NULL
    assert lib.mb_row_plan(0, 0, 8, 64, 1, None) == MB_ERR_NULL


def test_binding_rejects_without_gpu_work():
    import torch
    x = torch.zeros(8)
    with pytest.raises(ValueError):
        mb.fused_add_relu_scale(x, x, x)          # CPU tensors are refused


def test_further_chains_argument_checks(lib):
    f = lib.fused_layernorm_act
    assert f(A, None, C, D, E, None, 0, 64, 1e-5, 2, 0, None) == MB_OK
    assert f(A, None, C, D, E, None, 4, 64, 1e-5, 3, 0, None) == MB_ERR_VALUE   # act
    assert f(A, None, C, D, E, None, 4, 64, 1e-5, 1, 9, None) == MB_ERR_DTYPE
    assert f(None, None, C, D, E, None, 4, 64, 1e-5, 1, 0, None) == MB_ERR_NULL
    assert f(A, B, C, D, E, E + 128, 4, 64, 1e-5, 1, 0, None) == MB_ERR_OVERLAP  # h over out
    assert f(A, B, C, D, E, B + 64, 4, 64, 1e-5, 1, 0, None) == MB_ERR_OVERLAP   # h over r
    assert f(A, B + 2, C, D, E, None, 4, 64, 1e-5, 1, 0, None) == MB_ERR_ALIGN
    s = lib.fused_row_softmax
    assert s(A, B, 0, 10, 0, None) == MB_OK
    assert s(A, B, 4, 0, 0, None) == MB_ERR_SHAPE
    assert s(A, A + 8, 4, 10, 0, None) == MB_ERR_OVERLAP
    assert s(A, None, 4, 10, 1, None) == MB_ERR_NULL
    assert s(A + 1, B, 4, 10, 1, None) == MB_ERR_ALIGN
    g = lib.fused_bias_relu_branch_mean_epilogue_bf16
    assert g(A, B, C, D, E, 0, 64, 1.1, 0.1, None) == MB_OK
    assert g(A, B, C, D, A + 2, 2, 64, 1.1, 0.1, None) == MB_ERR_OVERLAP
    assert g(A + 1, B, C, D, E, 2, 64, 1.1, 0.1, None) == MB_ERR_ALIGN


def test_layernorm_ex_argument_checks(lib):
    """Dropout probability, statistics pointers and their overlaps are all
    checked on the host."""
    f = lib.fused_layernorm_act_ex
    F = 0x60000000                                  # statistics buffers
    G = F + 0x1000
    nan = float("nan")
    assert f(A, B, C, D, E, None, F, G, 0, 64, 1e-5, 1, 0.1, 1, 0, 0, None) == MB_OK
    for p in (-0.1, 1.0, 1.5, nan):
        assert f(A, B, C, D, E, None, None, None, 4, 64, 1e-5, 1, p, 1, 0, 0, None) == MB_ERR_VALUE
    assert f(A, B, C, D, E, None, F + 2, None, 4, 64, 1e-5, 1, 0.1, 1, 0, 0, None) == MB_ERR_ALIGN
    assert f(A, B, C, D, E, None, None, G + 1, 4, 64, 1e-5, 1, 0.1, 1, 0, 0, None) == MB_ERR_ALIGN
    assert f(A, B, C, D, E, None, A + 8, None, 4, 64, 1e-5, 1, 0.0, 1, 0, 0, None) == MB_ERR_OVERLAP
    assert f(A, B, C, D, E, None, E + 16, None, 4, 64, 1e-5, 1, 0.0, 1, 0, 0, None) == MB_ERR_OVERLAP
    assert f(A, B, C, D, E, None, F, F + 8, 4, 64, 1e-5, 1, 0.0, 1, 0, 0, None) == MB_ERR_OVERLAP
    assert f(A, B, C, D, E, F, None, F + 64, 4, 64, 1e-5, 1, 0.0, 1, 0, 0, None) == MB_ERR_OVERLAP
    assert f(A, B, C, D, E, None, None, None, 4, 64, 1e-5, 7, 0.1, 1, 0, 0, None) == MB_ERR_VALUE
    assert f(None, B, C, D, E, None, F, G, 4, 64, 1e-5, 1, 0.1, 1, 0, 0, None) == MB_ERR_NULL
    assert lib.mb_row_plan(9, 0, 4, 64, 1, (ctypes.c_int32 * 7)()) == MB_ERR_VALUE


def test_pointwise_bcast_argument_checks(lib):
    f = lib.fused_add_relu_scale_bcast
    assert f(A, B, C, D, 0, 64, 1, 1, 0.5, 0, None) == MB_OK
    assert f(A, B, C, D, 4, 0, 1, 1, 0.5, 0, None) == MB_ERR_SHAPE
    assert f(A, B, C, D, 4, 1 << 31, 1, 1, 0.5, 0, None) == MB_ERR_SHAPE
    assert f(A, B, C, D, -1, 64, 1, 1, 0.5, 0, None) == MB_ERR_SHAPE
    assert f(A, B, C, D, 4, 64, 2, 1, 0.5, 0, None) == MB_ERR_VALUE
    assert f(A, B, C, D, 4, 64, 1, 1, float("inf"), 0, None) == MB_ERR_VALUE
    assert f(A, B, C, D, 4, 64, 1, 1, 0.5, 5, None) == MB_ERR_DTYPE
    assert f(A, None, C, D, 4, 64, 1, 1, 0.5, 0, None) == MB_ERR_NULL
    assert f(A + 2, B, C, D, 4, 64, 1, 1, 0.5, 0, None) == MB_ERR_ALIGN
    assert f(A, B, C, A + 64, 4, 64, 1, 1, 0.5, 0, None) == MB_ERR_OVERLAP
    # a per-column b1 occupies cols elements only; a full one rows * cols
    assert f(A, D + 4 * 64, C, D, 4, 64, 0, 1, 0.5, 0, None) == MB_ERR_OVERLAP


def test_scale_mask_softmax_argument_checks(lib):
    f = lib.fused_scale_mask_softmax
    assert f(A, B, 0, 64, 0.125, 1, 4, 0, 0, None) == MB_OK
    assert f(A, B, 4, 64, float("nan"), 1, 4, 0, 0, None) == MB_ERR_VALUE
    assert f(A, B, 4, 64, 0.125, 2, 4, 0, 0, None) == MB_ERR_VALUE
    assert f(A, B, 4, 64, 0.125, 1, 0, 0, 0, None) == MB_ERR_VALUE      # period
    assert f(A, B, 4, 64, 0.125, 1, 4, -1, 0, None) == MB_ERR_VALUE     # offset
    assert f(A, A + 64, 4, 64, 0.125, 1, 4, 0, 0, None) == MB_ERR_OVERLAP
    assert f(A + 2, B, 4, 64, 0.125, 0, 1, 0, 0, None) == MB_ERR_ALIGN
    assert f(A, None, 4, 64, 0.125, 0, 1, 0, 1, None) == MB_ERR_NULL
    assert f(A, B, 4, 0, 0.125, 0, 1, 0, 0, None) == MB_ERR_SHAPE


def test_library_build_depends_on_its_build_script(tmp_path, monkeypatch):
    """A change to the build script (its flags or architecture) makes the
    library out of date, like a change to a source file."""
    import time
    from memory_bound_gb300 import build as b
    lib = tmp_path / "lib.so"
    lib.write_bytes(b"x")
    monkeypatch.setattr(b, "LIB", str(lib))
    future = time.time() + 3600
    os.utime(lib, (future, future))
    assert b._up_to_date()
    later = future + 60
    script = b.__file__
    st = os.stat(script)
    try:
        os.utime(script, (later, later))
        assert not b._up_to_date()
    finally:
        os.utime(script, (st.st_atime, st.st_mtime))


def test_dominant_kernel_fits_four_ctas_an_sm(tmp_path):
    """The two-slot staged bf16 LayerNorm kernel (the 32768 x 8192 bench row's
    kernel) compiles to at most 32 registers a thread, so four 512-thread CTAs
    share an SM; kernels added to its translation unit have pushed ptxas to 38
    (three CTAs) before.  Reads only ptxas's resource report."""
    import subprocess
    src = os.path.join(lib_build.CSRC, "rows_ln_bf16.cu")
    res = subprocess.run([lib_build.NVCC, *lib_build.ARCH, *lib_build.FLAGS, "-Xptxas", "-v",
                          "-c", src, "-o", str(tmp_path / "ln_bf16.o")],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-2000:]
    name = "rows_cta_kernelINS_11LnGeluChainItEELi2ELi8ELb1EE"
    blocks = re.split(r"Compiling entry function '", res.stderr)
    block = [b for b in blocks if b.split("'")[0].find(name) >= 0]
    assert len(block) == 1, "kernel not found in the ptxas report"
    regs = int(re.search(r"Used (\d+) registers", block[0]).group(1))
    assert regs <= 32, f"{regs} registers"
