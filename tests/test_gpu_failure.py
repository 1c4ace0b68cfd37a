"""Failure detection without a GPU fault: a kernel's bounded barrier wait is
made to run out (a barrier nothing completes, with a 2 ms limit); the kernel
must end, the device flag must reach the host through mb_device_error, and
the context must stay usable for ordinary calls afterwards."""
import ctypes
import time

import numpy as np
import pytest
import torch

import memory_bound_gb300 as mb
import oracle
import synth

from gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    from memory_bound_gb300 import build as lib_build
    lib_build.build()
    torch.cuda.set_device(0)
    lib = mb.load_library()
    assert mb.device_error() == 0                     # clean start (and clears)
    t0 = time.perf_counter()
    st = lib.mb_selftest_wait_timeout(2000, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    flags = ctypes.c_uint32(0)
    assert lib.mb_device_error(ctypes.byref(flags)) == 8      # MB_ERR_DEVICE
    assert flags.value == 1                                    # the wait-timeout bit
    assert time.perf_counter() - t0 < 30
    assert mb.device_error() == 0                              # read clears it
    # the context still works
    x, b1, b2 = (synth.normal(1201, k, (4096,)) for k in range(3))
    y = mb.fused_add_relu_scale(to_dev(x), to_dev(b1), to_dev(b2), 0.5)
    assert np.array_equal(to_host(y).view(np.uint32),
                          oracle.add_relu_scale(x, b1, b2, 0.5).view(np.uint32))
    assert lib.mb_selftest_wait_timeout(0, None) == 6          # MB_ERR_VALUE


def test_cluster_exchange_timeout_is_reported_and_context_survives():
    """The cluster exchange's bounded wait: one push never sent, the wait runs
    out after 2 ms, the flag is reported, and a long-row call (the cluster
    path) still works afterwards."""
    from memory_bound_gb300 import build as lib_build
    lib_build.build()
    torch.cuda.set_device(0)
    lib = mb.load_library()
    assert mb.device_error() == 0
    t0 = time.perf_counter()
    assert lib.mb_selftest_exchange_timeout(2000, torch.cuda.current_stream().cuda_stream) == 0
    flags = ctypes.c_uint32(0)
    assert lib.mb_device_error(ctypes.byref(flags)) == 8
    assert flags.value == 1
    assert time.perf_counter() - t0 < 30
    assert mb.device_error() == 0
    x = synth.normal(1301, 0, (3, 65536))
    y = mb.fused_row_softmax(to_dev(x))
    want = oracle.row_softmax(x).astype(np.float64)
    assert np.all(np.abs(to_host(y).astype(np.float64) - want) <= 1e-5 * want + 2.0 ** -126)
    assert lib.mb_selftest_exchange_timeout(2000000, None) == 6
