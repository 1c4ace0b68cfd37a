"""Helpers for the GPU parity tests: host <-> device transfer of the
generator's arrays and the comparison rules.

Tolerances (the oracle is the reference):
  pointwise chain          bit-exact (0 ulp; the bar is <= 1 ulp)
  fp32 row chains          |gpu - oracle| <= 1e-5 * max(|oracle|, 1)
  bf16 outputs             |gpu - oracle| <= 1e-2 * max(|oracle|, 1e-2)
"""
import numpy as np
import torch

RTOL_F32, FLOOR_F32 = 1e-5, 1.0
RTOL_BF16, FLOOR_BF16 = 1e-2, 1e-2


def to_dev(a, bf16=False, device="cuda"):
    if bf16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host(t):
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_to_f64(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_bitexact(got, want, what=""):
    g = np.ascontiguousarray(got)
    w = np.ascontiguousarray(want)
    assert g.shape == w.shape, (g.shape, w.shape)
    gb = g.view(np.uint32 if g.dtype == np.float32 else np.uint16)
    wb = w.view(np.uint32 if w.dtype == np.float32 else np.uint16)
    bad = np.flatnonzero(gb.reshape(-1) != wb.reshape(-1))
    assert bad.size == 0, (f"{what}: {bad.size} elements differ, first at {bad[0]}: "
                           f"gpu {g.reshape(-1)[bad[0]]!r} oracle {w.reshape(-1)[bad[0]]!r}")


def max_ulp_f32(got, want):
    """Largest distance in units in the last place (at the oracle value)."""
    g = np.asarray(got, np.float32).view(np.int32).astype(np.int64)
    w = np.asarray(want, np.float32).view(np.int32).astype(np.int64)
    g = np.where(g < 0, -(g & 0x7FFFFFFF), g)
    w = np.where(w < 0, -(w & 0x7FFFFFFF), w)
    return int(np.abs(g - w).max()) if g.size else 0


def assert_close(got, want, bf16=False, what=""):
    """The tolerance rule above; returns (max abs err, max err / limit)."""
    if bf16:
        g, w = bf16_to_f64(got), bf16_to_f64(want)
        rtol, floor = RTOL_BF16, FLOOR_BF16
    else:
        g, w = np.asarray(got, np.float64), np.asarray(want, np.float64)
        rtol, floor = RTOL_F32, FLOOR_F32
    assert g.shape == w.shape, (g.shape, w.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - w)
    lim = rtol * np.maximum(np.abs(w), floor)
    ratio = err / lim
    worst = int(np.argmax(ratio)) if ratio.size else 0
    assert not np.any(err > lim), (
        f"{what}: {int(np.sum(err > lim))} elements out of tolerance; worst flat index "
        f"{worst}: gpu {g.reshape(-1)[worst]!r} oracle {w.reshape(-1)[worst]!r}")
    return (float(err.max()) if err.size else 0.0, float(ratio.max()) if ratio.size else 0.0)


def guarded_empty(shape, dtype, guard=64, device="cuda"):
    """An output tensor with `guard` canary elements on both sides (in one
    allocation); returns (buffer, view).  check_guard() verifies the canaries."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * guard, dtype=dtype, device=device)
    if dtype == torch.bfloat16:
        buf.view(torch.int16).fill_(0x7FA5)
    else:
        buf.view(torch.int32).fill_(0x7FA5A5A5)
    return buf, buf[guard:guard + n].view(shape)


def check_guard(buf, guard=64):
    if buf.dtype == torch.bfloat16:
        v = buf.view(torch.int16)
        sentinel = 0x7FA5
    else:
        v = buf.view(torch.int32)
        sentinel = 0x7FA5A5A5
    head, tail = v[:guard], v[-guard:]
    assert bool((head == sentinel).all()) and bool((tail == sentinel).all()), "write outside the output"


# Worst-case figures of the whole-tensor checks, printed at the end of the
# run by the terminal-summary hook in conftest.py.
PARITY_REPORT = []


def report(what, **fields):
    PARITY_REPORT.append((what, fields))


def max_rel_above(got, want, bf16=False, floor=1e-3):
    """Largest pure relative error over the elements whose oracle value is at
    least ``floor`` in magnitude (the fp32 bar carries an absolute floor below
    1; this is the figure without it)."""
    g = bf16_to_f64(got) if bf16 else np.asarray(got, np.float64)
    w = bf16_to_f64(want) if bf16 else np.asarray(want, np.float64)
    big = np.abs(w) >= floor
    return float((np.abs(g - w)[big] / np.abs(w[big])).max()) if big.any() else 0.0
