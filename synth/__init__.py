"""Seeded, counter-based synthetic inputs.

This module holds no arithmetic of the fused chains: it only draws numbers.
Both the CUDA path's tests and benchmark and the CPU oracle's tests read their
inputs from here, so that the two sides see identical host arrays.

Definition (written from the published SplitMix64 generator and the
Box-Muller transform):

* ``mix64(z)`` is SplitMix64's output function::

      z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
      z = (z ^ (z >> 27)) * 0x94D049BB133111EB
      return z ^ (z >> 31)                      (all arithmetic mod 2**64)

* a stream is named by ``(seed, tensor_id)``; its key is
  ``K = mix64(seed * G + tensor_id + 1)`` with ``G = 0x9E3779B97F4A7C15``
  (SplitMix64's increment), and its ``i``-th 64-bit draw is
  ``mix64(K + (i + 1) * G)`` -- SplitMix64 run from state ``K``, addressed by
  counter so any element can be computed on its own;
* a uniform double in [0, 1) is ``(d >> 11) * 2**-53``;
* element ``k`` of an N(mu, sigma) tensor uses draws ``2k`` and ``2k+1``:
  ``u1 = ((d_2k >> 11) + 1) * 2**-53`` (in (0, 1]),
  ``u2 = (d_2k+1 >> 11) * 2**-53``, ``z = sqrt(-2 ln u1) cos(2 pi u2)``,
  value ``mu + sigma z`` (sigma is the standard deviation);
* element ``k`` of a U(a, b) tensor is ``a + (b - a) u`` with ``u`` from draw
  ``k``;
* the double is rounded to fp32 (nearest, ties to even); bf16 tensors are then
  rounded from that fp32 value to bf16 (nearest, ties to even) and returned as
  raw uint16 bit patterns.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1

# Elements generated per chunk; chunks are independent (counter-based), so
# they run on a thread pool (numpy releases the GIL in its ufuncs).
_CHUNK = 1 << 21


def mix64_int(z):
    """SplitMix64 output function on a Python int (reference for tests)."""
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def stream_key(seed, tensor_id):
    return mix64_int((seed * GOLDEN + tensor_id + 1) & _MASK)


def _mix64_np(z):
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def draws(seed, tensor_id, start, count):
    """64-bit draws ``start .. start+count-1`` of stream (seed, tensor_id)."""
    key = np.uint64(stream_key(seed, tensor_id))
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix64_np(key + i * np.uint64(GOLDEN))


def _u53(d):
    return (d >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _normal_chunk(seed, tid, k0, count, mean, std):
    d = draws(seed, tid, 2 * k0, 2 * count)
    u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = _u53(d[1::2])
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return (mean + std * z).astype(np.float32)


def _uniform_chunk(seed, tid, k0, count, lo, hi):
    u = _u53(draws(seed, tid, k0, count))
    return (lo + (hi - lo) * u).astype(np.float32)


def _fill(fn, n, seed, tid, a, b):
    out = np.empty(n, np.float32)
    starts = range(0, n, _CHUNK)

    def job(k0):
        c = min(_CHUNK, n - k0)
        out[k0:k0 + c] = fn(seed, tid, k0, c, a, b)

    if n <= _CHUNK:
        if n:
            job(0)
    else:
        workers = min(16, os.cpu_count() or 1)
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(job, starts))
    return out


def f32_to_bf16_bits(a):
    """Round fp32 values to bf16 (nearest, ties to even); raw uint16 bits.
    Inputs here are always finite."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h):
    """Exact widening of raw bf16 bits to fp32."""
    return (np.asarray(h, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal(seed, tensor_id, shape, mean=0.0, std=1.0, dtype="f32"):
    n = int(np.prod(shape)) if len(shape) else 1
    v = _fill(_normal_chunk, n, seed, tensor_id, mean, std).reshape(shape)
    return f32_to_bf16_bits(v) if dtype == "bf16" else v


def uniform(seed, tensor_id, shape, lo=0.0, hi=1.0, dtype="f32"):
    n = int(np.prod(shape)) if len(shape) else 1
    v = _fill(_uniform_chunk, n, seed, tensor_id, lo, hi).reshape(shape)
    return f32_to_bf16_bits(v) if dtype == "bf16" else v
