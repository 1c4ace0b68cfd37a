"""The seeded input generator: its published building blocks, its counter
addressing, golden first values (drift check) and the workload table."""
import json
import math
import os

import numpy as np
import pytest

import synth
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_splitmix64_published_vector():
    # SplitMix64 from state 0: the first three outputs of the reference
    # generator (state += 0x9E3779B97F4A7C15, then the output mix).
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = [synth.mix64_int(synth.GOLDEN * i) for i in (1, 2, 3)]
    assert got == want


def test_counter_addressing_matches_scalar_definition():
    key = synth.stream_key(5, 3)
    want = [synth.mix64_int(key + (i + 1) * synth.GOLDEN) for i in range(40)]
    got = synth.draws(5, 3, 0, 40).tolist()
    assert got == want
    assert synth.draws(5, 3, 17, 10).tolist() == want[17:27]


def _scalar_normal(seed, tid, k, mean, std):
    key = synth.stream_key(seed, tid)
    d1 = synth.mix64_int(key + (2 * k + 1) * synth.GOLDEN)
    d2 = synth.mix64_int(key + (2 * k + 2) * synth.GOLDEN)
    u1 = ((d1 >> 11) + 1) * 2.0 ** -53
    u2 = (d2 >> 11) * 2.0 ** -53
    z = math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)
    return np.float32(mean + std * z)


def test_vectorised_normal_matches_scalar_definition():
    n = (1 << 21) + 77      # spans two chunks of the thread pool
    v = synth.normal(9, 1, (n,), 0.25, 2.0)
    for k in (0, 1, 2, 1000, (1 << 21) - 1, 1 << 21, n - 1):
        assert v[k] == _scalar_normal(9, 1, k, 0.25, 2.0), k


def test_uniform_matches_scalar_definition():
    v = synth.uniform(2, 2, (100,), 0.5, 1.5)
    key = synth.stream_key(2, 2)
    for k in (0, 50, 99):
        d = synth.mix64_int(key + (k + 1) * synth.GOLDEN)
        assert v[k] == np.float32(0.5 + 1.0 * ((d >> 11) * 2.0 ** -53))


def test_distribution_moments():
    z = synth.normal(1, 0, (1 << 20,))
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1.0) < 5e-3
    u = synth.uniform(1, 1, (1 << 20,), 0.5, 1.5)
    assert u.min() >= 0.5 and u.max() < 1.5 and abs(u.mean() - 1.0) < 2e-3


def test_bf16_rounding_of_inputs():
    f = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 3.0e-39], np.float32)
    got = synth.f32_to_bf16_bits(f)
    assert got.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0021]
    assert np.array_equal(synth.bf16_bits_to_f32(got)[:4],
                          np.array([1.0, 1.0, 1.0 + 2 ** -6, -2.5], np.float32))


def test_golden_first_values():
    """Drift check: the first values of every workload tensor, written by
    tests/golden/make_synth_golden.py."""
    with open(os.path.join(GOLDEN, "synth_first_values.json")) as f:
        gold = json.load(f)
    for w in W.ALL:
        for t in w.tensors:
            rows = 1 if (w.chain != "add_relu_scale" and not t.per_column) else None
            a = w.generate(t, rows=rows).reshape(-1)[:6]
            got = [int(v) for v in (a if a.dtype == np.uint16 else a.view(np.uint32))]
            assert got == gold[w.name][t.name], (w.name, t.name)


@pytest.mark.parametrize("w", W.ALL + W.NEXT, ids=lambda w: w.name)
def test_workload_ideal_bytes(w):
    # read-once / write-once bytes of one call, from the workload shapes
    want = {
        "pointwise_f32_4096": 4 * 4096 * 4,
        "pointwise_f32_4Mi": 4 * 4 * 1024 * 1024 * 4,
        "inductor_f32_1024x1024": 2 * 1024 * 1024 * 4 + 3 * 1024 * 4,
        "ln_gelu_f32_8192x4096": 3 * 8192 * 4096 * 4 + 2 * 4096 * 4,
        "ln_gelu_bf16_32768x8192": 3 * 32768 * 8192 * 2 + 2 * 8192 * 2,
        "softmax_f32_131072x4096": 2 * 131072 * 4096 * 4,
        "lnact_res_h_bf16_32768x8192": 4 * 32768 * 8192 * 2 + 2 * 8192 * 2,
        "lnact_relu_f32_8192x4096": 2 * 8192 * 4096 * 4 + 2 * 4096 * 4,
        "inductor_bf16_1024x1024": 2 * 1024 * 1024 * 2 + 3 * 1024 * 2,
        "lnact_relu_dropout_f32_8192x4096": 2 * 8192 * 4096 * 4 + 2 * 4096 * 4,
        "pointwise_bcast_f32_4096x1024": 2 * 4096 * 1024 * 4 + 2 * 1024 * 4,
        # 32 heads x (1 + 2 + ... + 4096) unmasked keys read, every output written
        "softmax_scale_causal_f32_131072x4096": (32 * 4096 * 4097 // 2 + 131072 * 4096) * 4,
        "ln_gelu_f32_8192x4099": 3 * 8192 * 4099 * 4 + 2 * 4099 * 4,
    }[w.name]
    assert w.ideal_bytes() == want
