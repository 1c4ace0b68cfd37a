"""The bench's CPU legs without a GPU: the single-core oracle baseline and the
same oracle spread over spawned processes, on a small sample."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_cpu_baselines_on_a_small_sample():
    sample = bench.cpu_sample(0.01)
    gbs, secs, desc = bench.cpu_baseline(sample)
    assert gbs > 0 and secs > 0 and "pointwise_f32_4Mi" in desc
    pg, ps = bench.cpu_baseline_all_cores(sample, 2)
    assert pg > 0 and ps > 0


def test_host_info():
    h = bench.host_info()
    assert h["cores_available"] >= 1 and h["cpu"]


def test_plan_chain_names_every_row_workload():
    """Every row workload maps to a plan-query chain name the binding
    accepts; the pointwise chains have none."""
    from synth import workloads as W
    names = {"ln", "inductor", "lnact_res", "lnact", "softmax", "lnact_res_dropout",
             "lnact_dropout", "lnact_res_h", "softmax_mask"}
    for w in W.ALL + W.NEXT:
        got = bench.plan_chain(w)
        if w.chain.startswith("add_relu_scale"):
            assert got is None, w.name
        else:
            assert got in names, (w.name, got)
    assert bench.plan_chain(W.LNACT_RELU_DROP_F32) == "lnact_dropout"
    assert bench.plan_chain(W.LNACT_RES_BF16) == "lnact_res_h"
