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


def test_spread_and_kernel_summary():
    """The per-kernel distribution over replays and the compact summary that
    ends the JSON line (every measured workload, the hot-L2 rates)."""
    mean, med, p10, p90 = bench.spread([1.0, 2.0, 3.0, 4.0, 10.0])
    assert mean == 4.0 and med == 3.0 and p10 <= med <= p90
    e = {"us_per_call": 3.0, "us_per_call_p10_p90": [2.0, 5.0], "gbs": 100.0,
         "frac_of_measured_hbm": 0.5, "frac_of_size_matched_copy": 0.9}
    s = bench.kernel_summary({"a": e}, {"b": e}, {"c": {"us_per_call": 1.5}})
    assert s["a"] == [3.0, 2.0, 5.0, 100.0, 0.5, 0.9] and s["b"] == s["a"]
    assert len(s["fields"]) == len(s["a"])
    assert s["hot_l2_us_per_call"] == {"c": 1.5}
