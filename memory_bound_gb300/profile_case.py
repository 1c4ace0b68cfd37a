"""Run one fused chain on a chosen shape a few times (for ncu captures).

    python -m memory_bound_gb300.profile_case ln_bf16 8192 8192 --iters 3

Chains: pointwise_f32, pointwise_bf16, pointwise_bcast_f32, inductor_f32,
ln_f32, ln_bf16, lnrelu_f32 (LayerNorm -> ReLU, no residual), lnrelu_drop_f32
and lnrelu_drop_bf16 (with dropout p = 0.1), softmax_f32, softmax_bf16.
Inputs are seeded synthetic tensors from synth; nothing is checked here (the
tests do that).  Keep ncu captures small: a few hundred MB on the device.
"""
import argparse
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import memory_bound_gb300 as mb  # noqa: E402
import synth  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("chain")
    ap.add_argument("rows", type=int)
    ap.add_argument("cols", type=int)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--path", default="auto")
    ap.add_argument("--ctas", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    a = ap.parse_args(argv)
    from memory_bound_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    bf16 = a.chain.endswith("bf16")
    dt = "bf16" if bf16 else "f32"

    def t(tid, shape, lo=0.0, hi=1.0, uniform=False):
        fn = synth.uniform if uniform else synth.normal
        h = fn(99, tid, shape, lo, hi, dtype=dt)
        if bf16:
            return torch.from_numpy(h.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(h).to(dev)

    mb.set_row_path(a.path, a.ctas, a.stages)
    if a.chain == "pointwise_bcast_f32":
        x, b1, b2 = t(0, (a.rows, a.cols)), t(1, (a.cols,)), t(2, (a.cols,))
        out = torch.empty_like(x)
        run = lambda: mb.fused_add_relu_scale(x, b1, b2, 0.5, out=out)
    elif a.chain.startswith("lnrelu"):
        x = t(0, (a.rows, a.cols))
        w, b = t(2, (a.cols,), 0.5, 1.5, True), t(3, (a.cols,), 0, 0.1)
        out = torch.empty_like(x)
        p = 0.1 if "drop" in a.chain else 0.0
        run = lambda: mb.fused_layernorm_act(x, None, w, b, 1e-5, act="relu", out=out, p=p,
                                             seed=2024)
    elif a.chain.startswith("pointwise"):
        n = a.rows * a.cols
        x, b1, b2 = t(0, (n,)), t(1, (n,)), t(2, (n,))
        out = torch.empty_like(x)
        run = lambda: mb.fused_add_relu_scale(x, b1, b2, 0.5, out=out)
    elif a.chain == "inductor_f32":
        x = t(0, (a.rows, a.cols))
        bias, gamma, beta = t(1, (a.cols,), 0, 0.1), t(2, (a.cols,), 0.5, 1.5, True), t(3, (a.cols,), 0, 0.1)
        out = torch.empty_like(x)
        run = lambda: mb.fused_bias_relu_branch_mean_epilogue(x, bias, gamma, beta, 1.1, 0.1, out=out)
    elif a.chain.startswith("softmax"):
        x = t(0, (a.rows, a.cols))
        out = torch.empty_like(x)
        run = lambda: mb.fused_row_softmax(x, out=out)
    else:
        x, r = t(0, (a.rows, a.cols)), t(1, (a.rows, a.cols))
        w, b = t(2, (a.cols,), 0.5, 1.5, True), t(3, (a.cols,), 0, 0.1)
        out = torch.empty_like(x)
        run = lambda: mb.fused_residual_layernorm_gelu(x, r, w, b, 1e-5, out=out)
    for _ in range(a.iters):
        run()
    torch.cuda.synchronize()
    kind = ("lnact_dropout" if a.chain.startswith("lnrelu_drop") else
            "lnact" if a.chain.startswith("lnrelu") else
            "ln" if a.chain.startswith("ln") else
            "softmax" if a.chain.startswith("softmax") else "inductor")
    print("plan:", mb.row_plan(kind, dt, a.rows, a.cols)
          if not a.chain.startswith("pointwise") else "pointwise")


if __name__ == "__main__":
    main()
