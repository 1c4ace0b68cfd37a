"""The synthetic workloads, by name, with their seeds and tensor ids.

Shapes and distributions are the pages' example workloads:

* pointwise chain ``relu(x + b1) * 0.5 + b2`` on full-size fp32 ``randn``
  tensors of 4 * 1024 * 1024 elements ([P1] §3.1), and a 4096-element small
  case;
* the TorchInductor example on ``x`` f32[1024, 1024] with f32[1024] ``bias``,
  ``gamma``, ``beta`` ([P4] "model");
* residual + LayerNorm + GeLU-tanh rows ([P2] §2.3) at hidden 4096 fp32 and
  hidden 8192 bf16;
* for the further chains (NEXT): row softmax on [P1] §4.1's attention-score
  matrix, the LayerNorm family with a residual-stream output or a ReLU, the
  TorchInductor chain in bf16, [P2] §2.1's LayerNorm -> ReLU -> Dropout, the
  pointwise chain with per-column b1 / b2, and [P1] §4.1-4.2's score matrix
  scaled and causally masked.

N(mu, s) takes ``s`` as the standard deviation.  Tensor ids are assigned in
the order each workload lists its tensors.
"""
from dataclasses import dataclass, field

import numpy as np

from . import normal, uniform


@dataclass(frozen=True)
class Tensor:
    name: str
    tid: int
    dist: str          # "normal" or "uniform"
    a: float           # mean (normal) or low (uniform)
    b: float           # std (normal) or high (uniform)
    per_column: bool   # a length-cols vector broadcast over rows


@dataclass(frozen=True)
class Workload:
    name: str
    chain: str         # "add_relu_scale" | "add_relu_scale_bcast" | "inductor" |
    #                    "ln_gelu" | "lnact" | "softmax" | "softmax_mask"
    dtype: str         # "f32" | "bf16"
    rows: int          # 1 for the pointwise chain
    cols: int          # n for the pointwise chain
    seed: int
    tensors: tuple
    params: dict = field(default_factory=dict)

    @property
    def elem_bytes(self):
        return 2 if self.dtype == "bf16" else 4

    def shape(self, t):
        if t.per_column:
            return (self.cols,)
        if self.chain == "add_relu_scale":
            return (self.cols,)
        return (self.rows, self.cols)

    def ideal_bytes(self, rows=None):
        """Read-once / write-once bytes of one call (optionally for a prefix
        of ``rows`` rows).  A causally masked softmax reads only the unmasked
        keys of each row and writes every output."""
        rows = self.rows if rows is None else rows
        eb = self.elem_bytes
        if self.params.get("causal"):
            per, off = self.params["period"], self.params["offset"]
            i = np.arange(rows, dtype=np.int64)
            read = int(np.minimum(self.cols, i % per + off + 1).sum())
            return (read + rows * self.cols) * eb
        full = sum(1 for t in self.tensors if not t.per_column)
        percol = sum(1 for t in self.tensors if t.per_column)
        outs = 2 if self.params.get("write_h") else 1
        return rows * self.cols * eb * (full + outs) + percol * self.cols * eb

    def generate(self, tensor, rows=None):
        """Host array for one tensor (uint16 bit patterns for bf16).
        ``rows`` limits row-shaped tensors to their first rows."""
        shape = self.shape(tensor)
        if rows is not None and not tensor.per_column and len(shape) == 2:
            shape = (rows, shape[1])
        fn = normal if tensor.dist == "normal" else uniform
        return fn(self.seed, tensor.tid, shape, tensor.a, tensor.b, self.dtype)

    def generate_all(self, rows=None):
        return {t.name: self.generate(t, rows) for t in self.tensors}


def _pointwise(name, n, seed):
    return Workload(name, "add_relu_scale", "f32", 1, n, seed, (
        Tensor("x", 0, "normal", 0.0, 1.0, False),
        Tensor("b1", 1, "normal", 0.0, 1.0, False),
        Tensor("b2", 2, "normal", 0.0, 1.0, False),
    ), {"scale": 0.5})


POINTWISE_TINY = _pointwise("pointwise_f32_4096", 4096, 0)
POINTWISE_4M = _pointwise("pointwise_f32_4Mi", 4 * 1024 * 1024, 1)

INDUCTOR_1024 = Workload("inductor_f32_1024x1024", "inductor", "f32", 1024, 1024, 2, (
    Tensor("x", 0, "normal", 0.0, 1.0, False),
    Tensor("bias", 1, "normal", 0.0, 0.1, True),
    Tensor("gamma", 2, "uniform", 0.5, 1.5, True),
    Tensor("beta", 3, "normal", 0.0, 0.1, True),
), {"x_scale": 1.1, "branch_scale": 0.1})


def _ln(name, dtype, rows, hidden, seed):
    return Workload(name, "ln_gelu", dtype, rows, hidden, seed, (
        Tensor("x", 0, "normal", 0.0, 1.0, False),
        Tensor("r", 1, "normal", 0.0, 1.0, False),
        Tensor("w", 2, "uniform", 0.5, 1.5, True),
        Tensor("b", 3, "normal", 0.0, 0.1, True),
    ), {"eps": 1e-5})


LN_F32 = _ln("ln_gelu_f32_8192x4096", "f32", 8192, 4096, 3)
LN_BF16 = _ln("ln_gelu_bf16_32768x8192", "bf16", 32768, 8192, 4)

# Rows marked "next" in the scope table: the same shapes, other chains.
# Row softmax on the attention-score matrix of "PyTorch operator fusion in
# practice" §4.1 (batch 1, 32 heads, seq_len 4096: [32*4096, 4096] fp32).
SOFTMAX_F32 = Workload("softmax_f32_131072x4096", "softmax", "f32", 32 * 4096, 4096, 5, (
    Tensor("x", 0, "normal", 0.0, 1.0, False),
), {})
# Residual + LayerNorm + GeLU that also writes the residual stream h = x + r.
LNACT_RES_BF16 = Workload("lnact_res_h_bf16_32768x8192", "lnact", "bf16", 32768, 8192, 6, (
    Tensor("x", 0, "normal", 0.0, 1.0, False),
    Tensor("r", 1, "normal", 0.0, 1.0, False),
    Tensor("w", 2, "uniform", 0.5, 1.5, True),
    Tensor("b", 3, "normal", 0.0, 0.1, True),
), {"eps": 1e-5, "act": "gelu_tanh", "residual": True, "write_h": True})
# Plain LayerNorm -> ReLU (no residual), fp32.
LNACT_RELU_F32 = Workload("lnact_relu_f32_8192x4096", "lnact", "f32", 8192, 4096, 7, (
    Tensor("x", 0, "normal", 0.0, 1.0, False),
    Tensor("w", 2, "uniform", 0.5, 1.5, True),
    Tensor("b", 3, "normal", 0.0, 0.1, True),
), {"eps": 1e-5, "act": "relu", "residual": False, "write_h": False})
INDUCTOR_BF16 = Workload("inductor_bf16_1024x1024", "inductor", "bf16", 1024, 1024, 8,
                         INDUCTOR_1024.tensors, {"x_scale": 1.1, "branch_scale": 0.1})
# "Operator fusion and kernel optimisation" §2.1: LayerNorm -> ReLU ->
# Dropout(p = 0.1) in one kernel, fp32, on the same rows as the plain chain.
LNACT_RELU_DROP_F32 = Workload("lnact_relu_dropout_f32_8192x4096", "lnact", "f32", 8192, 4096, 9,
                               LNACT_RELU_F32.tensors,
                               {"eps": 1e-5, "act": "relu", "residual": False, "write_h": False,
                                "p": 0.1, "seed": 2024, "offset": 0})
# The pointwise chain with bias-like operands: x [4096, 1024] (4 Mi fp32
# elements, as the plain chain) and b1, b2 per column.
POINTWISE_BCAST_F32 = Workload("pointwise_bcast_f32_4096x1024", "add_relu_scale_bcast", "f32",
                               4096, 1024, 10, (
                                   Tensor("x", 0, "normal", 0.0, 1.0, False),
                                   Tensor("b1", 1, "normal", 0.0, 1.0, True),
                                   Tensor("b2", 2, "normal", 0.0, 1.0, True),
                               ), {"scale": 0.5})
# The same score matrix as an attention layer's softmax sees it (§4.1-4.2 of
# the same page): scaled by 1/sqrt(64) and causally masked, 4096 queries per
# head, keys aligned to the queries (offset 0).
SOFTMAX_CAUSAL_F32 = Workload("softmax_scale_causal_f32_131072x4096", "softmax_mask", "f32",
                              32 * 4096, 4096, 11, SOFTMAX_F32.tensors,
                              {"scale": 0.125, "causal": True, "period": 4096, "offset": 0})
# Residual + LayerNorm + GeLU on rows whose length is not a whole number of
# 16-byte vectors (4099 fp32 values, 16396 bytes): consecutive rows start 0,
# 12, 8 and 4 bytes past a 16-byte boundary, so each row is read as a short
# head, whole 16-byte vectors and a short tail.
LN_F32_RAGGED = _ln("ln_gelu_f32_8192x4099", "f32", 8192, 4099, 12)
NEXT = (SOFTMAX_F32, LNACT_RES_BF16, LNACT_RELU_F32, INDUCTOR_BF16, LNACT_RELU_DROP_F32,
        POINTWISE_BCAST_F32, SOFTMAX_CAUSAL_F32, LN_F32_RAGGED)

ALL = (POINTWISE_TINY, POINTWISE_4M, INDUCTOR_1024, LN_F32, LN_BF16)
BY_NAME = {w.name: w for w in ALL + NEXT}


def sample_rows(rows, count, seed=12345):
    """``count`` distinct row indices spread over ``rows``: the first, the
    last, and a seeded random choice in between (sorted)."""
    count = min(count, rows)
    picks = {0, rows - 1}
    rng = np.random.default_rng(seed)
    while len(picks) < count:
        picks.add(int(rng.integers(0, rows)))
    return np.array(sorted(picks), dtype=np.int64)
