"""Capture a sequence of fused-chain calls into one CUDA graph and replay it.

The chains neither allocate nor synchronise, so a step of several calls on
fixed buffers can be captured once and replayed: one launch of the graph
instead of one host launch per kernel, which is what makes small,
launch-bound chains (a few microseconds of work each) run back to back on
the GPU ("Operator fusion and kernel optimisation: from CUDA Graph to
FlashAttention" §4.3: capture a kernel sequence once, then launch the graph).
New inputs are copied into the captured buffers between replays.

    step = ChainGraph(lambda: (mb.fused_add_relu_scale(x, b1, b2, out=y),
                               mb.fused_residual_layernorm_gelu(y2, r, w, b, out=o)))
    x.copy_(next_x); step.replay()
"""
import torch


class ChainGraph:
    """`fn` (a callable issuing library calls on fixed tensors) run `warmup`
    times on the current stream, so that launch plans and kernel attributes
    are settled outside the capture, then captured into a CUDA graph on a
    side stream.  ``replay()`` launches the graph on the current stream."""

    def __init__(self, fn, warmup=1):
        for _ in range(max(1, int(warmup))):
            fn()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="thread_local"):
            fn()
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()
