"""memory_bound_gb300 -- fused memory-bound operator chains for GB300 (sm_103a).

A thin Python binding over the C ABI of ``libmemory_bound.so``
(``include/memory_bound.h``).  The functions here only marshal arguments:
torch tensors in, device pointers, sizes and the current CUDA stream out.
Every step of every chain runs in the library's CUDA kernels; there is no
fallback of any kind, and calling a chain without the built library raises.

    fused_add_relu_scale(x, b1, b2, scale=0.5, out=None)
    fused_residual_layernorm_gelu(x, r, w, b, eps=1e-5, out=None)
    fused_bias_relu_branch_mean_epilogue(x, bias, gamma, beta,
                                         x_scale=1.1, branch_scale=0.1, out=None)
    fused_layernorm_act(x, r, w, b, eps=1e-5, act="gelu_tanh", want_h=False)   # r may be None
    fused_row_softmax(x, out=None)

``graph.ChainGraph`` captures a sequence of these calls into one CUDA graph
for replay.

``raw`` exposes the C entry points themselves (plain integers for pointers
and streams) for callers that manage their own memory.
"""
from ._binding import (  # noqa: F401
    ACTIVATIONS, MB_BF16, MB_F32, MB_MAX_COLS, MBError, ROW_PATHS, device_error,
    fused_add_relu_scale, fused_bias_relu_branch_mean_epilogue, fused_layernorm_act,
    fused_residual_layernorm_gelu, fused_row_softmax, library_path, load_library, raw, row_plan,
    set_launch_overlap, set_pointwise_shape, set_row_path, status_string,
)
from . import graph  # noqa: F401,E402
