"""Packed (varlen) width-4 depthwise causal convolution + SiLU for GB300.

The compute runs in ``libvcd.so`` (hand-written CUDA for sm_103a behind a C ABI,
declared in ``include/vcd.h``). This package marshals torch tensors into that
ABI; it has no CPU fallback. Importing it does not load the library; the first
call does, and raises if the library has not been built.
"""
from .binding import (  # noqa: F401
    VCD_OK, VCD_ERR_INVALID_ARG, VCD_ERR_WORKSPACE_TOO_SMALL, VCD_ERR_MISALIGNED, VCD_ERR_CUDA,
    VcdError, conv1d_bwd, conv1d_bwd_call_workspace_size, conv1d_bwd_exact,
    conv1d_bwd_exact_workspace_size, conv1d_bwd_noalloc,
    conv1d_bwd_route_workspace_size,
    conv1d_bwd_workspace_size, conv1d_fwd, conv1d_fwd_exact, conv1d_fwd_workspace_size,
    conv1d_status_string, conv1d_wait_fault, library_path, load_library,
)
from .functional import (  # noqa: F401,E402
    CakeCausalConv1dFunction, cake_causal_conv1d_train_backward,
    cake_causal_conv1d_train_backward_workspace, cake_causal_conv1d_train_backward_workspace_bytes,
    cake_causal_conv1d_train_forward, cake_causal_conv1d_train_forward_workspace,
    cake_causal_conv1d_train_forward_workspace_bytes, causal_conv1d,
)
