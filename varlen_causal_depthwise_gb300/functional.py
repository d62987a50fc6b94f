"""torch-level API with the FlashInfer pages' names and contracts.

Pages: "flashinfer.cake_causal_conv1d_train.cake_causal_conv1d_train_forward"
(Parameters, Returns), "...cake_causal_conv1d_train_backward" (description,
Parameters, Returns) and "...CakeCausalConv1dFunction" (class description).
The function names and keyword arguments are kept as the pages give them so code
written against those pages runs unchanged; every computation happens in the
CUDA library (``binding``), this module only checks contracts, picks output
dtypes and manages the optional workspaces.
"""
import torch

from . import binding

_FWD_WS = {}   # (device index, stream handle) -> uint8 workspace of the forward (size 0)
_BWD_WS = {}   # (device index, stream handle) -> uint8 workspace of the backward


def _check_x(x, name="x"):
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be a BF16 tensor")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not (x.dim() == 2 or (x.dim() == 3 and x.shape[0] == 1)):
        raise ValueError(f"{name} must be [S, C] or [1, S, C], got {tuple(x.shape)}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if x.shape[-1] % 8 != 0:
        raise ValueError(f"C must be a multiple of 8, got {x.shape[-1]}")


def _check_params(x, weight, cu_seqlens, bias):
    C = x.shape[-1]
    if weight.dim() != 2 or weight.shape[0] != C or weight.shape[1] != 4:
        raise ValueError(f"weight must be [C, 4] = [{C}, 4] (width 4 only), got {tuple(weight.shape)}")
    if weight.dtype not in (torch.float32, torch.bfloat16) or not weight.is_contiguous():
        raise ValueError("weight must be a contiguous FP32 or BF16 tensor")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int32 vector [num_docs + 1]")
    if cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens needs at least one element")
    if bias is not None:
        if bias.shape != (C,) or bias.dtype not in (torch.float32, torch.bfloat16) \
                or not bias.is_contiguous():
            raise ValueError(f"bias must be a contiguous FP32 or BF16 [{C}] tensor")
    for t in (weight, cu_seqlens, bias):
        if t is not None and t.device != x.device:
            raise ValueError("all tensors must be on x's device")


def _stream_key(device):
    return (device.index, torch.cuda.current_stream(device).cuda_stream)


def cake_causal_conv1d_train_forward_workspace_bytes():
    """Bytes of the forward workspace: 0 (the forward keeps no counters)."""
    return binding.conv1d_fwd_workspace_size(0, 8)


def cake_causal_conv1d_train_forward_workspace(device=None):
    """A forward workspace: an empty uint8 tensor, accepted and ignored."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    return torch.empty(cake_causal_conv1d_train_forward_workspace_bytes(), dtype=torch.uint8,
                       device=dev)


def cake_causal_conv1d_train_backward_workspace_bytes(S, C):
    """Bytes of backward workspace for S tokens and C channels; the same for
    every route and device."""
    return binding.conv1d_bwd_workspace_size(S, C)


def cake_causal_conv1d_train_backward_workspace(S, C, device=None):
    dev = torch.device("cuda") if device is None else torch.device(device)
    return torch.empty(cake_causal_conv1d_train_backward_workspace_bytes(S, C), dtype=torch.uint8,
                       device=dev)


def _bwd_workspace(x, S, C, workspace, policy):
    need = binding.conv1d_bwd_route_workspace_size(S, C, policy)
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"workspace holds {workspace.numel() * workspace.element_size()} "
                             f"bytes, {need} needed")
        return workspace
    if torch.cuda.is_current_stream_capturing():
        # inside a graph capture: a buffer of the call's own (the graph's pool keeps it)
        return torch.empty(need, dtype=torch.uint8, device=x.device)
    key = _stream_key(x.device)
    ws = _BWD_WS.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
        _BWD_WS[key] = ws
    return ws


def cake_causal_conv1d_train_forward(x, weight, cu_seqlens, *, bias=None, out=None,
                                     workspace=None):
    """y = bf16(silu(sum_k weight[c, k] x[t - 3 + k, c] + bias[c])), zero history
    before each document's first token (forward page, Returns)."""
    _check_x(x)
    _check_params(x, weight, cu_seqlens, bias)
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous BF16 tensor of x's shape")
    if x.numel() == 0:
        return out
    return binding.conv1d_fwd(x, weight, cu_seqlens, bias=bias, y=out, workspace=workspace)


def cake_causal_conv1d_train_backward(x, weight, cu_seqlens, dy, *, bias=None,
                                      silu_grad_preactivation="bf16", workspace=None, dx=None,
                                      dweight=None, dbias=None):
    """(dx, dweight) or (dx, dweight, dbias) with a bias (backward page, Returns).
    Output dtypes default to the parameters'; dbias needs bias."""
    _check_x(x)
    _check_x(dy, "dy")
    if dy.shape != x.shape:
        raise ValueError("dy must have x's shape")
    _check_params(x, weight, cu_seqlens, bias)
    if silu_grad_preactivation not in ("bf16", "fp32"):
        raise ValueError("silu_grad_preactivation must be 'bf16' or 'fp32'")
    if dbias is not None and bias is None:
        raise ValueError("dbias needs bias")
    S, C = int(x.shape[-2]), int(x.shape[-1])
    if dx is None:
        dx = torch.empty_like(x)
    if dweight is None:
        dweight = torch.empty(C, 4, dtype=weight.dtype, device=x.device)
    if bias is not None and dbias is None:
        dbias = torch.empty(C, dtype=bias.dtype, device=x.device)
    ws = _bwd_workspace(x, S, C, workspace, silu_grad_preactivation) if S > 0 else workspace
    binding.conv1d_bwd(x, dy, weight, cu_seqlens, bias=bias, policy=silu_grad_preactivation,
                       dx=dx, dweight=dweight, dbias=dbias, workspace=ws)
    return (dx, dweight) if bias is None else (dx, dweight, dbias)


class CakeCausalConv1dFunction(torch.autograd.Function):
    """Autograd wrapper saving only (x, weight, cu_seqlens, bias); its backward
    runs cake_causal_conv1d_train_backward on the incoming gradient (made a
    contiguous BF16 tensor first) and returns the gradients of weight and bias in
    the parameters' dtypes (CakeCausalConv1dFunction page)."""

    @staticmethod
    def forward(ctx, x, weight, cu_seqlens, bias=None, silu_grad_preactivation="bf16"):
        y = cake_causal_conv1d_train_forward(x, weight, cu_seqlens, bias=bias)
        ctx.save_for_backward(x, weight, cu_seqlens, bias)
        ctx.policy = silu_grad_preactivation
        return y

    @staticmethod
    def backward(ctx, grad_y):
        x, weight, cu_seqlens, bias = ctx.saved_tensors
        dy = grad_y.to(torch.bfloat16).contiguous()
        grads = cake_causal_conv1d_train_backward(x, weight, cu_seqlens, dy, bias=bias,
                                                  silu_grad_preactivation=ctx.policy)
        dx, dweight = grads[0], grads[1]
        dbias = grads[2] if bias is not None else None
        return (dx if ctx.needs_input_grad[0] else None,
                dweight if ctx.needs_input_grad[1] else None,
                None,
                dbias if bias is not None and ctx.needs_input_grad[3] else None,
                None)


def causal_conv1d(x, weight, cu_seqlens, bias=None, silu_grad_preactivation="bf16"):
    """Differentiable packed causal depthwise conv (width 4) + SiLU."""
    return CakeCausalConv1dFunction.apply(x, weight, cu_seqlens, bias, silu_grad_preactivation)
