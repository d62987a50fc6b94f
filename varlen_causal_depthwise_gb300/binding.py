"""ctypes binding of ``libvcd.so`` (the C ABI declared in ``include/vcd.h``).

Argument marshalling only: tensors become device pointers, dtypes become
``vcd_dtype`` codes, the current torch stream becomes the ``cudaStream_t``.
Every step of the operation runs in the library's CUDA kernels; there is no
CPU fallback, and a missing library raises instead of degrading.
"""
import ctypes
import os

import torch

VCD_OK = 0
VCD_ERR_INVALID_ARG = 1
VCD_ERR_WORKSPACE_TOO_SMALL = 2
VCD_ERR_MISALIGNED = 3
VCD_ERR_CUDA = 4

VCD_BF16 = 0
VCD_FP32 = 1
POLICIES = {"bf16": 0, "fp32": 1}

_DTYPE = {torch.bfloat16: VCD_BF16, torch.float32: VCD_FP32}

_lib = None

# name -> (restype, argtypes); the same set include/vcd.h declares.
_vp, _i64, _int, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "conv1d_fwd_workspace_size": (_int, [_i64, _i64, ctypes.POINTER(_sz)]),
    "conv1d_bwd_workspace_size": (_int, [_i64, _i64, ctypes.POINTER(_sz)]),
    "conv1d_bwd_route_workspace_size": (_int, [_i64, _i64, _int, ctypes.POINTER(_sz)]),
    "conv1d_bwd_call_workspace_size": (_int, [_i64, _i64, _i64, _int, _int, ctypes.POINTER(_sz)]),
    "conv1d_fwd": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _i64, _vp, _int, _vp, _vp, _sz,
                          _vp]),
    "conv1d_fwd_exact": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _i64, _vp, _int, _vp, _vp]),
    "conv1d_bwd": (_int, [_vp, _vp, _i64, _i64, _vp, _int, _vp, _i64, _vp, _int, _int, _vp,
                          _vp, _int, _vp, _int, _vp, _sz, _vp]),
    "conv1d_bwd_exact_workspace_size": (_int, [_i64, _i64, ctypes.POINTER(_sz)]),
    "conv1d_bwd_exact": (_int, [_vp, _vp, _i64, _i64, _vp, _int, _vp, _i64, _vp, _int, _int, _vp,
                                _vp, _int, _vp, _int, _vp, _sz, _vp]),
    "conv1d_bwd_noalloc": (_int, [_vp, _vp, _i64, _i64, _vp, _int, _vp, _i64, _vp, _int, _int,
                                  _vp, _vp, _int, _vp, _int, _vp]),
    "conv1d_wait_fault": (_int, [ctypes.POINTER(_int)]),
    "conv1d_status_string": (ctypes.c_char_p, [_int]),
}

# include/vcd_stream.h: the bandwidth-ceiling kernel (no part of the operation).
STREAM_SIGNATURES = {
    "vcd_stream_copy": (_int, [_vp, _vp, _vp, _sz, _int, _vp]),
}


class VcdError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {conv1d_status_string(status)} (status {status})")


def library_path():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvcd.so")


def load_library():
    """Load libvcd.so once; raise if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m varlen_causal_depthwise_gb300.build`"
                " (or __graft_entry__.build()); there is no CPU fallback")
        lib = ctypes.CDLL(path)
        for name, (res, args) in {**SIGNATURES, **STREAM_SIGNATURES}.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def conv1d_status_string(status):
    return load_library().conv1d_status_string(int(status)).decode()


def _check(status, where):
    if status != VCD_OK:
        raise VcdError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dt(t):
    if t is None:
        return VCD_FP32
    if t.dtype not in _DTYPE:
        raise TypeError(f"unsupported dtype {t.dtype}; FP32 or BF16 expected")
    return _DTYPE[t.dtype]


def _stream(stream, device):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _require(t, name, dtypes, device, shape=None):
    """The C ABI sees only a pointer: the layout the kernels assume is checked
    here (CUDA, on x's device, contiguous, dtype, shape)."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, x on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must be one of {dtypes}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _sc(x):
    if x.dim() == 3 and x.shape[0] == 1:
        return int(x.shape[1]), int(x.shape[2])
    if x.dim() != 2:
        raise ValueError(f"x must be [S, C] or [1, S, C], got {tuple(x.shape)}")
    return int(x.shape[0]), int(x.shape[1])


def conv1d_fwd_workspace_size(S, C):
    n = ctypes.c_size_t(0)
    _check(load_library().conv1d_fwd_workspace_size(int(S), int(C), ctypes.byref(n)),
           "conv1d_fwd_workspace_size")
    return n.value


def conv1d_bwd_workspace_size(S, C):
    n = ctypes.c_size_t(0)
    _check(load_library().conv1d_bwd_workspace_size(int(S), int(C), ctypes.byref(n)),
           "conv1d_bwd_workspace_size")
    return n.value


def conv1d_bwd_route_workspace_size(S, C, policy="bf16"):
    """Bytes one policy's program needs (at most conv1d_bwd_workspace_size)."""
    if policy not in POLICIES:
        raise ValueError(f"policy must be 'bf16' or 'fp32', got {policy!r}")
    n = ctypes.c_size_t(0)
    _check(load_library().conv1d_bwd_route_workspace_size(int(S), int(C), POLICIES[policy],
                                                          ctypes.byref(n)),
           "conv1d_bwd_route_workspace_size")
    return n.value


def conv1d_bwd_call_workspace_size(S, C, num_docs, policy="bf16", has_bias=True):
    """Bytes one backward call needs exactly (its launch shape's partial rows)."""
    if policy not in POLICIES:
        raise ValueError(f"policy must be 'bf16' or 'fp32', got {policy!r}")
    n = ctypes.c_size_t(0)
    _check(load_library().conv1d_bwd_call_workspace_size(int(S), int(C), int(num_docs),
                                                         POLICIES[policy], int(bool(has_bias)),
                                                         ctypes.byref(n)),
           "conv1d_bwd_call_workspace_size")
    return n.value


def conv1d_fwd(x, weight, cu_seqlens, bias=None, y=None, workspace=None, stream=None):
    """y = bf16(silu(causal width-4 depthwise conv(x) + bias)), per document.

    x: BF16 CUDA tensor [S, C] or [1, S, C]; weight [C, 4] FP32/BF16;
    cu_seqlens int32 [num_docs + 1]; bias [C] FP32/BF16 or None.
    Returns y (allocated when not given)."""
    lib = load_library()
    S, C = _sc(x)
    dev = x.device
    _require(x, "x", (torch.bfloat16,), dev)
    _require(weight, "weight", (torch.float32, torch.bfloat16), dev, (C, 4))
    _require(cu_seqlens, "cu_seqlens", (torch.int32,), dev)
    _require(bias, "bias", (torch.float32, torch.bfloat16), dev, (C,))
    if y is None:
        y = torch.empty_like(x)
    _require(y, "y", (torch.bfloat16,), dev, x.shape)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        st = lib.conv1d_fwd(_ptr(x), S, C, _ptr(weight), _dt(weight), _ptr(cu_seqlens),
                            cu_seqlens.numel() - 1, _ptr(bias), _dt(bias), _ptr(y),
                            _ptr(workspace), nbytes, _stream(stream, dev))
    _check(st, "conv1d_fwd")
    return y


def conv1d_fwd_exact(x, weight, cu_seqlens, bias=None, y=None, stream=None):
    """conv1d_fwd with every element of y within one BF16 ulp of the exact
    value (the exactness-guarded route; slower). Same arguments."""
    lib = load_library()
    S, C = _sc(x)
    dev = x.device
    _require(x, "x", (torch.bfloat16,), dev)
    _require(weight, "weight", (torch.float32, torch.bfloat16), dev, (C, 4))
    _require(cu_seqlens, "cu_seqlens", (torch.int32,), dev)
    _require(bias, "bias", (torch.float32, torch.bfloat16), dev, (C,))
    if y is None:
        y = torch.empty_like(x)
    _require(y, "y", (torch.bfloat16,), dev, x.shape)
    with torch.cuda.device(dev):
        st = lib.conv1d_fwd_exact(_ptr(x), S, C, _ptr(weight), _dt(weight), _ptr(cu_seqlens),
                                  cu_seqlens.numel() - 1, _ptr(bias), _dt(bias), _ptr(y),
                                  _stream(stream, dev))
    _check(st, "conv1d_fwd_exact")
    return y


def conv1d_bwd_exact_workspace_size(S, C):
    n = ctypes.c_size_t(0)
    _check(load_library().conv1d_bwd_exact_workspace_size(int(S), int(C), ctypes.byref(n)),
           "conv1d_bwd_exact_workspace_size")
    return n.value


def conv1d_bwd_exact(x, dy, weight, cu_seqlens, bias=None, policy="bf16", dx=None, dweight=None,
                     dbias=None, workspace=None, stream=None, want_dbias=None):
    """conv1d_bwd with every element of dx within one BF16 ulp of the exact
    value (the exactness-guarded route; slower). Same arguments; the workspace
    is conv1d_bwd_exact_workspace_size(S, C) bytes (allocated when omitted)."""
    S, C = _sc(x)
    if workspace is None:
        workspace = torch.empty(conv1d_bwd_exact_workspace_size(S, C), dtype=torch.uint8,
                                device=x.device)
    return conv1d_bwd(x, dy, weight, cu_seqlens, bias, policy, dx, dweight, dbias, workspace,
                      stream, want_dbias, _entry="conv1d_bwd_exact")


def conv1d_bwd(x, dy, weight, cu_seqlens, bias=None, policy="bf16", dx=None, dweight=None,
               dbias=None, workspace=None, stream=None, want_dbias=None, _entry="conv1d_bwd"):
    """Gradients of the forward: returns (dx, dweight, dbias or None).

    Output dtypes default to the parameters' dtypes. ``workspace`` (uint8, at
    least conv1d_bwd_call_workspace_size(S, C, num_docs, policy, bias is not
    None) bytes; conv1d_bwd_route_workspace_size(S, C, policy) always suffices)
    is allocated when omitted."""
    lib = load_library()
    S, C = _sc(x)
    if policy not in POLICIES:
        raise ValueError(f"policy must be 'bf16' or 'fp32', got {policy!r}")
    dev = x.device
    _require(x, "x", (torch.bfloat16,), dev)
    _require(dy, "dy", (torch.bfloat16,), dev, x.shape)
    _require(weight, "weight", (torch.float32, torch.bfloat16), dev, (C, 4))
    _require(cu_seqlens, "cu_seqlens", (torch.int32,), dev)
    _require(bias, "bias", (torch.float32, torch.bfloat16), dev, (C,))
    if dx is None:
        dx = torch.empty_like(x)
    if dweight is None:
        dweight = torch.empty(C, 4, dtype=weight.dtype, device=dev)
    if want_dbias is None:
        want_dbias = bias is not None
    if dbias is None and want_dbias:
        dbias = torch.empty(C, dtype=bias.dtype if bias is not None else torch.float32,
                            device=dev)
    _require(dx, "dx", (torch.bfloat16,), dev, x.shape)
    _require(dweight, "dweight", (torch.float32, torch.bfloat16), dev, (C, 4))
    _require(dbias, "dbias", (torch.float32, torch.bfloat16), dev, (C,))
    if workspace is None:
        workspace = torch.empty(conv1d_bwd_route_workspace_size(S, C, policy), dtype=torch.uint8,
                                device=dev)
    _require(workspace, "workspace", (torch.uint8,), dev)
    nbytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        st = getattr(lib, _entry)(_ptr(x), _ptr(dy), S, C, _ptr(weight), _dt(weight),
                                  _ptr(cu_seqlens), cu_seqlens.numel() - 1, _ptr(bias), _dt(bias),
                                  POLICIES[policy], _ptr(dx), _ptr(dweight), _dt(dweight),
                                  _ptr(dbias), _dt(dbias), _ptr(workspace), nbytes,
                                  _stream(stream, dev))
    _check(st, _entry)
    return dx, dweight, dbias


def conv1d_bwd_noalloc(x, dy, weight, cu_seqlens, bias=None, policy="bf16", dx=None,
                       dweight=None, dbias=None, stream=None, want_dbias=None):
    """conv1d_bwd for callers that cannot give the library device memory: the
    partial rows live in the library's fixed scratch array (see include/vcd.h).
    Outputs not passed in are allocated here by torch, as in conv1d_bwd; the
    library call itself allocates nothing."""
    lib = load_library()
    S, C = _sc(x)
    if policy not in POLICIES:
        raise ValueError(f"policy must be 'bf16' or 'fp32', got {policy!r}")
    dev = x.device
    _require(x, "x", (torch.bfloat16,), dev)
    _require(dy, "dy", (torch.bfloat16,), dev, x.shape)
    _require(weight, "weight", (torch.float32, torch.bfloat16), dev, (C, 4))
    _require(cu_seqlens, "cu_seqlens", (torch.int32,), dev)
    _require(bias, "bias", (torch.float32, torch.bfloat16), dev, (C,))
    if dx is None:
        dx = torch.empty_like(x)
    if dweight is None:
        dweight = torch.empty(C, 4, dtype=weight.dtype, device=dev)
    if want_dbias is None:
        want_dbias = bias is not None
    if dbias is None and want_dbias:
        dbias = torch.empty(C, dtype=bias.dtype if bias is not None else torch.float32,
                            device=dev)
    _require(dx, "dx", (torch.bfloat16,), dev, x.shape)
    _require(dweight, "dweight", (torch.float32, torch.bfloat16), dev, (C, 4))
    _require(dbias, "dbias", (torch.float32, torch.bfloat16), dev, (C,))
    with torch.cuda.device(dev):
        st = lib.conv1d_bwd_noalloc(_ptr(x), _ptr(dy), S, C, _ptr(weight), _dt(weight),
                                    _ptr(cu_seqlens), cu_seqlens.numel() - 1, _ptr(bias),
                                    _dt(bias), POLICIES[policy], _ptr(dx), _ptr(dweight),
                                    _dt(dweight), _ptr(dbias), _dt(dbias), _stream(stream, dev))
    _check(st, "conv1d_bwd_noalloc")
    return dx, dweight, dbias


def stream_copy(a, out, b=None, blocks_per_sm=2, stream=None):
    """out = a (or a XOR b) byte for byte through vcd_stream_copy: the traffic
    of a forward (a -> out) or a backward (a, b -> out) call with no
    arithmetic. Tensors: CUDA, contiguous, same byte size."""
    n = a.numel() * a.element_size()
    for t, name in ((a, "a"), (out, "out"), (b, "b")):
        if t is None:
            continue
        _require(t, name, (t.dtype,), a.device)
        if t.numel() * t.element_size() != n:
            raise ValueError(f"{name} must hold {n} bytes")
    st = load_library().vcd_stream_copy(_ptr(a), _ptr(b), _ptr(out), n, int(blocks_per_sm),
                                        _stream(stream, a.device))
    _check(st, "vcd_stream_copy")


def conv1d_wait_fault():
    """True if a backward kernel gave up waiting on a staged tile since the
    last call (never in normal operation); clears the flag. Synchronous."""
    flag = _int(0)
    _check(load_library().conv1d_wait_fault(ctypes.byref(flag)), "conv1d_wait_fault")
    return bool(flag.value)
