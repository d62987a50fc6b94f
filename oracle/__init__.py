"""FP64 CPU oracle for the packed width-4 depthwise causal convolution + SiLU.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package. The CUDA
library never calls it and shares no code with it.

The C source (``vcd_oracle.c``) holds the definitions, written from the FlashInfer
API pages "cake_causal_conv1d_train_forward" (Parameters, Returns) and
"cake_causal_conv1d_train_backward" (Parameters: silu_grad_preactivation;
Returns). This module only marshals arrays through ctypes.

Parity pins (all in ``tests/test_oracle_pins.py``): a dense banded-matrix
formulation, torch FP64 ``conv1d`` per document with autograd, central finite
differences, closed forms (tap orientation, SiLU identities), BF16 rounding
against torch and hand-placed midpoints, empty documents, S == 0, document
shuffling, and a hand-worked fixture in ``tests/golden/``.
"""
import ctypes
import os

import numpy as np
import torch

from . import build as _build

POLICY = {"bf16": 0, "fp32": 1}

_lib = None
_D = ctypes.POINTER(ctypes.c_double)
_U16 = ctypes.POINTER(ctypes.c_uint16)
_I32 = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


def load(path=None):
    """Load (building first if needed) the oracle library; returns the CDLL."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(_build.build()))
    return _lib


def _declare(lib):
    lib.vcd_oracle_fwd.argtypes = [_i64, _i64, _U16, _D, _D, _I32, _i64, _D, _D]
    lib.vcd_oracle_fwd_at.argtypes = [_i64, _i64, _U16, _D, _D, _I32, _i64, _i64, _I64, _I64,
                                      _D, _D]
    lib.vcd_oracle_bwd.argtypes = [_i64, _i64, _U16, _U16, _D, _D, _I32, _i64, ctypes.c_int,
                                   _D, _D, _D, _D, _D, _D]
    lib.vcd_oracle_bwd_dx_at.argtypes = [_i64, _i64, _U16, _U16, _D, _D, _I32, _i64,
                                         ctypes.c_int, _i64, _I64, _I64, _D, _D]
    lib.vcd_oracle_bwd_params_at.argtypes = [_i64, _i64, _U16, _U16, _D, _D, _I32, _i64,
                                             ctypes.c_int, _i64, _I64, _D, _D, _D, _D]
    for name in ("vcd_oracle_round_bf16", "vcd_oracle_silu", "vcd_oracle_silu_grad"):
        getattr(lib, name).argtypes = [ctypes.c_double]
        getattr(lib, name).restype = ctypes.c_double
    for name in ("vcd_oracle_fwd", "vcd_oracle_fwd_at", "vcd_oracle_bwd",
                 "vcd_oracle_bwd_dx_at", "vcd_oracle_bwd_params_at"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


# ------------------------------------------------------------ marshalling ---

def _bits(t):
    """BF16 CPU tensor -> contiguous uint16 numpy array of its bit patterns."""
    t = torch.as_tensor(t)
    assert t.dtype == torch.bfloat16, t.dtype
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy()
                                .view(np.uint16))


def _f64(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return np.ascontiguousarray(t.detach().cpu().double().numpy())
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _i32(t):
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.int32))


def _i64a(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _p(a, ctype):
    return None if a is None else a.ctypes.data_as(ctype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (status {rc})")


def _shape(x):
    x = torch.as_tensor(x)
    if x.dim() == 3:
        x = x.reshape(x.shape[-2], x.shape[-1])
    return x, int(x.shape[0]), int(x.shape[1])


# ------------------------------------------------------------------- API ---

def fwd(x, weight, cu_seqlens, bias=None, lib=None):
    """Full forward. Returns (y, allowance), both float64 numpy [S, C]."""
    lib = lib or load()
    x, S, C = _shape(x)
    xb, w, b, cu = _bits(x), _f64(weight).reshape(-1), _f64(bias), _i32(cu_seqlens)
    y = np.zeros((S, C), np.float64)
    a = np.zeros((S, C), np.float64)
    rc = lib.vcd_oracle_fwd(S, C, _p(xb, _U16), _p(w, _D), _p(b, _D), _p(cu, _I32),
                            len(cu) - 1, _p(y, _D), _p(a, _D))
    _check(rc, "fwd")
    return y, a


def fwd_at(x, weight, cu_seqlens, ts, cs, bias=None, lib=None):
    """Forward at the listed (t, c) pairs. Returns (y, allowance) 1-D float64."""
    lib = lib or load()
    x, S, C = _shape(x)
    xb, w, b, cu = _bits(x), _f64(weight).reshape(-1), _f64(bias), _i32(cu_seqlens)
    ts, cs = _i64a(ts), _i64a(cs)
    y = np.zeros(len(ts), np.float64)
    a = np.zeros(len(ts), np.float64)
    rc = lib.vcd_oracle_fwd_at(S, C, _p(xb, _U16), _p(w, _D), _p(b, _D), _p(cu, _I32),
                               len(cu) - 1, len(ts), _p(ts, _I64), _p(cs, _I64), _p(y, _D),
                               _p(a, _D))
    _check(rc, "fwd_at")
    return y, a


def bwd(x, dy, weight, cu_seqlens, bias=None, policy="bf16", lib=None, magnitudes=False):
    """Full backward. Returns (dx, dx_allowance, dweight [C,4], dbias [C] or None),
    plus (dweight_mag, dbias_mag) -- the sums of |term| -- with magnitudes=True."""
    lib = lib or load()
    x, S, C = _shape(x)
    dy, _, _ = _shape(dy)
    xb, gb = _bits(x), _bits(dy)
    w, b, cu = _f64(weight).reshape(-1), _f64(bias), _i32(cu_seqlens)
    dx = np.zeros((S, C), np.float64)
    a = np.zeros((S, C), np.float64)
    dw = np.zeros((C, 4), np.float64)
    db = np.zeros(C, np.float64) if bias is not None else None
    mw = np.zeros((C, 4), np.float64)
    mb = np.zeros(C, np.float64)
    rc = lib.vcd_oracle_bwd(S, C, _p(xb, _U16), _p(gb, _U16), _p(w, _D), _p(b, _D),
                            _p(cu, _I32), len(cu) - 1, POLICY[policy], _p(dx, _D), _p(a, _D),
                            _p(dw, _D), _p(db, _D), _p(mw, _D), _p(mb, _D))
    _check(rc, "bwd")
    if magnitudes:
        return dx, a, dw, db, mw, (mb if bias is not None else None)
    return dx, a, dw, db


def bwd_dx_at(x, dy, weight, cu_seqlens, ts, cs, bias=None, policy="bf16", lib=None):
    """dx at the listed (t, c) pairs. Returns (dx, allowance) 1-D float64."""
    lib = lib or load()
    x, S, C = _shape(x)
    dy, _, _ = _shape(dy)
    xb, gb = _bits(x), _bits(dy)
    w, b, cu = _f64(weight).reshape(-1), _f64(bias), _i32(cu_seqlens)
    ts, cs = _i64a(ts), _i64a(cs)
    dx = np.zeros(len(ts), np.float64)
    a = np.zeros(len(ts), np.float64)
    rc = lib.vcd_oracle_bwd_dx_at(S, C, _p(xb, _U16), _p(gb, _U16), _p(w, _D), _p(b, _D),
                                  _p(cu, _I32), len(cu) - 1, POLICY[policy], len(ts),
                                  _p(ts, _I64), _p(cs, _I64), _p(dx, _D), _p(a, _D))
    _check(rc, "bwd_dx_at")
    return dx, a


def bwd_params_at(x, dy, weight, cu_seqlens, cs, bias=None, policy="bf16", lib=None,
                  magnitudes=False):
    """dweight [n,4] and dbias [n] (None without bias) for the listed channels,
    plus their magnitude sums with magnitudes=True."""
    lib = lib or load()
    x, S, C = _shape(x)
    dy, _, _ = _shape(dy)
    xb, gb = _bits(x), _bits(dy)
    w, b, cu = _f64(weight).reshape(-1), _f64(bias), _i32(cu_seqlens)
    cs = _i64a(cs)
    dw = np.zeros((len(cs), 4), np.float64)
    db = np.zeros(len(cs), np.float64) if bias is not None else None
    mw = np.zeros((len(cs), 4), np.float64)
    mb = np.zeros(len(cs), np.float64)
    rc = lib.vcd_oracle_bwd_params_at(S, C, _p(xb, _U16), _p(gb, _U16), _p(w, _D), _p(b, _D),
                                      _p(cu, _I32), len(cu) - 1, POLICY[policy], len(cs),
                                      _p(cs, _I64), _p(dw, _D), _p(db, _D), _p(mw, _D),
                                      _p(mb, _D))
    _check(rc, "bwd_params_at")
    if magnitudes:
        return dw, db, mw, (mb if bias is not None else None)
    return dw, db


def round_bf16(v, lib=None):
    lib = lib or load()
    return lib.vcd_oracle_round_bf16(float(v))


def silu(v, lib=None):
    lib = lib or load()
    return lib.vcd_oracle_silu(float(v))


def silu_grad(v, lib=None):
    lib = lib or load()
    return lib.vcd_oracle_silu_grad(float(v))
