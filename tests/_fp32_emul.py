"""FP32 evaluations of the operation, in numpy, in several evaluation orders.

The oracle returns, beside each y and dx value, an allowance: its bound on the
error any FP32 evaluation of the same formulas can make. These emulations are
such evaluations -- different summation orders, fused and unfused
multiply-adds, three ways of forming the sigmoid -- so they pin the allowance
from both sides:

* below: no emulated FP32 result may lie further from the FP64 value than the
  allowance (an allowance that forgets an error source fails);
* above: summed over many elements, the allowance may exceed the largest error
  the emulations actually make by a bounded factor (an allowance inflated well
  past the errors FP32 can make fails).

Each FP32 operation is rounded once to float32 (a fused multiply-add forms the
exact product in float64 -- 24 + 24 bits fit in 53 -- adds in float64 and
rounds to float32). Nothing here shares code with the oracle or the CUDA
library; the document structure comes from cu_seqlens directly.
"""
import numpy as np
import torch

F32 = np.float32


def f32(v):
    return np.asarray(v, dtype=np.float64).astype(F32)


def fma(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(F32)


def mul(a, b):
    return (a * b).astype(F32)


def add(a, b):
    return (a + b).astype(F32)


def rne_bf16(v):
    """float32 -> nearest BF16 (ties to even) -> float32, by torch's cast."""
    return torch.from_numpy(np.ascontiguousarray(v, dtype=F32)).to(torch.bfloat16).float().numpy()


LOG2E = F32(1.4426950408889634)


def sigmoid(p, how):
    """Three FP32 routes to 1 / (1 + e^-p)."""
    one = F32(1.0)
    if how == "exp2":             # 2^(-p log2 e) with the argument rounded, then 1 / (1 + e)
        e = np.exp2(mul(-p, np.full_like(p, LOG2E))).astype(F32)
        return (one / add(e, np.full_like(p, one))).astype(F32)
    if how == "exp":              # e^-p, then 1 / (1 + e)
        e = np.exp(-p).astype(F32)
        return (one / add(e, np.full_like(p, one))).astype(F32)
    if how == "split":            # the overflow-free form: e^p / (1 + e^p) for p < 0
        e = np.exp(-np.abs(p)).astype(F32)
        d = add(e, np.full_like(p, one))
        pos = (one / d).astype(F32)
        neg = (e / d).astype(F32)
        return np.where(p >= 0, pos, neg).astype(F32)
    raise ValueError(how)


SIGMOIDS = ("exp2", "exp", "split")


def silu(p, how):
    return mul(p, sigmoid(p, how))


def silu_grad(p, how, fused):
    """s (1 + p (1 - s)): as two FMAs (s + s (p - p s)) or unfused."""
    s = sigmoid(p, how)
    if fused:
        t = fma(-p, s, p)
        return fma(s, t, s)
    one = np.full_like(p, F32(1.0))
    return mul(s, add(one, mul(p, add(one, -s))))


def doc_start(cu, S):
    """start[t] = first token of t's document (cu_seqlens is sorted; the last
    index i with cu[i] <= t)."""
    cu = np.asarray(cu, dtype=np.int64)
    t = np.arange(S)
    i = np.searchsorted(cu, t, side="right") - 1
    return cu[i]


def taps(x, start):
    """X[k][t, c] = x[t - 3 + k, c] inside t's document, else 0 (float32)."""
    S = x.shape[0]
    out = []
    t = np.arange(S)
    for k in range(4):
        j = t - 3 + k
        ok = j >= start
        v = np.zeros_like(x)
        v[ok] = x[j[ok]]
        out.append(v)
    return out


ORDERS = ("chain", "reverse", "pairwise")


def pre32(X, w, b, order):
    """FP32 preactivation in one of three orders. X: taps, w [C, 4] f32, b [C] f32."""
    S, C = X[0].shape
    bb = np.broadcast_to(b, (S, C)).astype(F32)
    if order == "chain":          # b, then taps 0..3 by FMA
        acc = bb
        for k in range(4):
            acc = fma(np.broadcast_to(w[:, k], (S, C)), X[k], acc)
        return acc
    if order == "reverse":        # products rounded, added from tap 3 down, bias last
        acc = np.zeros((S, C), F32)
        for k in (3, 2, 1, 0):
            acc = add(acc, mul(np.broadcast_to(w[:, k], (S, C)), X[k]))
        return add(acc, bb)
    if order == "pairwise":       # (w0 x0 + w1 x1) + (w2 x2 + w3 x3), then the bias
        p = [mul(np.broadcast_to(w[:, k], (S, C)), X[k]) for k in range(4)]
        return add(add(add(p[0], p[1]), add(p[2], p[3])), bb)
    raise ValueError(order)


def forward_variants(x, w, b, cu):
    """FP32 y (before any BF16 rounding) for every (order, sigmoid) pair."""
    x = f32(x)
    S, C = x.shape
    w = f32(w)
    b = np.zeros(C, F32) if b is None else f32(b)
    X = taps(x, doc_start(cu, S))
    out = []
    for order in ORDERS:
        p = pre32(X, w, b, order)
        for how in SIGMOIDS:
            out.append(silu(p, how))
    return out


def dx_from_dpre(d, w, start, order):
    """dx[t] = sum_k w[k] dpre[t + 3 - k] over t + 3 - k < S in t's document."""
    S, C = d.shape
    t = np.arange(S)
    terms = []
    for k in range(4):
        j = t + 3 - k
        ok = j < S
        ok[ok] = start[j[ok]] == start[ok]
        v = np.zeros_like(d)
        v[ok] = d[j[ok]]
        terms.append((k, v))
    W = lambda k: np.broadcast_to(w[:, k], (S, C))
    if order == "chain":          # w3 d[t], then w2, w1, w0 by FMA (gather form)
        acc = mul(W(3), terms[3][1])
        for k in (2, 1, 0):
            acc = fma(W(k), terms[k][1], acc)
        return acc
    acc = np.zeros((S, C), F32)   # products rounded, added from tap 0 up
    for k in (0, 1, 2, 3):
        acc = add(acc, mul(W(k), terms[k][1]))
    return acc


def backward_dx_variants(x, dy, w, b, cu, policy):
    """FP32 dx (before BF16 rounding) for a set of evaluation routes."""
    x, dy = f32(x), f32(dy)
    S, C = x.shape
    w = f32(w)
    b = np.zeros(C, F32) if b is None else f32(b)
    start = doc_start(cu, S)
    X = taps(x, start)
    out = []
    for order in ORDERS:
        pre = pre32(X, w, b, order)
        p = rne_bf16(pre) if policy == "bf16" else pre
        for how in SIGMOIDS:
            for fused in (True, False):
                d = mul(dy, silu_grad(p, how, fused))
                for dorder in ("chain", "sum"):
                    if not fused and dorder == "sum" and how != "exp":
                        continue          # keep the count of routes moderate
                    out.append(dx_from_dpre(d, w, start, dorder))
    return out
