"""Independent checks ("pins") for the FP64 oracle.

Each pin computes the same quantity a different way from the oracle's per-element
loops, so a plausible slip in the oracle (wrong tap, sign, index, mask, rounding)
fails at least one of them:

* ``pin_banded``      dense per-document banded matrix A_w: pre = A_w x + b,
                      dx = A_w^T dpre, dweight from the tap masks (numpy / torch).
* ``pin_conv1d``      torch FP64 ``conv1d(groups=C, padding=3)`` run on each
                      document alone, SiLU and gradients by torch autograd.
* ``pin_fd``          central finite differences of sum(dy * y) in weight and bias.
* ``pin_rounding``    round-to-nearest-even BF16 against torch's float32 -> bf16
                      cast and hand-placed midpoints.
* ``pin_silu``        SiLU / SiLU' against torch FP64 and closed-form identities.
* ``pin_golden``      a hand-worked example stored under tests/golden/.
* ``pin_allowances``  the oracle's FP32-error allowances for y and dx against
                      FP32 evaluations emulated in numpy in many evaluation
                      orders (tests/_fp32_emul.py): never below an emulated
                      error, and in aggregate at most ALLOW_RATIO_MAX times the
                      largest emulated errors.

They take the oracle library as an argument so the mutation test can run them
against deliberately broken copies of the oracle.
"""
import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from varlen_causal_depthwise_gb300 import synth
import _fp32_emul

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------- helpers --

def rne_bf16_bits(v):
    """RNE of float64 values to BF16 by integer operations on the binary64
    pattern (normal BF16 range only). Independent of the oracle's frexp/nearbyint
    route."""
    v = np.asarray(v, dtype=np.float64)
    bits = v.view(np.uint64).copy()
    drop = np.uint64(45)                          # 52 - 7 fraction bits dropped
    lsb = (bits >> drop) & np.uint64(1)
    bits = bits + (np.uint64(1) << np.uint64(44)) - np.uint64(1) + lsb
    bits = bits & ~((np.uint64(1) << drop) - np.uint64(1))
    return bits.view(np.float64)


def tap_masks(S, lengths):
    """M[k][t, j] = 1 iff token j feeds tap k of token t inside t's document."""
    M = np.zeros((4, S, S))
    a = 0
    for n in lengths:
        for t in range(a, a + n):
            for k in range(4):
                j = t - 3 + k
                if j >= a:
                    M[k, t, j] = 1.0
        a += n
    return M


def as64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def silu_and_grad_torch(p):
    """SiLU and its derivative by torch autograd, FP64."""
    pt = torch.tensor(p, dtype=torch.float64, requires_grad=True)
    y = F.silu(pt)
    (g,) = torch.autograd.grad(y.sum(), pt)
    return y.detach().numpy(), g.numpy()


def small_case(S, C, lengths, seed, bias=True, w_dtype=torch.float32, x_sigma=1.0):
    return synth.custom(S, C, lengths, seed=seed, x_sigma=x_sigma, weight_dtype=w_dtype,
                        bias_dtype=torch.float32 if bias else None)


def random_lengths(S, rng, max_len=9, empty_p=0.2):
    out, tot = [], 0
    while tot < S:
        n = 0 if rng.random() < empty_p else int(rng.integers(1, max_len + 1))
        n = min(n, S - tot)
        out.append(n)
        tot += n
    if rng.random() < 0.5:
        out.insert(int(rng.integers(0, len(out) + 1)), 0)
    return out


# -------------------------------------------------------------------- pins --

def pin_banded(lib, seed, policy):
    """Oracle fwd/bwd vs the dense banded-matrix formulation."""
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 40))
    C = 8 * int(rng.integers(1, 3))
    lengths = random_lengths(S, rng)
    w = small_case(S, C, lengths, seed, bias=bool(rng.integers(0, 2)))
    x, dy, W, b = as64(w.x), as64(w.dy), as64(w.weight), as64(w.bias)
    M = tap_masks(S, lengths)
    pre = np.stack([sum(W[c, k] * (M[k] @ x[:, c]) for k in range(4)) for c in range(C)], 1)
    if b is not None:
        pre = pre + b[None, :]
    y, _ = silu_and_grad_torch(pre)
    p = rne_bf16_bits(pre) if policy == "bf16" else pre
    _, g = silu_and_grad_torch(p)
    dpre = dy * g
    dx = np.stack([sum(W[c, k] * (M[k].T @ dpre[:, c]) for k in range(4)) for c in range(C)], 1)
    dW = np.array([[dpre[:, c] @ (M[k] @ x[:, c]) for k in range(4)] for c in range(C)])
    db = dpre.sum(0)

    yo, _ = oracle.fwd(w.x, w.weight, w.cu_seqlens, w.bias, lib=lib)
    dxo, _, dWo, dbo = oracle.bwd(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, policy, lib=lib)
    np.testing.assert_allclose(yo, y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dxo, dx, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dWo, dW, rtol=1e-11, atol=1e-11)
    if b is not None:
        np.testing.assert_allclose(dbo, db, rtol=1e-11, atol=1e-11)


def pin_conv1d(lib, seed):
    """Oracle vs torch FP64 conv1d per document + autograd (exact policy)."""
    rng = np.random.default_rng(1000 + seed)
    lengths = [int(v) for v in rng.integers(0, 30, size=int(rng.integers(1, 6)))]
    S = sum(lengths)
    if S == 0:
        lengths, S = [5], 5
    C = 16
    w = small_case(S, C, lengths, seed)
    W = w.weight.double().clone().requires_grad_(True)
    B = w.bias.double().clone().requires_grad_(True)
    X = w.x.double().clone().requires_grad_(True)
    outs, a = [], 0
    for n in lengths:
        if n == 0:
            continue
        seg = X[a:a + n].t().unsqueeze(0)                       # [1, C, n]
        pre = F.conv1d(seg, W.unsqueeze(1), B, padding=3, groups=C)[0, :, :n]
        outs.append(F.silu(pre).t())
        a += n
    Y = torch.cat(outs, 0)
    loss = (Y * w.dy.double()).sum()
    gX, gW, gB = torch.autograd.grad(loss, (X, W, B))

    yo, _ = oracle.fwd(w.x, w.weight, w.cu_seqlens, w.bias, lib=lib)
    dxo, _, dWo, dbo = oracle.bwd(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, "fp32", lib=lib)
    np.testing.assert_allclose(yo, Y.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dxo, gX.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dWo, gW.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dbo, gB.numpy(), rtol=1e-10, atol=1e-11)


def pin_fd(lib, seed):
    """Central finite differences of L = sum(dy * y) in weight and bias."""
    rng = np.random.default_rng(2000 + seed)
    S = 24
    lengths = random_lengths(S, rng, max_len=10)
    C = 8
    w = small_case(S, C, lengths, seed)
    W = as64(w.weight)
    B = as64(w.bias)
    dy = as64(w.dy)

    def loss(Wv, Bv):
        y, _ = oracle.fwd(w.x, Wv, w.cu_seqlens, Bv, lib=lib)
        return float((y * dy).sum())

    _, _, dWo, dbo = oracle.bwd(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, "fp32", lib=lib)
    for c in range(C):
        for k in range(4):
            h = 1e-6 * max(1.0, abs(W[c, k]))
            Wp, Wm = W.copy(), W.copy()
            Wp[c, k] += h
            Wm[c, k] -= h
            fd = (loss(Wp, B) - loss(Wm, B)) / (2 * h)
            assert abs(fd - dWo[c, k]) <= 1e-7 * max(1.0, abs(dWo[c, k])), (c, k, fd, dWo[c, k])
        h = 1e-6
        Bp, Bm = B.copy(), B.copy()
        Bp[c] += h
        Bm[c] -= h
        fd = (loss(W, Bp) - loss(W, Bm)) / (2 * h)
        assert abs(fd - dbo[c]) <= 1e-7 * max(1.0, abs(dbo[c])), (c, fd, dbo[c])


def pin_rounding(lib):
    """BF16 RNE: torch's float32 -> bf16 cast on float32 inputs, and exact
    midpoints / just-off-midpoint doubles placed by hand."""
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
        np.ldexp(rng.random(200), -130),                  # subnormal bf16 range
        [3.3895313892515355e38, 3.39e38, -1.0, 0.0, -0.0],
    ]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.bfloat16).double().numpy()
    got = np.array([oracle.round_bf16(float(v), lib=lib) for v in vals])
    np.testing.assert_array_equal(got, want)
    cases = [
        (1.0 + 2.0 ** -8, 1.0),                           # tie -> even (down)
        (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),           # tie -> even (up)
        (1.0 + 2.0 ** -8 + 2.0 ** -40, 1.0 + 2.0 ** -7),  # just above a tie (double only)
        (1.0 + 2.0 ** -8 - 2.0 ** -40, 1.0),
        (-(1.0 + 3 * 2.0 ** -8), -(1.0 + 2.0 ** -6)),
        (2.0 ** -127 + 2.0 ** -134, 2.0 ** -127),         # subnormal tie -> even
        (2.0 ** 128 * (1 - 2.0 ** -9), math.inf),         # rounds past the max -> inf
    ]
    for v, r in cases:
        assert oracle.round_bf16(v, lib=lib) == r, (v, r)


def pin_silu(lib):
    ps = np.concatenate([np.linspace(-30, 30, 601), [0.0, 1e-300, -1e-300, 700.0, -700.0]])
    y, g = silu_and_grad_torch(ps)
    got_y = np.array([oracle.silu(p, lib=lib) for p in ps])
    got_g = np.array([oracle.silu_grad(p, lib=lib) for p in ps])
    np.testing.assert_allclose(got_y, y, rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(got_g, g, rtol=1e-12, atol=1e-15)
    for p in (0.3, 2.0, 7.5, 40.0):
        # sigmoid(p) + sigmoid(-p) = 1  =>  silu(p) - silu(-p) = p
        assert abs(oracle.silu(p, lib=lib) - oracle.silu(-p, lib=lib) - p) <= 1e-15 * max(1, p)
        # silu'(p) + silu'(-p) = 1
        assert abs(oracle.silu_grad(p, lib=lib) + oracle.silu_grad(-p, lib=lib) - 1) <= 1e-15
    assert oracle.silu(0.0, lib=lib) == 0.0 and oracle.silu_grad(0.0, lib=lib) == 0.5


def pin_golden(lib, name="hand_example.json"):
    """Hand-derived preactivations and gradient structure (see the fixture)."""
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    x = torch.tensor(g["x"], dtype=torch.float32).to(torch.bfloat16).reshape(-1, 1)
    dy = torch.tensor(g["dy"], dtype=torch.float32).to(torch.bfloat16).reshape(-1, 1)
    W = torch.tensor([g["weight"]], dtype=torch.float64)
    B = torch.tensor([g["bias"]], dtype=torch.float64)
    cu = torch.tensor(g["cu_seqlens"], dtype=torch.int32)
    pre = np.array(g["pre"], dtype=np.float64)
    y_want, grad = silu_and_grad_torch(pre)
    y, _ = oracle.fwd(x, W, cu, B, lib=lib)
    np.testing.assert_allclose(y[:, 0], y_want, rtol=1e-15, atol=0)
    dpre = np.array(g["dy"]) * grad
    dx, _, dW, db = oracle.bwd(x, dy, W, cu, B, "fp32", lib=lib)
    dx_want = np.array(g["dx_coeff"], dtype=np.float64) @ dpre
    np.testing.assert_allclose(dx[:, 0], dx_want, rtol=1e-14, atol=1e-15)
    xv = np.array(g["x"], dtype=np.float64)
    for k in range(4):
        want = sum(dpre[t] * xv[j] for t, j in g["dweight_pairs"][str(k)])
        assert abs(dW[0, k] - want) <= 1e-14 * max(1, abs(want)), (k, dW[0, k], want)
    assert abs(db[0] - dpre.sum()) <= 1e-14 * max(1, abs(dpre.sum()))


# Summed over the elements of a case, the allowance may exceed the largest
# error of the emulated FP32 evaluations by at most this factor. The oracle's
# allowances sit at 26-42 on the cases below; any one of their constants made
# 64 times larger moves its case to 93-2200.
ALLOW_RATIO_MAX = 75.0

_ALLOW_CASES = None


def _allow_cases():
    """Two problems of 8192 x 32 (long documents at sigma 1, documents of 0-5
    tokens at sigma 2) with the emulated FP32 results, computed once."""
    global _ALLOW_CASES
    if _ALLOW_CASES is None:
        cases = []
        for seed, (docs, sigma) in enumerate([(("uniform", 1, 200, 2), 1.0),
                                              (("uniform", 0, 5, 0), 2.0)]):
            S, C = 8192, 32
            lengths = synth.doc_lengths(docs, S, np.random.default_rng(seed))
            w = synth.custom(S, C, lengths, seed=seed, x_sigma=sigma)
            cu = w.cu_seqlens.numpy()
            x, dy = w.x.float().numpy(), w.dy.float().numpy()
            W, b = w.weight.float().numpy(), w.bias.float().numpy()
            ys = _fp32_emul.forward_variants(x, W, b, cu)
            dxs = {pol: _fp32_emul.backward_dx_variants(x, dy, W, b, cu, pol)
                   for pol in ("bf16", "fp32")}
            cases.append((w, ys, dxs))
        _ALLOW_CASES = cases
    return _ALLOW_CASES


def _check_allowance(ref, allow, variants, what):
    err = np.max([np.abs(v.astype(np.float64) - ref) for v in variants], axis=0)
    bad = err > allow
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements where an FP32 evaluation is "
                           f"further from the FP64 value than the allowance")
    ratio = float(allow.sum() / err.sum())
    assert ratio <= ALLOW_RATIO_MAX, f"{what}: allowance {ratio:.1f}x the FP32 errors seen"
    return ratio


def pin_allowances(lib):
    """The y and dx allowances against emulated FP32 evaluations."""
    ratios = {}
    for i, (w, ys, dxs) in enumerate(_allow_cases()):
        y, ya = oracle.fwd(w.x, w.weight, w.cu_seqlens, w.bias, lib=lib)
        ratios[f"case{i} y"] = _check_allowance(y, ya, ys, f"case {i} y")
        for pol in ("bf16", "fp32"):
            dx, da, _, _ = oracle.bwd(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, pol, lib=lib)
            ratios[f"case{i} {pol} dx"] = _check_allowance(dx, da, dxs[pol], f"case {i} {pol} dx")
    return ratios
