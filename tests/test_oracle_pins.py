"""Pins the FP64 oracle to the pages' definitions by independent routes (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from varlen_causal_depthwise_gb300 import synth
import _pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("policy", ["bf16", "fp32"])
def test_banded_matrix(lib, seed, policy):
    _pins.pin_banded(lib, seed, policy)


@pytest.mark.parametrize("seed", range(4))
def test_torch_conv1d_per_document(lib, seed):
    _pins.pin_conv1d(lib, seed)


@pytest.mark.parametrize("seed", range(2))
def test_finite_differences(lib, seed):
    _pins.pin_fd(lib, seed)


def test_bf16_rounding(lib):
    _pins.pin_rounding(lib)


def test_silu_closed_forms(lib):
    _pins.pin_silu(lib)


def test_golden_hand_example(lib):
    _pins.pin_golden(lib)


def test_tap_orientation(lib):
    """weight = e3, bias 0 gives silu(x); weight = e0 gives silu(x[t-3] + b) inside
    a document and silu(b) on its first three tokens."""
    w = _pins.small_case(20, 8, [7, 0, 13], seed=3)
    W = torch.zeros(8, 4)
    W[:, 3] = 1
    y, _ = oracle.fwd(w.x, W, w.cu_seqlens, None)
    want, _ = _pins.silu_and_grad_torch(_pins.as64(w.x))
    np.testing.assert_allclose(y, want, rtol=1e-15)
    W = torch.zeros(8, 4)
    W[:, 0] = 1
    y, _ = oracle.fwd(w.x, W, w.cu_seqlens, w.bias)
    x, b = _pins.as64(w.x), _pins.as64(w.bias)
    for t in range(20):
        start = 0 if t < 7 else 7
        pre = b + (x[t - 3] if t - 3 >= start else 0.0)
        np.testing.assert_allclose(y[t], _pins.silu_and_grad_torch(pre)[0], rtol=1e-15)


def test_document_start_is_zero_history(lib):
    """Every document's first token sees only itself: pre = w3 x + b."""
    w = synth.make("tiny", S=512, C=16)
    y, _ = oracle.fwd(w.x, w.weight, w.cu_seqlens, w.bias)
    x, W, b = _pins.as64(w.x), _pins.as64(w.weight), _pins.as64(w.bias)
    for s in w.cu_seqlens[:-1].tolist():
        if s < w.S:
            want, _ = _pins.silu_and_grad_torch(W[:, 3] * x[s] + b)
            np.testing.assert_allclose(y[s], want, rtol=1e-14)


def test_empty_documents_change_nothing(lib):
    lengths = [5, 0, 0, 9, 0, 3, 0]
    w = _pins.small_case(17, 8, lengths, seed=11)
    cu2 = synth.cu_from_lengths([n for n in lengths if n])
    a = oracle.fwd(w.x, w.weight, w.cu_seqlens, w.bias)[0]
    b = oracle.fwd(w.x, w.weight, cu2, w.bias)[0]
    np.testing.assert_array_equal(a, b)
    for pol in ("bf16", "fp32"):
        r1 = oracle.bwd(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, pol)
        r2 = oracle.bwd(w.x, w.dy, w.weight, cu2, w.bias, pol)
        for u, v in zip(r1, r2):
            np.testing.assert_array_equal(u, v)


def test_documents_are_independent(lib):
    """Each document run alone gives the same rows; shuffling documents permutes
    y and dx and leaves dweight / dbias unchanged (up to summation order)."""
    lengths = [6, 1, 11, 4]
    w = _pins.small_case(22, 8, lengths, seed=5)
    y, _ = oracle.fwd(w.x, w.weight, w.cu_seqlens, w.bias)
    dx, _, dW, db = oracle.bwd(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, "bf16")
    bounds = np.cumsum([0] + lengths)
    for i, n in enumerate(lengths):
        a = bounds[i]
        cu = torch.tensor([0, n], dtype=torch.int32)
        yi, _ = oracle.fwd(w.x[a:a + n], w.weight, cu, w.bias)
        np.testing.assert_array_equal(yi, y[a:a + n])
    order = [2, 0, 3, 1]
    idx = np.concatenate([np.arange(bounds[i], bounds[i + 1]) for i in order])
    cu = synth.cu_from_lengths([lengths[i] for i in order])
    y2, _ = oracle.fwd(w.x[idx], w.weight, cu, w.bias)
    dx2, _, dW2, db2 = oracle.bwd(w.x[idx], w.dy[idx], w.weight, cu, w.bias, "bf16")
    np.testing.assert_array_equal(y2, y[idx])
    np.testing.assert_array_equal(dx2, dx[idx])
    np.testing.assert_allclose(dW2, dW, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(db2, db, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("cu", [[0], [0, 0], [0, 0, 0, 0]])
def test_empty_sequence(lib, cu):
    x = torch.zeros(0, 8, dtype=torch.bfloat16)
    W = torch.randn(8, 4)
    b = torch.randn(8)
    cu = torch.tensor(cu, dtype=torch.int32)
    y, _ = oracle.fwd(x, W, cu, b)
    assert y.shape == (0, 8)
    dx, _, dW, db = oracle.bwd(x, x, W, cu, b, "bf16")
    assert dx.shape == (0, 8)
    assert not dW.any() and not db.any()


def test_policy_plumbing(lib):
    """With weight e3 and no bias pre = x is BF16-exact, so both policies agree
    bit for bit; with general weights the bf16 policy equals the exact gradient
    evaluated at bf16(pre)."""
    w = _pins.small_case(30, 8, [30], seed=9, bias=False)
    W = torch.zeros(8, 4)
    W[:, 3] = 1
    a = oracle.bwd(w.x, w.dy, W, w.cu_seqlens, None, "bf16")
    b = oracle.bwd(w.x, w.dy, W, w.cu_seqlens, None, "fp32")
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[2], b[2])
    dx_bf, _, _, _ = oracle.bwd(w.x, w.dy, w.weight, w.cu_seqlens, None, "bf16")
    dx_ex, _, _, _ = oracle.bwd(w.x, w.dy, w.weight, w.cu_seqlens, None, "fp32")
    assert np.abs(dx_bf - dx_ex).max() > 0      # the policies really differ


def test_sampled_entry_points_match_full(lib):
    w = synth.make("boundary", S=300, C=24)
    y, ya = oracle.fwd(w.x, w.weight, w.cu_seqlens, w.bias)
    rng = np.random.default_rng(0)
    ts, cs = rng.integers(0, 300, 200), rng.integers(0, 24, 200)
    ys, yas = oracle.fwd_at(w.x, w.weight, w.cu_seqlens, ts, cs, w.bias)
    np.testing.assert_array_equal(ys, y[ts, cs])
    np.testing.assert_array_equal(yas, ya[ts, cs])
    for pol in ("bf16", "fp32"):
        dx, da, dW, db = oracle.bwd(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, pol)
        dxs, das = oracle.bwd_dx_at(w.x, w.dy, w.weight, w.cu_seqlens, ts, cs, w.bias, pol)
        np.testing.assert_array_equal(dxs, dx[ts, cs])
        np.testing.assert_array_equal(das, da[ts, cs])
        chans = [0, 5, 23]
        dWs, dbs = oracle.bwd_params_at(w.x, w.dy, w.weight, w.cu_seqlens, chans, w.bias, pol)
        np.testing.assert_array_equal(dWs, dW[chans])
        np.testing.assert_array_equal(dbs, db[chans])


def test_allowances_against_fp32_evaluations(lib):
    """Every emulated FP32 evaluation of y and dx lies within the oracle's
    allowance, and the allowance is not inflated far past those errors."""
    ratios = _pins.pin_allowances(lib)
    assert min(ratios.values()) >= 1.0, ratios


def test_allowance_is_small_where_well_conditioned(lib):
    """The FP32 allowance stays far below a BF16 ulp except near cancellation."""
    w = synth.make("tiny", S=256, C=32)
    y, ya = oracle.fwd(w.x, w.weight, w.cu_seqlens, w.bias)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -126))) - 7)
    frac = np.mean(ya > 0.25 * ulp)
    assert frac < 0.01, frac


def test_malformed_cu_seqlens_rejected(lib):
    x = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(8, 4)
    for cu in ([1, 4], [0, 3], [0, 3, 2, 4]):
        with pytest.raises(ValueError):
            oracle.fwd(x, W, torch.tensor(cu, dtype=torch.int32), None)


def test_parameter_dtype_independence(lib):
    """The weight and bias dtypes are storage only: with values that BF16
    represents exactly, every (weight, bias) dtype pair gives the same y, dx,
    dweight and dbias."""
    w = _pins.small_case(40, 16, [15, 0, 25], seed=4)
    Wv = w.weight.to(torch.bfloat16).float()          # BF16-representable values
    bv = w.bias.to(torch.bfloat16).float()
    ref = None
    for wdt in (torch.float32, torch.bfloat16):
        for bdt in (torch.float32, torch.bfloat16):
            W, b = Wv.to(wdt), bv.to(bdt)
            y, _ = oracle.fwd(w.x, W, w.cu_seqlens, b)
            dx, _, dW, db = oracle.bwd(w.x, w.dy, W, w.cu_seqlens, b, "bf16")
            out = (y, dx, dW, db)
            if ref is None:
                ref = out
            for u, v in zip(out, ref):
                np.testing.assert_array_equal(u, v)
