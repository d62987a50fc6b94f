"""The comparison rules themselves (CPU): at the "large" workload's full length
(S = 262144, the longest sums of the five workloads) a plausible GPU result
passes, and planted mistakes in a BF16 gradient -- a factor of 2 on one entry,
truncation instead of rounding, two channels swapped, one entry a BF16 ulp
off -- fail. The "GPU" values are the oracle's FP64 gradients with FP32-sized
noise at the policy's rel-L2 level, rounded as the reduce kernel rounds."""
import numpy as np
import pytest
import torch

import oracle
from varlen_causal_depthwise_gb300 import synth
from _check import REL_L2, bf16_close, grads_close, rne_bf16


@pytest.fixture(scope="module")
def large_grads():
    w = synth.make("large", C=16)                      # full S, 16 channels
    assert w.S == 262144
    chans = np.arange(16)
    dw, db = oracle.bwd_params_at(w.x, w.dy, w.weight, w.cu_seqlens, chans, w.bias, "fp32")
    return dw, db


def _fake_gpu(ref, policy, rng):
    """FP32 values within the policy's rel-L2 of ref (noise at 40% of it)."""
    rms = np.sqrt(np.mean(ref ** 2))
    f = ref + rng.standard_normal(ref.shape) * 0.4 * REL_L2[policy] * rms
    return f.astype(np.float32)


def test_plausible_result_passes(large_grads):
    dw, db = large_grads
    rng = np.random.default_rng(0)
    f_w, f_b = _fake_gpu(dw, "fp32", rng), _fake_gpu(db, "fp32", rng)
    grads_close(f_w, f_b, dw, db, "fp32", "plausible", dw_bf16=rne_bf16(f_w),
                db_bf16=rne_bf16(f_b))


@pytest.mark.parametrize("mistake", ["double_one", "truncate", "swap_channels", "one_ulp",
                                     "double_fp32"])
def test_planted_mistakes_fail(large_grads, mistake):
    dw, db = large_grads
    rng = np.random.default_rng(1)
    f_w, f_b = _fake_gpu(dw, "fp32", rng), _fake_gpu(db, "fp32", rng)
    g_w = rne_bf16(f_w)
    if mistake == "double_one":
        g_w[3, 1] *= 2.0
    elif mistake == "truncate":                        # round toward zero
        bits = f_w.view(np.uint32) & np.uint32(0xFFFF0000)
        g_w = bits.view(np.float32).astype(np.float64)
    elif mistake == "swap_channels":
        g_w[[2, 5]] = g_w[[5, 2]]
    elif mistake == "one_ulp":
        v = torch.tensor(g_w[7, 2], dtype=torch.bfloat16)
        g_w[7, 2] = float(torch.nextafter(v, torch.tensor(np.inf, dtype=torch.bfloat16)))
    elif mistake == "double_fp32":                     # both outputs wrong together
        f_w = (f_w * 2).astype(np.float32)
        g_w = rne_bf16(f_w)
    with pytest.raises(AssertionError):
        grads_close(f_w, f_b, dw, db, "fp32", mistake, dw_bf16=g_w, db_bf16=rne_bf16(f_b))


def test_strict_floor():
    """The 1-ulp rule plus allowance passes, but too many elements that need
    the allowance fail the strict floor."""
    ref = np.linspace(1.0, 2.0, 100000)
    ulp = 2.0 ** -7
    gpu = ref.copy()
    allow = np.zeros_like(ref)
    idx = np.arange(0, 100000, 1000)                   # 100 elements, 1e-3 of them
    gpu[idx] += 1.5 * ulp
    allow[idx] = ulp
    with pytest.raises(AssertionError, match="strict"):
        bf16_close(gpu, ref, allow, "too many")
    gpu2 = ref.copy()
    gpu2[idx[:10]] += 1.5 * ulp                        # 1e-4: within the floor
    assert bf16_close(gpu2, ref, allow, "few") == pytest.approx(1 - 1e-4)
    with pytest.raises(AssertionError):
        bf16_close(gpu2, ref, allow, "exact", strict_miss_fraction=0)
