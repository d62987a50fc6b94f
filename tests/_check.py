"""Comparison rules between the CUDA library and the FP64 oracle.

* y and dx (BF16): |g - r| <= ulp_bf16(r) + allowance, where the allowance is
  the oracle's bound on FP32 evaluation error (zero for well-conditioned
  elements; pinned against emulated FP32 evaluations). The strict rule
  (allowance 0) must also hold on all but a small fraction of the elements:
  STRICT_MISS_FRACTION, or STRICT_MISS_MIN elements in a small case.
* FP32 dweight / dbias: rel-L2 against the oracle of the same SiLU' policy,
  5e-5 under "bf16" and 5e-7 under "fp32" (the backward page states about
  3e-5 and 2e-7).
* BF16 dweight / dbias come from another call of the same route asking for
  BF16 outputs. Both calls sum the same partial rows in the same order, so
  (i) each BF16 value must be the round-to-nearest-even of the FP32 output of
  the FP32 call -- exactly, except that under the "fp32" policy (an FP64
  total rounded once to each dtype) an FP32 value lying on a BF16 rounding
  midpoint admits either neighbour -- and (ii) elementwise
  |g - r| <= ulp_bf16(r) + BF16_GRAD_RMS_FACTOR * tol * rms(r), tol the
  policy's rel-L2 bound: a BF16 gradient is one rounding away from an FP32
  value whose error is of the order of tol times the typical gradient.
"""
import numpy as np
import torch

REL_L2 = {"bf16": 5e-5, "fp32": 5e-7}
STRICT_MISS_FRACTION = 2e-4
STRICT_MISS_MIN = 2
BF16_GRAD_RMS_FACTOR = 8.0


def ulp_bf16(r):
    a = np.abs(np.asarray(r, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126.0), -126.0)
    return np.exp2(e - 7.0)


def bf16_close(gpu, ref, allow, what, strict_miss_fraction=STRICT_MISS_FRACTION):
    """Assert the BF16 rule and the floor on strict passes; returns the strict
    1-ulp pass fraction. strict_miss_fraction=0 demands every element strict."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    allow = np.zeros_like(ref) if allow is None else np.asarray(allow, dtype=np.float64)
    err = np.abs(gpu - ref)
    ulp = ulp_bf16(ref)
    ok = err <= ulp + allow
    if not ok.all():
        bad = np.flatnonzero(~ok.reshape(-1))
        i = bad[np.argmax((err - ulp - allow).reshape(-1)[bad])]
        raise AssertionError(
            f"{what}: {bad.size} of {ok.size} elements outside 1 ulp + allowance; worst flat "
            f"index {i}: gpu {gpu.reshape(-1)[i]!r} ref {ref.reshape(-1)[i]!r} "
            f"ulp {ulp.reshape(-1)[i]!r} allowance {allow.reshape(-1)[i]!r}")
    strict = err <= ulp
    misses = int(strict.size - np.count_nonzero(strict))
    limit = 0 if strict_miss_fraction == 0 else max(STRICT_MISS_MIN,
                                                    int(strict_miss_fraction * strict.size))
    assert misses <= limit, (f"{what}: {misses} of {strict.size} elements miss the strict "
                             f"1-ulp bound (at most {limit} may)")
    return float(np.mean(strict)) if strict.size else 1.0


def rel_l2(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(gpu - ref) / (den if den > 0 else 1.0))


def rne_bf16(v):
    """FP32 values -> nearest BF16 (ties to even), as float64."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.bfloat16).double().numpy()


def bf16_midpoint(f):
    """True where the FP32 value f lies exactly halfway between two BF16 values."""
    bits = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    return (bits & np.uint32(0xFFFF)) == np.uint32(0x8000)


def bf16_grad_close(g, f, ref, policy, what):
    """BF16 gradient g against the same route's FP32 output f and the oracle's
    value ref (rules (i) and (ii) of the module docstring)."""
    g = np.asarray(g, dtype=np.float64)
    f32 = np.asarray(f, dtype=np.float32)
    ref = np.asarray(ref, dtype=np.float64)
    want = rne_bf16(f32)
    same = g == want
    if policy == "fp32":
        # a midpoint FP32 value came from an FP64 total on one side of it
        up = np.nextafter(f32, np.float32(np.inf), dtype=np.float32)
        down = np.nextafter(f32, np.float32(-np.inf), dtype=np.float32)
        mid = bf16_midpoint(f32)
        same |= mid & ((g == rne_bf16(up)) | (g == rne_bf16(down)))
    if not same.all():
        i = np.flatnonzero(~same.reshape(-1))[0]
        raise AssertionError(f"{what}: BF16 output {g.reshape(-1)[i]!r} is not the rounding of "
                             f"the FP32 output {float(f32.reshape(-1)[i])!r} (flat index {i}, "
                             f"{int((~same).sum())} such)")
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bound = ulp_bf16(ref) + BF16_GRAD_RMS_FACTOR * REL_L2[policy] * rms
    err = np.abs(g - ref)
    bad = err > bound
    if bad.any():
        i = np.flatnonzero(bad.reshape(-1))[0]
        raise AssertionError(f"{what}: BF16 gradient {g.reshape(-1)[i]!r} vs oracle "
                             f"{ref.reshape(-1)[i]!r} beyond 1 ulp + {BF16_GRAD_RMS_FACTOR} x "
                             f"tol x rms ({int(bad.sum())} such)")


def grads_close(dw, db, ref_dw, ref_db, policy, what, dw_bf16=None, db_bf16=None):
    """FP32 dweight / dbias by rel-L2; the BF16 outputs of a second call of the
    same route (dw_bf16 / db_bf16, optional) by bf16_grad_close. Returns the
    rel-L2 errors."""
    out = {}
    e = rel_l2(dw, ref_dw)
    assert e <= REL_L2[policy], f"{what} dweight rel-L2 {e:.3g} > {REL_L2[policy]}"
    out["dweight_rel_l2"] = e
    if dw_bf16 is not None:
        bf16_grad_close(dw_bf16, dw, ref_dw, policy, f"{what} BF16 dweight")
    if ref_db is not None:
        e = rel_l2(db, ref_db)
        assert e <= REL_L2[policy], f"{what} dbias rel-L2 {e:.3g} > {REL_L2[policy]}"
        out["dbias_rel_l2"] = e
        if db_bf16 is not None:
            bf16_grad_close(db_bf16, db, ref_db, policy, f"{what} BF16 dbias")
    return out
