"""Comparison rules between the CUDA library and the FP64 oracle.

* BF16 outputs (y, dx, BF16 dweight / dbias): |g - r| <= ulp_bf16(r) + allowance,
  where the allowance is the oracle's bound on FP32 evaluation error (zero for
  well-conditioned elements). The strict fraction (allowance 0) is reported.
* FP32 dweight / dbias: rel-L2 against the oracle of the same SiLU' policy,
  5e-5 under "bf16" and 5e-7 under "fp32" (the pages state about 3e-5 and 2e-7).
* BF16 dweight / dbias: 1 ulp plus the worst-case error of summing n = S terms
  in FP32 in any order, (n - 1) u sum|term| with u = 2^-24 (the classical bound
  for recursive summation); it only matters for entries that nearly cancel.
"""
import numpy as np

REL_L2 = {"bf16": 5e-5, "fp32": 5e-7}


def ulp_bf16(r):
    a = np.abs(np.asarray(r, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126.0), -126.0)
    return np.exp2(e - 7.0)


def bf16_close(gpu, ref, allow, what):
    """Assert the BF16 rule; returns the strict 1-ulp pass fraction."""
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
    return float(np.mean(err <= ulp))


def rel_l2(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(gpu - ref) / (den if den > 0 else 1.0))


U32 = 2.0 ** -24


def grads_close(dw, db, ref_dw, ref_db, policy, bf16_out_w, bf16_out_b, what, mag_dw=None,
                mag_db=None, n_terms=0):
    """FP32 outputs by rel-L2, BF16 outputs by the 1-ulp rule (+ summation bound)."""
    out = {}
    sum_allow = lambda m: None if m is None else max(n_terms - 1, 0) * U32 * np.asarray(m)
    if bf16_out_w:
        out["dweight_strict"] = bf16_close(dw, ref_dw, sum_allow(mag_dw), f"{what} dweight")
    else:
        e = rel_l2(dw, ref_dw)
        assert e <= REL_L2[policy], f"{what} dweight rel-L2 {e:.3g} > {REL_L2[policy]}"
        out["dweight_rel_l2"] = e
    if ref_db is not None:
        if bf16_out_b:
            out["dbias_strict"] = bf16_close(db, ref_db, sum_allow(mag_db), f"{what} dbias")
        else:
            e = rel_l2(db, ref_db)
            assert e <= REL_L2[policy], f"{what} dbias rel-L2 {e:.3g} > {REL_L2[policy]}"
            out["dbias_rel_l2"] = e
    return out
