// vcd_dfloat.cuh -- "double-float" arithmetic: a value held as the
// unevaluated sum hi + lo of two FP32 numbers (|lo| at most half an ulp of
// hi), about 48 significant bits, from FP32 operations and the error-free
// transformations of Knuth (two-sum) and Dekker (two-product, here one FMA).
//
// The exactness-guarded backward recomputes the few dx elements whose FP32
// value it cannot certify; those need SiLU' and the four-term sum well beyond
// FP32 accuracy. FP64 would give that, but runs at a small fraction of FP32's
// rate on GB300, so the recomputation uses these FP32 pairs instead.
#pragma once
#include <stdint.h>

namespace vcd {

struct dfloat {
    float hi, lo;
};

__device__ __forceinline__ dfloat df_of(float v) { return {v, 0.0f}; }

// a + b = s + e exactly (any magnitudes).
__device__ __forceinline__ dfloat df_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bv = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bv)), __fsub_rn(b, bv));
    return {s, e};
}

// a + b = s + e exactly, for |a| >= |b| (or a == 0).
__device__ __forceinline__ dfloat df_fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// a b = p + e exactly (barring underflow).
__device__ __forceinline__ dfloat df_two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ dfloat df_neg(dfloat a) { return {-a.hi, -a.lo}; }

// a + b with both parts' errors carried (relative error about 2^-47).
__device__ __forceinline__ dfloat df_add(dfloat a, dfloat b) {
    dfloat s = df_two_sum(a.hi, b.hi);
    const dfloat t = df_two_sum(a.lo, b.lo);
    s.lo = __fadd_rn(s.lo, t.hi);
    s = df_fast_two_sum(s.hi, s.lo);
    s.lo = __fadd_rn(s.lo, t.lo);
    return df_fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ dfloat df_mul(dfloat a, dfloat b) {
    dfloat p = df_two_prod(a.hi, b.hi);
    p.lo = __fmaf_rn(a.hi, b.lo, p.lo);
    p.lo = __fmaf_rn(a.lo, b.hi, p.lo);
    return df_fast_two_sum(p.hi, p.lo);
}

__device__ __forceinline__ dfloat df_mul_f(dfloat a, float b) {
    dfloat p = df_two_prod(a.hi, b);
    p.lo = __fmaf_rn(a.lo, b, p.lo);
    return df_fast_two_sum(p.hi, p.lo);
}

// 1 / d for d in [1, 2]: the FP32 reciprocal and one Newton step r + r (1 - d r)
// carried out in pairs (doubles the 24 correct bits).
__device__ __forceinline__ dfloat df_recip(dfloat d) {
    const float r0 = __frcp_rn(d.hi);
    const dfloat e = df_add(df_of(1.0f), df_neg(df_mul_f(d, r0)));
    return df_add(df_of(r0), df_mul_f(e, r0));
}

// ln 2 in three FP32 parts: kDfLn2A has 17 significant bits, so k kDfLn2A is
// exact for |k| < 128; the three sum to ln 2 within 2^-69.
constexpr float kDfLn2A = 0x1.62e4p-1f;
constexpr float kDfLn2B = 0x1.7f7d1cp-20f;
constexpr float kDfLn2C = 0x1.ef357ap-45f;
constexpr float kDfInvLn2 = 0x1.715476p+0f;

// 1/n! for n = 0..12 as FP32 pairs (hi, lo), hi the nearest float.
__device__ __forceinline__ dfloat df_inv_factorial(int n) {
    switch (n) {
        case 0: case 1: return {1.0f, 0.0f};
        case 2: return {0x1p-1f, 0.0f};
        case 3: return {0x1.555556p-3f, -0x1.555556p-28f};
        case 4: return {0x1.555556p-5f, -0x1.555556p-30f};
        case 5: return {0x1.111112p-7f, -0x1.ddddde0p-32f};
        case 6: return {0x1.6c16c2p-10f, -0x1.27d27ep-35f};
        case 7: return {0x1.a01a02p-13f, -0x1.7f97fap-39f};
        case 8: return {0x1.a01a02p-16f, -0x1.7f97fap-42f};
        case 9: return {0x1.71de3ap-19f, 0x1.55b1ccp-45f};
        case 10: return {0x1.27e4fcp-22f, -0x1.10ec14p-47f};
        case 11: return {0x1.ae6456p-26f, 0x1.fd5138p-52f};
        default: return {0x1.1eed8ep-29f, 0x1.ff1b12p-54f};
    }
}

// e^y for -87 <= y <= 0: y = k ln 2 + r with |r| <= ln(2)/2 (r in pairs,
// ln 2 in three parts), e^r from its Taylor series to r^12 (truncation below
// 2^-52), scaled by 2^k. Relative error about 2^-46.
__device__ __forceinline__ dfloat df_exp_nonpos(dfloat y) {
    const float kf = rintf(__fmul_rn(y.hi, kDfInvLn2));
    const float r0 = __fmaf_rn(-kf, kDfLn2A, y.hi);                  // exact (Sterbenz)
    dfloat r = df_two_sum(r0, y.lo);
    r = df_add(r, df_neg(df_two_prod(kf, kDfLn2B)));
    r = df_add(r, df_of(-__fmul_rn(kf, kDfLn2C)));
    dfloat poly = df_inv_factorial(12);
#pragma unroll
    for (int n = 11; n >= 0; --n) poly = df_add(df_mul(poly, r), df_inv_factorial(n));
    const int k = (int)kf;
    return {ldexpf(poly.hi, k), ldexpf(poly.lo, k)};
}

// silu'(p) = s (1 + p (1 - s)), s = sigmoid(p), with e = e^-|p| <= 1 so that
// both s and 1 - s come out of 1 / (1 + e) without cancellation: for p >= 0,
// s = 1 / (1 + e) and 1 - s = e / (1 + e); for p < 0 the other way round.
// Relative error about 2^-44 (absolute where silu' crosses zero near
// p = -1.28). For |p| > 87, e^-|p| is below FP32's range and taken as 0.
__device__ __forceinline__ dfloat df_silu_grad(dfloat p) {
    const bool neg = p.hi < 0.0f;
    const dfloat ap = neg ? df_neg(p) : p;
    const dfloat e = ap.hi > 87.0f ? df_of(0.0f) : df_exp_nonpos(df_neg(ap));
    const dfloat r = df_recip(df_add(df_of(1.0f), e));
    const dfloat er = df_mul(e, r);
    const dfloat s = neg ? er : r;
    const dfloat oms = neg ? r : er;
    return df_mul(s, df_add(df_of(1.0f), df_mul(p, oms)));
}

}  // namespace vcd
