/*
 * vcd_oracle.c -- plain FP64 CPU oracle for the packed (varlen) width-4
 * depthwise causal convolution + SiLU, training forward and backward.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline /
 * reference legs of the benchmark load this library. The CUDA library shares
 * no code, header, table or helper with it, and neither includes the other.
 *
 * What it computes follows the FlashInfer API pages
 *   F = "flashinfer.cake_causal_conv1d_train.cake_causal_conv1d_train_forward"
 *   B = "flashinfer.cake_causal_conv1d_train.cake_causal_conv1d_train_backward"
 * and is written as the plain definitions, one output element at a time,
 * single-threaded, in double precision:
 *
 *   start(t)      first token of the document holding token t: the documents
 *                 are [cu[i], cu[i+1]); a repeated value is an empty
 *                 document (F, Parameters: cu_seqlens).
 *   xm(t, j)      x[j] if start(t) <= j <= t, else 0: zero history before a
 *                 document's first token (F, Returns).
 *   pre(t,c)      bias[c] + sum_k weight[c,k] * xm(t, t-3+k); weight[c,3]
 *                 multiplies the current token, weight[c,0] the token three
 *                 back (F, Parameters: weight, bias).
 *   y(t,c)        silu(pre) = pre * sigmoid(pre) (F, Returns). The oracle
 *                 returns the unrounded FP64 value.
 *   p(t,c)        the point SiLU' is evaluated at: bf16(pre) under the "bf16"
 *                 policy, pre itself under "fp32" (B, Parameters:
 *                 silu_grad_preactivation). bf16() is round-to-nearest-even.
 *   dpre(t,c)     dy * silu'(p), silu'(p) = s (1 + p (1 - s)), s = sigmoid(p).
 *   dx(t,c)       sum_k weight[c,k] * dpre(t+3-k, c) over t+3-k < S in the
 *                 same document as t (B, Returns; the formula is split over
 *                 two bullets there, read as the adjoint of pre).
 *   dweight[c,k]  sum_t dpre(t,c) * xm(t, t-3+k)   (B, Returns)
 *   dbias[c]      sum_t dpre(t,c)                   (B, Returns)
 *
 * Sums use Neumaier-compensated summation so the FP64 values are exact to a
 * few units of 2^-53 relative to the sum of magnitudes.
 *
 * Besides each y / dx value the oracle can return an ALLOWANCE: a first-order
 * bound on the error that any FP32 evaluation of the same formulas can make
 * (unit roundoff u = 2^-24, transcendental functions accurate to a few u).
 * It only matters where the result cancels (|pre| << sum |terms|) or, under
 * the "bf16" policy, where pre lies within FP32 error of a BF16 rounding
 * midpoint so that bf16(pre) has two defensible values. The tests accept a
 * GPU value g for a reference r when |g - r| <= ulp_bf16(r) + allowance.
 * The constants are stated next to the code that uses them.
 *
 * Inputs: x and dy are raw BF16 bit patterns (uint16, [S, C] row-major);
 * weight [C, 4] and bias [C] are doubles (the caller widens FP32 or BF16
 * values exactly); cu_seqlens is int32 [num_docs + 1].
 *
 * Status codes: 0 ok, 1 invalid argument (bad sizes, malformed cu_seqlens,
 * index out of range).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORC_OK 0
#define ORC_BAD 1

#define POLICY_BF16 0
#define POLICY_FP32 1

/* FP32 unit roundoff used by the allowances. */
static const double U32 = 5.9604644775390625e-08; /* 2^-24 */

/* ---------------------------------------------------------------- BF16 --- */

/* BF16 is the top 16 bits of an IEEE binary32 pattern. */
static double bf16_value(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a double to the nearest BF16 value, ties to even, returned as a
 * double. BF16: 8 significant bits, exponent range of binary32 (normal
 * numbers down to 2^-126, subnormal spacing 2^-133, largest finite value
 * (2 - 2^-7) * 2^127; anything that rounds beyond it is infinite). */
double vcd_oracle_round_bf16(double v) {
    if (v != v || v == 0.0 || isinf(v)) return v;
    double a = fabs(v);
    int e;
    frexp(a, &e);             /* a = m * 2^e, 0.5 <= m < 1 */
    int lead = e - 1;         /* exponent of the leading bit */
    if (lead < -126) lead = -126;
    double spacing = ldexp(1.0, lead - 7);
    double r = nearbyint(a / spacing) * spacing; /* default mode: ties to even */
    if (r >= ldexp(1.0, 128)) r = INFINITY;
    return copysign(r, v);
}

/* ------------------------------------------------------- compensated sum -- */

typedef struct { double s, c; } nsum;

static void nsum_add(nsum* a, double v) {
    double t = a->s + v;
    if (fabs(a->s) >= fabs(v)) a->c += (a->s - t) + v;
    else a->c += (v - t) + a->s;
    a->s = t;
}

static double nsum_get(const nsum* a) { return a->s + a->c; }

/* ---------------------------------------------------------------- SiLU --- */

static double sigmoid(double p) {
    if (p >= 0.0) return 1.0 / (1.0 + exp(-p));
    double e = exp(p);
    return e / (1.0 + e);
}

static double silu(double p) { return p * sigmoid(p); }

/* d/dp [p sigmoid(p)] = s + p s (1 - s), with 1 - s = sigmoid(-p). */
static double silu_grad(double p) {
    double s = sigmoid(p);
    double one_minus_s = sigmoid(-p);
    return s * (1.0 + p * one_minus_s);
}

/* Sum of the magnitudes of the terms of silu_grad's formula; the FP32
 * evaluation error of silu'(p) is bounded relative to it. */
static double silu_grad_mag(double p) {
    double s = sigmoid(p);
    return s * (1.0 + fabs(p) * sigmoid(-p));
}

/* ------------------------------------------------------------- problem --- */

typedef struct {
    int64_t S, C, num_docs;
    const uint16_t* x;
    const uint16_t* dy;   /* may be NULL for forward-only use */
    const double* w;      /* [C][4] */
    const double* b;      /* [C] or NULL */
    const int32_t* cu;    /* [num_docs + 1] */
} problem;

/* cu_seqlens contract (F, Parameters: cu_seqlens): cu[0] == 0,
 * non-decreasing, cu[num_docs] == S. */
static int check_problem(const problem* P) {
    if (P->S < 0 || P->C <= 0 || P->num_docs < 0 || !P->cu || !P->w) return ORC_BAD;
    if (P->S > 0 && !P->x) return ORC_BAD;
    if (P->num_docs == 0) return P->S == 0 ? ORC_OK : ORC_BAD;
    if (P->cu[0] != 0 || (int64_t)P->cu[P->num_docs] != P->S) return ORC_BAD;
    for (int64_t i = 0; i < P->num_docs; ++i)
        if (P->cu[i + 1] < P->cu[i]) return ORC_BAD;
    return ORC_OK;
}

/* First token of the document holding t: cu[i] for the i with
 * cu[i] <= t < cu[i+1] (unique; empty documents never hold a token). */
static int64_t doc_start(const problem* P, int64_t t) {
    int64_t lo = 0, hi = P->num_docs; /* cu[lo] <= t < cu[hi] */
    while (hi - lo > 1) {
        int64_t mid = lo + (hi - lo) / 2;
        if ((int64_t)P->cu[mid] <= t) lo = mid; else hi = mid;
    }
    return P->cu[lo];
}

static double x_at(const problem* P, int64_t t, int64_t c) {
    return bf16_value(P->x[t * P->C + c]);
}

static double dy_at(const problem* P, int64_t t, int64_t c) {
    return bf16_value(P->dy[t * P->C + c]);
}

/* xm(t, j): x[j] when j lies in t's document at or before t, else 0. */
static double xm(const problem* P, int64_t t, int64_t j, int64_t c) {
    if (j < doc_start(P, t) || j > t) return 0.0;
    return x_at(P, j, c);
}

/* pre(t, c) and the sum of the magnitudes of its terms. */
static double pre_at(const problem* P, int64_t t, int64_t c, double* mag) {
    nsum acc = {0.0, 0.0};
    double m = 0.0;
    if (P->b) { nsum_add(&acc, P->b[c]); m += fabs(P->b[c]); }
    for (int k = 0; k < 4; ++k) {
        double term = P->w[c * 4 + k] * xm(P, t, t - 3 + k, c); /* exact in FP64 */
        nsum_add(&acc, term);
        m += fabs(term);
    }
    if (mag) *mag = m;
    return nsum_get(&acc);
}

/* FP32 evaluation error bound of pre: at most 8 roundings (4 products,
 * 4 additions, fused or not) each <= u * sum|terms|; 10 u for margin. */
static double pre_allow(double mag) { return 10.0 * U32 * mag; }

/* Point where SiLU' is evaluated, and the largest change of silu'(p) that an
 * FP32 evaluation of pre can cause (allowance). */
static double policy_point(double pre, double e_pre, int policy, double* dgrad) {
    if (policy == POLICY_FP32) {
        /* |silu''| <= 1/2 everywhere, so an error e in pre moves silu' by
         * at most e / 2. */
        *dgrad = 0.5 * e_pre;
        return pre;
    }
    double p = vcd_oracle_round_bf16(pre);
    double lo = vcd_oracle_round_bf16(pre - e_pre);
    double hi = vcd_oracle_round_bf16(pre + e_pre);
    double g = silu_grad(p), d = 0.0;
    if (lo != p) d = fmax(d, fabs(silu_grad(lo) - g));
    if (hi != p) d = fmax(d, fabs(silu_grad(hi) - g));
    *dgrad = d;
    return p;
}

/* dpre(t, c) and a bound on |FP32 dpre - dpre|. */
static double dpre_at(const problem* P, int64_t t, int64_t c, int policy, double* allow) {
    double mag;
    double pre = pre_at(P, t, c, &mag);
    double e_pre = pre_allow(mag);
    double dgrad;
    double p = policy_point(pre, e_pre, policy, &dgrad);
    double g = dy_at(P, t, c);
    double d = g * silu_grad(p);
    if (allow) {
        /* silu' itself: a few roundings plus approximate exp and reciprocal,
         * (16 + 2|p|) u relative to its magnitude (the 2|p| covers the
         * rounding of the exponent's argument). Then one multiply by dy. */
        double e_grad = (16.0 + 2.0 * fabs(p)) * U32 * silu_grad_mag(p);
        *allow = fabs(g) * (dgrad + e_grad) + 2.0 * U32 * fabs(d);
    }
    return d;
}

/* ------------------------------------------------------------- forward --- */

static int fwd_elem(const problem* P, int64_t t, int64_t c, double* y, double* allow) {
    if (t < 0 || t >= P->S || c < 0 || c >= P->C) return ORC_BAD;
    double mag;
    double pre = pre_at(P, t, c, &mag);
    double v = silu(pre);
    *y = v;
    if (allow) {
        /* |silu'| <= 1.1 carries the pre error; the SiLU evaluation adds
         * (16 + 2|pre|) u relative. */
        *allow = 1.1 * pre_allow(mag) + (16.0 + 2.0 * fabs(pre)) * U32 * fabs(v);
    }
    return ORC_OK;
}

int vcd_oracle_fwd(int64_t S, int64_t C, const uint16_t* x, const double* w, const double* b,
                   const int32_t* cu, int64_t num_docs, double* y, double* y_allow) {
    problem P = {S, C, num_docs, x, NULL, w, b, cu};
    if (check_problem(&P) != ORC_OK || (S > 0 && !y)) return ORC_BAD;
    for (int64_t t = 0; t < S; ++t)
        for (int64_t c = 0; c < C; ++c)
            fwd_elem(&P, t, c, &y[t * C + c], y_allow ? &y_allow[t * C + c] : NULL);
    return ORC_OK;
}

int vcd_oracle_fwd_at(int64_t S, int64_t C, const uint16_t* x, const double* w, const double* b,
                      const int32_t* cu, int64_t num_docs, int64_t n, const int64_t* ts,
                      const int64_t* cs, double* y, double* y_allow) {
    problem P = {S, C, num_docs, x, NULL, w, b, cu};
    if (check_problem(&P) != ORC_OK || n < 0) return ORC_BAD;
    for (int64_t i = 0; i < n; ++i)
        if (fwd_elem(&P, ts[i], cs[i], &y[i], y_allow ? &y_allow[i] : NULL) != ORC_OK)
            return ORC_BAD;
    return ORC_OK;
}

/* ------------------------------------------------------------ backward --- */

static int dx_elem(const problem* P, int64_t t, int64_t c, int policy, double* dx, double* allow) {
    if (t < 0 || t >= P->S || c < 0 || c >= P->C) return ORC_BAD;
    int64_t s = doc_start(P, t);
    nsum acc = {0.0, 0.0};
    double e = 0.0, mag = 0.0;
    for (int k = 0; k < 4; ++k) {
        int64_t j = t + 3 - k;                   /* token whose pre used x[t] via tap k */
        if (j >= P->S || doc_start(P, j) != s) continue;
        double a;
        double d = dpre_at(P, j, c, policy, &a);
        double wk = P->w[c * 4 + k];
        nsum_add(&acc, wk * d);
        e += fabs(wk) * a;
        mag += fabs(wk * d);
    }
    *dx = nsum_get(&acc);
    /* dpre errors carried through the taps, plus the 4-term FP32 sum. */
    if (allow) *allow = e + 8.0 * U32 * mag;
    return ORC_OK;
}

/* dweight [4] and dbias of channel c; with non-NULL mag4 / magb also the sums
 * of the magnitudes of their terms, sum_t |dpre * xm| and sum_t |dpre|. */
static int params_channel(const problem* P, int64_t c, int policy, double* dw4, double* db,
                          double* mag4, double* magb) {
    if (c < 0 || c >= P->C) return ORC_BAD;
    nsum acc[4] = {{0, 0}, {0, 0}, {0, 0}, {0, 0}};
    nsum accb = {0.0, 0.0};
    double m[4] = {0, 0, 0, 0}, mb = 0.0;
    for (int64_t t = 0; t < P->S; ++t) {
        double d = dpre_at(P, t, c, policy, NULL);
        for (int k = 0; k < 4; ++k) {
            double term = d * xm(P, t, t - 3 + k, c);
            nsum_add(&acc[k], term);
            m[k] += fabs(term);
        }
        nsum_add(&accb, d);
        mb += fabs(d);
    }
    for (int k = 0; k < 4; ++k) {
        dw4[k] = nsum_get(&acc[k]);
        if (mag4) mag4[k] = m[k];
    }
    if (db) *db = nsum_get(&accb);
    if (magb) *magb = mb;
    return ORC_OK;
}

static int check_bwd(const problem* P, int policy) {
    if (check_problem(P) != ORC_OK) return ORC_BAD;
    if (P->S > 0 && !P->dy) return ORC_BAD;
    if (policy != POLICY_BF16 && policy != POLICY_FP32) return ORC_BAD;
    return ORC_OK;
}

/* Full backward: dx [S, C] (+ allowance), dweight [C, 4], dbias [C]
 * (dbias may be NULL), and optionally the magnitude sums of the gradients'
 * terms (dweight_mag [C, 4], dbias_mag [C]; NULL to skip). S == 0 gives zero
 * gradients (B, Returns). */
int vcd_oracle_bwd(int64_t S, int64_t C, const uint16_t* x, const uint16_t* dy, const double* w,
                   const double* b, const int32_t* cu, int64_t num_docs, int policy, double* dx,
                   double* dx_allow, double* dweight, double* dbias, double* dweight_mag,
                   double* dbias_mag) {
    problem P = {S, C, num_docs, x, dy, w, b, cu};
    if (check_bwd(&P, policy) != ORC_OK || !dweight || (S > 0 && !dx)) return ORC_BAD;
    for (int64_t t = 0; t < S; ++t)
        for (int64_t c = 0; c < C; ++c)
            dx_elem(&P, t, c, policy, &dx[t * C + c], dx_allow ? &dx_allow[t * C + c] : NULL);
    for (int64_t c = 0; c < C; ++c)
        params_channel(&P, c, policy, &dweight[c * 4], dbias ? &dbias[c] : NULL,
                       dweight_mag ? &dweight_mag[c * 4] : NULL, dbias_mag ? &dbias_mag[c] : NULL);
    return ORC_OK;
}

int vcd_oracle_bwd_dx_at(int64_t S, int64_t C, const uint16_t* x, const uint16_t* dy,
                         const double* w, const double* b, const int32_t* cu, int64_t num_docs,
                         int policy, int64_t n, const int64_t* ts, const int64_t* cs, double* dx,
                         double* dx_allow) {
    problem P = {S, C, num_docs, x, dy, w, b, cu};
    if (check_bwd(&P, policy) != ORC_OK || n < 0) return ORC_BAD;
    for (int64_t i = 0; i < n; ++i)
        if (dx_elem(&P, ts[i], cs[i], policy, &dx[i], dx_allow ? &dx_allow[i] : NULL) != ORC_OK)
            return ORC_BAD;
    return ORC_OK;
}

/* dweight / dbias for a list of channels: dweight [n, 4], dbias [n], and
 * optionally their magnitude sums (same shapes; NULL to skip). */
int vcd_oracle_bwd_params_at(int64_t S, int64_t C, const uint16_t* x, const uint16_t* dy,
                             const double* w, const double* b, const int32_t* cu,
                             int64_t num_docs, int policy, int64_t n, const int64_t* cs,
                             double* dweight, double* dbias, double* dweight_mag,
                             double* dbias_mag) {
    problem P = {S, C, num_docs, x, dy, w, b, cu};
    if (check_bwd(&P, policy) != ORC_OK || n < 0) return ORC_BAD;
    for (int64_t i = 0; i < n; ++i)
        if (params_channel(&P, cs[i], policy, &dweight[i * 4], dbias ? &dbias[i] : NULL,
                           dweight_mag ? &dweight_mag[i * 4] : NULL,
                           dbias_mag ? &dbias_mag[i] : NULL) != ORC_OK)
            return ORC_BAD;
    return ORC_OK;
}

/* Scalar entry points so the tests can pin SiLU and SiLU' against closed
 * forms and a library routine. */
double vcd_oracle_silu(double p) { return silu(p); }
double vcd_oracle_silu_grad(double p) { return silu_grad(p); }
