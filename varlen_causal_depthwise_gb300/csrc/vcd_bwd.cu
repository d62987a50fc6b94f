// vcd_bwd.cu -- backward of the packed width-4 depthwise causal convolution +
// SiLU (FlashInfer page "cake_causal_conv1d_train_backward", description,
// Parameters: silu_grad_preactivation, Returns):
//
//   pre      recomputed in FP32 from x (nothing but x, weight, cu_seqlens and
//            bias is saved by the forward)
//   p        bf16(pre) under the "bf16" policy, pre under "fp32"
//   dpre     dy * silu'(p), FP32
//   dx[t]    bf16(sum_k w[k] dpre[t + 3 - k]) over the same document
//   dw[k]    sum_t dpre[t] x[t - 3 + k]  (zero history)
//   db       sum_t dpre[t]
//
// Main kernel: one warp per chunk of work units (32 * kBwdVec channels x L
// tokens each, vcd_plan.h), walking its tokens forward once, in one of three
// launch shapes picked per call (12 warps per SM with up to 168 registers a
// thread, 16 warps with 128, or 12 warps with shared memory for the "fp32"
// policy's compensated chunk sums; BwdGeom below). x and dy stream through a
// per-warp shared-memory ring of kBwdNs stages: one lane issues two 2D
// tensor-map copies (TMA) per batch of kBwdU tokens onto the stage's
// mbarrier, kBwdNs - 1 batches ahead. Registers hold the x of the three
// previous tokens and their dpre, so each token gives pre, dpre, its dweight /
// dbias products, and dx of the token three back in gather form:
//   dx[t-3] = w3 dpre[t-3] + w2 dpre[t-2] + w1 dpre[t-1] + w0 dpre[t].
// A batch without a document start in positions q-2 .. q+U-1 (one bit mask
// per batch from cu_seqlens) takes a mask-free path; otherwise each term is
// predicated on "no document start in between". The unit reads x over
// [begin-3, end+3) and dy over [begin, end+3), writes dx over [begin, end),
// and keeps dweight / dbias in registers; at its end each lane writes its
// channels' five FP32 sums into the chunk's partial row (or folds them into
// the chunk's compensated sums). HBM traffic: 6 bytes per element.
//
// Reduce kernel: launched with programmatic stream serialization, it waits on
// griddepcontrol for the main kernel and sums the partial rows of each channel
// in a fixed order (FP32, or compensated FP32 pairs under the "fp32" policy),
// so the gradients are bitwise reproducible for a given (S, C) and route.
//
// The exactness-guarded route (conv1d_bwd_exact) runs the main kernel with
// EXACT = true and a third kernel that recomputes the listed dx elements.
#include <atomic>

#include <cuda_runtime.h>
#include <stdint.h>

#include "vcd_device.cuh"
#include "vcd_dfloat.cuh"
#include "vcd_kernels.h"
#include "vcd_plan.h"

namespace vcd {
namespace {

#ifndef VCD_BWD_PACKED
#define VCD_BWD_PACKED 0
#endif
#ifndef VCD_BWD_PACKED_ACC
#define VCD_BWD_PACKED_ACC 0
#endif
constexpr bool kPK = VCD_BWD_PACKED != 0;                 // packed FP32x2 arithmetic
constexpr bool kPA = kPK || VCD_BWD_PACKED_ACC != 0;      // ... for dweight / dbias / dx
constexpr int kNP = kBwdVec / 2;                          // channel pairs per lane
constexpr int kBwdColCh = 32 * kBwdVec;                   // channels per unit column
constexpr int kBwdRowBytes = 2 * kBwdColCh;               // bytes of a token's row segment

// Geometry of a launch shape (vcd_plan.h): warps per CTA (one CTA per SM),
// ring stages and tokens per batch.
template <int SHAPE> struct BwdGeom;
template <> struct BwdGeom<kBwdWide> { static constexpr int kWarps = 12, kNs = 3, kU = 12; };
template <> struct BwdGeom<kBwdDeep> { static constexpr int kWarps = 16, kNs = 2, kU = 8; };
template <> struct BwdGeom<kBwdChunked> { static constexpr int kWarps = 12, kNs = 3, kU = 8; };
template <int SHAPE> struct BwdShapeT : BwdGeom<SHAPE> {
    using G = BwdGeom<SHAPE>;
    static constexpr int kThreads = 32 * G::kWarps;
    static constexpr int kTensorBytes = G::kU * kBwdRowBytes;   // one tensor's rows of one stage
    static constexpr int kStageBytes = 2 * kTensorBytes;        // x rows, then dy rows
    static constexpr int kWarpBytes = G::kNs * kStageBytes;
    static constexpr int kSmemBytes = G::kWarps * kWarpBytes;
    static_assert(G::kU % 2 == 0 && G::kU <= 30 && G::kNs >= 2, "batch geometry");
    static_assert(kSmemBytes <= 227 * 1024, "ring exceeds the shared memory of one CTA");
    static_assert(kBwdShapeWarps[SHAPE] == G::kWarps, "plan and kernel disagree on the shape");
    // Chunks of several units (SEG): each lane's compensated chunk sums, hi
    // and lo of its 5 * kBwdVec values, after the rings ([warp][value][lane]).
    static constexpr int kAccFloats = 2 * kPartialStride * kBwdVec;
    static constexpr int kAccBytes = G::kWarps * kAccFloats * 32 * 4;
    // the TMA ring's barriers: one 8-byte mbarrier per stage of each warp
    static constexpr int kBarBytes = G::kWarps * G::kNs * 8;
    template <bool SEG> static constexpr int smem_bytes() {
        return kSmemBytes + (SEG ? kAccBytes : 0) + kBarBytes;
    }
};
// Units of several per chunk are the "fp32" policy's, a multiple of
// kFp32UnitAlign tokens long (vcd_plan.h); a multiple of the batch puts every
// unit boundary at the same position of a batch.
static_assert(kFp32UnitAlign % BwdGeom<kBwdChunked>::kU == 0, "unit boundaries must align");
static_assert(BwdShapeT<kBwdChunked>::smem_bytes<true>() <= 227 * 1024, "accumulators do not fit");
static_assert(BwdShapeT<kBwdWide>::smem_bytes<false>() <= 227 * 1024, "ring and barriers do not fit");



// Set when a kernel gave up waiting on a TMA tile (mbar_wait_bounded); the
// outputs of that call are then incomplete. Never set in normal operation;
// conv1d_wait_fault() reads it.
__device__ int g_vcd_wait_fault = 0;

constexpr int kPolicyBF16 = 0;
constexpr int kPolicyFP32 = 1;

__device__ __forceinline__ bool bit(uint32_t m, int i) { return (m >> i) & 1u; }

template <int POLICY, bool PK = kPK>
__device__ __forceinline__ float2 grad_at(float2 pre) {
    if (POLICY == kPolicyBF16) return silu_grad2<PK>(round_bf16x2(pre));
    return silu_grad2_accurate(pre);
}

// SEG: a warp's chunk holds several units (the "fp32" policy's short units),
// whose sums it adds into compensated accumulators in shared memory at each
// unit boundary; the chunk writes one partial row. Without SEG every chunk is
// a single unit, the unit-boundary logic compiles away, and the unit's
// register sums are its row.
// EXACT: the exactness-guarded route (conv1d_bwd_exact), every batch through
// one predicated path with checks (below); instantiated with BIAS =
// kRouteRuntime (dtypes read at run time).
constexpr float kU24 = 0x1p-24f;                  // FP32 unit roundoff
constexpr float kExactScale = 0x1p-11f;           // magnitudes are kept scaled by this
// Absolute error bound of silu_grad_accurate_nc (about 12 2^-24 for every
// p), with margin.
constexpr float kExactGradErr = 0x1p-24f * 24.0f;
// A dx whose FP32 value v is within 2^-9 |v| of the exact value rounds to
// BF16 within one ulp of it (|v| < 2^8 ulp(v), so the rounding's half ulp
// plus 2^-9 |v| stays below one ulp); larger error bounds are recomputed.
constexpr float kExactAccept = 0x1p-9f;

// The transposed narrow column (vcd_plan.h, narrow_plan): assignment k of
// that column. Lane gi + g s (g = the column's four-channel groups) takes
// group gi of piece s % h of chunk k q + s / h, a stretch of P tokens that it
// walks alone: its own copies of x and dy (8-byte cp.async into its bytes of
// the warp's ring, the layout of a full column's stage), its own cu_seqlens
// cursor, and every token through one branch-free path (the main loop's
// arithmetic, each term selected by operand). At the end the lanes of a
// chunk's later pieces hand their five FP32 sums per channel to the chunk's
// first piece, which adds them in piece order (compensated when the chunk
// holds several units, the "fp32" policy's) and writes the chunk's partial
// row. Out of line: the main loop's register allocation stays as it is.
template <int SHAPE, bool W_BF16, int BIAS, int POLICY>
__device__ __noinline__ void bwd_narrow(const BwdArgs& a, int64_t k, uint32_t ring_s,
                                        const unsigned char* ring, int lane) {
    using SH = BwdShapeT<SHAPE>;
    constexpr int kU = SH::kU, kNs = SH::kNs;
    const int64_t S = a.plan.S, C = a.plan.C;
    const int g = (int)a.plan.ng, h = (int)a.plan.h, nq = (int)a.plan.q;
    const int gi = lane % g, s = lane / g;
    const int64_t chunk = k * nq + s / h;
    const int piece = s % h;
    const bool valid = s < nq * h && chunk < a.plan.chunks;
    const int64_t c0 = a.plan.nfull * kBwdColCh + gi * kBwdVec;
    const int64_t span = a.plan.per * a.plan.L;                 // tokens of a chunk
    const int64_t P = (span + h - 1) / h;                       // of a piece
    int64_t t0 = 0, t1 = 0;
    if (valid) {
        const int64_t cs = chunk * span, ce = cs + span < S ? cs + span : S;
        t0 = cs + piece * P < ce ? cs + piece * P : ce;
        t1 = t0 + P < ce ? t0 + P : ce;
    }
    // relative tokens r (token q0 + r), as in the main loop: dweight and dx
    // for r in [3, r_end); x read over [q0, t_du), dy over [t0, t_du) (dpre
    // of the three tokens after the piece enters its last dx)
    const int64_t q0 = t0 - 3;
    const int64_t t_du = valid ? (t1 + 3 < S ? t1 + 3 : S) : 0;
    const int r_end = (int)(t1 - q0);
    const int nb = (int)((P + 6 + kU - 1) / kU);                // warp-uniform
    const bool with_bias = BIAS == kRouteRuntime ? a.bias_kind != kBiasNone : BIAS != kBiasNone;
    const int32_t* __restrict__ cu = a.cu_seqlens;
    const int ncu = (int)(a.num_docs + 1);

    const unsigned char* const xg = static_cast<const unsigned char*>(a.x) + (q0 * C + c0) * 2;
    const unsigned char* const gg = static_cast<const unsigned char*>(a.dy) + (q0 * C + c0) * 2;
    const int64_t rowb = C * 2;
    auto issue = [&](int i, int slot) {
        if (i < nb) {
            const uint32_t st = ring_s + slot * SH::kStageBytes + lane * (2 * kBwdVec);
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                const int r = i * kU + j;
                const int64_t t = q0 + r;
                const bool okx = valid && t >= 0 && t < t_du;
                const bool okg = okx && r >= 3;
                const int64_t off = (int64_t)r * rowb;
                cp_async8(st + j * kBwdRowBytes, okx ? xg + off : a.x, okx);
                cp_async8(st + SH::kTensorBytes + j * kBwdRowBytes, okg ? gg + off : a.dy, okg);
            }
        }
        cp_async_commit();
    };
    __syncwarp();                        // the previous assignment's reads of the ring are done
#pragma unroll
    for (int i = 0; i < kNs - 1; ++i) issue(i, i);

    float2 w[4][kNP], b[kNP];
    if constexpr (BIAS == kRouteRuntime)
        load_taps_rt(a.weight, a.bias, a.weight_bf16 != 0, a.bias_kind, c0, valid, w, b);
    else
        load_taps<W_BF16, BIAS, kNP>(a.weight, a.bias, c0, valid, w, b);
    LaneDocs doc;
    doc.init(cu, ncu, (int)q0 - 2);
    uint32_t carry = doc.starts(cu, ncu, (int)q0 - 2, 2);               // bits of q0-2, q0-1

    float2 xc[3][kNP], dc[3][kNP], dw[4][kNP], db[kNP];
#pragma unroll
    for (int p = 0; p < kNP; ++p) {
#pragma unroll
        for (int j = 0; j < 3; ++j) xc[j][p] = dc[j][p] = zero2();
#pragma unroll
        for (int j = 0; j < 4; ++j) dw[j][p] = zero2();
        db[p] = zero2();
    }
    __nv_bfloat16* dxq = static_cast<__nv_bfloat16*>(a.dx) + (q0 - 3) * C + c0;   // token q0 - 3

    int slot = 0;
    for (int i = 0; i < nb; ++i) {
        cp_async_wait<kNs - 2>();        // this lane's copies of batch i have landed
        __syncwarp();
        issue(i + kNs - 1, slot == 0 ? kNs - 1 : slot - 1);
        const int r0 = i * kU;
        const uint32_t nw = doc.starts(cu, ncu, (int)(q0 + r0), kU);
        const uint32_t M = carry | (nw << 2);                            // bit i <-> token q - 2 + i
        carry = nw >> (kU - 2);
        const unsigned char* sx = ring + slot * SH::kStageBytes + lane * (2 * kBwdVec);
        const unsigned char* sg = sx + SH::kTensorBytes;
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            const int r = r0 + j;
            uint32_t xv[kNP], gv[kNP], o[kNP];
            lds_pairs<kBwdVec>(sx + j * kBwdRowBytes, xv);
            lds_pairs<kBwdVec>(sg + j * kBwdRowBytes, gv);
            // The lanes' masks differ (each walks its own tokens), so every
            // term is selected by operand, never branched around: a term
            // outside the document or the piece multiplies a selected zero
            // (same values as skipping it, whatever the excluded x or dy
            // holds). dy is zero-filled outside [t0, t_du), so dpre there is 0.
            const bool m1 = !bit(M, j + 2);
            const bool m2 = m1 && !bit(M, j + 1);
            const bool m3 = m2 && !bit(M, j);
            const bool k1 = !bit(M, j);
            const bool k2 = k1 && !bit(M, j + 1);
            const bool k3 = k2 && !bit(M, j + 2);
            const bool acc = r >= 3 && r < r_end;
            const bool emit = r >= 6 && r - 3 < r_end;
#pragma unroll
            for (int p = 0; p < kNP; ++p) {
                const float2 xf = bf16x2_to_float2(xv[p]);
                const float2 gf = bf16x2_to_float2(gv[p]);
                const float2 x0 = m3 ? xc[0][p] : zero2();
                const float2 x1 = m2 ? xc[1][p] : zero2();
                const float2 x2 = m1 ? xc[2][p] : zero2();
                float2 pre = fma2<true>(w[0][p], x0, b[p]);
                pre = fma2<true>(w[1][p], x1, pre);
                pre = fma2<true>(w[2][p], x2, pre);
                pre = fma2<true>(w[3][p], xf, pre);
                const float2 d = mul2<true>(gf, grad_at<POLICY, true>(pre));
                const float2 da = acc ? d : zero2();
                dw[0][p] = fma2<true>(da, x0, dw[0][p]);
                dw[1][p] = fma2<true>(da, x1, dw[1][p]);
                dw[2][p] = fma2<true>(da, x2, dw[2][p]);
                dw[3][p] = fma2<true>(da, xf, dw[3][p]);
                if (with_bias) db[p] = add2<true>(db[p], da);
                const float2 e1 = k1 ? dc[1][p] : zero2();
                const float2 e2 = k2 ? dc[2][p] : zero2();
                const float2 e3 = k3 ? d : zero2();
                float2 gsum = mul2<true>(w[3][p], dc[0][p]);
                gsum = fma2<true>(w[2][p], e1, gsum);
                gsum = fma2<true>(w[1][p], e2, gsum);
                gsum = fma2<true>(w[0][p], e3, gsum);
                o[p] = float2_to_bf16x2(gsum);
                xc[0][p] = xc[1][p];
                xc[1][p] = xc[2][p];
                xc[2][p] = xf;
                dc[0][p] = dc[1][p];
                dc[1][p] = dc[2][p];
                dc[2][p] = d;
            }
            if (emit) st_pairs<kBwdVec>(dxq + (int64_t)r * C, o);
        }
        slot = slot + 1 == kNs ? 0 : slot + 1;
    }
    cp_async_wait<0>();                  // nothing in flight into the ring past this point

    // The chunk's row: pieces 1 .. h-1 (lanes lane + g, lane + 2g, ...) added
    // into piece 0's sums in piece order. Units of the "fp32" policy's chunks
    // go through a compensated sum, as the main loop's chunks do.
    const bool comp = a.plan.per > 1;
    float own[kPartialStride * kBwdVec], hi[kPartialStride * kBwdVec], lo[kPartialStride * kBwdVec];
#pragma unroll
    for (int f = 0; f < kPartialStride * kBwdVec; ++f) {
        const int ch = f / kPartialStride, kk = f % kPartialStride;
        const float2 v = kk < 4 ? dw[kk][ch / 2] : db[ch / 2];
        own[f] = hi[f] = (ch & 1) ? v.y : v.x;
        lo[f] = 0.0f;
    }
    for (int j = 1; j < h; ++j) {
        const int src = lane + j * g < 32 ? lane + j * g : lane;
#pragma unroll
        for (int f = 0; f < kPartialStride * kBwdVec; ++f) {
            const float v = __shfl_sync(kFull, own[f], src);
            if (comp) acc_two_sum(hi[f], lo[f], v);
            else hi[f] = __fadd_rn(hi[f], v);
        }
    }
    if (valid && piece == 0) {
        float2* dst = reinterpret_cast<float2*>(
            a.partials + ((chunk * a.plan.ncols + a.plan.nfull) * kBwdColCh + gi * kBwdVec) * kPartialStride);
#pragma unroll
        for (int f = 0; f < kPartialStride * kBwdVec / 2; ++f)
            dst[f] = make_float2(__fadd_rn(hi[2 * f], lo[2 * f]), __fadd_rn(hi[2 * f + 1], lo[2 * f + 1]));
    }
}

// NARROW: the plan transposes the last column (a.plan.nnarrow > 0); its
// assignments run bwd_narrow. A separate instantiation, so that the other
// kernels' register allocation does not carry that path.
template <int SHAPE, bool W_BF16, int BIAS, int POLICY, bool SEG, bool EXACT = false, bool NARROW = false>
__global__ void __launch_bounds__(BwdShapeT<SHAPE>::kThreads, 1)
    bwd_main_kernel(const __grid_constant__ BwdArgs a) {
    using SH = BwdShapeT<SHAPE>;
    constexpr int kBwdU = SH::kU, kBwdNs = SH::kNs;
    constexpr int kBwdTensorBytes = SH::kTensorBytes, kBwdStageBytes = SH::kStageBytes;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    unsigned char* const ring = smem + wid * SH::kWarpBytes;
    const uint32_t ring_s = smem_u32(ring);
    const int64_t warp0 = (int64_t)blockIdx.x * SH::kWarps + wid;
    const int64_t nwarps = (int64_t)gridDim.x * SH::kWarps;
    const int64_t S = a.plan.S, C = a.plan.C, L = a.plan.L;
    const int64_t ncols = a.plan.ncols;
    __nv_bfloat16* __restrict__ dx = static_cast<__nv_bfloat16*>(a.dx);
    const int32_t* __restrict__ cu = a.cu_seqlens;
    const int ncu = (int)(a.num_docs + 1);
    const int Ci = (int)C;                               // row stride, elements
    const bool with_bias = BIAS == kRouteRuntime ? a.bias_kind != kBiasNone : BIAS != kBiasNone;
    // The mask-free path in packed FP32x2 instructions (two channels per
    // instruction, the same rounding as two scalar ones, so the same bits)
    // where that is faster, measured: the chunked shape and the deep shape
    // without a bias (large fp32 2313 -> 2244 us, mid 80 -> 76 us); the wide
    // shape and the masked paths run slower packed (register pressure).
    constexpr bool kFastPk = kPK || SHAPE == kBwdChunked || (SHAPE == kBwdDeep && BIAS == kBiasNone);
    constexpr bool kFastPa = kPA || kFastPk;

    // Assignment. Each column's units are cut into chunks of `per` consecutive
    // units (the plan's, from constants), and a warp streams a whole chunk as
    // one segment: a pipeline restart happens per chunk, not per unit. Chunks
    // are dealt row-major (consecutive warps take consecutive columns of the
    // same chunk), so warps running side by side read whole token rows. Chunk
    // (chunk, col) owns partial row chunk * ncols + col, whichever warp
    // computes it. Without SEG every chunk is one unit.
    const int64_t rows = a.plan.rows;
    const int64_t per = SEG ? a.plan.per : 1;
    const int64_t nfull = NARROW ? a.plan.nfull : ncols;
    const int64_t n_full_asg = nfull * a.plan.chunks;           // then the transposed column's
    const int64_t n_asg = NARROW ? n_full_asg + a.plan.nnarrow : n_full_asg;
    float* const acc = reinterpret_cast<float*>(smem + SH::kSmemBytes) +
                       wid * SH::kAccFloats * 32 + lane;        // SEG: [value][lane] of this warp
    // TMA ring: this warp's stage barriers, initialised once (one arrival per
    // phase: the producer lane's expect_tx); phase parities in `phases`.
    const uint32_t bars = smem_u32(smem + SH::kSmemBytes + (SEG ? SH::kAccBytes : 0)) +
                          wid * kBwdNs * 8;
    uint32_t phases = 0;
    bool fault = false;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kBwdNs; ++s) mbar_init(bars + 8 * s, 1);
        mbar_init_fence();
    }
    __syncwarp();
    for (int64_t asg = warp0; asg < n_asg; asg += nwarps) {
        // The transposed column's assignments sit evenly spaced among the
        // others (one in `stride`), so that no SM holds more than one of
        // their warps: their lanes' scattered 8-byte copies and stores load
        // the SM's L1 several times more per token than a full column's.
        int64_t fa = asg;                                        // full-column assignment
        if constexpr (NARROW) {
            const int64_t nn = a.plan.nnarrow, stride = n_asg / nn;
            const int64_t ks = asg / stride;
            if (asg % stride == 0 && ks < nn) {
                bwd_narrow<SHAPE, W_BF16, BIAS, POLICY>(a, ks, ring_s, ring, lane);
                continue;
            }
            fa = asg - (ks + 1 < nn ? ks + 1 : nn);
        }
        const int64_t col = fa % nfull, chunk = fa / nfull;
        const int64_t row0 = chunk * per;
        const int64_t row1 = !SEG ? row0 + 1 : row0 + per < rows ? row0 + per : rows;
        const int64_t c0 = col * kBwdColCh + lane * kBwdVec;
        const bool active = c0 < C;
        const int64_t t_begin = row0 * L;
        const int64_t t_end = row1 * L < S ? row1 * L : S;
        const int64_t u_end = t_end + 3 < S ? t_end + 3 : S;     // dpre needed below u_end
        const int64_t q0 = t_begin - 3;                          // 3 warm-up tokens
        // relative token indices (token q0 + r): outputs and dweight for r in
        // [3, r_end), dpre for r in [3, r_du), batches while r - 3 < r_end;
        // unit row0 + k starts at r = 3 + k L
        const int r_end = (int)(t_end - q0);
        const int r_du = (int)(u_end - q0);
        const int nb = (r_end + 3 + kBwdU - 1) / kBwdU;
        const int Li = (int)L;
        int r_next = SEG && row1 - row0 > 1 ? 3 + Li : INT_MAX;   // where the next unit starts

        // The first batches' copies go out before the taps and the document
        // lookup, whose dependent loads then overlap them.

        __syncwarp();                    // the previous unit's reads of the ring are done
        auto issue = [&](int i, int slot) {
            // Tiles of tokens q0 + i U .. + U - 1 x the column's 128 channels
            // (rows outside [0, S) and channels past C arrive as zeros; the
            // x and dy rows outside what the unit uses are never read).
            if (i < nb && lane == 0) {
                const uint32_t st = ring_s + slot * kBwdStageBytes, bar = bars + 8 * slot;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, kBwdStageBytes);
                const int c = (int)(col * kBwdColCh), t = (int)q0 + i * kBwdU;
                tma_load_2d(st, &a.tmap_x, c, t, bar);
                tma_load_2d(st + kBwdTensorBytes, &a.tmap_dy, c, t, bar);
            }
        };
#pragma unroll
        for (int s = 0; s < kBwdNs - 1; ++s) issue(s, s);

        float2 w[4][kNP], b[kNP];
        if constexpr (BIAS == kRouteRuntime)
            load_taps_rt(a.weight, a.bias, a.weight_bf16 != 0, a.bias_kind, c0, active, w, b);
        else
            load_taps<W_BF16, BIAS, kNP>(a.weight, a.bias, c0, active, w, b);
        DocCursor doc;
        doc.init(cu, ncu, (int)q0 - 2, lane);
        uint32_t carry = doc.starts(cu, ncu, (int)q0 - 2, 2, lane);            // bits of q0-2, q0-1

        float2 xc[3][kNP], dc[3][kNP];    // x and dpre of tokens q-3, q-2, q-1
        float2 dw[4][kNP], db[kNP];       // this unit's FP32 sums
        float2 ec[3][kNP];                // EXACT: bounds on the error of those dpre
        uint32_t xn = 0;                  // EXACT: this chunk's listed elements (warp-uniform)
        uint64_t* const xlist = EXACT ? a.xlist + asg * a.xcap : nullptr;
#pragma unroll
        for (int p = 0; p < kNP; ++p) {
#pragma unroll
            for (int k = 0; k < 3; ++k) xc[k][p] = dc[k][p] = ec[k][p] = zero2();
#pragma unroll
            for (int k = 0; k < 4; ++k) dw[k][p] = zero2();
            db[p] = zero2();
        }

        // This lane's sums in row order: channel c0 + i's five values at
        // 5 i .. 5 i + 4 (dweight taps 0..3, dbias).
        auto sum_at = [&](int f) -> float {
            const int ch = f / kPartialStride, k = f % kPartialStride;
            const float2 v = k < 4 ? dw[k][ch / 2] : db[ch / 2];
            return (ch & 1) ? v.y : v.x;
        };
        auto clear_sums = [&]() {
#pragma unroll
            for (int p = 0; p < kNP; ++p) {
#pragma unroll
                for (int k = 0; k < 4; ++k) dw[k][p] = zero2();
                db[p] = zero2();
            }
        };
        // SEG: the finished unit's sums into the chunk's accumulators.
        auto fold_unit = [&]() {
#pragma unroll
            for (int f = 0; f < kPartialStride * kBwdVec; ++f)
                acc_two_sum(acc[(2 * f) * 32], acc[(2 * f + 1) * 32], sum_at(f));
            clear_sums();
        };
        if (SEG) {
#pragma unroll
            for (int f = 0; f < SH::kAccFloats; ++f) acc[f * 32] = 0.0f;
        }
        // Write the chunk's partial row ([kBwdColCh channels][5] FP32; this
        // lane's kBwdVec channels are 5 * kBwdVec consecutive floats): the
        // register sums of its one unit, or the rounded compensated sums.
        auto write_row = [&]() {
            if (SEG) fold_unit();
            if (active) {
                float2* dst = reinterpret_cast<float2*>(
                    a.partials + ((chunk * ncols + col) * kBwdColCh + lane * kBwdVec) * kPartialStride);
#pragma unroll
                for (int i = 0; i < kBwdVec * kPartialStride / 2; ++i) {
                    float v[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int f = 2 * i + h;
                        v[h] = SEG ? __fadd_rn(acc[(2 * f) * 32], acc[(2 * f + 1) * 32]) : sum_at(f);
                    }
                    dst[i] = make_float2(v[0], v[1]);
                }
            }
            if (!SEG) clear_sums();
            if (EXACT && lane == 0) a.xcount[asg] = xn;
        };
        // SEG: token r (at position 3 of its batch) starts the next unit.
        auto unit_boundary = [&](int r) {
            if (SEG && r == r_next) {
                fold_unit();
                r_next = r_next + Li < r_end ? r_next + Li : INT_MAX;
            }
        };

        // EXACT: one token of the guarded route. As the general path, plus:
        //  - "bf16" policy: a preactivation within its FP32 error bound
        //    (4 2^-24 mag, mag = the magnitude of its terms) of a BF16
        //    rounding midpoint is summed exactly before it is rounded, so p
        //    is the rounding of the exact preactivation;
        //  - SiLU' by the accurate, cancellation-free evaluation for both
        //    policies;
        //  - a bound on each dpre's error (e: SiLU' evaluation kExactGradErr
        //    times |dy|, the product's rounding, and under "fp32" the
        //    preactivation's error times max|silu''| = 1/2) and on dx's:
        //    sum |w| e + 5 2^-24 sum |w dpre|. A dx whose bound exceeds
        //    kExactAccept of its value goes to the chunk's list (its BF16
        //    rounding might miss the 1-ulp bound) and is recomputed afterwards
        //    in double-float arithmetic.
        auto exact_token = [&](int r, const uint32_t (&xv)[kNP], const uint32_t (&gv)[kNP], bool m1,
                               bool m2, bool m3, bool k1, bool k2, bool k3, bool has_d, bool acc,
                               bool emit, uint32_t (&o)[kNP]) {
            float2 pre[kNP], mag[kNP], xf[kNP], gf[kNP];
            uint32_t flip = 0;                       // bit 2p + h: preactivation needs its exact sum
#pragma unroll
            for (int p = 0; p < kNP; ++p) {
                xf[p] = bf16x2_to_float2(xv[p]);
                gf[p] = bf16x2_to_float2(gv[p]);
                const float2 xs[4] = {xc[0][p], xc[1][p], xc[2][p], xf[p]};
                const bool on[4] = {m3, m2, m1, true};
                pre[p] = b[p];
                mag[p] = make_float2(fabsf(b[p].x) * kExactScale, fabsf(b[p].y) * kExactScale);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (!on[k]) continue;
                    pre[p] = fma2<false>(w[k][p], xs[k], pre[p]);
                    mag[p].x = __fmaf_rn(fabsf(w[k][p].x) * kExactScale, fabsf(xs[k].x), mag[p].x);
                    mag[p].y = __fmaf_rn(fabsf(w[k][p].y) * kExactScale, fabsf(xs[k].y), mag[p].y);
                }
                if (POLICY == kPolicyBF16 && has_d) {
                    // |pre - midpoint of its BF16 interval| (exact: Sterbenz) vs 4 2^-24 mag
                    const float e_pre[2] = {mag[p].x * kExactScale, mag[p].y * kExactScale};
                    const float pv[2] = {pre[p].x, pre[p].y};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float mid = __uint_as_float((__float_as_uint(pv[h]) & 0xffff0000u) | 0x8000u);
                        if (fabsf(__fsub_rn(pv[h], mid)) <= e_pre[h]) flip |= 1u << (2 * p + h);
                    }
                }
            }
            float2 pt[kNP];                           // the point SiLU' is taken at
#pragma unroll
            for (int p = 0; p < kNP; ++p) pt[p] = POLICY == kPolicyBF16 ? round_bf16x2(pre[p]) : pre[p];
            if (POLICY == kPolicyBF16 && __any_sync(kFull, flip != 0)) {
#pragma unroll
                for (int e = 0; e < 2 * kNP; ++e) {
                    if (!((flip >> e) & 1u)) continue;
                    const int p = e >> 1;
                    const bool hi = e & 1;
                    const float wk[4] = {hi ? w[0][p].y : w[0][p].x, hi ? w[1][p].y : w[1][p].x,
                                         hi ? w[2][p].y : w[2][p].x, hi ? w[3][p].y : w[3][p].x};
                    const float xk[4] = {hi ? xc[0][p].y : xc[0][p].x, hi ? xc[1][p].y : xc[1][p].x,
                                         hi ? xc[2][p].y : xc[2][p].x, hi ? xf[p].y : xf[p].x};
                    const bool on[4] = {m3, m2, m1, true};
                    const double pe = exact_preactivation(hi ? b[p].y : b[p].x, wk, xk, on);
                    const float pr = __bfloat162float(__double2bfloat16(pe));
                    if (hi) pt[p].y = pr; else pt[p].x = pr;
                }
            }
            uint32_t doubt = 0;                       // bit 2p + h: dx of channel 2p + h is listed
#pragma unroll
            for (int p = 0; p < kNP; ++p) {
                float2 d = zero2(), ed = zero2();
                if (has_d) {
                    const float2 g = make_float2(silu_grad_accurate_nc(pt[p].x),
                                                 silu_grad_accurate_nc(pt[p].y));
                    d = mul2<false>(gf[p], g);
                    ed.x = __fmaf_rn(fabsf(gf[p].x), kExactGradErr, kU24 * fabsf(d.x));
                    ed.y = __fmaf_rn(fabsf(gf[p].y), kExactGradErr, kU24 * fabsf(d.y));
                    if (POLICY == kPolicyFP32) {          // |silu''| <= 1/2 times 4 2^-24 mag
                        ed.x = __fmaf_rn(fabsf(gf[p].x), mag[p].x * (0.5f * kExactScale), ed.x);
                        ed.y = __fmaf_rn(fabsf(gf[p].y), mag[p].y * (0.5f * kExactScale), ed.y);
                    }
                }
                if (acc) {
                    if (m3) dw[0][p] = fma2<kPA>(d, xc[0][p], dw[0][p]);
                    if (m2) dw[1][p] = fma2<kPA>(d, xc[1][p], dw[1][p]);
                    if (m1) dw[2][p] = fma2<kPA>(d, xc[2][p], dw[2][p]);
                    dw[3][p] = fma2<kPA>(d, xf[p], dw[3][p]);
                    if (with_bias) db[p] = add2<kPA>(db[p], d);
                }
                float2 g = mul2<kPA>(w[3][p], dc[0][p]);
                if (k1) g = fma2<kPA>(w[2][p], dc[1][p], g);
                if (k2) g = fma2<kPA>(w[1][p], dc[2][p], g);
                if (k3) g = fma2<kPA>(w[0][p], d, g);
                o[p] = float2_to_bf16x2(g);
                // error bound of this dx: the dpre errors carried by |w|, and
                // 5 roundings' worth of the terms' magnitude
                const float2 ds[4] = {dc[0][p], dc[1][p], dc[2][p], d};
                const float2 es[4] = {ec[0][p], ec[1][p], ec[2][p], ed};
                const bool in[4] = {true, k1, k2, k3};
                const int tap[4] = {3, 2, 1, 0};
                float ex = 0.0f, ey = 0.0f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (!in[i]) continue;
                    const float2 aw = make_float2(fabsf(w[tap[i]][p].x), fabsf(w[tap[i]][p].y));
                    ex = __fmaf_rn(aw.x, __fmaf_rn(5.0f * kU24, fabsf(ds[i].x), es[i].x), ex);
                    ey = __fmaf_rn(aw.y, __fmaf_rn(5.0f * kU24, fabsf(ds[i].y), es[i].y), ey);
                }
                if (emit && ex > kExactAccept * fabsf(g.x)) doubt |= 1u << (2 * p);
                if (emit && ey > kExactAccept * fabsf(g.y)) doubt |= 2u << (2 * p);
                xc[0][p] = xc[1][p];
                xc[1][p] = xc[2][p];
                xc[2][p] = xf[p];
                dc[0][p] = dc[1][p];
                dc[1][p] = dc[2][p];
                dc[2][p] = d;
                ec[0][p] = ec[1][p];
                ec[1][p] = ec[2][p];
                ec[2][p] = ed;
            }
            if (__any_sync(kFull, doubt != 0)) {
                // list dx[t - 3] of the doubtful channels, warp-aggregated
                const uint32_t below = (1u << lane) - 1u;
                const uint64_t t3 = (uint64_t)(q0 + r - 3);      // the token whose dx this is
#pragma unroll
                for (int e = 0; e < 2 * kNP; ++e) {
                    const bool mine = (doubt >> e) & 1u;
                    const uint32_t bal = __ballot_sync(kFull, mine);
                    if (bal == 0) continue;
                    const uint32_t pos = xn + __popc(bal & below);
                    if (mine && pos < (uint32_t)a.xcap)
                        xlist[pos] = (t3 << 32) | (uint64_t)(c0 + e);
                    xn += __popc(bal);
                }
            }
        };

        __nv_bfloat16* dxp = dx + (q0 - 3) * C + c0;   // dx row of relative token -3
        const int64_t dstep = C;

        int slot = 0;
        for (int i = 0; i < nb; ++i) {
            if (!mbar_wait_bounded(bars + 8 * slot, (phases >> slot) & 1u)) {
                fault = true;
                break;
            }
            phases ^= 1u << slot;
            __syncwarp();
            issue(i + kBwdNs - 1, slot == 0 ? kBwdNs - 1 : slot - 1);
            const int r0 = i * kBwdU;
            const int64_t q = q0 + r0;
            const uint32_t nw = doc.starts(cu, ncu, (int)q, kBwdU, lane);
            __nv_bfloat16* dxq = dxp + (int64_t)r0 * dstep;  // dx row of token q - 3
            const uint32_t M = carry | (nw << 2);            // bit i <-> token q - 2 + i
            carry = nw >> (kBwdU - 2);
            const unsigned char* sx = ring + slot * kBwdStageBytes + lane * (2 * kBwdVec);
            const unsigned char* sg = sx + kBwdTensorBytes;

            // an interior batch: every token accumulates and emits dx three
            // tokens back (a unit boundary, if any, is at position 3)
            const bool interior = r0 >= 6 && r0 + kBwdU <= r_end;
            if constexpr (EXACT) {
                // not unrolled: the guarded body is long, and kBwdU copies of
                // it overflow the instruction cache (measured)
#pragma unroll 1
                for (int j = 0; j < kBwdU; ++j) {
                    const int r = r0 + j;
                    if (j == 3) unit_boundary(r);
                    uint32_t xv[kNP], gv[kNP], o[kNP];
                    lds_pairs<kBwdVec>(sx + j * kBwdRowBytes, xv);
                    lds_pairs<kBwdVec>(sg + j * kBwdRowBytes, gv);
                    const bool m1 = !bit(M, j + 2);
                    const bool m2 = m1 && !bit(M, j + 1);
                    const bool m3 = m2 && !bit(M, j);
                    const bool k1 = !bit(M, j);
                    const bool k2 = k1 && !bit(M, j + 1);
                    const bool k3 = k2 && !bit(M, j + 2);
                    const bool has_d = r >= 3 && r < r_du;
                    const bool acc = r >= 3 && r < r_end;
                    const bool emit = active && r >= 6 && r - 3 < r_end;
                    exact_token(r, xv, gv, m1, m2, m3, k1, k2, k3, has_d, acc, emit, o);
                    if (emit) st_pairs<kBwdVec>(dxq + j * Ci, o);
                }
            } else if (M == 0 && interior) {
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    if (j == 3) unit_boundary(r0 + j);
                    uint32_t xv[kNP], gv[kNP], o[kNP];
                    lds_pairs<kBwdVec>(sx + j * kBwdRowBytes, xv);
                    lds_pairs<kBwdVec>(sg + j * kBwdRowBytes, gv);
#pragma unroll
                    for (int p = 0; p < kNP; ++p) {
                        const float2 xf = bf16x2_to_float2(xv[p]);
                        const float2 gf = bf16x2_to_float2(gv[p]);
                        float2 pre = fma2<kFastPk>(w[0][p], xc[0][p], b[p]);
                        pre = fma2<kFastPk>(w[1][p], xc[1][p], pre);
                        pre = fma2<kFastPk>(w[2][p], xc[2][p], pre);
                        pre = fma2<kFastPk>(w[3][p], xf, pre);
                        const float2 d = mul2<kFastPk>(gf, grad_at<POLICY, kFastPk>(pre));
                        dw[0][p] = fma2<kFastPa>(d, xc[0][p], dw[0][p]);
                        dw[1][p] = fma2<kFastPa>(d, xc[1][p], dw[1][p]);
                        dw[2][p] = fma2<kFastPa>(d, xc[2][p], dw[2][p]);
                        dw[3][p] = fma2<kFastPa>(d, xf, dw[3][p]);
                        if (with_bias) db[p] = add2<kFastPa>(db[p], d);
                        float2 g = mul2<kFastPa>(w[3][p], dc[0][p]);
                        g = fma2<kFastPa>(w[2][p], dc[1][p], g);
                        g = fma2<kFastPa>(w[1][p], dc[2][p], g);
                        g = fma2<kFastPa>(w[0][p], d, g);
                        o[p] = float2_to_bf16x2(g);
                        xc[0][p] = xc[1][p];
                        xc[1][p] = xc[2][p];
                        xc[2][p] = xf;
                        dc[0][p] = dc[1][p];
                        dc[1][p] = dc[2][p];
                        dc[2][p] = d;
                    }
                    if (active) st_pairs<kBwdVec>(dxq + j * Ci, o);
                }
            } else if (SHAPE != kBwdWide && interior) {
                // Document starts inside: bit i of N1 / N2 / N3 is set when no
                // document starts at bit i / at bits i, i+1 / at bits i..i+2
                // of M, so each term's predicate is one bit of one mask. (The
                // wide shape runs long documents only, and leaves its rare
                // batches with a start to the general path below: a third
                // copy of the loop makes its kernels spill.)
                const uint32_t N1 = ~M, N2 = ~(M | (M >> 1)), N3 = ~(M | (M >> 1) | (M >> 2));
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    if (j == 3) unit_boundary(r0 + j);
                    uint32_t xv[kNP], gv[kNP], o[kNP];
                    lds_pairs<kBwdVec>(sx + j * kBwdRowBytes, xv);
                    lds_pairs<kBwdVec>(sg + j * kBwdRowBytes, gv);
                    // tap k of token t sees x[t-3+k] iff no start in (t-3+k, t];
                    // dx[t-3] sees dpre[t-3+i] iff no start in (t-3, t-3+i]
                    const bool m1 = bit(N1, j + 2), m2 = bit(N2, j + 1), m3 = bit(N3, j);
                    const bool k1 = bit(N1, j), k2 = bit(N2, j);
#pragma unroll
                    for (int p = 0; p < kNP; ++p) {
                        const float2 xf = bf16x2_to_float2(xv[p]);
                        const float2 gf = bf16x2_to_float2(gv[p]);
                        float2 pre = b[p];
                        if (m3) pre = fma2<kPK>(w[0][p], xc[0][p], pre);
                        if (m2) pre = fma2<kPK>(w[1][p], xc[1][p], pre);
                        if (m1) pre = fma2<kPK>(w[2][p], xc[2][p], pre);
                        pre = fma2<kPK>(w[3][p], xf, pre);
                        const float2 d = mul2<kPK>(gf, grad_at<POLICY>(pre));
                        if (m3) dw[0][p] = fma2<kPA>(d, xc[0][p], dw[0][p]);
                        if (m2) dw[1][p] = fma2<kPA>(d, xc[1][p], dw[1][p]);
                        if (m1) dw[2][p] = fma2<kPA>(d, xc[2][p], dw[2][p]);
                        dw[3][p] = fma2<kPA>(d, xf, dw[3][p]);
                        if (with_bias) db[p] = add2<kPA>(db[p], d);
                        float2 g = mul2<kPA>(w[3][p], dc[0][p]);
                        if (k1) g = fma2<kPA>(w[2][p], dc[1][p], g);
                        if (k2) g = fma2<kPA>(w[1][p], dc[2][p], g);
                        if (m3) g = fma2<kPA>(w[0][p], d, g);
                        o[p] = float2_to_bf16x2(g);
                        xc[0][p] = xc[1][p];
                        xc[1][p] = xc[2][p];
                        xc[2][p] = xf;
                        dc[0][p] = dc[1][p];
                        dc[1][p] = dc[2][p];
                        dc[2][p] = d;
                    }
                    if (active) st_pairs<kBwdVec>(dxq + j * Ci, o);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int r = r0 + j;
                    if (j == 3) unit_boundary(r);
                    uint32_t xv[kNP], gv[kNP], o[kNP];
                    lds_pairs<kBwdVec>(sx + j * kBwdRowBytes, xv);
                    lds_pairs<kBwdVec>(sg + j * kBwdRowBytes, gv);
                    // tap k of token t sees x[t-3+k] iff no start in (t-3+k, t]
                    const bool m1 = !bit(M, j + 2);
                    const bool m2 = m1 && !bit(M, j + 1);
                    const bool m3 = m2 && !bit(M, j);
                    // dx[t-3] sees dpre[t-3+i] iff no start in (t-3, t-3+i]
                    const bool k1 = !bit(M, j);
                    const bool k2 = k1 && !bit(M, j + 1);
                    const bool k3 = k2 && !bit(M, j + 2);
                    const bool has_d = r >= 3 && r < r_du;
                    const bool acc = r >= 3 && r < r_end;
                    const bool emit = active && r >= 6 && r - 3 < r_end;
#pragma unroll
                    for (int p = 0; p < kNP; ++p) {
                        const float2 xf = bf16x2_to_float2(xv[p]);
                        const float2 gf = bf16x2_to_float2(gv[p]);
                        float2 pre = b[p];
                        if (m3) pre = fma2<kPK>(w[0][p], xc[0][p], pre);
                        if (m2) pre = fma2<kPK>(w[1][p], xc[1][p], pre);
                        if (m1) pre = fma2<kPK>(w[2][p], xc[2][p], pre);
                        pre = fma2<kPK>(w[3][p], xf, pre);
                        float2 d = zero2();
                        if (has_d) d = mul2<kPK>(gf, grad_at<POLICY>(pre));
                        if (acc) {
                            if (m3) dw[0][p] = fma2<kPA>(d, xc[0][p], dw[0][p]);
                            if (m2) dw[1][p] = fma2<kPA>(d, xc[1][p], dw[1][p]);
                            if (m1) dw[2][p] = fma2<kPA>(d, xc[2][p], dw[2][p]);
                            dw[3][p] = fma2<kPA>(d, xf, dw[3][p]);
                            if (with_bias) db[p] = add2<kPA>(db[p], d);
                        }
                        float2 g = mul2<kPA>(w[3][p], dc[0][p]);
                        if (k1) g = fma2<kPA>(w[2][p], dc[1][p], g);
                        if (k2) g = fma2<kPA>(w[1][p], dc[2][p], g);
                        if (k3) g = fma2<kPA>(w[0][p], d, g);
                        o[p] = float2_to_bf16x2(g);
                        xc[0][p] = xc[1][p];
                        xc[1][p] = xc[2][p];
                        xc[2][p] = xf;
                        dc[0][p] = dc[1][p];
                        dc[1][p] = dc[2][p];
                        dc[2][p] = d;
                    }
                    if (emit) st_pairs<kBwdVec>(dxq + j * Ci, o);
                }
            }
            slot = slot + 1 == kBwdNs ? 0 : slot + 1;
        }

        if (fault) break;
        write_row();
    }
    if (fault) {
        // A tile never arrived: flag it, and give the stages still in flight
        // a bounded wait of their own before the warp leaves, so that no copy
        // lands in shared memory the CTA has released.
        if (lane == 0) atomicExch(&g_vcd_wait_fault, 1);
#pragma unroll
        for (int s = 0; s < kBwdNs; ++s) mbar_wait_bounded(bars + 8 * s, (phases >> s) & 1u);
    }
    // Let the reduce kernel's CTAs be scheduled; its griddepcontrol.wait still
    // waits for this whole grid to finish and its writes to be visible.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- reduce ---

// The value hi + lo (|lo| at most half an ulp of hi, hi = fl(hi + lo)) in
// BF16, rounded to nearest-even as the exact sum would be: hi's own rounding
// unless hi lies exactly halfway between two BF16 values and lo decides the
// side.
__device__ __forceinline__ __nv_bfloat16 pair_to_bf16(float hi, float lo) {
    const uint32_t u = __float_as_uint(hi);
    if ((u & 0xffffu) != 0x8000u || lo == 0.0f) return __float2bfloat16_rn(hi);
    const bool away = (lo > 0.0f) == (hi > 0.0f);            // the sum's magnitude exceeds |hi|
    const uint32_t r = away ? (u & 0xffff0000u) + 0x10000u : (u & 0xffff0000u);
    return __ushort_as_bfloat16((unsigned short)(r >> 16));
}

// Reduce: output (channel c, value k) is the sum over the R chunk rows of its
// column. A CTA handles 32 outputs with n threads each (n = red_slices(R)):
// thread s sums the fixed row slice [s R / n, (s + 1) R / n) in row order,
// then thread 0 of the output adds the n slice sums in slice order. The order
// depends on R only, so the result is bitwise reproducible per (S, C, route).
// n grows with R (at least 8 rows a slice, at most 16 slices) so that each
// thread's chain of dependent loads stays short.
// COMP (the "fp32" policy): every addition is compensated (two-sum into a
// hi / lo pair), so the total is the rows' exact sum to about R 2^-48
// relative to the sum of their magnitudes before its one final rounding --
// what an FP64 accumulator would give, at FP32 rates (FP64 arithmetic runs at
// a small fraction of FP32's on GB300).
constexpr int kRedOutputs = 32;
constexpr int kRedMaxSlices = 16;

inline int red_slices(int64_t rows) {
    int n = 1;
    while (n < kRedMaxSlices && rows >= 8 * (int64_t)n) n *= 2;
    return n;
}

template <bool COMP>
__global__ void __launch_bounds__(kRedOutputs * kRedMaxSlices, 4) bwd_reduce_kernel(const BwdArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float part_hi[kRedMaxSlices][kRedOutputs];
    __shared__ float part_lo[kRedMaxSlices][kRedOutputs];
    const BwdPlan& P = a.plan;
    const int nsl = blockDim.x / kRedOutputs;
    const int o = threadIdx.x % kRedOutputs;          // consecutive threads: consecutive outputs
    const int sl = threadIdx.x / kRedOutputs;
    const int64_t idx = (int64_t)blockIdx.x * kRedOutputs + o;
    const bool valid = idx < P.C * kPartialStride;
    const int64_t c = valid ? idx / kPartialStride : 0;
    const int k = (int)(idx % kPartialStride);
    const int64_t col = c / kBwdColCh, ci = c % kBwdColCh;
    const float* src = a.partials + (col * kBwdColCh + ci) * kPartialStride + k;
    const int64_t stride = P.ncols * kBwdColCh * kPartialStride;
    const int64_t R = P.chunks;
    const int64_t r0 = R * sl / nsl, r1 = R * (sl + 1) / nsl;
    float hi = 0.0f, lo = 0.0f;
    const bool wanted = valid && !(k == 4 && a.dbias == nullptr);
    if (wanted) {
        // batches of 8 independent loads; rows past r1 read nothing and add
        // zero, which leaves every sum and its order unchanged
        const int n = (int)(r1 - r0);
        const float* q = src + r0 * stride;
        for (int r = 0; r < n; r += 8) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[j] = r + j < n ? __ldcg(q) : 0.0f;
                q += stride;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (COMP) acc_two_sum(hi, lo, v[j]);
                else hi += v[j];
            }
        }
    }
    part_hi[sl][o] = hi;
    part_lo[sl][o] = lo;
    __syncthreads();
    if (sl != 0 || !wanted) return;
    hi = part_hi[0][o];
    lo = part_lo[0][o];
    for (int j = 1; j < nsl; ++j) {
        if (COMP) {
            acc_two_sum(hi, lo, part_hi[j][o]);
            lo = __fadd_rn(lo, part_lo[j][o]);
        } else {
            hi += part_hi[j][o];
        }
    }
    void* base = k < 4 ? a.dweight : a.dbias;
    const int64_t at = k < 4 ? c * 4 + k : c;
    const bool bf16 = (k < 4 ? a.dweight_bf16 : a.dbias_bf16) != 0;
    if (COMP) {
        // normalise: s = fl(hi + lo) and the exact remainder e
        const float s = __fadd_rn(hi, lo);
        const float bv = __fsub_rn(s, hi);
        const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bv)), __fsub_rn(lo, bv));
        if (bf16) reinterpret_cast<__nv_bfloat16*>(base)[at] = pair_to_bf16(s, e);
        else reinterpret_cast<float*>(base)[at] = s;
    } else {
        if (bf16) reinterpret_cast<__nv_bfloat16*>(base)[at] = __float2bfloat16_rn(hi);
        else reinterpret_cast<float*>(base)[at] = hi;
    }
}

// ------------------------------------------------------- exact fix-up ---

// The document holding t: its first token s0 (the last cu_seqlens entry
// <= t) and the first token past t where another document starts (the first
// entry > t; no such entry: S). Token j > t is in t's document iff j < next.
// Clamped so that a malformed array cannot send a read out of range.
__device__ void doc_of(const int32_t* __restrict__ cu, int ncu, int64_t t, int64_t S, int64_t& s0,
                       int64_t& next) {
    int lo = 0, hi = ncu;                                   // cu[lo] <= t < cu[hi] when sorted
    while (hi - lo > 1) {
        const int mid = lo + (hi - lo) / 2;
        if ((int64_t)__ldg(cu + mid) <= t) lo = mid; else hi = mid;
    }
    const int64_t s = __ldg(cu + lo);
    s0 = s < 0 ? 0 : s > t ? t : s;
    const int64_t n = hi < ncu ? (int64_t)__ldg(cu + hi) : S;
    next = n > t ? n : t + 1;
}

__device__ float param_at(const void* base, bool bf16, int64_t i) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
    return reinterpret_cast<const float*>(base)[i];
}

// dx[t, c] of the policy from the inputs, to about 2^-44 before its one
// rounding to BF16: each preactivation summed exactly (exact_preactivation),
// SiLU' at the policy's point in double-float arithmetic, the products with
// dy and the weights and the four-term sum in double-float.
__device__ __nv_bfloat16 dx_exact(const BwdArgs& a, int64_t t, int64_t c) {
    const int64_t S = a.plan.S, C = a.plan.C;
    const int32_t* cu = a.cu_seqlens;
    const int ncu = (int)(a.num_docs + 1);
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    const __nv_bfloat16* dy = static_cast<const __nv_bfloat16*>(a.dy);
    const bool wb = a.weight_bf16 != 0;
    float wk[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) wk[k] = param_at(a.weight, wb, c * 4 + k);
    const float bias = a.bias_kind == kBiasNone ? 0.0f : param_at(a.bias, a.bias_kind == kBiasBF16, c);
    int64_t s0, next;
    doc_of(cu, ncu, t, S, s0, next);
    dfloat acc = df_of(0.0f);
    for (int k = 0; k < 4; ++k) {
        const int64_t j = t + 3 - k;                         // the token whose pre used x[t] via tap k
        if (j >= S || j >= next) continue;                   // past the end, or in a later document
        float xs[4];
        bool on[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int64_t i = j - 3 + m;
            on[m] = i >= s0;
            xs[m] = on[m] ? __bfloat162float(x[i * C + c]) : 0.0f;
        }
        const double pre = exact_preactivation(bias, wk, xs, on);
        dfloat p;
        if (a.policy == kPolicyBF16) {
            p = df_of(__bfloat162float(__double2bfloat16(pre)));
        } else {
            p.hi = (float)pre;
            p.lo = (float)(pre - (double)p.hi);
        }
        const dfloat dpre = df_mul_f(df_silu_grad(p), __bfloat162float(dy[j * C + c]));
        acc = df_add(acc, df_mul_f(dpre, wk[k]));
    }
    return pair_to_bf16(acc.hi, acc.lo);
}

// Recomputes the dx elements the guarded main kernel listed, one list (one
// chunk of one column) per CTA; a list that overflowed its room means every
// element of its chunk.
__global__ void __launch_bounds__(256) bwd_exact_fixup_kernel(const BwdArgs a) {
    const BwdPlan& P = a.plan;
    const int64_t lists = P.ncols * P.chunks;
    __nv_bfloat16* dx = static_cast<__nv_bfloat16*>(a.dx);
    for (int64_t id = blockIdx.x; id < lists; id += gridDim.x) {
        const uint32_t n = a.xcount[id];
        if (n <= (uint64_t)a.xcap) {
            const uint64_t* list = a.xlist + id * a.xcap;
            for (uint32_t e = threadIdx.x; e < n; e += blockDim.x) {
                const uint64_t v = list[e];
                const int64_t t = (int64_t)(v >> 32), c = (int64_t)(v & 0xffffffffu);
                if (t < P.S && c < P.C) dx[t * P.C + c] = dx_exact(a, t, c);
            }
        } else {
            const int64_t col = id % P.ncols, chunk = id / P.ncols;
            const int64_t r0 = chunk * P.per, r1 = r0 + P.per < P.rows ? r0 + P.per : P.rows;
            const int64_t t0 = r0 * P.L, t1 = r1 * P.L < P.S ? r1 * P.L : P.S;
            const int64_t c0 = col * kBwdColCh;
            const int64_t nc = P.C - c0 < kBwdColCh ? P.C - c0 : kBwdColCh;
            for (int64_t e = threadIdx.x; e < (t1 - t0) * nc; e += blockDim.x) {
                const int64_t t = t0 + e / nc, c = c0 + e % nc;
                dx[t * P.C + c] = dx_exact(a, t, c);
            }
        }
    }
}

// -------------------------------------------------------------- launch ---

template <int SHAPE, bool W_BF16, int BIAS, int POLICY, bool SEG, bool EXACT = false, bool NARROW = false>
int prepare_main_t() {
    // Once per (instantiation, device): allow the dynamic shared memory and
    // read the occupancy; both are host-side queries. The cache entries are
    // atomic (host threads may get here at once; each stores the same value).
    using SH = BwdShapeT<SHAPE>;
    constexpr int kSmem = SH::template smem_bytes<SEG>();
    static std::atomic<int> occ[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    const int known = occ[dev].load(std::memory_order_relaxed);
    if (known > 0) return known;
    if (cudaFuncSetAttribute(bwd_main_kernel<SHAPE, W_BF16, BIAS, POLICY, SEG, EXACT, NARROW>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, bwd_main_kernel<SHAPE, W_BF16, BIAS, POLICY, SEG, EXACT, NARROW>,
                                                      SH::kThreads, kSmem) != cudaSuccess)
        return 0;
    occ[dev].store(n, std::memory_order_relaxed);
    return n;
}

template <int SHAPE, bool W_BF16, int BIAS, int POLICY, bool SEG, bool EXACT = false, bool NARROW = false>
cudaError_t launch_main_form(const BwdArgs& a, int sm_count, cudaStream_t stream) {
    using SH = BwdShapeT<SHAPE>;
    if ((a.plan.nnarrow > 0) != NARROW) return cudaErrorInvalidValue;
    const int occ = prepare_main_t<SHAPE, W_BF16, BIAS, POLICY, SEG, EXACT, NARROW>();
    if (occ <= 0) return cudaErrorInvalidConfiguration;
    const int64_t n_asg = a.plan.nfull * a.plan.chunks + a.plan.nnarrow;
    const int64_t ctas_needed = (n_asg + SH::kWarps - 1) / SH::kWarps;
    const int64_t resident = (int64_t)sm_count * occ;
    const int64_t grid = ctas_needed < resident ? ctas_needed : resident;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(grid > 0 ? grid : 1));
    cfg.blockDim = dim3(SH::kThreads);
    cfg.dynamicSmemBytes = SH::template smem_bytes<SEG>();
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, bwd_main_kernel<SHAPE, W_BF16, BIAS, POLICY, SEG, EXACT, NARROW>, a);
}

// Chunks of several units come only from the "fp32" policy, which runs the
// chunked shape; every other route has one unit per chunk.
// Plans with the transposed narrow column take the NARROW instantiations.
template <int SHAPE, bool W_BF16, int BIAS, int POLICY>
cudaError_t launch_main_t(const BwdArgs& a, int sm_count, cudaStream_t stream) {
    const bool narrow = a.plan.nnarrow > 0;
    if constexpr (SHAPE != kBwdWide && POLICY == kPolicyFP32) {
        if (a.plan.per > 1)
            return narrow ? launch_main_form<SHAPE, W_BF16, BIAS, POLICY, true, false, true>(a, sm_count, stream)
                          : launch_main_form<SHAPE, W_BF16, BIAS, POLICY, true>(a, sm_count, stream);
    }
    if (a.plan.per > 1) return cudaErrorInvalidValue;
    return narrow ? launch_main_form<SHAPE, W_BF16, BIAS, POLICY, false, false, true>(a, sm_count, stream)
                  : launch_main_form<SHAPE, W_BF16, BIAS, POLICY, false>(a, sm_count, stream);
}

template <bool COMP>
cudaError_t launch_reduce_t(const BwdArgs& a, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    const int64_t n = a.plan.C * kPartialStride;
    cfg.gridDim = dim3((unsigned)((n + kRedOutputs - 1) / kRedOutputs));
    cfg.blockDim = dim3(kRedOutputs * red_slices(a.plan.chunks));
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bwd_reduce_kernel<COMP>, a);
}

// cuTensorMapEncodeTiled from the driver (looked up once through the runtime,
// so the library needs no link-time dependency on the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || p == nullptr)
            return nullptr;
        f = reinterpret_cast<EncodeTiledFn>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

}  // namespace

cudaError_t encode_bf16_rows(CUtensorMap* m, const void* base, int64_t S, int64_t C, int cols,
                             int rows) {
    EncodeTiledFn f = encode_tiled();
    if (f == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)S};
    const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
    const cuuint32_t box[2] = {(cuuint32_t)cols, (cuuint32_t)rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Reads (and clears) the flag a backward kernel sets when it gave up waiting
// on a tile. Synchronous.
cudaError_t read_wait_fault(int* flag) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_vcd_wait_fault, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_vcd_wait_fault, &zero, sizeof(int));
    return e;
}

namespace {
cudaError_t encode_maps(BwdArgs& a) {
    const int rows = a.shape == kBwdWide ? BwdGeom<kBwdWide>::kU
                     : a.shape == kBwdDeep ? BwdGeom<kBwdDeep>::kU : BwdGeom<kBwdChunked>::kU;
    cudaError_t e = encode_bf16_rows(&a.tmap_x, a.x, a.plan.S, a.plan.C, kBwdColCh, rows);
    if (e == cudaSuccess) e = encode_bf16_rows(&a.tmap_dy, a.dy, a.plan.S, a.plan.C, kBwdColCh, rows);
    return e;
}
}  // namespace

cudaError_t launch_bwd_exact(const BwdArgs& args, int sm_count, cudaStream_t stream) {
    BwdArgs a = args;
    cudaError_t e = encode_maps(a);
    if (e != cudaSuccess) return e;
    const bool fp32 = a.policy == kPolicyFP32;
    if (fp32 && a.plan.per > 1)
        e = launch_main_form<kBwdChunked, false, kRouteRuntime, kPolicyFP32, true, true>(a, sm_count, stream);
    else if (fp32)
        e = launch_main_form<kBwdChunked, false, kRouteRuntime, kPolicyFP32, false, true>(a, sm_count, stream);
    else if (a.plan.per == 1)
        e = launch_main_form<kBwdChunked, false, kRouteRuntime, kPolicyBF16, false, true>(a, sm_count, stream);
    else
        e = cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    e = fp32 ? launch_reduce_t<true>(a, stream) : launch_reduce_t<false>(a, stream);
    if (e != cudaSuccess) return e;
    const int64_t lists = a.plan.ncols * a.plan.chunks;
    const int64_t grid = lists < (int64_t)sm_count * 8 ? lists : (int64_t)sm_count * 8;
    bwd_exact_fixup_kernel<<<(unsigned)(grid > 0 ? grid : 1), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdArgs& args, int sm_count, cudaStream_t stream) {
    BwdArgs a = args;
    {
        const cudaError_t e = encode_maps(a);
        if (e != cudaSuccess) return e;
    }
    typedef cudaError_t (*L)(const BwdArgs&, int, cudaStream_t);
#define VCD_ROW(SH, WB, POL) {launch_main_t<SH, WB, kBiasNone, POL>, launch_main_t<SH, WB, kBiasF32, POL>, \
                              launch_main_t<SH, WB, kBiasBF16, POL>}
    // [weight dtype][bias kind]. The wide shape serves "bf16"-policy calls with
    // a bias only (bwd_shape), so it has no no-bias and no "fp32" kernels.
    static const L wide_bf16[2][3] = {
        {nullptr, launch_main_t<kBwdWide, false, kBiasF32, kPolicyBF16>, launch_main_t<kBwdWide, false, kBiasBF16, kPolicyBF16>},
        {nullptr, launch_main_t<kBwdWide, true, kBiasF32, kPolicyBF16>, launch_main_t<kBwdWide, true, kBiasBF16, kPolicyBF16>}};
    // The deep shape serves "bf16"-policy calls without a bias on longer
    // documents only; the chunked one "fp32" calls and short documents.
    static const L deep_bf16[2][3] = {{launch_main_t<kBwdDeep, false, kBiasNone, kPolicyBF16>, nullptr, nullptr},
                                      {launch_main_t<kBwdDeep, true, kBiasNone, kPolicyBF16>, nullptr, nullptr}};
    static const L chunked_bf16[2][3] = {VCD_ROW(kBwdChunked, false, kPolicyBF16),
                                         VCD_ROW(kBwdChunked, true, kPolicyBF16)};
    static const L fp32_t[2][3] = {VCD_ROW(kBwdChunked, false, kPolicyFP32),
                                   VCD_ROW(kBwdChunked, true, kPolicyFP32)};
#undef VCD_ROW
    const int wi = a.weight_bf16 ? 1 : 0;
    const bool fp32 = a.policy == kPolicyFP32;
    const L fn = fp32 ? (a.shape == kBwdChunked ? fp32_t[wi][a.bias_kind] : nullptr)
                      : a.shape == kBwdWide ? wide_bf16[wi][a.bias_kind]
                      : a.shape == kBwdChunked ? chunked_bf16[wi][a.bias_kind] : deep_bf16[wi][a.bias_kind];
    if (fn == nullptr) return cudaErrorInvalidValue;     // a shape bwd_shape never picks
    cudaError_t e = fn(a, sm_count, stream);
    if (e != cudaSuccess) return e;
    return fp32 ? launch_reduce_t<true>(a, stream) : launch_reduce_t<false>(a, stream);
}

}  // namespace vcd
