// vcd_fwd.cu -- forward of the packed width-4 depthwise causal convolution +
// SiLU (FlashInfer page "cake_causal_conv1d_train_forward", Returns):
//
//   y[t, c] = bf16(silu(sum_k w[c, k] x[t - 3 + k, c] + b[c]))
//
// with zero history before each document's first token.
//
// One warp per work unit (128 channels x L tokens, vcd_plan.h); a lane owns 4
// channels (kFwdVec). The warp streams its 256-byte row segments into a
// shared-memory ring, kFwdNs - 1 batches of kFwdU tokens ahead of the
// arithmetic, so the loads in flight cost no registers: per-lane 16-byte
// cp.async in the streaming shape, one tensor-map copy (TMA) per batch onto
// the stage's mbarrier for short documents and the exact route. The three previous
// tokens of x stay in registers as FP32. Document starts come from a warp-wide
// walk over cu_seqlens as one bit mask per batch (positions q-2 .. q+U-1); a
// batch with no start in it takes a mask-free path, otherwise each tap is
// predicated on "no document start between that token and the current one",
// which is the zero history. Both paths apply the taps in the same order, so a
// token's result does not depend on where batches fall.
//
// Memory-bound: 4 bytes of HBM traffic per element (read x, write y).
#include <atomic>
#include <type_traits>

#include <cuda_runtime.h>
#include <stdint.h>

#include "vcd_device.cuh"
#include "vcd_kernels.h"
#include "vcd_plan.h"

namespace vcd {
namespace {

#ifndef VCD_FWD_PACKED
#define VCD_FWD_PACKED 1
#endif
#ifndef VCD_FWD_PACKED_SILU
#define VCD_FWD_PACKED_SILU 0
#endif
constexpr bool kPK = VCD_FWD_PACKED != 0;              // packed FP32x2 arithmetic (taps)
constexpr bool kPKS = VCD_FWD_PACKED_SILU != 0;        // ... (SiLU)
constexpr int kFwdColCh = 32 * kFwdVec;               // channels per unit column
constexpr int kFwdRowBytes = 2 * kFwdColCh;            // bytes of a token's row segment

// Batch geometry of a forward shape (vcd_plan.h): tokens per batch and ring
// stages. Short documents take 16-token batches in 2 stages: their per-batch
// cu_seqlens walk and masks are the cost, so fewer, longer batches pay
// (131072 x 1032: 8 x 3 104.5 us, 8 x 4 106.6, 12 x 3 104.3, 16 x 2 100.4;
// measured).
// kTma: the stages arrive by tensor-map copies (one per batch, issued by one
// lane, onto an mbarrier) instead of per-lane cp.async -- faster where most
// batches walk cu_seqlens and take the masked path (short documents: 110 ->
// 104 us at 131072 x 1032), slower for streaming 4-token batches (65536 x
// 6144: 254 -> 267 us; measured on GB300).
template <int SHAPE> struct FwdGeom;
// kCtas: resident CTAs per SM the launch bounds promise (the exactness check
// needs more registers).
template <> struct FwdGeom<kFwdStream> {
    static constexpr int kU = 4, kNs = 6, kCtas = kFwdCtasPerSm; static constexpr bool kTma = false;
};
template <> struct FwdGeom<kFwdShortDocs> {
    static constexpr int kU = 16, kNs = 2, kCtas = kFwdCtasPerSm; static constexpr bool kTma = true;
};
template <> struct FwdGeom<kFwdExact> {
    static constexpr int kU = 8, kNs = 3, kCtas = 2; static constexpr bool kTma = true;
};
template <int SHAPE> struct FwdShapeT : FwdGeom<SHAPE> {
    using G = FwdGeom<SHAPE>;
    static constexpr int kStageBytes = G::kU * kFwdRowBytes;
    static constexpr int kWarpBytes = G::kNs * kStageBytes;
    static constexpr int kRingBytes = kWarpsPerCta * kWarpBytes;
    // the TMA ring's barriers, one 8-byte mbarrier per stage of each warp
    static constexpr int kSmemBytes = kRingBytes + (G::kTma ? kWarpsPerCta * G::kNs * 8 : 0);
    static_assert(G::kU % 2 == 0 && G::kU <= 30 && G::kNs >= 2, "batch geometry");
};

__device__ __forceinline__ bool bit(uint32_t m, int i) { return (m >> i) & 1u; }

// Set when a forward kernel gave up waiting on a tile (mbar_wait_bounded);
// never in normal operation. conv1d_wait_fault() reads it.
__device__ int g_vcd_fwd_wait_fault = 0;

// Routes by instantiation. The main loop is the same code for every route,
// but the compiler schedules it differently per instantiation, and that moves
// the time by up to 12% (measured on GB300): an instantiation specialised on
// the dtypes is fastest for FP32 weights and for BF16 weights without a bias,
// while BF16 weights with a bias run fastest through the one that takes the
// dtypes at run time (65536 x 6144: 289 -> 260 us; 262144 x 8192: 1450 ->
// 1342 us).

// A shape that stages by tensor-map copies gets the map with its arguments
// (the streaming shape keeps the plain, smaller argument block).
struct FwdTmaArgs : FwdArgs {
    CUtensorMap tmap_x;       // x as [S rows, C channels], boxes of a batch x 128 channels
};
template <int SHAPE>
using FwdParams = typename std::conditional<FwdGeom<SHAPE>::kTma, FwdTmaArgs, FwdArgs>::type;

// The exactness check of conv1d_fwd_exact. An element's FP32 result y32 (an
// FMA chain for pre, then SiLU from exp2 / reciprocal) is within 2^-10 |y| of
// the exact y -- so that its BF16 rounding is within 3/4 of a BF16 ulp --
// whenever mag (1 + |pre|) <= 4096 |pre|, mag = |b| + sum |w_k x_k| the
// magnitude of the preactivation's terms: the chain errs by at most
// 4 2^-24 mag, which SiLU carries into y with relative gain |1 + pre (1 - s)|
// <= 1 + |pre|, and the SiLU evaluation adds at most (8 + |pre|) 2^-24
// relative. The kernel tests the sufficient condition mag 2^-11 <= min(|pre|,
// 1) with the magnitudes pre-scaled by 2^-11, and recomputes the elements
// that fail it from their exactly summed preactivation.
constexpr float kExactMagScale = 0x1p-11f;

template <int SHAPE, bool W_BF16, int BIAS>
__global__ void __launch_bounds__(kThreadsPerCta, FwdGeom<SHAPE>::kCtas)
    fwd_kernel(const __grid_constant__ FwdParams<SHAPE> a) {
    constexpr bool kTma = FwdGeom<SHAPE>::kTma;
    constexpr int kFwdU = FwdShapeT<SHAPE>::kU;                 // tokens per batch
    constexpr int kFwdNs = FwdShapeT<SHAPE>::kNs;               // ring stages
    constexpr int kFwdStageBytes = FwdShapeT<SHAPE>::kStageBytes;
    constexpr int kFwdWarpBytes = FwdShapeT<SHAPE>::kWarpBytes;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    unsigned char* const ring = smem + wid * kFwdWarpBytes;
    const uint32_t ring_s = smem_u32(ring);
    const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerCta + wid;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
    const int64_t S = a.plan.S, C = a.plan.C, L = a.plan.L;
    const int64_t units = a.plan.units, ncols = a.plan.ncols;
    const __nv_bfloat16* __restrict__ x = static_cast<const __nv_bfloat16*>(a.x);
    __nv_bfloat16* __restrict__ y = static_cast<__nv_bfloat16*>(a.y);
    const int32_t* __restrict__ cu = a.cu_seqlens;
    const int ncu = (int)(a.num_docs + 1);
    const int Ci = (int)C;                               // row stride, elements
    // TMA: this warp's stage barriers (one arrival per phase: the producer
    // lane's expect_tx), initialised once; phase parities in `phases`
    const uint32_t bars = smem_u32(smem + FwdShapeT<SHAPE>::kRingBytes) + wid * kFwdNs * 8;
    uint32_t phases = 0;
    bool fault = false;
    if (kTma) {
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < kFwdNs; ++s) mbar_init(bars + 8 * s, 1);
            mbar_init_fence();
        }
        __syncwarp();
    }

    for (int64_t u = warp0; u < units; u += nwarps) {
        const int64_t col = u % ncols, row = u / ncols;
        const int64_t c0 = col * kFwdColCh + lane * kFwdVec;
        const bool active = c0 < C;
        const int64_t t_begin = row * L;
        const int64_t t_end = t_begin + L < S ? t_begin + L : S;
        const int64_t q0 = t_begin - 3;                         // 3 warm-up tokens
        const int n_rel = (int)(t_end - q0);                    // relative tokens 0 .. n_rel-1
        const int nb = (n_rel + kFwdU - 1) / kFwdU;

        RowStream<1, kFwdRowBytes, int64_t> rs;
        if (!kTma) {
            const __nv_bfloat16* const bases[1] = {x};
            const int64_t lows[1] = {q0 > 0 ? q0 : 0};
            rs.init(bases, C, col, q0, lows, t_end, lane);
        }
        auto issue = [&](int i, int slot) {
            if constexpr (kTma) {
                // the tile of tokens q0 + i U .. + U - 1 x the column's 128
                // channels (rows outside [0, S) and channels past C arrive as
                // zeros; rows past the unit are never read)
                if (i < nb && lane == 0) {
                    const uint32_t bar = bars + 8 * slot;
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(bar, kFwdStageBytes);
                    tma_load_2d(ring_s + slot * kFwdStageBytes, &a.tmap_x, (int)(col * kFwdColCh),
                                (int)q0 + i * kFwdU, bar);
                }
            } else {
                if (i < nb) {
                    const uint32_t d[1] = {ring_s + slot * kFwdStageBytes};
                    rs.stage<kFwdU>(d, i * kFwdU, x);
                }
                cp_async_commit();
            }
        };
        __nv_bfloat16* yp = y + q0 * C + c0;                   // y row of relative token 0
        const int64_t ystep = C;

        // The taps and the document lookup (a chain of dependent loads) go
        // after the first batches' copies, whose latency they then overlap;
        // the exact shape keeps them first (its registers are tighter).
        float2 w[4][2], b[2];
        DocCursor doc;
        uint32_t carry;
        auto setup = [&]() {
            if (BIAS == kRouteRuntime)
                load_taps_rt(a.weight, a.bias, a.weight_bf16 != 0, a.bias_kind, c0, active, w, b);
            else
                load_taps<W_BF16, BIAS, 2>(a.weight, a.bias, c0, active, w, b);
            doc.init(cu, ncu, (int)q0 - 2, lane);
            carry = doc.starts(cu, ncu, (int)q0 - 2, 2, lane);               // bits of q0-2, q0-1
        };
        if constexpr (SHAPE == kFwdExact) setup();
        __syncwarp();                    // the previous unit's reads of the ring are done
#pragma unroll
        for (int s = 0; s < kFwdNs - 1; ++s) issue(s, s);
        if constexpr (SHAPE != kFwdExact) setup();
        float2 xc[3][2];                                              // x[q-3], x[q-2], x[q-1]
#pragma unroll
        for (int k = 0; k < 3; ++k) xc[k][0] = xc[k][1] = zero2();


        int slot = 0;                    // ring stage of batch i
        for (int i = 0; i < nb; ++i) {
            if constexpr (kTma) {
                if (!mbar_wait_bounded(bars + 8 * slot, (phases >> slot) & 1u)) {
                    fault = true;
                    break;
                }
                phases ^= 1u << slot;
            } else {
                cp_async_wait<kFwdNs - 2>();
            }
            __syncwarp();
            issue(i + kFwdNs - 1, slot == 0 ? kFwdNs - 1 : slot - 1);   // (i + Ns - 1) % Ns
            const int r0 = i * kFwdU;                    // relative index of the batch
            const int64_t q = q0 + r0;
            const uint32_t nw = doc.starts(cu, ncu, (int)q, kFwdU, lane);
            const uint32_t M = carry | (nw << 2);        // bit i <-> token q - 2 + i
            carry = nw >> (kFwdU - 2);
            const unsigned char* st = ring + slot * kFwdStageBytes + lane * (2 * kFwdVec);
            __nv_bfloat16* yq = yp + (int64_t)r0 * ystep;

            if constexpr (SHAPE == kFwdExact) {
                // every batch through one predicated path, each element checked
                // (the repair out of line keeps the unrolled loop small enough
                // for the instruction cache)
#pragma unroll
                for (int j = 0; j < kFwdU; ++j) {
                    const int r = r0 + j;
                    const uint2 xv = lds64(st + j * kFwdRowBytes);
                    const float2 xf[2] = {bf16x2_to_float2(xv.x), bf16x2_to_float2(xv.y)};
                    const bool m1 = !bit(M, j + 2);
                    const bool m2 = m1 && !bit(M, j + 1);
                    const bool m3 = m2 && !bit(M, j);
                    float2 yv[2];
                    uint32_t doubt = 0;                  // bit 2p + h: channel 2p + h needs recomputing
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        float2 pre = b[p];
                        float2 mag = make_float2(fabsf(b[p].x) * kExactMagScale, fabsf(b[p].y) * kExactMagScale);
                        const float2 xs[4] = {xc[0][p], xc[1][p], xc[2][p], xf[p]};
                        const bool on[4] = {m3, m2, m1, true};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if (!on[k]) continue;
                            pre = fma2<false>(w[k][p], xs[k], pre);
                            mag.x = __fmaf_rn(fabsf(w[k][p].x) * kExactMagScale, fabsf(xs[k].x), mag.x);
                            mag.y = __fmaf_rn(fabsf(w[k][p].y) * kExactMagScale, fabsf(xs[k].y), mag.y);
                        }
                        yv[p] = silu2<false>(pre);
                        if (mag.x > fminf(fabsf(pre.x), 1.0f)) doubt |= 1u << (2 * p);
                        if (mag.y > fminf(fabsf(pre.y), 1.0f)) doubt |= 2u << (2 * p);
                    }
                    if (__any_sync(kFull, doubt != 0)) {
                        // rare: those elements from their exactly summed
                        // preactivation (one FP32 rounding), then SiLU
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (!((doubt >> e) & 1u)) continue;
                            const int p = e >> 1;
                            const bool hi = e & 1;
                            const float bb = hi ? b[p].y : b[p].x;
                            const float wk[4] = {hi ? w[0][p].y : w[0][p].x, hi ? w[1][p].y : w[1][p].x,
                                                 hi ? w[2][p].y : w[2][p].x, hi ? w[3][p].y : w[3][p].x};
                            const float xk[4] = {hi ? xc[0][p].y : xc[0][p].x, hi ? xc[1][p].y : xc[1][p].x,
                                                 hi ? xc[2][p].y : xc[2][p].x, hi ? xf[p].y : xf[p].x};
                            const bool on[4] = {m3, m2, m1, true};
                            const float pe = (float)exact_preactivation(bb, wk, xk, on);
                            const float ye = silu2<false>(make_float2(pe, pe)).x;
                            if (hi) yv[p].y = ye; else yv[p].x = ye;
                        }
                    }
                    uint32_t o[2];
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        o[p] = float2_to_bf16x2(yv[p]);
                        xc[0][p] = xc[1][p];
                        xc[1][p] = xc[2][p];
                        xc[2][p] = xf[p];
                    }
                    if (active && r >= 3 && r < n_rel) st_stream(yq + j * Ci, make_uint2(o[0], o[1]));
                }
            } else if (M == 0 && r0 >= 3 && r0 + kFwdU <= n_rel) {      // every token stored
#pragma unroll
                for (int j = 0; j < kFwdU; ++j) {
                    const uint2 xv = lds64(st + j * kFwdRowBytes);
                    const float2 xf[2] = {bf16x2_to_float2(xv.x), bf16x2_to_float2(xv.y)};
                    uint32_t o[2];
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        float2 pre = fma2<kPK>(w[0][p], xc[0][p], b[p]);
                        pre = fma2<kPK>(w[1][p], xc[1][p], pre);
                        pre = fma2<kPK>(w[2][p], xc[2][p], pre);
                        pre = fma2<kPK>(w[3][p], xf[p], pre);
                        o[p] = float2_to_bf16x2(silu2<kPKS>(pre));
                        xc[0][p] = xc[1][p];
                        xc[1][p] = xc[2][p];
                        xc[2][p] = xf[p];
                    }
                    if (active) st_stream(yq + j * Ci, make_uint2(o[0], o[1]));
                }
            } else if (SHAPE == kFwdShortDocs && r0 >= 3 && r0 + kFwdU <= n_rel) {
                // Short documents put a start in most batches. bit i of N1 /
                // N2 / N3: no document start at bit i / at bits i, i+1 / at
                // bits i..i+2 of M. (The streaming shape leaves the rare
                // batches with a start to the general path below: a third
                // copy of the loop slows its mask-free path, measured.)
                const uint32_t N1 = ~M, N2 = ~(M | (M >> 1)), N3 = ~(M | (M >> 1) | (M >> 2));
#pragma unroll
                for (int j = 0; j < kFwdU; ++j) {
                    const uint2 xv = lds64(st + j * kFwdRowBytes);
                    const float2 xf[2] = {bf16x2_to_float2(xv.x), bf16x2_to_float2(xv.y)};
                    // tap k of token t sees x[t-3+k] iff no document starts in (t-3+k, t]
                    const bool m1 = bit(N1, j + 2), m2 = bit(N2, j + 1), m3 = bit(N3, j);
                    uint32_t o[2];
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        float2 pre = b[p];
                        if (m3) pre = fma2<kPK>(w[0][p], xc[0][p], pre);
                        if (m2) pre = fma2<kPK>(w[1][p], xc[1][p], pre);
                        if (m1) pre = fma2<kPK>(w[2][p], xc[2][p], pre);
                        pre = fma2<kPK>(w[3][p], xf[p], pre);
                        o[p] = float2_to_bf16x2(silu2<kPKS>(pre));
                        xc[0][p] = xc[1][p];
                        xc[1][p] = xc[2][p];
                        xc[2][p] = xf[p];
                    }
                    if (active) st_stream(yq + j * Ci, make_uint2(o[0], o[1]));
                }
            } else {
#pragma unroll
                for (int j = 0; j < kFwdU; ++j) {
                    const int r = r0 + j;
                    const uint2 xv = lds64(st + j * kFwdRowBytes);
                    const float2 xf[2] = {bf16x2_to_float2(xv.x), bf16x2_to_float2(xv.y)};
                    // tap k of token t sees x[t-3+k] iff no document starts in (t-3+k, t]
                    const bool m1 = !bit(M, j + 2);
                    const bool m2 = m1 && !bit(M, j + 1);
                    const bool m3 = m2 && !bit(M, j);
                    uint32_t o[2];
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        float2 pre = b[p];
                        if (m3) pre = fma2<kPK>(w[0][p], xc[0][p], pre);
                        if (m2) pre = fma2<kPK>(w[1][p], xc[1][p], pre);
                        if (m1) pre = fma2<kPK>(w[2][p], xc[2][p], pre);
                        pre = fma2<kPK>(w[3][p], xf[p], pre);
                        o[p] = float2_to_bf16x2(silu2<kPKS>(pre));
                        xc[0][p] = xc[1][p];
                        xc[1][p] = xc[2][p];
                        xc[2][p] = xf[p];
                    }
                    if (active && r >= 3 && r < n_rel) st_stream(yq + j * Ci, make_uint2(o[0], o[1]));
                }
            }
            slot = slot + 1 == kFwdNs ? 0 : slot + 1;
        }
        if (kTma && fault) break;
    }
    if (kTma && fault) {
        // a tile never arrived: flag it and give the stages still in flight a
        // bounded wait before the warp leaves
        if (lane == 0) atomicExch(&g_vcd_fwd_wait_fault, 1);
#pragma unroll
        for (int s = 0; s < kFwdNs; ++s) mbar_wait_bounded(bars + 8 * s, (phases >> s) & 1u);
    }
}

template <int SHAPE, bool W_BF16, int BIAS>
int prepare_t() {
    // Once per (instantiation, device): allow the dynamic shared memory and
    // read the occupancy; both are host-side queries. The cache entries are
    // atomic (host threads may get here at once; each stores the same value).
    static std::atomic<int> occ[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    const int known = occ[dev].load(std::memory_order_relaxed);
    if (known > 0) return known;
    constexpr int kSmem = FwdShapeT<SHAPE>::kSmemBytes;
    if (cudaFuncSetAttribute(fwd_kernel<SHAPE, W_BF16, BIAS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_kernel<SHAPE, W_BF16, BIAS>, kThreadsPerCta,
                                                      kSmem) != cudaSuccess)
        return 0;
    occ[dev].store(n, std::memory_order_relaxed);
    return n;
}

template <int SHAPE, bool W_BF16, int BIAS>
cudaError_t launch_fwd_t(const FwdArgs& args, int sm_count, cudaStream_t stream) {
    FwdParams<SHAPE> a;
    static_cast<FwdArgs&>(a) = args;
    if constexpr (FwdGeom<SHAPE>::kTma) {
        const cudaError_t e = encode_bf16_rows(&a.tmap_x, a.x, a.plan.S, a.plan.C, kFwdColCh,
                                               FwdGeom<SHAPE>::kU);
        if (e != cudaSuccess) return e;
    }
    const int occ = prepare_t<SHAPE, W_BF16, BIAS>();
    if (occ <= 0) return cudaErrorInvalidConfiguration;
    const int64_t ctas_needed = (a.plan.units + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t resident = (int64_t)sm_count * occ;
    const int64_t grid = ctas_needed < resident ? ctas_needed : resident;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(grid > 0 ? grid : 1));
    cfg.blockDim = dim3(kThreadsPerCta);
    cfg.dynamicSmemBytes = FwdShapeT<SHAPE>::kSmemBytes;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, fwd_kernel<SHAPE, W_BF16, BIAS>, a);
}

}  // namespace

cudaError_t read_fwd_wait_fault(int* flag) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_vcd_fwd_wait_fault, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_vcd_fwd_wait_fault, &zero, sizeof(int));
    return e;
}

cudaError_t launch_fwd_exact(const FwdArgs& a, int sm_count, cudaStream_t stream) {
    return launch_fwd_t<kFwdExact, false, kRouteRuntime>(a, sm_count, stream);
}

cudaError_t launch_fwd(const FwdArgs& a, int sm_count, cudaStream_t stream) {
    typedef cudaError_t (*L)(const FwdArgs&, int, cudaStream_t);
    // [shape][weight dtype][bias kind]
#define VCD_ROW(SH) {{launch_fwd_t<SH, false, kBiasNone>, launch_fwd_t<SH, false, kBiasF32>, \
                      launch_fwd_t<SH, false, kBiasBF16>},                                      \
                     {launch_fwd_t<SH, true, kBiasNone>, launch_fwd_t<SH, false, kRouteRuntime>,  \
                      launch_fwd_t<SH, false, kRouteRuntime>}}
    static const L launch[2][2][3] = {VCD_ROW(kFwdStream), VCD_ROW(kFwdShortDocs)};
#undef VCD_ROW
    const int shape = fwd_shape(a.plan.S, a.num_docs);
    return launch[shape][a.weight_bf16 ? 1 : 0][a.bias_kind](a, sm_count, stream);
}

}  // namespace vcd
