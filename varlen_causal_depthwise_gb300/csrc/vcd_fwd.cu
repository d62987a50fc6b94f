// vcd_fwd.cu -- forward of the packed width-4 depthwise causal convolution +
// SiLU (FlashInfer page "cake_causal_conv1d_train_forward", Returns):
//
//   y[t, c] = bf16(silu(sum_k w[c, k] x[t - 3 + k, c] + b[c]))
//
// with zero history before each document's first token.
//
// One warp per work unit (128 channels x L tokens, vcd_plan.h); a lane owns 4
// channels (kFwdVec). The warp streams its 256-byte row segments into a shared-memory
// ring with cp.async, kFwdNs - 1 batches of kFwdU tokens ahead of the
// arithmetic, so the loads in flight cost no registers. The three previous
// tokens of x stay in registers as FP32. Document starts come from a warp-wide
// walk over cu_seqlens as one bit mask per batch (positions q-2 .. q+U-1); a
// batch with no start in it takes a mask-free path, otherwise each tap is
// predicated on "no document start between that token and the current one",
// which is the zero history. Both paths apply the taps in the same order, so a
// token's result does not depend on where batches fall.
//
// Memory-bound: 4 bytes of HBM traffic per element (read x, write y).
#include <atomic>

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
// stages.
template <int SHAPE> struct FwdGeom;
template <> struct FwdGeom<kFwdStream> { static constexpr int kU = 4, kNs = 6; };
template <> struct FwdGeom<kFwdShortDocs> { static constexpr int kU = 8, kNs = 3; };
template <int SHAPE> struct FwdShapeT : FwdGeom<SHAPE> {
    using G = FwdGeom<SHAPE>;
    static constexpr int kStageBytes = G::kU * kFwdRowBytes;
    static constexpr int kWarpBytes = G::kNs * kStageBytes;
    static constexpr int kSmemBytes = kWarpsPerCta * kWarpBytes;
    static_assert(G::kU % 2 == 0 && G::kU <= 30 && G::kNs >= 2, "batch geometry");
};

__device__ __forceinline__ bool bit(uint32_t m, int i) { return (m >> i) & 1u; }

// The taps and the bias with their dtypes chosen at run time (one uniform
// branch per unit), for the instantiation that serves routes by run-time
// dtype.
__device__ __forceinline__ void load_taps_rt(const void* weight, const void* bias, bool w_bf16,
                                             int bias_kind, int64_t c0, bool active,
                                             float2 (&w)[4][2], float2 (&b)[2]) {
    if (w_bf16) {
        if (bias_kind == kBiasF32) load_taps<true, kBiasF32, 2>(weight, bias, c0, active, w, b);
        else if (bias_kind == kBiasBF16) load_taps<true, kBiasBF16, 2>(weight, bias, c0, active, w, b);
        else load_taps<true, kBiasNone, 2>(weight, bias, c0, active, w, b);
    } else {
        if (bias_kind == kBiasF32) load_taps<false, kBiasF32, 2>(weight, bias, c0, active, w, b);
        else if (bias_kind == kBiasBF16) load_taps<false, kBiasBF16, 2>(weight, bias, c0, active, w, b);
        else load_taps<false, kBiasNone, 2>(weight, bias, c0, active, w, b);
    }
}

// Routes by instantiation. The main loop is the same code for every route,
// but the compiler schedules it differently per instantiation, and that moves
// the time by up to 12% (measured on GB300): an instantiation specialised on
// the dtypes is fastest for FP32 weights and for BF16 weights without a bias,
// while BF16 weights with a bias run fastest through the one that takes the
// dtypes at run time (65536 x 6144: 289 -> 260 us; 262144 x 8192: 1450 ->
// 1342 us).
constexpr int kRouteRuntime = -1;     // W_BF16 / BIAS template value: dtypes read at run time

template <int SHAPE, bool W_BF16, int BIAS>
__global__ void __launch_bounds__(kThreadsPerCta, kFwdCtasPerSm) fwd_kernel(const FwdArgs a) {
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

    for (int64_t u = warp0; u < units; u += nwarps) {
        const int64_t col = u % ncols, row = u / ncols;
        const int64_t c0 = col * kFwdColCh + lane * kFwdVec;
        const bool active = c0 < C;
        const int64_t t_begin = row * L;
        const int64_t t_end = t_begin + L < S ? t_begin + L : S;
        const int64_t q0 = t_begin - 3;                         // 3 warm-up tokens
        const int n_rel = (int)(t_end - q0);                    // relative tokens 0 .. n_rel-1
        const int nb = (n_rel + kFwdU - 1) / kFwdU;

        float2 w[4][2], b[2];
        if (BIAS == kRouteRuntime)
            load_taps_rt(a.weight, a.bias, a.weight_bf16 != 0, a.bias_kind, c0, active, w, b);
        else
            load_taps<W_BF16, BIAS, 2>(a.weight, a.bias, c0, active, w, b);
        DocCursor doc;
        doc.init(cu, ncu, (int)q0 - 2, lane);
        uint32_t carry = doc.starts(cu, ncu, (int)q0 - 2, 2, lane);            // bits of q0-2, q0-1
        float2 xc[3][2];                                              // x[q-3], x[q-2], x[q-1]
#pragma unroll
        for (int k = 0; k < 3; ++k) xc[k][0] = xc[k][1] = zero2();

        RowStream<1, kFwdRowBytes, int64_t> rs;
        {
            const __nv_bfloat16* const bases[1] = {x};
            const int64_t lows[1] = {q0 > 0 ? q0 : 0};
            rs.init(bases, C, col, q0, lows, t_end, lane);
        }
        __nv_bfloat16* yp = y + q0 * C + c0;                   // y row of relative token 0
        const int64_t ystep = C;

        __syncwarp();                    // the previous unit's reads of the ring are done
#pragma unroll
        for (int s = 0; s < kFwdNs - 1; ++s) {
            if (s < nb) {
                const uint32_t d[1] = {ring_s + s * kFwdStageBytes};
                rs.stage<kFwdU>(d, s * kFwdU, x);
            }
            cp_async_commit();
        }

        int slot = 0;                    // ring stage of batch i
        for (int i = 0; i < nb; ++i) {
            cp_async_wait<kFwdNs - 2>();
            __syncwarp();
            {
                const int nx = i + kFwdNs - 1;
                const int nslot = slot == 0 ? kFwdNs - 1 : slot - 1;   // (i + Ns - 1) % Ns
                if (nx < nb) {
                    const uint32_t d[1] = {ring_s + nslot * kFwdStageBytes};
                    rs.stage<kFwdU>(d, nx * kFwdU, x);
                }
                cp_async_commit();
            }
            const int r0 = i * kFwdU;                    // relative index of the batch
            const int64_t q = q0 + r0;
            const uint32_t nw = doc.starts(cu, ncu, (int)q, kFwdU, lane);
            const uint32_t M = carry | (nw << 2);        // bit i <-> token q - 2 + i
            carry = nw >> (kFwdU - 2);
            const unsigned char* st = ring + slot * kFwdStageBytes + lane * (2 * kFwdVec);
            __nv_bfloat16* yq = yp + (int64_t)r0 * ystep;

            if (M == 0 && r0 >= 3 && r0 + kFwdU <= n_rel) {      // every token stored
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
cudaError_t launch_fwd_t(const FwdArgs& a, int sm_count, cudaStream_t stream) {
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
