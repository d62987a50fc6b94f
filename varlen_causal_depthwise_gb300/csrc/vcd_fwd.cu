// vcd_fwd.cu -- forward of the packed width-4 depthwise causal convolution +
// SiLU (FlashInfer page "cake_causal_conv1d_train_forward", Returns):
//
//   y[t, c] = bf16(silu(sum_k w[c, k] x[t - 3 + k, c] + b[c]))
//
// with zero history before each document's first token.
//
// One warp per work unit (32 groups of kFwdVec channels x L tokens, see
// vcd_plan.h). Each lane streams its slice of every token row with one vector
// load (16 bytes for 8 channels), keeps the three previous tokens of its
// channels in registers as FP32, and writes its BF16 slice of y per token. Loads run one batch of U tokens
// ahead of the arithmetic (two register buffers, ping-pong). A document start
// clears the register window, which is exactly the zero history; the starts
// come from a warp-cooperative walk over cu_seqlens, one 32-bit mask per
// batch. Memory-bound: 4 bytes of HBM traffic per element (read x, write y).
#include <cuda_runtime.h>
#include <stdint.h>

#include "vcd_device.cuh"
#include "vcd_kernels.h"
#include "vcd_plan.h"

namespace vcd {
namespace {

#ifndef VCD_FWD_U
#define VCD_FWD_U 4
#endif
constexpr int kFwdU = VCD_FWD_U;   // tokens per batch (loads run one batch ahead)
constexpr int kPairs = kFwdVec / 2;

template <int VEC> struct VecType;
template <> struct VecType<8> { typedef uint4 T; };
template <> struct VecType<4> { typedef uint2 T; };
typedef VecType<kFwdVec>::T XVec;

__device__ __forceinline__ __attribute__((unused)) uint32_t word(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__device__ __forceinline__ uint32_t word(const uint2& v, int i) { return i == 0 ? v.x : v.y; }
__device__ __forceinline__ void set_word(uint4& v, int i, uint32_t w) {
    if (i == 0) v.x = w; else if (i == 1) v.y = w; else if (i == 2) v.z = w; else v.w = w;
}
__device__ __forceinline__ void set_word(uint2& v, int i, uint32_t w) {
    if (i == 0) v.x = w; else v.y = w;
}
__device__ __forceinline__ XVec zero_vec() {
    XVec v;
#pragma unroll
    for (int i = 0; i < kPairs; ++i) set_word(v, i, 0u);
    return v;
}

template <bool W_BF16, int BIAS>
struct FwdLane {
    float2 w[4][kPairs];   // w[k][q]: tap k of channels (2q, 2q + 1) of the lane
    float2 b[kPairs];
    float2 win[3][kPairs]; // x[t-3], x[t-2], x[t-1] of the lane's channels

    __device__ __forceinline__ void load_params(const FwdArgs& a, int64_t g, bool active) {
#pragma unroll
        for (int q = 0; q < kPairs; ++q) {
            b[q] = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k][q] = make_float2(0.f, 0.f);
        }
        if (!active) return;
        const int64_t c0 = g * kFwdVec;
#pragma unroll
        for (int q = 0; q < kPairs; ++q) {
            if (W_BF16) {
                // channels 2q, 2q + 1: 2 x 4 BF16 taps = one 16-byte vector
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                    reinterpret_cast<const __nv_bfloat16*>(a.weight) + (c0 + 2 * q) * 4));
                const float2 e01 = bf16x2_to_float2(v.x), e23 = bf16x2_to_float2(v.y);
                const float2 o01 = bf16x2_to_float2(v.z), o23 = bf16x2_to_float2(v.w);
                w[0][q] = make_float2(e01.x, o01.x);
                w[1][q] = make_float2(e01.y, o01.y);
                w[2][q] = make_float2(e23.x, o23.x);
                w[3][q] = make_float2(e23.y, o23.y);
            } else {
                const float4* wp = reinterpret_cast<const float4*>(a.weight) + c0 + 2 * q;
                const float4 e = __ldg(wp), o = __ldg(wp + 1);
                w[0][q] = make_float2(e.x, o.x);
                w[1][q] = make_float2(e.y, o.y);
                w[2][q] = make_float2(e.z, o.z);
                w[3][q] = make_float2(e.w, o.w);
            }
            if (BIAS == kBiasF32)
                b[q] = __ldg(reinterpret_cast<const float2*>(a.bias) + c0 / 2 + q);
            else if (BIAS == kBiasBF16)
                b[q] = bf16x2_to_float2(__ldg(reinterpret_cast<const uint32_t*>(a.bias) + c0 / 2 + q));
        }
    }

    __device__ __forceinline__ void clear_window() {
#pragma unroll
        for (int k = 0; k < 3; ++k)
#pragma unroll
            for (int q = 0; q < kPairs; ++q) win[k][q] = make_float2(0.f, 0.f);
    }

    // One token: y from the window and the current x, then slide the window.
    __device__ __forceinline__ XVec token(const XVec& xv) {
        XVec out;
#pragma unroll
        for (int q = 0; q < kPairs; ++q) {
            const float2 xf = bf16x2_to_float2(word(xv, q));
            float2 pre = fma2(w[0][q], win[0][q], b[q]);
            pre = fma2(w[1][q], win[1][q], pre);
            pre = fma2(w[2][q], win[2][q], pre);
            pre = fma2(w[3][q], xf, pre);
            set_word(out, q, float2_to_bf16x2(silu2(pre)));
            win[0][q] = win[1][q];
            win[1][q] = win[2][q];
            win[2][q] = xf;
        }
        return out;
    }
};

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint2* p, const uint2& v) { __stcs(p, v); }

template <bool W_BF16, int BIAS>
__global__ void __launch_bounds__(kThreadsPerCta, 2) fwd_kernel(const FwdArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const Plan& P = a.plan;
    const int64_t vrow = P.C / kFwdVec;                 // vectors per token row
    const XVec* __restrict__ x = reinterpret_cast<const XVec*>(a.x);
    XVec* __restrict__ y = reinterpret_cast<XVec*>(a.y);
    const int64_t ncu = a.num_docs + 1;

    for (int64_t u = warp0; u < P.units; u += nwarps) {
        const int64_t col = u % P.ncols, row = u / P.ncols;
        const int64_t g = col * 32 + lane;
        const bool active = g < P.groups;
        const int64_t t_begin = row * P.L;
        const int64_t t_end = t_begin + P.L < P.S ? t_begin + P.L : P.S;

        FwdLane<W_BF16, BIAS> st;
        st.load_params(a, g, active);
        st.clear_window();

        int64_t p = t_begin >= 3 ? t_begin - 3 : 0;   // window warm-up from here
        int64_t ci = lower_bound_warp(a.cu_seqlens, ncu, p, lane);
        const XVec* xp = x + g;
        XVec* yp = y + g;

        XVec bufA[kFwdU], bufB[kFwdU];
        auto load = [&](XVec (&buf)[kFwdU], int64_t q) {
#pragma unroll
            for (int j = 0; j < kFwdU; ++j)
                buf[j] = (active && q + j < t_end) ? ld_stream(xp + (q + j) * vrow) : zero_vec();
        };
        auto step = [&](const XVec (&buf)[kFwdU], int64_t q) {
            const uint32_t starts = doc_starts(a.cu_seqlens, ncu, ci, q, kFwdU, lane);
            if (starts == 0 && q >= t_begin && q + kFwdU <= t_end) {
#pragma unroll
                for (int j = 0; j < kFwdU; ++j) {
                    const XVec o = st.token(buf[j]);
                    if (active) st_stream(yp + (q + j) * vrow, o);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kFwdU; ++j) {
                    if (q + j >= t_end) break;
                    if (starts & (1u << j)) st.clear_window();
                    const XVec o = st.token(buf[j]);
                    if (active && q + j >= t_begin) st_stream(yp + (q + j) * vrow, o);
                }
            }
        };

        load(bufA, p);
        for (;;) {
            load(bufB, p + kFwdU);
            step(bufA, p);
            p += kFwdU;
            if (p >= t_end) break;
            load(bufA, p + kFwdU);
            step(bufB, p);
            p += kFwdU;
            if (p >= t_end) break;
        }
    }
}

template <bool W_BF16, int BIAS>
cudaError_t launch_fwd_t(const FwdArgs& a, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsPerCta);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, fwd_kernel<W_BF16, BIAS>, a);
}

template <bool W_BF16, int BIAS>
int occupancy_t() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_kernel<W_BF16, BIAS>,
                                                      kThreadsPerCta, 0) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, int sm_count, cudaStream_t stream) {
    typedef cudaError_t (*L)(const FwdArgs&, int, cudaStream_t);
    typedef int (*O)();
    static const L launch[2][3] = {
        {launch_fwd_t<false, kBiasNone>, launch_fwd_t<false, kBiasF32>, launch_fwd_t<false, kBiasBF16>},
        {launch_fwd_t<true, kBiasNone>, launch_fwd_t<true, kBiasF32>, launch_fwd_t<true, kBiasBF16>}};
    static const O occ[2][3] = {
        {occupancy_t<false, kBiasNone>, occupancy_t<false, kBiasF32>, occupancy_t<false, kBiasBF16>},
        {occupancy_t<true, kBiasNone>, occupancy_t<true, kBiasF32>, occupancy_t<true, kBiasBF16>}};
    const int wi = a.weight_bf16 ? 1 : 0;
    const int bi = a.bias_kind;
    const int64_t ctas_needed = (a.plan.units + kWarpsPerCta - 1) / kWarpsPerCta;
    int64_t resident = (int64_t)sm_count * occ[wi][bi]();
    int64_t grid = ctas_needed < resident ? ctas_needed : resident;
    if (grid < 1) grid = 1;
    return launch[wi][bi](a, (int)grid, stream);
}

}  // namespace vcd
