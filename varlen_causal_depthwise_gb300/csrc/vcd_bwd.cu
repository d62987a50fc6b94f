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
// Main kernel: one warp per work unit (32 groups of 4 channels x L tokens,
// vcd_plan.h), walking its tokens forward once. The x window (three previous
// tokens, cleared at a document start) gives pre and the dweight products; dx
// is produced three tokens late: each new dpre[u] is scattered into the three
// pending dx accumulators of tokens u-1, u-2, u-3 unless a document start lies
// between, and dx[u-3] is then complete. The unit reads x over [begin-3,
// end+3) and dy over [begin, end+3), writes dx over [begin, end), and keeps
// dweight / dbias in registers; at its end each lane writes its channels' five
// FP32 sums into the unit's partial row. HBM traffic: 6 bytes per element.
//
// Reduce kernel: launched with programmatic stream serialization, it waits on
// griddepcontrol for the main kernel and sums the partial rows of each channel
// in row order (FP32, or FP64 under the "fp32" policy), so the gradients are
// bitwise reproducible for a given (S, C) and route.
#include <cuda_runtime.h>
#include <stdint.h>

#include "vcd_device.cuh"
#include "vcd_kernels.h"
#include "vcd_plan.h"

namespace vcd {
namespace {

#ifndef VCD_BWD_U
#define VCD_BWD_U 4
#endif
constexpr int kBwdU = VCD_BWD_U;        // tokens per batch (loads run one batch ahead)
constexpr int kBP = kBwdVec / 2;        // channel pairs per lane
constexpr int kFoldBatches = 8;         // "fp32" policy: fold partial sums every 8 batches
constexpr int kColChannels = 32 * kBwdVec;

constexpr int kPolicyBF16 = 0;
constexpr int kPolicyFP32 = 1;

// Neumaier-compensated running sum of float2 values (the "fp32" policy's
// outer accumulation level).
struct CompSum2 {
    float2 s, c;
    __device__ __forceinline__ void zero() { s = c = make_float2(0.f, 0.f); }
    __device__ __forceinline__ static void add1(float& s, float& c, float v) {
        const float t = s + v;
        c += fabsf(s) >= fabsf(v) ? (s - t) + v : (v - t) + s;
        s = t;
    }
    __device__ __forceinline__ void add(float2 v) {
        add1(s.x, c.x, v.x);
        add1(s.y, c.y, v.y);
    }
    __device__ __forceinline__ float2 get() const { return add2(s, c); }
};

template <bool W_BF16, int BIAS, int POLICY>
struct BwdLane {
    float2 w[4][kBP];
    float2 b[kBP];
    float2 xw[3][kBP];   // x[u-3], x[u-2], x[u-1], zero before the document start
    float2 pd[3][kBP];   // pending dx of tokens u-1, u-2, u-3
    uint32_t live;       // bit i: pd[i] still receives contributions
    float2 dw[4][kBP];   // dweight partial sums (inner level under "fp32")
    float2 db[kBP];
    CompSum2 odw[4][kBP];   // outer level, "fp32" policy only (unused otherwise)
    CompSum2 odb[kBP];

    __device__ __forceinline__ void load_params(const BwdArgs& a, int64_t g, bool active) {
#pragma unroll
        for (int q = 0; q < kBP; ++q) {
            b[q] = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k][q] = make_float2(0.f, 0.f);
        }
        if (!active) return;
        const int64_t c0 = g * kBwdVec;
#pragma unroll
        for (int q = 0; q < kBP; ++q) {
            if (W_BF16) {
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

    __device__ __forceinline__ void reset() {
        live = 0;
#pragma unroll
        for (int q = 0; q < kBP; ++q) {
#pragma unroll
            for (int k = 0; k < 3; ++k) xw[k][q] = pd[k][q] = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 4; ++k) dw[k][q] = make_float2(0.f, 0.f);
            db[q] = make_float2(0.f, 0.f);
            if (POLICY == kPolicyFP32) {
#pragma unroll
                for (int k = 0; k < 4; ++k) odw[k][q].zero();
                odb[q].zero();
            }
        }
    }

    // "fp32" policy: move the inner sums into the compensated outer sums.
    __device__ __forceinline__ void fold() {
        if (POLICY != kPolicyFP32) return;
#pragma unroll
        for (int q = 0; q < kBP; ++q) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                odw[k][q].add(dw[k][q]);
                dw[k][q] = make_float2(0.f, 0.f);
            }
            odb[q].add(db[q]);
            db[q] = make_float2(0.f, 0.f);
        }
    }

    __device__ __forceinline__ void doc_start() {
#pragma unroll
        for (int k = 0; k < 3; ++k)
#pragma unroll
            for (int q = 0; q < kBP; ++q) xw[k][q] = make_float2(0.f, 0.f);
        live = 0;
    }

    // Warm-up token (before the unit's range): only slides the x window.
    __device__ __forceinline__ void halo(uint2 xv) {
#pragma unroll
        for (int q = 0; q < kBP; ++q) {
            xw[0][q] = xw[1][q];
            xw[1][q] = xw[2][q];
            xw[2][q] = bf16x2_to_float2(q == 0 ? xv.x : xv.y);
        }
    }

    // Token u inside [begin, end + 3): dpre, dweight / dbias (if ACC), the
    // scatter into pending dx, and dx[u - 3] as packed BF16.
    template <bool ACC, bool ALL_LIVE>
    __device__ __forceinline__ uint2 token(uint2 xv, uint2 gv) {
        uint32_t out[kBP];
#pragma unroll
        for (int q = 0; q < kBP; ++q) {
            const float2 xf = bf16x2_to_float2(q == 0 ? xv.x : xv.y);
            const float2 gf = bf16x2_to_float2(q == 0 ? gv.x : gv.y);
            float2 pre = fma2(w[0][q], xw[0][q], b[q]);
            pre = fma2(w[1][q], xw[1][q], pre);
            pre = fma2(w[2][q], xw[2][q], pre);
            pre = fma2(w[3][q], xf, pre);
            float2 sg;
            if (POLICY == kPolicyBF16) sg = silu_grad2(round_bf16x2(pre));
            else sg = silu_grad2_precise(pre);
            const float2 d = mul2(gf, sg);
            if (ACC) {
                dw[0][q] = fma2(d, xw[0][q], dw[0][q]);
                dw[1][q] = fma2(d, xw[1][q], dw[1][q]);
                dw[2][q] = fma2(d, xw[2][q], dw[2][q]);
                dw[3][q] = fma2(d, xf, dw[3][q]);
                if (BIAS != kBiasNone) db[q] = add2(db[q], d);
            }
            if (ALL_LIVE || (live & 1u)) pd[0][q] = fma2(w[2][q], d, pd[0][q]);
            if (ALL_LIVE || (live & 2u)) pd[1][q] = fma2(w[1][q], d, pd[1][q]);
            if (ALL_LIVE || (live & 4u)) pd[2][q] = fma2(w[0][q], d, pd[2][q]);
            out[q] = float2_to_bf16x2(pd[2][q]);
            pd[2][q] = pd[1][q];
            pd[1][q] = pd[0][q];
            pd[0][q] = mul2(w[3][q], d);
            xw[0][q] = xw[1][q];
            xw[1][q] = xw[2][q];
            xw[2][q] = xf;
        }
        live = ((live << 1) | 1u) & 7u;
        return make_uint2(out[0], out[1]);
    }

    // Final sums of channel pair q, element e (0: .x, 1: .y): dw0..3, db.
    __device__ __forceinline__ void result(int q, float (&r)[2][5]) const {
        float2 v[5];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            v[k] = POLICY == kPolicyFP32 ? odw[k][q].get() : dw[k][q];
        v[4] = POLICY == kPolicyFP32 ? odb[q].get() : db[q];
#pragma unroll
        for (int k = 0; k < 5; ++k) {
            r[0][k] = v[k].x;
            r[1][k] = v[k].y;
        }
    }
};

__device__ __forceinline__ void st_stream2(uint2* p, uint2 v) { __stcs(p, v); }

template <bool W_BF16, int BIAS, int POLICY>
__global__ void __launch_bounds__(kThreadsPerCta, 2) bwd_main_kernel(const BwdArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const Plan& P = a.plan;
    const int64_t vrow = P.C / kBwdVec;
    const uint2* __restrict__ x = reinterpret_cast<const uint2*>(a.x);
    const uint2* __restrict__ dy = reinterpret_cast<const uint2*>(a.dy);
    uint2* __restrict__ dx = reinterpret_cast<uint2*>(a.dx);
    const int64_t ncu = a.num_docs + 1;

    for (int64_t u = warp0; u < P.units; u += nwarps) {
        const int64_t col = u % P.ncols, row = u / P.ncols;
        const int64_t g = col * 32 + lane;
        const bool active = g < P.groups;
        const int64_t t_begin = row * P.L;
        const int64_t t_end = t_begin + P.L < P.S ? t_begin + P.L : P.S;
        const int64_t u_end = t_end + 3 < P.S ? t_end + 3 : P.S;

        BwdLane<W_BF16, BIAS, POLICY> st;
        st.load_params(a, g, active);
        st.reset();

        int64_t p = t_begin >= 3 ? t_begin - 3 : 0;
        int64_t ci = lower_bound_warp(a.cu_seqlens, ncu, p, lane);
        const uint2* xp = x + g;
        const uint2* gp = dy + g;
        uint2* dxp = dx + g;

        uint2 xA[kBwdU], gA[kBwdU], xB[kBwdU], gB[kBwdU];
        auto load = [&](uint2 (&xb)[kBwdU], uint2 (&gb)[kBwdU], int64_t q) {
#pragma unroll
            for (int j = 0; j < kBwdU; ++j) {
                const int64_t t = q + j;
                xb[j] = (active && t < u_end) ? ld_stream(xp + t * vrow) : make_uint2(0, 0);
                gb[j] = (active && t >= t_begin && t < u_end) ? ld_stream(gp + t * vrow)
                                                              : make_uint2(0, 0);
            }
        };
        int nb = 0;
        auto step = [&](const uint2 (&xb)[kBwdU], const uint2 (&gb)[kBwdU], int64_t q) {
            const uint32_t starts = doc_starts(a.cu_seqlens, ncu, ci, q, kBwdU, lane);
            if (starts == 0 && st.live == 7u && q >= t_begin + 3 && q + kBwdU <= t_end) {
                // Steady state: no document start, every token accumulates and emits.
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const uint2 o = st.template token<true, true>(xb[j], gb[j]);
                    if (active) st_stream2(dxp + (q + j - 3) * vrow, o);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t t = q + j;
                    if (t >= u_end) break;
                    if (starts & (1u << j)) st.doc_start();
                    if (t < t_begin) {
                        st.halo(xb[j]);
                        continue;
                    }
                    const uint2 o = t < t_end ? st.template token<true, false>(xb[j], gb[j])
                                              : st.template token<false, false>(xb[j], gb[j]);
                    if (active && t - 3 >= t_begin) st_stream2(dxp + (t - 3) * vrow, o);
                }
            }
            if (POLICY == kPolicyFP32 && ++nb == kFoldBatches) {
                st.fold();
                nb = 0;
            }
        };

        load(xA, gA, p);
        for (;;) {
            load(xB, gB, p + kBwdU);
            step(xA, gA, p);
            p += kBwdU;
            if (p >= u_end) break;
            load(xA, gA, p + kBwdU);
            step(xB, gB, p);
            p += kBwdU;
            if (p >= u_end) break;
        }
        st.fold();

        // dx of the last (up to) three tokens: pd[2] = dx[u_end - 3],
        // pd[1] = dx[u_end - 2], pd[0] = dx[u_end - 1].
#pragma unroll
        for (int i = 2; i >= 0; --i) {
            const int64_t t = u_end - 1 - i;
            if (active && t >= t_begin && t < t_end)
                st_stream2(dxp + t * vrow, make_uint2(float2_to_bf16x2(st.pd[i][0]),
                                                      float2_to_bf16x2(st.pd[i][1])));
        }

        // Partial row of this unit: [32 * kBwdVec channels][5] FP32.
        if (active) {
            float r[kBwdVec][5];
#pragma unroll
            for (int q = 0; q < kBP; ++q) {
                float rq[2][5];
                st.result(q, rq);
#pragma unroll
                for (int k = 0; k < 5; ++k) {
                    r[2 * q][k] = rq[0][k];
                    r[2 * q + 1][k] = rq[1][k];
                }
            }
            float4* dst = reinterpret_cast<float4*>(a.partials + (u * kColChannels + lane * kBwdVec) * kPartialStride);
            const float* flat = &r[0][0];
#pragma unroll
            for (int i = 0; i < kBwdVec * kPartialStride / 4; ++i)
                dst[i] = make_float4(flat[4 * i], flat[4 * i + 1], flat[4 * i + 2], flat[4 * i + 3]);
        }
    }
    // Let the reduce kernel's CTAs be scheduled; its griddepcontrol.wait still
    // waits for this whole grid to finish and its writes to be visible.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- reduce ---

template <typename T> __device__ __forceinline__ void store_out(void* base, int64_t i, T v, bool bf16);

template <> __device__ __forceinline__ void store_out<float>(void* base, int64_t i, float v, bool bf16) {
    if (bf16) reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
    else reinterpret_cast<float*>(base)[i] = v;
}
template <> __device__ __forceinline__ void store_out<double>(void* base, int64_t i, double v, bool bf16) {
    if (bf16) reinterpret_cast<__nv_bfloat16*>(base)[i] = __double2bfloat16(v);
    else reinterpret_cast<float*>(base)[i] = (float)v;
}

// One thread per (channel, value): sums the unit rows of the channel's column
// in row order 0, 1, ..., rows - 1.
template <typename ACC>
__global__ void __launch_bounds__(256) bwd_reduce_kernel(const BwdArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const Plan& P = a.plan;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= P.C * kPartialStride) return;
    const int64_t c = idx / kPartialStride;
    const int k = (int)(idx % kPartialStride);
    if (k == 4 && a.dbias == nullptr) return;
    const int64_t col = c / kColChannels, ci = c % kColChannels;
    const float* src = a.partials + (col * kColChannels + ci) * kPartialStride + k;
    const int64_t stride = P.ncols * kColChannels * kPartialStride;
    ACC acc = 0;
    int64_t r = 0;
    for (; r + 8 <= P.rows; r += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + (r + j) * stride);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc += (ACC)v[j];
    }
    for (; r < P.rows; ++r) acc += (ACC)__ldcg(src + r * stride);
    if (k < 4) store_out<ACC>(a.dweight, c * 4 + k, acc, a.dweight_bf16 != 0);
    else store_out<ACC>(a.dbias, c, acc, a.dbias_bf16 != 0);
}

// -------------------------------------------------------------- launch ---

template <bool W_BF16, int BIAS, int POLICY>
cudaError_t launch_main_t(const BwdArgs& a, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsPerCta);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, bwd_main_kernel<W_BF16, BIAS, POLICY>, a);
}

template <bool W_BF16, int BIAS, int POLICY>
int occupancy_t() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, bwd_main_kernel<W_BF16, BIAS, POLICY>,
                                                      kThreadsPerCta, 0) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

template <typename ACC>
cudaError_t launch_reduce_t(const BwdArgs& a, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    const int64_t n = a.plan.C * kPartialStride;
    cfg.gridDim = dim3((unsigned)((n + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bwd_reduce_kernel<ACC>, a);
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, int sm_count, cudaStream_t stream) {
    typedef cudaError_t (*L)(const BwdArgs&, int, cudaStream_t);
    typedef int (*O)();
#define VCD_ROW(WB, POL) {launch_main_t<WB, kBiasNone, POL>, launch_main_t<WB, kBiasF32, POL>, launch_main_t<WB, kBiasBF16, POL>}
#define VCD_OROW(WB, POL) {occupancy_t<WB, kBiasNone, POL>, occupancy_t<WB, kBiasF32, POL>, occupancy_t<WB, kBiasBF16, POL>}
    static const L launch[2][2][3] = {{VCD_ROW(false, kPolicyBF16), VCD_ROW(false, kPolicyFP32)},
                                      {VCD_ROW(true, kPolicyBF16), VCD_ROW(true, kPolicyFP32)}};
    static const O occ[2][2][3] = {{VCD_OROW(false, kPolicyBF16), VCD_OROW(false, kPolicyFP32)},
                                   {VCD_OROW(true, kPolicyBF16), VCD_OROW(true, kPolicyFP32)}};
#undef VCD_ROW
#undef VCD_OROW
    const int wi = a.weight_bf16 ? 1 : 0;
    const int pi = a.policy == kPolicyFP32 ? 1 : 0;
    const int bi = a.bias_kind;
    const int64_t ctas_needed = (a.plan.units + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t resident = (int64_t)sm_count * occ[wi][pi][bi]();
    int64_t grid = ctas_needed < resident ? ctas_needed : resident;
    if (grid < 1) grid = 1;
    cudaError_t e = launch[wi][pi][bi](a, (int)grid, stream);
    if (e != cudaSuccess) return e;
    return pi ? launch_reduce_t<double>(a, stream) : launch_reduce_t<float>(a, stream);
}

}  // namespace vcd
