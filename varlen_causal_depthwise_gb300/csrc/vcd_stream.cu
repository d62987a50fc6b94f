// vcd_stream.cu -- vcd_stream_copy (include/vcd_stream.h): the traffic of a
// forward or backward call with no arithmetic, for the bandwidth ceiling the
// kernels are measured against.
//
// A grid of blocks_per_sm x SMs CTAs of 512 threads strides over the buffer;
// each thread keeps four independent 16-byte loads (eight with b) in flight
// before it stores, so the memory system sees as many outstanding requests as
// the convolution's rings keep.
#include <atomic>

#include <cuda_runtime.h>
#include <stdint.h>

#include "vcd_stream.h"

namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 4;

template <bool TWO>
__global__ void __launch_bounds__(kThreads) stream_copy_kernel(const uint4* __restrict__ a,
                                                              const uint4* __restrict__ b,
                                                              uint4* __restrict__ out, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < n; i += kUnroll * stride) {
        uint4 v[kUnroll];
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) v[j] = __ldcs(a + i + j * stride);
        if (TWO) {
#pragma unroll
            for (int j = 0; j < kUnroll; ++j) {
                const uint4 u = __ldcs(b + i + j * stride);
                v[j] = make_uint4(v[j].x ^ u.x, v[j].y ^ u.y, v[j].z ^ u.z, v[j].w ^ u.w);
            }
        }
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) out[i + j * stride] = v[j];
    }
    for (; i < n; i += stride) {
        uint4 v = __ldcs(a + i);
        if (TWO) {
            const uint4 u = __ldcs(b + i);
            v = make_uint4(v.x ^ u.x, v.y ^ u.y, v.z ^ u.z, v.w ^ u.w);
        }
        out[i] = v;
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" int vcd_stream_copy(const void* a, const void* b, void* out, size_t bytes,
                               int blocks_per_sm, cudaStream_t stream) {
    if (bytes % 16 != 0 || blocks_per_sm < 1 || blocks_per_sm > 4) return 1;
    if (bytes == 0) return 0;
    if (!a || !out) return 1;
    if (!aligned16(a) || !aligned16(out) || (b && !aligned16(b))) return 3;
    static std::atomic<int> sms_cache[64];
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 4;
    if (dev >= 0 && dev < 64) sms = sms_cache[dev].load(std::memory_order_relaxed);
    if (sms <= 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return 4;
        if (dev >= 0 && dev < 64) sms_cache[dev].store(sms, std::memory_order_relaxed);
    }
    const int64_t n = (int64_t)(bytes / 16);
    const dim3 grid((unsigned)(sms * blocks_per_sm));
    if (b)
        stream_copy_kernel<true><<<grid, kThreads, 0, stream>>>(
            static_cast<const uint4*>(a), static_cast<const uint4*>(b), static_cast<uint4*>(out), n);
    else
        stream_copy_kernel<false><<<grid, kThreads, 0, stream>>>(
            static_cast<const uint4*>(a), nullptr, static_cast<uint4*>(out), n);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}
