// vcd_noalloc.cu -- conv1d_bwd_noalloc: the backward for callers that cannot
// allocate device memory, with its partial-row scratch in a fixed array that
// lives in the library's own device image instead of a caller workspace.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library is loaded holds VCD_NOALLOC_SCRATCH_BYTES of it until the process
// exits. In host code its name is only a host-side stand-in, so the device
// address comes from cudaGetSymbolAddress with the device current. A call
// made outside stream capture looks it up afresh (a host-side query), so a
// device reset, after which the array may live at another address, is
// followed; a call made while its stream is capturing uses the address the
// last call outside capture found on that device.
#include <atomic>

#include <cuda_runtime.h>
#include <stdint.h>

#include "vcd.h"
#include "vcd_kernels.h"
#include "vcd_plan.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[VCD_NOALLOC_SCRATCH_BYTES];

std::atomic<void*> g_scratch_addr[vcd::kMaxDevices];

// Device address of g_bwd_scratch on the current device.
int scratch_address(cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= vcd::kMaxDevices) return VCD_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return VCD_ERR_CUDA;
    void* p = cap == cudaStreamCaptureStatusNone
                  ? nullptr : g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) {
            g_scratch_addr[dev].store(nullptr, std::memory_order_release);
            return VCD_ERR_CUDA;
        }
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return VCD_OK;
}

}  // namespace

extern "C" int conv1d_bwd_noalloc(const void* x, const void* dy, int64_t S, int64_t C,
                                  const void* weight, int weight_dtype,
                                  const int32_t* cu_seqlens, int64_t num_docs, const void* bias,
                                  int bias_dtype, int policy, void* dx, void* dweight,
                                  int dweight_dtype, void* dbias, int dbias_dtype,
                                  cudaStream_t stream) {
    // The arguments first, as in conv1d_bwd: a bad call is refused before any
    // CUDA call (the scratch lookup below) can fail on its own.
    const int chk = vcd::check_bwd_args(x, dy, S, C, weight, weight_dtype, cu_seqlens, num_docs,
                                        bias, bias_dtype, policy, dx, dweight, dweight_dtype,
                                        dbias, dbias_dtype);
    if (chk != VCD_OK) return chk;
    void* scratch = nullptr;
    if (S > 0) {
        if (vcd::bwd_workspace_bytes_for(S, C, policy) > (uint64_t)VCD_NOALLOC_SCRATCH_BYTES)
            return VCD_ERR_WORKSPACE_TOO_SMALL;   // shape needs more than the fixed scratch
        const int st = scratch_address(stream, &scratch);
        if (st != VCD_OK) return st;
    }
    // The partial rows are written in full before the reduce reads them, so
    // whatever an earlier call left in the array does not matter.
    return conv1d_bwd(x, dy, S, C, weight, weight_dtype, cu_seqlens, num_docs, bias, bias_dtype,
                      policy, dx, dweight, dweight_dtype, dbias, dbias_dtype, scratch,
                      scratch ? (size_t)VCD_NOALLOC_SCRATCH_BYTES : 0, stream);
}
