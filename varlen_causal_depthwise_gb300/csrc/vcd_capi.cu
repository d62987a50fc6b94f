// vcd_capi.cu -- the extern "C" entry points declared in include/vcd.h:
// argument checks, the S == 0 cases, the work-unit plan, and the launches.
// Nothing here allocates, synchronizes or reads device memory on the host.
#include <atomic>

#include <cuda_runtime.h>
#include <stdint.h>

#include "vcd.h"
#include "vcd_kernels.h"
#include "vcd_plan.h"

namespace {

// SM count of the current device (cached; a host-side attribute query). Host
// threads may make their first calls at once: the cache entries are atomic,
// and filling one twice stores the same value.
int sm_count_of_current(int* sms) {
    static std::atomic<int> cache[vcd::kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return VCD_ERR_CUDA;
    if (dev >= 0 && dev < vcd::kMaxDevices) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *sms = c;
            return VCD_OK;
        }
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return VCD_ERR_CUDA;
    if (dev >= 0 && dev < vcd::kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
    *sms = n;
    return VCD_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool dtype_ok(int d) { return d == VCD_BF16 || d == VCD_FP32; }

// Shape rules of the forward page (Parameters: x, cu_seqlens): C % 8 == 0,
// S fits the int32 cu_seqlens, and a non-empty sequence has documents.
int check_shape(int64_t S, int64_t C, int64_t num_docs) {
    if (S < 0 || C <= 0 || C % 8 != 0 || num_docs < 0) return VCD_ERR_INVALID_ARG;
    // token positions, document indices and per-batch row offsets stay in 32 bits
    if (S > INT32_MAX - 64 || num_docs > INT32_MAX - 1 || C > ((int64_t)1 << 26))
        return VCD_ERR_INVALID_ARG;
    if (S > 0 && num_docs == 0) return VCD_ERR_INVALID_ARG;
    return VCD_OK;
}

// Inputs shared by both directions (x, weight, cu_seqlens, bias).
int check_inputs(const void* x, const void* weight, int weight_dtype, const int32_t* cu,
                 const void* bias, int bias_dtype) {
    if (!x || !weight || !cu) return VCD_ERR_INVALID_ARG;
    if (!dtype_ok(weight_dtype) || (bias && !dtype_ok(bias_dtype))) return VCD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(weight, 16) || (bias && !aligned(bias, 16)) || !aligned(cu, 4))
        return VCD_ERR_MISALIGNED;
    return VCD_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? VCD_OK : VCD_ERR_CUDA; }

}  // namespace

namespace vcd {

// Every argument check of the backward except the workspace's, in conv1d_bwd's
// order; the tensors themselves are checked only when S > 0 (an empty
// sequence may pass NULL for them).
int check_bwd_args(const void* x, const void* dy, int64_t S, int64_t C, const void* weight,
                   int weight_dtype, const int32_t* cu_seqlens, int64_t num_docs, const void* bias,
                   int bias_dtype, int policy, const void* dx, const void* dweight,
                   int dweight_dtype, const void* dbias, int dbias_dtype) {
    int st = check_shape(S, C, num_docs);
    if (st != VCD_OK) return st;
    if (policy != VCD_SILU_GRAD_BF16 && policy != VCD_SILU_GRAD_FP32) return VCD_ERR_INVALID_ARG;
    if (!dtype_ok(weight_dtype) || (bias && !dtype_ok(bias_dtype))) return VCD_ERR_INVALID_ARG;
    if (!dweight || !dtype_ok(dweight_dtype)) return VCD_ERR_INVALID_ARG;
    if (dbias && (!bias || !dtype_ok(dbias_dtype))) return VCD_ERR_INVALID_ARG;  // dbias needs bias
    const uintptr_t dwa = dweight_dtype == VCD_BF16 ? 2 : 4, dba = dbias_dtype == VCD_BF16 ? 2 : 4;
    if (!aligned(dweight, dwa) || (dbias && !aligned(dbias, dba))) return VCD_ERR_MISALIGNED;
    if (S == 0) return VCD_OK;
    st = check_inputs(x, weight, weight_dtype, cu_seqlens, bias, bias_dtype);
    if (st != VCD_OK) return st;
    if (!dy || !dx) return VCD_ERR_INVALID_ARG;
    if (!aligned(dy, 16) || !aligned(dx, 16)) return VCD_ERR_MISALIGNED;
    if (dx == x || dx == dy) return VCD_ERR_INVALID_ARG;
    return VCD_OK;
}

}  // namespace vcd

extern "C" {

int conv1d_fwd_workspace_size(int64_t S, int64_t C, size_t* bytes) {
    if (!bytes || check_shape(S, C, S > 0 ? 1 : 0) != VCD_OK) return VCD_ERR_INVALID_ARG;
    *bytes = 0;
    return VCD_OK;
}

int conv1d_bwd_workspace_size(int64_t S, int64_t C, size_t* bytes) {
    if (!bytes || check_shape(S, C, S > 0 ? 1 : 0) != VCD_OK) return VCD_ERR_INVALID_ARG;
    *bytes = (size_t)vcd::bwd_workspace_bytes(S, C);
    return VCD_OK;
}

int conv1d_bwd_route_workspace_size(int64_t S, int64_t C, int policy, size_t* bytes) {
    if (!bytes || check_shape(S, C, S > 0 ? 1 : 0) != VCD_OK) return VCD_ERR_INVALID_ARG;
    if (policy != VCD_SILU_GRAD_BF16 && policy != VCD_SILU_GRAD_FP32) return VCD_ERR_INVALID_ARG;
    *bytes = (size_t)vcd::bwd_workspace_bytes_for(S, C, policy);
    return VCD_OK;
}

int conv1d_bwd_call_workspace_size(int64_t S, int64_t C, int64_t num_docs, int policy,
                                   int has_bias, size_t* bytes) {
    if (!bytes || check_shape(S, C, num_docs) != VCD_OK) return VCD_ERR_INVALID_ARG;
    if (policy != VCD_SILU_GRAD_BF16 && policy != VCD_SILU_GRAD_FP32) return VCD_ERR_INVALID_ARG;
    *bytes = (size_t)vcd::bwd_call_workspace_bytes(S, C, num_docs, policy, has_bias != 0);
    return VCD_OK;
}

}  // extern "C"

namespace {

// conv1d_fwd and conv1d_fwd_exact: the same checks, then the route.
int fwd_call(const void* x, int64_t S, int64_t C, const void* weight, int weight_dtype,
             const int32_t* cu_seqlens, int64_t num_docs, const void* bias, int bias_dtype,
             void* y, cudaStream_t stream, bool exact) {
    int st = check_shape(S, C, num_docs);
    if (st != VCD_OK) return st;
    if (!dtype_ok(weight_dtype) || (bias && !dtype_ok(bias_dtype))) return VCD_ERR_INVALID_ARG;
    if (S == 0) return VCD_OK;                       // empty output, no launch
    st = check_inputs(x, weight, weight_dtype, cu_seqlens, bias, bias_dtype);
    if (st != VCD_OK) return st;
    if (!y) return VCD_ERR_INVALID_ARG;
    if (!aligned(y, 16)) return VCD_ERR_MISALIGNED;
    if (y == x) return VCD_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = sm_count_of_current(&sms)) != VCD_OK) return st;

    vcd::FwdArgs a;
    a.x = x;
    a.weight = weight;
    a.bias = bias;
    a.cu_seqlens = cu_seqlens;
    a.num_docs = num_docs;
    a.y = y;
    a.weight_bf16 = weight_dtype == VCD_BF16;
    a.bias_kind = !bias ? vcd::kBiasNone : bias_dtype == VCD_BF16 ? vcd::kBiasBF16 : vcd::kBiasF32;
    a.plan = vcd::fwd_plan(S, C);
    return cuda_status(exact ? vcd::launch_fwd_exact(a, sms, stream) : vcd::launch_fwd(a, sms, stream));
}

}  // namespace

extern "C" {

int conv1d_fwd(const void* x, int64_t S, int64_t C, const void* weight, int weight_dtype,
               const int32_t* cu_seqlens, int64_t num_docs, const void* bias, int bias_dtype,
               void* y, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    return fwd_call(x, S, C, weight, weight_dtype, cu_seqlens, num_docs, bias, bias_dtype, y, stream,
                    false);
}

int conv1d_fwd_exact(const void* x, int64_t S, int64_t C, const void* weight, int weight_dtype,
                     const int32_t* cu_seqlens, int64_t num_docs, const void* bias, int bias_dtype,
                     void* y, cudaStream_t stream) {
    return fwd_call(x, S, C, weight, weight_dtype, cu_seqlens, num_docs, bias, bias_dtype, y, stream,
                    true);
}

int conv1d_bwd_exact_workspace_size(int64_t S, int64_t C, size_t* bytes) {
    if (!bytes || check_shape(S, C, S > 0 ? 1 : 0) != VCD_OK) return VCD_ERR_INVALID_ARG;
    *bytes = (size_t)vcd::bwd_exact_workspace_bytes(S, C);
    return VCD_OK;
}

}  // extern "C"

namespace {

// conv1d_bwd and conv1d_bwd_exact: the same checks, then the route.
int bwd_call(const void* x, const void* dy, int64_t S, int64_t C, const void* weight,
             int weight_dtype, const int32_t* cu_seqlens, int64_t num_docs, const void* bias,
             int bias_dtype, int policy, void* dx, void* dweight, int dweight_dtype, void* dbias,
             int dbias_dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream,
             bool exact) {
    int st = vcd::check_bwd_args(x, dy, S, C, weight, weight_dtype, cu_seqlens, num_docs, bias,
                                 bias_dtype, policy, dx, dweight, dweight_dtype, dbias, dbias_dtype);
    if (st != VCD_OK) return st;
    if (S == 0) {                                    // zero gradients, no kernel
        const size_t dwa = dweight_dtype == VCD_BF16 ? 2 : 4, dba = dbias_dtype == VCD_BF16 ? 2 : 4;
        cudaError_t e = cudaMemsetAsync(dweight, 0, (size_t)C * 4 * dwa, stream);
        if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, (size_t)C * dba, stream);
        return cuda_status(e);
    }
    const int weight_bf16 = weight_dtype == VCD_BF16;
    const int bias_kind = !bias ? vcd::kBiasNone : bias_dtype == VCD_BF16 ? vcd::kBiasBF16 : vcd::kBiasF32;
    const int shape = exact ? vcd::kBwdChunked : vcd::bwd_shape(S, num_docs, policy, bias != nullptr);
    const vcd::ExactLayout xl = vcd::exact_layout(S, C, policy);
    const uint64_t need = exact ? xl.total : vcd::bwd_workspace_bytes_for(S, C, policy, shape);
    if (!workspace || workspace_bytes < need) return VCD_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 16)) return VCD_ERR_MISALIGNED;
    int sms = 0;
    if ((st = sm_count_of_current(&sms)) != VCD_OK) return st;

    vcd::BwdArgs a;
    a.x = x;
    a.dy = dy;
    a.weight = weight;
    a.bias = bias;
    a.cu_seqlens = cu_seqlens;
    a.num_docs = num_docs;
    a.dx = dx;
    a.partials = static_cast<float*>(workspace);
    a.dweight = dweight;
    a.dbias = dbias;
    a.weight_bf16 = weight_bf16;
    a.bias_kind = bias_kind;
    a.policy = policy;
    a.dweight_bf16 = dweight_dtype == VCD_BF16;
    a.dbias_bf16 = dbias_dtype == VCD_BF16;
    a.shape = shape;
    a.plan = vcd::bwd_plan(S, C, policy, shape, !exact);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    a.xlist = exact ? reinterpret_cast<uint64_t*>(ws + xl.list_offset) : nullptr;
    a.xcount = exact ? reinterpret_cast<uint32_t*>(ws + xl.count_offset) : nullptr;
    a.xcap = exact ? xl.cap : 0;
    return cuda_status(exact ? vcd::launch_bwd_exact(a, sms, stream) : vcd::launch_bwd(a, sms, stream));
}

}  // namespace

extern "C" {

int conv1d_bwd(const void* x, const void* dy, int64_t S, int64_t C, const void* weight,
               int weight_dtype, const int32_t* cu_seqlens, int64_t num_docs, const void* bias,
               int bias_dtype, int policy, void* dx, void* dweight, int dweight_dtype,
               void* dbias, int dbias_dtype, void* workspace, size_t workspace_bytes,
               cudaStream_t stream) {
    return bwd_call(x, dy, S, C, weight, weight_dtype, cu_seqlens, num_docs, bias, bias_dtype, policy,
                    dx, dweight, dweight_dtype, dbias, dbias_dtype, workspace, workspace_bytes, stream,
                    false);
}

int conv1d_bwd_exact(const void* x, const void* dy, int64_t S, int64_t C, const void* weight,
                     int weight_dtype, const int32_t* cu_seqlens, int64_t num_docs, const void* bias,
                     int bias_dtype, int policy, void* dx, void* dweight, int dweight_dtype,
                     void* dbias, int dbias_dtype, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
    return bwd_call(x, dy, S, C, weight, weight_dtype, cu_seqlens, num_docs, bias, bias_dtype, policy,
                    dx, dweight, dweight_dtype, dbias, dbias_dtype, workspace, workspace_bytes, stream,
                    true);
}

int conv1d_wait_fault(int* flag) {
    if (!flag) return VCD_ERR_INVALID_ARG;
    int f = 0, b = 0;
    const cudaError_t e = vcd::read_fwd_wait_fault(&f);
    const cudaError_t e2 = vcd::read_wait_fault(&b);
    if (e != cudaSuccess || e2 != cudaSuccess) return VCD_ERR_CUDA;
    *flag = f | b;
    return VCD_OK;
}

const char* conv1d_status_string(int status) {
    switch (status) {
        case VCD_OK: return "ok";
        case VCD_ERR_INVALID_ARG: return "invalid argument";
        case VCD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case VCD_ERR_MISALIGNED: return "misaligned pointer";
        case VCD_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

}  // extern "C"
