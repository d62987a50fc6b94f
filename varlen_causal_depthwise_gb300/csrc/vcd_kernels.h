// vcd_kernels.h -- argument blocks and launchers of the CUDA kernels; the C ABI
// (vcd_capi.cu) validates arguments and calls these.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vcd_plan.h"

namespace vcd {

enum BiasKind { kBiasNone = 0, kBiasF32 = 1, kBiasBF16 = 2 };

constexpr int kMaxDevices = 64;

struct FwdArgs {
    const void* x;            // BF16 [S, C]
    const void* weight;       // [C, 4] FP32 or BF16
    const void* bias;         // [C] or nullptr
    const int32_t* cu_seqlens;
    int64_t num_docs;
    void* y;                  // BF16 [S, C]
    int weight_bf16;
    int bias_kind;            // BiasKind
    Plan plan;                // fwd_plan(S, C)
};

struct BwdArgs {
    const void* x;            // BF16 [S, C]
    const void* dy;           // BF16 [S, C]
    const void* weight;
    const void* bias;
    const int32_t* cu_seqlens;
    int64_t num_docs;
    void* dx;                 // BF16 [S, C]
    float* partials;          // [units][kColChannels][5] FP32
    void* dweight;            // [C, 4]
    void* dbias;              // [C] or nullptr
    int weight_bf16;
    int bias_kind;
    int policy;               // 0: SiLU' at bf16(pre), 1: at the FP32 pre
    int dweight_bf16;
    int dbias_bf16;
    int shape;                // BwdShape
    BwdPlan plan;             // bwd_plan(S, C, policy, shape)
    // The exactness-guarded route (conv1d_bwd_exact): per chunk a list of
    // xcap dx elements (token << 32 | channel) whose FP32 value it could not
    // certify, and their count (may exceed xcap: then the whole chunk is
    // recomputed); null otherwise.
    uint64_t* xlist;
    uint32_t* xcount;
    int64_t xcap;
    // 2D tensor maps of x and dy ([S rows, C channels] BF16, boxes of the
    // shape's batch of tokens x 128 channels), filled by launch_bwd.
    CUtensorMap tmap_x;
    CUtensorMap tmap_dy;
};

cudaError_t launch_fwd(const FwdArgs& a, int sm_count, cudaStream_t stream);
// The exactness-guarded forward (conv1d_fwd_exact).
cudaError_t launch_fwd_exact(const FwdArgs& a, int sm_count, cudaStream_t stream);
// The forward's wait-fault flag, read and cleared; synchronous.
cudaError_t read_fwd_wait_fault(int* flag);
// A [S, C] BF16 tensor as a 2D tensor map (channels innermost) with boxes of
// `rows` tokens x `cols` channels; elements outside the tensor read as zero.
cudaError_t encode_bf16_rows(CUtensorMap* m, const void* base, int64_t S, int64_t C, int cols,
                             int rows);
// conv1d_bwd's argument checks, all but the workspace's (vcd_capi.cu); a
// vcd_status code.
int check_bwd_args(const void* x, const void* dy, int64_t S, int64_t C, const void* weight,
                   int weight_dtype, const int32_t* cu_seqlens, int64_t num_docs, const void* bias,
                   int bias_dtype, int policy, const void* dx, const void* dweight,
                   int dweight_dtype, const void* dbias, int dbias_dtype);
// Main kernel, then the reduce kernel launched programmatically dependent on it.
cudaError_t launch_bwd(const BwdArgs& a, int sm_count, cudaStream_t stream);
// The exactness-guarded backward (conv1d_bwd_exact): the main kernel with
// its checks, the reduce, then the recomputation of the listed dx elements.
cudaError_t launch_bwd_exact(const BwdArgs& a, int sm_count, cudaStream_t stream);
// The backward's wait-fault flag (set, never in normal operation, when a
// kernel gave up waiting on a tile), read and cleared; synchronous.
cudaError_t read_wait_fault(int* flag);

}  // namespace vcd
