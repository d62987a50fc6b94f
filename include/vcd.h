/*
 * vcd.h -- C ABI of the packed (varlen) width-4 depthwise causal convolution
 * + SiLU, training forward and backward, for NVIDIA GB300 (sm_103a).
 *
 * The operation is the one defined on the FlashInfer API pages
 *   "flashinfer.cake_causal_conv1d_train.cake_causal_conv1d_train_forward"
 *   "flashinfer.cake_causal_conv1d_train.cake_causal_conv1d_train_backward"
 * (each entry point below cites the section it follows).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - S tokens (all documents packed back to back), C channels, C % 8 == 0.
 * - Activations x, y, dy, dx: BF16, [S, C] row-major (channels contiguous),
 *   device pointers, 16-byte aligned. A [1, S, C] tensor is the same memory.
 * - weight: [C, 4] row-major, FP32 or BF16, 16-byte aligned; weight[c, 3]
 *   multiplies the current token, weight[c, 0] the token three back.
 * - bias: optional [C], FP32 or BF16 (its dtype is independent of weight's),
 *   16-byte aligned.
 * - cu_seqlens: int32 [num_docs + 1] device array of document boundaries
 *   (cu_seqlens[0] == 0, non-decreasing, cu_seqlens[num_docs] == S; a repeated
 *   value is an empty document). The host never reads it.
 * - Ownership: the caller owns every buffer. The library allocates nothing,
 *   frees nothing, reads no device memory on the host and never synchronizes;
 *   every call only enqueues work on `stream`, so calls can be captured into a
 *   CUDA graph. Two calls that may run at the same time need two workspaces.
 * - Errors: arguments are checked before anything is enqueued; on any error
 *   no output is touched and a vcd_status code is returned. Malformed
 *   cu_seqlens contents (which the host cannot see) never cause an
 *   out-of-bounds access; the outputs are then unspecified.
 * - The functions use the CUDA device that is current on the calling thread.
 */
#ifndef VCD_H
#define VCD_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { VCD_BF16 = 0, VCD_FP32 = 1 } vcd_dtype;

/* Where SiLU' is evaluated in the backward ("silu_grad_preactivation" on the
 * backward page, Parameters): at the BF16-rounded recomputed preactivation,
 * or at the unrounded FP32 preactivation (with a final reduction as exact as
 * an FP64 one, in compensated FP32 arithmetic). */
typedef enum { VCD_SILU_GRAD_BF16 = 0, VCD_SILU_GRAD_FP32 = 1 } vcd_silu_policy;

typedef enum {
    VCD_OK = 0,
    VCD_ERR_INVALID_ARG = 1,          /* bad size, dtype, policy, NULL pointer */
    VCD_ERR_WORKSPACE_TOO_SMALL = 2,  /* workspace_bytes below the size query */
    VCD_ERR_MISALIGNED = 3,           /* a pointer breaks its alignment rule   */
    VCD_ERR_CUDA = 4                  /* a CUDA runtime call failed            */
} vcd_status;

/* Bytes of forward workspace for (S, C). The forward keeps no counters, so
 * this is 0 and conv1d_fwd accepts a NULL workspace. (Forward page,
 * Parameters: workspace.) Returns VCD_OK, or VCD_ERR_INVALID_ARG for S < 0,
 * C <= 0, C % 8 != 0 or bytes == NULL. */
int conv1d_fwd_workspace_size(int64_t S, int64_t C, size_t* bytes);

/* Bytes of backward workspace for (S, C): the FP32 partial rows of dweight
 * and dbias (backward page, Parameters: workspace). A function of (S, C)
 * alone: the maximum over every route (bias or not, dtypes, policy, launch
 * shape) and the same on every device, so one buffer serves every call of
 * that shape: one row of 128 channels x 5 FP32 values (2560 bytes) per chunk
 * of work of each 128-channel column, at most max(3072, ceil(C / 128)) rows. The kernel
 * writes every byte it later reads: the buffer needs no zeroing. Same errors
 * as the forward query. */
int conv1d_bwd_workspace_size(int64_t S, int64_t C, size_t* bytes);

/* Bytes of backward workspace one policy needs (backward page, Parameters:
 * workspace): the partial rows of the
 * "bf16" (policy 0) or "fp32" (policy 1) program for (S, C), the largest
 * over its launch shapes; at most conv1d_bwd_workspace_size(S, C). Every
 * conv1d_bwd call of that policy accepts a workspace of this size. Errors as
 * the queries above, plus VCD_ERR_INVALID_ARG for an unknown policy. */
int conv1d_bwd_route_workspace_size(int64_t S, int64_t C, int policy, size_t* bytes);

/* Bytes of backward workspace one call needs, exactly (backward page,
 * Parameters: workspace): the partial rows that
 * conv1d_bwd writes and reads for these arguments (has_bias: a bias is
 * passed). The call picks one of three launch shapes from them -- 12 warps
 * per SM with shared memory for chunk sums for the "fp32" policy and, under
 * either policy, when documents are shorter than 32 tokens on average
 * (num_docs * 32 >= S); otherwise under "bf16" 16 warps per SM without a
 * bias, 12 warps with more registers with one -- and the shape and C (a last
 * 128-channel column with at most 64 channels is transposed) set the number
 * of chunks. At most
 * conv1d_bwd_route_workspace_size(S, C, policy). Errors as
 * conv1d_bwd_route_workspace_size, plus VCD_ERR_INVALID_ARG for S > 0 with
 * num_docs <= 0. */
int conv1d_bwd_call_workspace_size(int64_t S, int64_t C, int64_t num_docs, int policy,
                                   int has_bias, size_t* bytes);

/* Forward (forward page, Returns):
 *   y[t, c] = bf16(silu(sum_k weight[c, k] * x[t - 3 + k, c] + bias[c]))
 * with zero history before each document's first token, FP32 arithmetic,
 * round-to-nearest-even to BF16.
 *   x         [S, C] BF16, read.
 *   weight    [C, 4] of weight_dtype, read.
 *   cu_seqlens, num_docs   document boundaries, read on the device.
 *   bias      [C] of bias_dtype or NULL (no bias), read.
 *   y         [S, C] BF16, written (may not alias x).
 *   workspace, workspace_bytes   ignored (size query gives 0); may be NULL.
 *   stream    CUDA stream the kernel is enqueued on.
 * S == 0 returns VCD_OK without launching. */
int conv1d_fwd(const void* x, int64_t S, int64_t C,
               const void* weight, int weight_dtype,
               const int32_t* cu_seqlens, int64_t num_docs,
               const void* bias, int bias_dtype,
               void* y,
               void* workspace, size_t workspace_bytes,
               cudaStream_t stream);

/* Forward with every element of y within one BF16 ulp of the exact value
 * (forward page, Returns: y = bf16(silu(...)), read as exact within one BF16
 * ulp). Same arguments, checks and outputs as conv1d_fwd but no workspace.
 * conv1d_fwd is within one ulp plus a first-order bound of FP32 rounding; it
 * can miss the strict bound where the preactivation nearly cancels (|pre| well
 * below the sum of its terms' magnitudes). This route checks each element
 * against a bound of its FP32 error and recomputes the doubtful ones (a few
 * in 10^4) from the exactly summed preactivation: slower than conv1d_fwd.
 * Preactivations below -87.3, where SiLU's FP32 evaluation flushes to zero
 * (|y| < 1.1e-36), keep that limit. */
int conv1d_fwd_exact(const void* x, int64_t S, int64_t C,
                     const void* weight, int weight_dtype,
                     const int32_t* cu_seqlens, int64_t num_docs,
                     const void* bias, int bias_dtype,
                     void* y, cudaStream_t stream);

/* Backward (backward page, description and Returns). Recomputes the FP32
 * preactivation from x, evaluates SiLU' at it per `policy`, and writes
 *   dx[t, c]      = bf16(sum_k weight[c, k] * dpre[t + 3 - k, c])  (same document)
 *   dweight[c, k] = sum_t dpre[t, c] * x[t - 3 + k, c]             (zero history)
 *   dbias[c]      = sum_t dpre[t, c]                               (if dbias != NULL)
 * with dpre = dy * silu'(p). Two launches on `stream`: the main kernel writes
 * dx and one FP32 partial row per chunk of work into the workspace, and a
 * reduce kernel, launched programmatically dependent on it, sums the rows in
 * a fixed order, so the gradients are bitwise identical for a given (S, C)
 * and route. Under VCD_SILU_GRAD_BF16 a chunk is one run of tokens summed in
 * FP32 and the reduce adds in FP32. Under VCD_SILU_GRAD_FP32 a chunk is
 * several runs of at most 256 tokens, each summed in FP32 and added into the
 * chunk's total with compensated (two-float) additions; the reduce adds the
 * chunk totals the same way, which keeps the sum as exact as an FP64
 * accumulator would before its one rounding to the output dtype.
 *   x, dy     [S, C] BF16, read.
 *   weight, cu_seqlens, num_docs, bias   as in conv1d_fwd (bias must be the
 *             forward's bias: it enters the preactivation).
 *   policy    vcd_silu_policy.
 *   dx        [S, C] BF16, written (may not alias x or dy).
 *   dweight   [C, 4] of dweight_dtype, written.
 *   dbias     [C] of dbias_dtype or NULL; non-NULL requires bias != NULL.
 *   workspace conv1d_bwd_workspace_size(S, C) bytes serve every route; the
 *             call itself checks only what its own route needs. 16-byte aligned.
 *   stream    CUDA stream both kernels are enqueued on.
 * S == 0 writes zero dweight (and dbias) with cudaMemsetAsync and launches
 * no kernel. */
int conv1d_bwd(const void* x, const void* dy, int64_t S, int64_t C,
               const void* weight, int weight_dtype,
               const int32_t* cu_seqlens, int64_t num_docs,
               const void* bias, int bias_dtype,
               int policy,
               void* dx, void* dweight, int dweight_dtype,
               void* dbias, int dbias_dtype,
               void* workspace, size_t workspace_bytes,
               cudaStream_t stream);

/* Bytes of workspace conv1d_bwd_exact needs for (S, C), either policy: the
 * partial rows of its launch shape, then per chunk of work a list of the dx
 * elements to recompute (room for one in 64 elements) and its count. Errors
 * as conv1d_bwd_workspace_size. */
int conv1d_bwd_exact_workspace_size(int64_t S, int64_t C, size_t* bytes);

/* Backward with every element of dx within one BF16 ulp of the exact value
 * under the policy (backward page, Parameters: silu_grad_preactivation: dx is
 * within one BF16 ulp of exact under both policies). Same arguments, checks
 * and outputs as conv1d_bwd, with a workspace of
 * conv1d_bwd_exact_workspace_size(S, C) bytes (no zeroing needed: every byte
 * read is written first). conv1d_bwd is within one ulp plus a first-order
 * bound of FP32 rounding; it can miss the strict bound where dx nearly
 * cancels, or, under "bf16", where the FP32 preactivation and the exact one
 * round to different BF16 values. This route takes the preactivations near a
 * BF16 rounding midpoint from their exact sum, evaluates SiLU' to about
 * 2^-22, bounds each dx's FP32 error, and recomputes the few (a few in 10^3)
 * that the bound cannot certify in double-float arithmetic (about 2^-44), in
 * a third launch after the reduce.
 * dweight and dbias are formed as in conv1d_bwd (same tolerances); under
 * "bf16" they use the exactly rounded preactivations. Slower than conv1d_bwd. */
int conv1d_bwd_exact(const void* x, const void* dy, int64_t S, int64_t C,
                     const void* weight, int weight_dtype,
                     const int32_t* cu_seqlens, int64_t num_docs,
                     const void* bias, int bias_dtype,
                     int policy,
                     void* dx, void* dweight, int dweight_dtype,
                     void* dbias, int dbias_dtype,
                     void* workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/* Size of the fixed device scratch used by conv1d_bwd_noalloc: 8 MiB. Under
 * either policy that holds the partial rows of every shape with
 * C <= 419328: at most max(3072, ceil(C / 128)) rows of 2560 bytes, i.e. at
 * most 7.9 MB while C <= 393216, and one row per 128-channel column above
 * that. */
#define VCD_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Backward without a workspace argument and without any allocation. The
 * pages have no counterpart to this entry point; it exists for callers that
 * cannot hand the library device memory of its own: code embedded in a host
 * program whose memory is owned by another allocator it cannot reach from C,
 * or code that must not call cudaMalloc/cudaFree once it is running (those
 * calls can stall every stream on the device). It computes exactly what
 * conv1d_bwd computes, with the same arguments minus workspace and
 * workspace_bytes, and keeps the partial rows in a fixed
 * VCD_NOALLOC_SCRATCH_BYTES array compiled into the library, which every GPU
 * that loads the library holds until the process exits.
 *   - Shapes whose partial rows exceed VCD_NOALLOC_SCRATCH_BYTES are refused
 *     with VCD_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   - A call with S > 0 made outside stream capture looks up the array's
 *     device address on the current device (cudaGetSymbolAddress, a host-side
 *     query) and remembers it for that device; a call made while `stream` is
 *     capturing uses the remembered address. Make one call on a device before
 *     capturing calls on it: a first call made during capture runs that lookup
 *     (and the kernels' one-time set-up: shared-memory attribute and occupancy
 *     queries) inside the capture. On GB300 with CUDA 13.0 such a first call
 *     was seen to succeed, its graph replaying the eager call's bits, but
 *     that order is not relied on.
 *   - Every call shares the one array. It needs no clearing (each call writes
 *     all the rows it reads), but two calls whose kernels may overlap on the
 *     GPU -- different streams, no ordering between them -- race on it and
 *     give wrong gradients; order such calls or use conv1d_bwd with separate
 *     workspaces.
 *   - Calls no allocating function (no cudaMalloc, cudaFree or library
 *     allocator). Other arguments and errors as in conv1d_bwd. */
int conv1d_bwd_noalloc(const void* x, const void* dy, int64_t S, int64_t C,
                       const void* weight, int weight_dtype,
                       const int32_t* cu_seqlens, int64_t num_docs,
                       const void* bias, int bias_dtype,
                       int policy,
                       void* dx, void* dweight, int dweight_dtype,
                       void* dbias, int dbias_dtype,
                       cudaStream_t stream);

/* The backward's main kernel stages x and dy through shared memory with
 * tensor-map copies (TMA) whose arrival it awaits on barriers; each wait gives
 * up after about a second of SM clocks (a copy takes microseconds), sets a
 * device-side flag and leaves that call's outputs incomplete. This reads the
 * flag into *flag (1 if any kernel gave up since the last read, else 0) and
 * clears it. Unlike every other entry point it reads device memory and waits
 * for the device (cudaMemcpyFromSymbol). No counterpart on the pages: a
 * diagnostic of this implementation. Returns VCD_OK, VCD_ERR_INVALID_ARG for
 * flag == NULL, or VCD_ERR_CUDA. */
int conv1d_wait_fault(int* flag);

/* Static description of a vcd_status code (never NULL). */
const char* conv1d_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* VCD_H */
