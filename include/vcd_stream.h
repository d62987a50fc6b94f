/*
 * vcd_stream.h -- a plain streaming kernel for measuring the HBM ceiling that
 * the convolution's kernels are compared against. The pages have no
 * counterpart: it computes nothing of the operation. It moves the same bytes
 * as a forward call (read n bytes, write n) or a backward call (read 2n,
 * write n) with 16-byte loads and stores and no other work, so its time is
 * what this GPU needs to move that traffic.
 */
#ifndef VCD_STREAM_H
#define VCD_STREAM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* out[i] = a[i] (b == NULL) or a[i] XOR b[i], over `bytes` bytes.
 *   a, b, out     device pointers, 16-byte aligned; b may be NULL; out may not
 *                 overlap a or b.
 *   bytes         a multiple of 16 (0 launches nothing).
 *   blocks_per_sm CTAs of 512 threads per SM in the grid (1..4).
 *   stream        CUDA stream the kernel is enqueued on.
 * Returns 0 (VCD_OK), 1 for a bad size, NULL pointer or blocks_per_sm, 3 for
 * a misaligned pointer, 4 if a CUDA call fails. Allocates nothing. */
int vcd_stream_copy(const void* a, const void* b, void* out, size_t bytes, int blocks_per_sm,
                    cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VCD_STREAM_H */
