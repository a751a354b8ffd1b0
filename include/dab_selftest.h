/*
 * dab_selftest.h -- device self-test entry point of libdab.so.
 *
 * Checks, on one 128-row tile, the five tensor-core operand forms that the
 * backward kernel of dab.h uses (same shared-memory layouts, matrix
 * descriptors and tensor-memory placements), so that a layout error shows up
 * as a wrong product of known matrices rather than as a wrong gradient.
 * Not part of the attention operation; the paper has no counterpart.
 */
#ifndef DAB_SELFTEST_H_
#define DAB_SELFTEST_H_

#include "dab.h"

#ifdef __cplusplus
extern "C" {
#endif

/* d = 64 or 128.  Device pointers, 16-byte aligned, caller-owned:
 *   x, y   bf16 [128][d] row-major
 *   z, pm  bf16 [128][128] row-major
 *   out0   f32 [128][128]  = x y^T
 *   out1   f32 [128][d]    = pm y
 *   out2   f32 [128][d]    = z y
 *   out3   f32 [128][128]  = x^T z     (d = 128)
 *          f32 [128][64]   = z^T x     (d = 64)
 *   status_ws  >= 256 bytes; its status word is read by dab_check_status().
 * Asynchronous on `stream`; argument errors are returned synchronously.     */
dab_status_t dab_selftest_mma(int d, const void* x, const void* y, const void* z,
                              const void* pm, float* out0, float* out1, float* out2,
                              float* out3, void* status_ws, cudaStream_t stream);

/* Dense bf16 tensor throughput of this build's own tcgen05 path, the
 * denominator against which the backward's throughput is quoted as a fraction
 * of the tensor peak.  Launches one CTA per SM; each issues `iters` x 4
 * back-to-back tcgen05.mma of M = 128, N = 256, K = 16 (bf16 x bf16 -> f32 in
 * tensor memory) from operands resident in shared memory, so the work is
 *     (SM count) * iters * 4 * 2 * 128 * 256 * 16  flops
 * and the caller times the launch on `stream` (CUDA events).  iters in
 * [1, 1<<22] (about a second at most).  status_ws: >= 256 bytes of device memory, caller-owned; its
 * status word (dab_check_status) reports a timed-out wait.  Asynchronous;
 * argument errors are returned synchronously.  Not part of the attention
 * operation; the paper has no counterpart.                                  */
dab_status_t dab_mma_peak(int iters, void* status_ws, cudaStream_t stream);

/* The SM count dab_mma_peak launches on (the current device), or -1.       */
int dab_mma_peak_grid(void);

#ifdef __cplusplus
}
#endif

#endif /* DAB_SELFTEST_H_ */
