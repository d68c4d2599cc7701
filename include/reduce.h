/*
 * reduce.h -- C ABI of the fp32 row reduction (same library as gemm.h).
 *
 *   out[r] = sum_{c < cols} x[r*ldx + c],   r < rows,
 *
 * fp32 inputs, fp32 accumulation, one fp32 result per row.  This is the
 * operation of the IREE page "[LLVMGPUVectorDistribute] Add support for
 * inter-subgroup multi_reduction": its two verification cases reduce a
 * 4096-element f32 vector to a scalar and a 4 x 4096 f32 matrix to 4 values
 * along the inner dimension (linalg.generic with arith.addf, initial value 0).
 * Its method -- each worker reduces its slice, the partial results of the
 * workers of one reduction are written to shared storage, re-read in a new
 * distribution, and reduced once more -- is done here at two levels: the
 * warps of a CTA (shuffles, then shared memory), and, for rows split across
 * CTAs, the CTAs of a row (partials in the workspace, reduced by the CTA that
 * arrives last, in split order).
 *
 * Summation order is fixed by the shapes and the SM count alone, so repeated
 * runs give bitwise-identical results.  Error bound (first order, u = 2^-24):
 *   |out[r] - exact| <= (L + splits + 18) * u * sum_c |x[r*ldx + c]|,
 * L = ceil(chunk / 4096) + 1 the longest sequential chain of one thread's
 * accumulators (chunk = elements of a row one CTA reduces; a thread keeps 16
 * fp32 accumulators), plus the depths of the trees that follow: 16
 * accumulators and the unaligned head/tail elements (5), 32 lanes (5),
 * 8 warps (3), and for a row split over `splits` CTAs the partials
 * (ceil(splits/32) sequential, then 32 lanes: at most splits + 5).
 *
 * Errors are status codes (gemm_status_t); nothing aborts or prints.
 */
#ifndef LGT_REDUCE_H
#define LGT_REDUCE_H

#include <stddef.h>
#include <stdint.h>

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of device workspace reduce_rows_f32 needs for rows x cols on a GPU
 * with `num_sms` SMs (0 = the current device's).  Zero when every row is
 * reduced by one CTA.  Otherwise it holds one fp32 partial per (row, split)
 * and one int32 arrival counter per row; it must be zero-filled before its
 * first use, and every successful run leaves the counters zero again. */
gemm_status_t reduce_rows_workspace_size(int64_t rows, int64_t cols, int32_t num_sms, size_t* bytes);

/* Enqueue out[r] = sum of row r of x on `stream` (a cudaStream_t; NULL =
 * legacy default stream), for the current device.
 *   x: device pointer, rows x cols fp32 with row pitch ldx elements
 *      (0 = cols; ldx >= cols), 4-byte aligned; read only.
 *   out: device pointer, rows fp32; written only.
 *   workspace: device memory of reduce_rows_workspace_size(rows, cols, 0)
 *      bytes (may be NULL when that is 0); owned by the caller; concurrent
 *      runs need distinct workspaces.
 * rows == 0 does nothing; cols == 0 writes zeros.  Returns
 * GEMM_ERR_INVALID_ARG (negative size, ldx < cols, NULL pointer),
 * GEMM_ERR_ALIGNMENT (x or out not 4-byte aligned), GEMM_ERR_WORKSPACE
 * (workspace missing or too small), GEMM_ERR_CUDA (no device, launch
 * failure). */
gemm_status_t reduce_rows_f32(const float* x, int64_t rows, int64_t cols, int64_t ldx, float* out, void* workspace,
                              size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LGT_REDUCE_H */
