/*
 * gbln.h - fused residual add + LayerNorm for GB300 (sm_103a): C ABI.
 *
 * The operation (lpqz.cn CUDA tutorial, sections 5.1-5.2): for each row of a
 * [rows, cols] matrix, h = x + residual, then
 *     mean = sum(h) / cols,  var = sum((h - mean)^2) / cols,
 *     y = (h - mean) / sqrt(var + eps) * gamma + beta,
 * all in one kernel that reads x and residual once and writes y (and h) once;
 * the statistics are merged in registers (per-thread chunks, combined with
 * the parallel form of Welford's update through warp shuffles and shared
 * memory), never written between passes.  The page builds it as the second
 * fused operator after attention, to show that a low-arithmetic-intensity
 * operator is set by the bytes it moves: the kernel is HBM-bound.
 *
 * Layout.  Row r of x starts at x + r * x_stride (elements), the same for
 * residual, y and h; columns are contiguous.  gamma and beta are float32
 * [cols].  mean and rstd (= 1 / sqrt(var + eps)) are float32 [rows].
 *
 * Constraints.  1 <= cols <= 16384; rows >= 0; strides >= cols; every pointer
 * aligned to its element size.  Rows move as 16-byte vectors when every
 * pointer is 16-byte aligned and every stride a multiple of 16 bytes, element
 * by element otherwise.  residual, h, gamma, beta, mean and rstd may be NULL:
 * no residual (h = x), h not stored, gamma = 1, beta = 0, statistics not stored.
 *
 * Ownership and errors are as for gbattn.h: the caller owns every buffer; the
 * library allocates nothing; argument errors return before any work is queued
 * (attn_last_error() says why); the call only queues work on `stream`.
 */
#ifndef GBLN_H
#define GBLN_H

#include <stddef.h>
#include <stdint.h>

#include "gbattn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int64_t rows, cols;
  int64_t x_stride, r_stride, y_stride, h_stride; /* elements between consecutive rows */
  float eps;
  attn_dtype_t dtype; /* element type of x, residual, y, h (ATTN_BF16 or ATTN_F32) */
} ln_params_t;

/*
 * y = LayerNorm(x + residual) * gamma + beta, per row, with h = x + residual
 * (rounded to dtype) optionally stored.  Arithmetic in float32.  Returns
 * ATTN_OK once the work is queued.
 */
attn_status_t ln_residual_fwd(const ln_params_t* p, const void* x, const void* residual, const float* gamma,
                              const float* beta, void* y, void* h, float* mean, float* rstd, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GBLN_H */
