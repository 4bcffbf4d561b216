/*
 * gq_norm.h -- RMS normalization fused with the Q8_0 quantization of the
 * normalized activations, the prologue of the prefill contraction (part of
 * libgq; conventions as in gq.h).
 *
 * Source: "Metal kernel capability table (Phase B ground truth)", section 6
 * "Norms / residual / GEMV family": rms_norm scales a row by its inverse RMS
 * and by (w + offset); rms_norm_q8 fuses the Q8 quantization into the norm
 * kernel, so the f32 normalized row is never written (there its block
 * scales came out wrong unless the threadgroup size and the row length were
 * multiples of 32; here K must be whole 32-blocks, checked before launch).
 */
#ifndef GQ_NORM_H
#define GQ_NORM_H

#include "gq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------------------
 * For every token t < M with x = X[t, 0..K):
 *   ss  = sum_j x_j^2, rounded ONCE to double (the exact sum: no summation
 *         order is involved),
 *   r   = sqrt(ss / K + eps)      (double; each operation rounded to nearest)
 *   inv = (float)(1.0 / r)        (double division, then rounded to f32)
 *   y_j = f32(f32(x_j * inv) * f32(w_j + offset))   (f32, rounded to nearest)
 * and then the Q8_0 rule of gq_quantize_q8_0 on every 32-block of y:
 *   amax = max |y|, d = amax / 127 (f32), q = clamp(round_half_away(y / d),
 *   -127, 127), q = 0 when d = 0.
 * Every step is fixed to the bit, so Xq and dx are bit-exact functions of
 * (X, w, offset, eps).
 *   X   f32[M][K] row-major, w f32[K] (the norm weight), read only.
 *   Xq  int8[M][K] and dx f32[M][K/32], overwritten: the layout
 *       gq_q4_0_gemm_q8act reads.
 *   All four pointers 16-byte aligned device memory.
 *   1 <= M, 32 <= K <= GQ_MAX_K, K % 32 == 0; eps finite and > 0, offset
 *   finite.
 * Errors (before any launch): GQ_ERR_NULL, GQ_ERR_ALIGN, GQ_ERR_SHAPE for M,
 * K, eps or offset out of range; after the launch, GQ_ERR_CUDA.
 * X must be finite: for a row holding an infinity or a NaN the codes are
 * unspecified (the kernel still reads and writes only its own row).
 * ------------------------------------------------------------------------ */
int gq_rmsnorm_quantize_q8_0(const float *X, const float *w, float offset, float eps, int8_t *Xq, float *dx,
                             int K, int M, gq_stream_t stream);

/* ---------------------------------------------------------------------------
 * The statistic of gq_rmsnorm_quantize_q8_0 alone: ss[t] = sum_j X[t][j]^2
 * rounded once to double, for every token t < M (the same device code as
 * the fused kernel's; exported so that the exact summation can be checked
 * on its own).  +infinity for a row holding an infinity and no NaN, NaN for
 * a row holding a NaN.
 *   X  f32[M][K] row-major, 16-byte aligned; ss f64[M], 16-byte aligned.
 *   1 <= M, 32 <= K <= GQ_MAX_K, K % 32 == 0.
 * Errors as gq_rmsnorm_quantize_q8_0's.
 * ------------------------------------------------------------------------ */
int gq_rmsnorm_sum_squares(const float *X, double *ss, int K, int M, gq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GQ_NORM_H */
