/*
 * gq_geglu.h -- the down projection of a gated GELU FFN with the gate
 * applied while its input is read (part of libgq; conventions as in gq.h).
 *
 * Source: "Metal kernel capability table (Phase B ground truth)", section 4
 * "FFN family": the fused GELU-tanh down kernels take the f32 gate and up
 * vectors and form gelu(gate) * up inside the down matvec, instead of a
 * separate elementwise GELU kernel writing h; finding F1: those fused
 * kernels lacked the +-15 clamp of the tanh argument that their separated
 * twins carry, and produced NaN for large gate values (here the clamp is
 * applied); finding F16: a fused down kernel read past the end of its gate
 * and up vectors when the FFN width was not whole blocks (here K must be
 * whole blocks, checked before launch).
 */
#ifndef GQ_GEGLU_H
#define GQ_GEGLU_H

#include "gq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------------------
 * y[i] = sum_j w_ij h_j,  h_j = gelu_tanh(g[j]) * u[j],
 *   gelu_tanh(a) = 0.5 a (1 + tanh(sqrt(2/pi) (a + 0.044715 a^3))), the tanh
 *   argument clamped to +-15; h_j is formed in f32.
 *   W_down  packed Q4_0 weights (gq_pack, format GQ_FORMAT_Q4_0), rows x K
 *           (rows = model width, K = FFN width), 16-byte aligned.
 *   g, u    f32[K] gate and up outputs (e.g. two gq_q4_0_matvec calls),
 *           16-byte aligned device memory; read only.
 *   y       f32[rows], 16-byte aligned, overwritten.
 *   M       batch size; must be 1.  1 <= rows, 32 <= K <= GQ_MAX_K, K % 32 == 0.
 * Errors (before any launch): GQ_ERR_NULL for a NULL pointer, GQ_ERR_ALIGN
 * for a misaligned one, GQ_ERR_SHAPE for rows/K/M out of range; after the
 * launch, GQ_ERR_CUDA.
 * Accuracy: with h_j the exact value of gelu_tanh(g_j) u_j,
 *   |y_i - sum_j w_ij h_j| <= 1e-5 sum_j |w_ij h_j|
 *                             + 2^-20 sum_j |w_ij| (|g_j u_j| + |h_j|)
 * (the second term bounds the f32 evaluation of h).
 * ------------------------------------------------------------------------ */
int gq_q4_0_geglu_down(const void *W_down, const float *g, const float *u, float *y, int rows, int K, int M,
                       gq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GQ_GEGLU_H */
