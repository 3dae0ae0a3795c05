/*
 * glu.h -- C ABI of the gated MLP activations SwiGLU and GeGLU, forward and backward,
 * with 64-bit indexing for long contexts (part of librope_qk.so).
 *
 * The operation.  In a layer's MLP, down_proj(act_fn(gate_proj(x)) * up_proj(x)) (TRL
 * docs, "training beyond 1M tokens", the per-layer memory section), with e =
 * gate_proj(x) and g = up_proj(x):
 *
 *     forward   h  = act(e) * g
 *     backward  dg = dh * act(e),   de = dh * g * act'(e)
 *
 * elementwise over rows x cols bf16 matrices, act = SiLU (SwiGLU) or GELU (GeGLU, the
 * exact erf form or the tanh form).  The unsloth.ai page "3x faster training with
 * packing" lists these kernels as updated with int64 indexing for long contexts
 * (section "Indexage int64 pour les kernels Triton"): a matrix may span more than 2^31
 * elements (1,048,576 tokens x 9,728, the intermediate width the TRL page uses, spans
 * 1.0e10), and every address is formed in 64 bits.
 *
 * Arithmetic.  bf16 inputs are widened exactly; act and act' are evaluated in forms
 * without cancellation (1 - sigmoid(x) = sigmoid(-x), Phi(x) = erfc(-x/sqrt2)/2,
 * (1 + tanh u)/2 = sigmoid(2u)).  Where every intermediate stays a normal binary32
 * number (|x| < 86 for SiLU, 12.5 for the erf form, 9.5 for the tanh form) they run in
 * binary32, exponentials and reciprocals from the special-function unit and erfc from a
 * fitted approximation (relative error < 4e-6 for |x| < 6.4, < 2e-5 up to 12.5);
 * farther out, and for NaN, the element's act, act' and products are evaluated in
 * binary64.  Every result is rounded once to bf16 (nearest even).  Results agree with a
 * binary64 evaluation rounded once to bf16 within one bf16 unit in the last place, plus
 * a few binary32 units of the magnitude of the terms summed in act'.
 *
 * Layout.  Each matrix is bf16 [rows][cols] with cols contiguous and a row stride in
 * elements (a multiple of 8; when rows > 1, at least cols and below cols + 2^31); cols
 * is a multiple of 8; pointers are 16-byte aligned; rows * cols / 8 < 2^31; each
 * matrix spans (rows - 1) * stride + cols < 2^56 elements.  The gate and up halves of one fused
 * [rows, 2*I] projection output are views with row stride 2*I.
 *
 * Aliasing.  An output may be exactly one of the inputs (same pointer and stride): it
 * is then overwritten in place element by element (e.g. h over g, or de over e and dg
 * over g, which needs no extra memory).  Otherwise every output must share no element
 * with any input, and the two outputs of the backward none with each other: either
 * their address ranges are disjoint, or they have the same row stride and sit side by
 * side inside it (the two halves of one [rows, 2I] buffer).
 *
 * Ownership, streams and errors as in rope_qk.h: device pointers owned by the caller,
 * no allocation, asynchronous on `stream`, ROPE_OK or a negative rope_status, checked
 * on the host before anything is launched.
 */
#ifndef GLU_H
#define GLU_H

#include <stdint.h>

#include "rope_qk.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum glu_kind {
    GLU_SWIGLU = 0,       /* act(x) = x * sigmoid(x)                                    */
    GLU_GEGLU = 1,        /* act(x) = x * Phi(x), Phi the standard normal CDF (erf form) */
    GLU_GEGLU_TANH = 2    /* act(x) = x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))     */
} glu_kind;

/* Forward: h = act(e) * g.  Strides in elements.  Returns ROPE_ERR_KIND for an unknown
 * kind, ROPE_ERR_SHAPE for negative sizes, cols not a multiple of 8, a row stride below
 * cols or at least cols + 2^31 (rows > 1), or rows * cols / 8 >= 2^31, ROPE_ERR_ALIGN,
 * ROPE_ERR_NULL, ROPE_ERR_OVERLAP. */
int glu_fwd(int32_t kind, const void *e, int64_t e_stride, const void *g, int64_t g_stride,
            void *h, int64_t h_stride, int64_t rows, int64_t cols, void *stream);

/* Backward: de = dh * g * act'(e), dg = dh * act(e).  Same rules as glu_fwd. */
int glu_bwd(int32_t kind, const void *dh, int64_t dh_stride, const void *e, int64_t e_stride,
            const void *g, int64_t g_stride, void *de, int64_t de_stride, void *dg,
            int64_t dg_stride, int64_t rows, int64_t cols, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GLU_H */
