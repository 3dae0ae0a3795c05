/*
 * CPU oracle for the gated MLP activations SwiGLU and GeGLU, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY (see rope_oracle.c): the plain definition the CUDA path is
 * checked against; it shares no code with the CUDA library.
 *
 * Sources (restated, nothing copied):
 *   [U1] unsloth.ai, "3x faster training with packing" (fr): the SwiGLU and GeGLU
 *        kernels were updated with int64 indexing for long contexts (bullet list and
 *        section "Indexage int64 pour les kernels Triton").
 *   [T]  TRL docs, "training beyond 1M tokens" (fr), the MLP line of a layer,
 *        down_proj(act_fn(gate_proj(x)) * up_proj(x)), at 1,048,576 tokens with an
 *        intermediate width of 9,728.
 *
 * Readings (the pages name the activations but print no formula):
 *   G1  e = gate_proj(x), g = up_proj(x); forward h = act(e) * g elementwise.
 *   G2  SwiGLU: act = SiLU, silu(x) = x * sigmoid(x), sigmoid(x) = 1 / (1 + exp(-x)).
 *   G3  GeGLU: act = GELU, exact form gelu(x) = x * Phi(x), Phi(x) = (1 + erf(x/sqrt 2))/2;
 *       and the tanh form gelu_t(x) = x/2 * (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 *   G4  backward, with dh = dL/dh: dg = dh * act(e), de = dh * g * act'(e), where
 *         silu'(x)   = sigmoid(x) * (1 + x (1 - sigmoid(x)))
 *         gelu'(x)   = Phi(x) + x * phi(x),  phi(x) = exp(-x^2/2) / sqrt(2 pi)
 *         gelu_t'(x) = (1 + t)/2 + x/2 (1 - t^2) sqrt(2/pi) (1 + 3 * 0.044715 x^2),
 *                      t = tanh(sqrt(2/pi) (x + 0.044715 x^3)).
 *   G5  every result is evaluated in binary64 from the exact bf16 inputs and rounded
 *       once to bf16 (round to nearest even), with each formula written so that no
 *       subtraction cancels in the tails (see activation()).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a binary64 value to bf16 directly (no intermediate binary32 rounding): keep 8
 * significant bits, round to nearest with ties to even (the default rounding mode of
 * nearbyint), subnormal spacing 2^-133 below 2^-126, infinity past the largest bf16. */
static uint16_t double_to_bf16(double v)
{
    if (isnan(v)) return 0x7fc0u;
    if (v == 0.0) return signbit(v) ? 0x8000u : 0x0000u;
    int e;
    frexp(v, &e);                        /* |v| = m * 2^e with m in [0.5, 1) */
    int q = e - 8;                       /* spacing of the bf16 numbers around |v| */
    if (q < -133) q = -133;
    double r = ldexp(nearbyint(ldexp(v, -q)), q);
    if (fabs(r) > 3.3895313892515355e38) return signbit(v) ? 0xff80u : 0x7f80u;
    float f = (float)r;                  /* exact: 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

uint16_t oracle_double_to_bf16(double v) { return double_to_bf16(v); }

static const double kSqrt2OverPi = 0.79788456080286535587989211986876;   /* sqrt(2/pi) */
static const double kInvSqrt2Pi = 0.39894228040143267793994605993438;    /* 1/sqrt(2 pi) */
static const double kInvSqrt2 = 0.70710678118654752440084436210485;      /* 1/sqrt(2) */
static const double kGeluTanhC = 0.044715;

/* 1 / (1 + exp(-x)), evaluated through exp(-|x|) so that it cannot overflow: for
 * x < 0 it is exp(x) / (1 + exp(x)), which keeps its value far in the left tail. */
static double sigmoid(double x)
{
    double t = exp(-fabs(x));
    return x >= 0.0 ? 1.0 / (1.0 + t) : t / (1.0 + t);
}

/* act(x) and act'(x) for kind 0 = SwiGLU, 1 = GeGLU (erf), 2 = GeGLU (tanh), written in
 * forms without cancellation in the tails (identical in exact arithmetic):
 *   1 - sigmoid(x) = sigmoid(-x);  Phi(x) = erfc(-x/sqrt 2) / 2;
 *   (1 + tanh u)/2 = sigmoid(2u);  (1 - tanh^2 u)/2 = 2 sigmoid(2u) sigmoid(-2u). */
static void activation(int32_t kind, double x, double *act, double *dact)
{
    if (kind == 0) {
        double s = sigmoid(x);
        *act = x * s;
        *dact = s * (1.0 + x * sigmoid(-x));
    } else if (kind == 1) {
        double Phi = 0.5 * erfc(-x * kInvSqrt2);
        double phi = exp(-0.5 * x * x) * kInvSqrt2Pi;
        *act = x * Phi;
        *dact = Phi + x * phi;
    } else {
        double u = kSqrt2OverPi * (x + kGeluTanhC * x * x * x);
        double sp = sigmoid(2.0 * u), sm = sigmoid(-2.0 * u);
        *act = x * sp;
        *dact = sp + 2.0 * x * sp * sm * kSqrt2OverPi * (1.0 + 3.0 * kGeluTanhC * x * x);
    }
}

/* act(x) and act'(x) in binary64, exposed for the pins. */
void oracle_glu_activation(int32_t kind, double x, double *act, double *dact)
{
    activation(kind, x, act, dact);
}

/* Forward over n elements: h[i] = bf16(act(e[i]) * g[i]). */
void oracle_glu_fwd(int32_t kind, const uint16_t *e, const uint16_t *g, uint16_t *h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double a, da;
        activation(kind, bf16_to_double(e[i]), &a, &da);
        h[i] = double_to_bf16(a * bf16_to_double(g[i]));
    }
}

/* Backward over n elements: dg = bf16(dh * act(e)), de = bf16(dh * g * act'(e)). */
void oracle_glu_bwd(int32_t kind, const uint16_t *dh, const uint16_t *e, const uint16_t *g,
                    uint16_t *de, uint16_t *dg, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double a, da;
        double x = bf16_to_double(e[i]);
        double gi = bf16_to_double(g[i]);
        double dhi = bf16_to_double(dh[i]);
        activation(kind, x, &a, &da);
        dg[i] = double_to_bf16(dhi * a);
        de[i] = double_to_bf16(dhi * gi * da);
    }
}
