/*
 * CPU oracle for packed variable-length QK rotary position embedding (RoPE).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * definition that the CUDA path is checked against.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline / reference arm may load it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (all statements restated, nothing copied):
 *   [U1] unsloth.ai, "3x faster training with packing" (fr),
 *        section "Kernel Triton QK RoPE fusionné avec packing":
 *        forward is  x*cos + rotate_half(x)*sin == x*cos + (x @ R)*sin with the
 *        block matrix R = [[0, I], [-I, 0]]; backward is dY*cos + (dY @ R^T)*sin,
 *        i.e. the same rotation with sin negated.
 *   [U2] same page, section "Packing non contaminé": position ids restart at
 *        every packed-sample boundary; the sequence-length metadata is kept.
 *   [U3] / [T] TRL docs, "training beyond 1M tokens" (fr), section on YaRN rescaling:
 *        names the rotary base `rope_theta` and describes the rescale as a linear map
 *        of positions (factor 4: 40,960 trained, 163,840 wanted).  The frequency
 *        formula itself is not printed on the pages; the standard RoFormer form is
 *        used (reading R3).
 *
 * Readings (the pages leave these steps open; each is stated once here):
 *   R1  pos(t) = t - cu[s] for the s with cu[s] <= t < cu[s+1]; tokens with no such
 *       s (t >= cu[n], or t < cu[0]) are outside every sequence and are not rotated.
 *       For a non-decreasing cu each token has at most one such s; an empty sequence
 *       (cu[s] == cu[s+1]) owns no token.
 *   R3  inverse frequencies w_j = RN32( pow(theta, -(2j)/d) / scale ), the power and
 *       the quotient taken in binary64 with the exponent formed as -(2.0*j)/d in
 *       binary64, j in [0, d/2).  scale is 1 for the plain rotation.
 *   R13 linear position rescaling ([T]: "position 100 000 becomes 25 000", factor 4):
 *       position p is read as p / scale, done by dividing every frequency by scale.
 *   R4  angle phi = RN32( (float)pos * w_j ): one binary32 multiply.
 *   R5  c = RN32(cos((double)phi)), s = RN32(sin((double)phi)) using the host
 *       libm in binary64 (the correctly rounded binary32 value except in cases
 *       within about 2^-50 of a rounding boundary).
 *   R6  with a = x_i, b = x_{i+h} (bf16 widened exactly), h = d/2, for i < h:
 *         y_i     = RNbf16( RN32( RN32(a*c) - RN32(b*s) ) )
 *         y_{i+h} = RNbf16( RN32( RN32(b*c) + RN32(a*s) ) )
 *       no fused multiply-add (build with -ffp-contract=off).  Backward uses -s.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC -lm
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---- bf16 <-> binary32 ------------------------------------------------- */

/* bf16 is the top 16 bits of a binary32; widening is exact. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to bf16, round-to-nearest, ties to even, on the bit pattern.
 * NaN stays NaN (quieted). Infinities and signed zeros are preserved. */
uint16_t oracle_float_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)          /* NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;            /* tie goes to the even result */
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

float oracle_bf16_to_float(uint16_t b) { return bf16_bits_to_float(b); }

/* ---- positions (R1, [U2]) ---------------------------------------------- */

/* pos_out[t] for t in [0, T): position of token t inside its packed sample, or -1
 * when the token lies in no sample.  Written as the definition: walk every sample
 * and number its tokens from zero.  Returns 0, or -1 if cu is not non-decreasing
 * or leaves [0, T]. */
int oracle_positions(const int32_t *cu, int32_t n_seqs, int64_t T, int32_t *pos_out)
{
    for (int64_t t = 0; t < T; ++t)
        pos_out[t] = -1;
    for (int32_t s = 0; s < n_seqs; ++s) {
        int64_t start = cu[s], end = cu[s + 1];
        if (start < 0 || end < start || end > T)
            return -1;
        for (int64_t t = start; t < end; ++t)
            pos_out[t] = (int32_t)(t - start);
    }
    return 0;
}

/* ---- frequencies and cos/sin (R3-R5, [U1], [U3]) ---------------------- */

void oracle_inv_freq_scaled(double theta, int32_t d, double scale, float *w_out)
{
    int32_t h = d / 2;
    for (int32_t j = 0; j < h; ++j) {
        double e = -(2.0 * (double)j) / (double)d;
        w_out[j] = (float)(pow(theta, e) / scale);
    }
}

void oracle_inv_freq(double theta, int32_t d, float *w_out)
{
    oracle_inv_freq_scaled(theta, d, 1.0, w_out);
}

void oracle_cos_sin_scaled(int32_t pos, double theta, int32_t d, double scale, float *c_out, float *s_out)
{
    int32_t h = d / 2;
    float w[512];
    oracle_inv_freq_scaled(theta, d, scale, w);
    for (int32_t j = 0; j < h; ++j) {
        float phi = (float)pos * w[j];
        c_out[j] = (float)cos((double)phi);
        s_out[j] = (float)sin((double)phi);
    }
}

void oracle_cos_sin(int32_t pos, double theta, int32_t d, float *c_out, float *s_out)
{
    oracle_cos_sin_scaled(pos, theta, d, 1.0, c_out, s_out);
}

/* ---- rotation (R6, [U1]) ----------------------------------------------- */

/* Rotate n_rows token rows.  x and y are bf16 bit patterns laid out [n_rows][H][d];
 * pos[r] is the position of row r, or -1 to copy the row through unchanged.
 * bwd != 0 applies the transpose rotation (sin negated).  x and y may alias.
 * d must be even and at most 1024. */
void oracle_rope_rows_scaled(const uint16_t *x, uint16_t *y, int64_t n_rows, const int32_t *pos,
                             int32_t H, int32_t d, double theta, double scale, int32_t bwd)
{
    int32_t h = d / 2;
    float c[512], s[512];
    for (int64_t r = 0; r < n_rows; ++r) {
        const uint16_t *xr = x + r * (int64_t)H * d;
        uint16_t *yr = y + r * (int64_t)H * d;
        if (pos[r] < 0) {
            if (yr != xr)
                memmove(yr, xr, sizeof(uint16_t) * (size_t)H * (size_t)d);
            continue;
        }
        oracle_cos_sin_scaled(pos[r], theta, d, scale, c, s);
        for (int32_t hd = 0; hd < H; ++hd) {
            const uint16_t *xh = xr + (int64_t)hd * d;
            uint16_t *yh = yr + (int64_t)hd * d;
            for (int32_t i = 0; i < h; ++i) {
                float a = bf16_bits_to_float(xh[i]);
                float b = bf16_bits_to_float(xh[i + h]);
                float sn = bwd ? -s[i] : s[i];
                float ac = a * c[i];
                float bs = b * sn;
                float bc = b * c[i];
                float as = a * sn;
                float lo = ac - bs;
                float hi = bc + as;
                yh[i] = oracle_float_to_bf16(lo);
                yh[i + h] = oracle_float_to_bf16(hi);
            }
        }
    }
}

void oracle_rope_rows(const uint16_t *x, uint16_t *y, int64_t n_rows, const int32_t *pos,
                      int32_t H, int32_t d, double theta, int32_t bwd)
{
    oracle_rope_rows_scaled(x, y, n_rows, pos, H, d, theta, 1.0, bwd);
}

/* Whole packed tensor: positions from cu (R1), then the rotation of every token
 * row.  x, y: [T][H][d] bf16 bits.  pos_scratch: caller-provided int32[T].
 * Returns 0, or -1 for an invalid cu. */
int oracle_rope_packed(const uint16_t *x, uint16_t *y, const int32_t *cu, int32_t n_seqs,
                       int64_t T, int32_t H, int32_t d, double theta, int32_t bwd,
                       int32_t *pos_scratch)
{
    if (oracle_positions(cu, n_seqs, T, pos_scratch) != 0)
        return -1;
    oracle_rope_rows(x, y, T, pos_scratch, H, d, theta, bwd);
    return 0;
}
