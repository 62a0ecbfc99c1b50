/*
 * Plain CPU oracle for the DiT elementwise hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * Every value is computed in IEEE double and rounded explicitly:
 *   RN16(v)  round-to-nearest-even to bfloat16 (8-bit significand, the fp32
 *            exponent range, subnormals kept, overflow to +-inf),
 *   RN32(v)  round-to-nearest-even to fp32 (a C cast from double).
 * bf16 values travel as uint16_t bit patterns.  Loops over rows use OpenMP;
 * each output element is computed by exactly one scalar expression, so the
 * thread count never changes a result.
 *
 * Sources (the web pages this path is taken from):
 *  - "[sglang] ERNIE-Image ... RoPE and GELU-mul fusion and RoPE cos/sin
 *    hoisting" (sglang PR #34306 analysis), section 1 (cos/sin computed once
 *    per forward as (B*S, rot_dim) rows), section 2 (rotate-half as
 *    round(round(x1*cos1) + round(-x2*sin1)), the eager chunk/neg/cat/mul/add
 *    chain) and section 3 (GEGLU up * gelu(gate) with the eager bf16
 *    activation rounding).
 *  - "SP: splitting activations alongside TP" (sequence-parallelism post),
 *    section "per-token normalisation and residual add" (RMSNorm rescales one
 *    token by its own features; the residual add pairs features of the same
 *    token) and the Pre-Norm layer figure (add, then normalise).
 *
 * Where the pages leave a step open, the reading taken is stated beside the
 * function.  Parity pins for every function live in the CPU test suite.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------ */
/* bf16 / fp32 rounding                                                */
/* ------------------------------------------------------------------ */

/* bf16 bit pattern -> exact double. */
EXPORT double dto_bf16_to_double(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* RN16 of a double: one correct rounding to the bf16 grid.
 * Grid spacing in binade [2^E, 2^(E+1)) is 2^(E-7); below 2^-126 the grid is
 * the subnormal one, spacing 2^-133.  NaN maps to a quiet NaN of the same
 * sign; values at or beyond (2 - 2^-8) * 2^127 round to infinity. */
EXPORT uint16_t dto_rn16(double v) {
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);          /* a = m * 2^e, m in [0.5, 1) */
    int E = e - 1;               /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;
    double q = ldexp(1.0, E - 7);
    double k = nearbyint(a / q); /* a/q is exact; default mode ties to even */
    double r = k * q;            /* exact: at most 9 significant bits */
    if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    float f = (float)r;          /* exact */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* RN32 of a double. */
EXPORT float dto_rn32(double v) { return (float)v; }

/* RN16(RN32(v)): the eager chain's "compute in fp32, store as bf16". */
EXPORT uint16_t dto_rn16_of_rn32(double v) { return dto_rn16((double)(float)v); }

/* Returns 1 when the floating-point environment keeps subnormals (no
 * flush-to-zero / denormals-are-zero), which every result here assumes. */
EXPORT int dto_fp_env_ok(void) {
    volatile float tiny = 0x1p-140f;
    volatile float one = 1.0f;
    volatile double dt = 0x1p-1060;
    return (tiny * one != 0.0f) && (dt * 1.0 != 0.0);
}

/* ------------------------------------------------------------------ */
/* Rotary cos/sin tables (ERNIE-Image page, section 1)                 */
/* ------------------------------------------------------------------ */

/* freqs is fp32 (S, B, 1, R) contiguous; the outputs are (B*S, R) rows, row
 * b*S + s, i.e. the (1, 0, 2, 3) permute followed by a reshape.  Each entry is
 * RN16(RN32(cos(f))): torch.cos on fp32 then .to(bf16), with the fp32 cos
 * idealised as correctly rounded (host libm cos in double, then one rounding
 * to fp32). */
EXPORT void dto_rope_cos_sin(const float* freqs, int64_t S, int64_t B, int64_t R,
                             uint16_t* cos_out, uint16_t* sin_out) {
    int64_t rows = B * S;
#pragma omp parallel for schedule(static)
    for (int64_t row = 0; row < rows; ++row) {
        int64_t b = row / S, s = row % S;
        const float* f = freqs + (s * B + b) * R;
        for (int64_t j = 0; j < R; ++j) {
            double a = (double)f[j];
            cos_out[row * R + j] = dto_rn16_of_rn32(cos(a));
            sin_out[row * R + j] = dto_rn16_of_rn32(sin(a));
        }
    }
}

/* fp64 tables with no rounding, for the invariant checks. */
EXPORT void dto_rope_cos_sin_f64(const double* freqs, int64_t S, int64_t B, int64_t R,
                                 double* cos_out, double* sin_out) {
    for (int64_t row = 0; row < B * S; ++row) {
        int64_t b = row / S, s = row % S;
        const double* f = freqs + (s * B + b) * R;
        for (int64_t j = 0; j < R; ++j) {
            cos_out[row * R + j] = cos(f[j]);
            sin_out[row * R + j] = sin(f[j]);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Rotate-half RoPE (ERNIE-Image page, section 2)                      */
/* ------------------------------------------------------------------ */

/* Rounding applied after each op of the eager chain: RN16 in bf16 mode, the
 * identity in exact (fp64) mode. */
static inline double round_op(double v, int exact) {
    return exact ? v : dto_bf16_to_double(dto_rn16(v));
}

/* One head row.  With h = rot/2, the eager chain splits the leading rot
 * columns into x1 = x[0:h], x2 = x[h:rot], builds cat(-x2, x1), and forms
 * x_rot*cos + rotated*sin, rounding each product and the sum:
 *   j <  h:  o[j] = R(R(x[j]*c[j]) + R(-x[j+h]*s[j]))
 *   h <= j < rot: o[j] = R(R(x[j]*c[j]) + R(x[j-h]*s[j]))
 *   j >= rot: o[j] = x[j]           (tail columns pass through) */
static void rope_row(const double* x, const double* c, const double* s, int64_t D,
                     int64_t rot, int exact, double* o) {
    int64_t h = rot / 2;
    for (int64_t j = 0; j < D; ++j) {
        if (j < h) {
            double p = round_op(x[j] * c[j], exact);
            double q = round_op(-x[j + h] * s[j], exact);
            o[j] = round_op(p + q, exact);
        } else if (j < rot) {
            double p = round_op(x[j] * c[j], exact);
            double q = round_op(x[j - h] * s[j], exact);
            o[j] = round_op(p + q, exact);
        } else {
            o[j] = x[j];
        }
    }
}

/* x, out: (B, S, H, D) with element strides (sx_b, sx_s, sx_h), D contiguous.
 * cos, sin: (B*S, rot) contiguous bf16, row b*S + s shared by all H heads. */
EXPORT void dto_rope_rotate_half(const uint16_t* x, int64_t B, int64_t S, int64_t H,
                                 int64_t D, int64_t sx_b, int64_t sx_s, int64_t sx_h,
                                 const uint16_t* cos_t, const uint16_t* sin_t, int64_t rot,
                                 uint16_t* out, int64_t so_b, int64_t so_s, int64_t so_h) {
#pragma omp parallel for schedule(static)
    for (int64_t tok = 0; tok < B * S; ++tok) {
        int64_t b = tok / S, s = tok % S;
        double* buf = (double*)malloc(sizeof(double) * (size_t)(2 * D + 2 * rot + 4));
        double *xr = buf, *orow = buf + D + 1, *cr = buf + 2 * D + 2, *sr = cr + rot + 1;
        for (int64_t j = 0; j < rot; ++j) {
            cr[j] = dto_bf16_to_double(cos_t[tok * rot + j]);
            sr[j] = dto_bf16_to_double(sin_t[tok * rot + j]);
        }
        for (int64_t hd = 0; hd < H; ++hd) {
            const uint16_t* xp = x + b * sx_b + s * sx_s + hd * sx_h;
            uint16_t* op = out + b * so_b + s * so_s + hd * so_h;
            for (int64_t j = 0; j < D; ++j) xr[j] = dto_bf16_to_double(xp[j]);
            rope_row(xr, cr, sr, D, rot, 0, orow);
            for (int64_t j = 0; j < D; ++j) op[j] = dto_rn16(orow[j]); /* already on grid */
        }
        free(buf);
    }
}

/* fp64 mode: contiguous (B, S, H, D) doubles, (B*S, rot) double tables. */
EXPORT void dto_rope_rotate_half_f64(const double* x, int64_t B, int64_t S, int64_t H,
                                     int64_t D, const double* cos_t, const double* sin_t,
                                     int64_t rot, double* out) {
    for (int64_t tok = 0; tok < B * S; ++tok)
        for (int64_t hd = 0; hd < H; ++hd)
            rope_row(x + (tok * H + hd) * D, cos_t + tok * rot, sin_t + tok * rot, D, rot,
                     1, out + (tok * H + hd) * D);
}

/* ------------------------------------------------------------------ */
/* GEGLU (ERNIE-Image page, section 3)                                 */
/* ------------------------------------------------------------------ */

/* gelu(x) = x * 1/2 * (1 + erf(x / sqrt 2)), the exact (erf) GELU that
 * F.gelu uses by default, evaluated through the equal form
 * 1/2 * x * erfc(-x / sqrt 2), which keeps relative accuracy for x << 0.
 * At x = -inf both forms evaluate to -inf * 0 = NaN under IEEE rules. */
EXPORT double dto_gelu_f64(double x) { return 0.5 * x * erfc(-x * M_SQRT1_2); }

/* The activation rounding: GELU computed in fp32 precision and stored as
 * bf16, RN16(RN32(gelu(x))). */
EXPORT uint16_t dto_gelu_bf16(uint16_t xb) {
    return dto_rn16_of_rn32(dto_gelu_f64(dto_bf16_to_double(xb)));
}

/* out[t,f] = RN16(up[t,f] * RN16(RN32(gelu(gate[t,f])))).  The product of two
 * bf16 values is exact in double, so the final rounding is a single one.
 * gate, up, out are (T, F) with row strides in elements. */
EXPORT void dto_gelu_and_mul(const uint16_t* gate, int64_t s_gate, const uint16_t* up,
                             int64_t s_up, uint16_t* out, int64_t s_out, int64_t T,
                             int64_t F) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t f = 0; f < F; ++f) {
            double g = dto_bf16_to_double(dto_gelu_bf16(gate[t * s_gate + f]));
            double u = dto_bf16_to_double(up[t * s_up + f]);
            out[t * s_out + f] = dto_rn16(u * g);
        }
    }
}

/* ------------------------------------------------------------------ */
/* RMSNorm fused with the residual add (sequence-parallelism post)     */
/* ------------------------------------------------------------------ */

/* One token row, pre-norm order: h = R(x + r) is the new residual stream;
 * y = R(h * (mean(h^2) + eps)^(-1/2) * w).  Exact mode drops every R. */
static void rmsnorm_row(const double* x, const double* r, const double* w, double eps,
                        int64_t C, int exact, double* h, double* y) {
    double ss = 0.0;
    for (int64_t c = 0; c < C; ++c) {
        h[c] = round_op(x[c] + r[c], exact);
        ss += h[c] * h[c];
    }
    double inv = 1.0 / sqrt(ss / (double)C + eps);
    for (int64_t c = 0; c < C; ++c) y[c] = round_op(h[c] * inv * w[c], exact);
}

/* x: (T, C) stride sx; residual: (T, C) stride sr, overwritten with h;
 * w: (C); out: (T, C) stride so.  eps is added inside the square root. */
EXPORT void dto_rmsnorm_residual(const uint16_t* x, int64_t sx, uint16_t* residual,
                                 int64_t sr, const uint16_t* w, double eps, uint16_t* out,
                                 int64_t so, int64_t T, int64_t C) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double* buf = (double*)malloc(sizeof(double) * (size_t)(5 * C + 5));
        double *xr = buf, *rr = xr + C + 1, *wr = rr + C + 1, *h = wr + C + 1, *y = h + C + 1;
        for (int64_t c = 0; c < C; ++c) {
            xr[c] = dto_bf16_to_double(x[t * sx + c]);
            rr[c] = dto_bf16_to_double(residual[t * sr + c]);
            wr[c] = dto_bf16_to_double(w[c]);
        }
        rmsnorm_row(xr, rr, wr, eps, C, 0, h, y);
        for (int64_t c = 0; c < C; ++c) {
            residual[t * sr + c] = dto_rn16(h[c]);
            out[t * so + c] = dto_rn16(y[c]);
        }
        free(buf);
    }
}

/* fp64 mode, contiguous (T, C). */
EXPORT void dto_rmsnorm_residual_f64(const double* x, const double* residual,
                                     const double* w, double eps, double* h_out,
                                     double* y_out, int64_t T, int64_t C) {
    for (int64_t t = 0; t < T; ++t)
        rmsnorm_row(x + t * C, residual + t * C, w, eps, C, 1, h_out + t * C, y_out + t * C);
}

/* ------------------------------------------------------------------ */
/* GEGLU after the gate_up projection (ERNIE-Image page, section 3)    */
/* ------------------------------------------------------------------ */

/* The MLP's gate_up = x W^T, with x (T, C) and W (N, C) bf16 (an nn.Linear
 * weight, output features in rows; for GEGLU N = 2F, gate rows first), is a
 * bf16 tensor: the exact dot products rounded once to bf16.  Each product of
 * two bf16 values is exact in double and the sum of C of them carries an error
 * below C * 2^-53 of the sum of magnitudes, far inside any rounding question
 * this file decides.  For the bounds used when the sum is accumulated in fp32
 * (in any order), also returns, per element,
 *   lo = RN16(dot - eps * sum|x w|),  hi = RN16(dot + eps * sum|x w|):
 * every fp32 accumulation whose error is below eps * sum|x w| rounds to a bf16
 * value between lo and hi. */
EXPORT void dto_gate_up_bf16(const uint16_t* x, int64_t T, int64_t C, const uint16_t* w,
                             int64_t N, double eps, uint16_t* exact, uint16_t* lo,
                             uint16_t* hi) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double* xr = (double*)malloc(sizeof(double) * (size_t)(C + 1));
        for (int64_t c = 0; c < C; ++c) xr[c] = dto_bf16_to_double(x[t * C + c]);
        for (int64_t n = 0; n < N; ++n) {
            double dot = 0.0, mag = 0.0;
            for (int64_t c = 0; c < C; ++c) {
                double p = xr[c] * dto_bf16_to_double(w[n * C + c]);
                dot += p;
                mag += fabs(p);
            }
            exact[t * N + n] = dto_rn16(dot);
            if (lo) lo[t * N + n] = dto_rn16(dot - eps * mag);
            if (hi) hi[t * N + n] = dto_rn16(dot + eps * mag);
        }
        free(xr);
    }
}

/* Threads the OpenMP loops use (reported beside the CPU timings). */
#ifdef _OPENMP
#include <omp.h>
EXPORT int dto_num_threads(void) { return omp_get_max_threads(); }
/* Threads for the following calls (the results do not depend on it). */
EXPORT void dto_set_num_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
#else
EXPORT int dto_num_threads(void) { return 1; }
EXPORT void dto_set_num_threads(int n) { (void)n; }
#endif
