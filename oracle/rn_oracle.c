/*
 * rn_oracle.c -- plain, slow, fp64 CPU oracle for bf16 row normalization.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA library is
 * checked against; nothing on the product path may call it.  It shares no
 * code, header, table or constant with the CUDA sources.
 *
 * What it computes (each function cites the passage it follows):
 *   - RMSNorm: "[Inductor] Codegen Gluon", section 3.1 "MVP: RMSNorm with
 *     TMA-Cached Reused Input": the reduction accumulates x*x over the row and
 *     the post-reduction pass computes x * rstd * weight.  The formula
 *     y = x * rsqrt(mean(x^2) + eps) * w is the plain reading of those two
 *     phases.
 *   - Fused per-head Q/K RMSNorm followed by neox RoPE, in place on packed
 *     QKV: "[pretuned] Optimize fused_qk_norm_rope on B200", section
 *     "Summary" (norm over the whole head, Q/K weights, RoPE, one store per
 *     half; partial rotary still normalises the non-rotary tail).
 *   - The rotary cos/sin table used as an input by the above, with binary32
 *     or bf16 entries.
 *   - L2Norm (x / max(||x||, eps)): "[Inductor] Codegen Gluon", section 3.2.
 *   - Fused residual add + RMSNorm: "TorchInductor: from ATen IR to Triton
 *     kernel", sections 14.3 and 14.27.
 *   - LayerNorm (mean and biased variance, then affine): "TorchInductor: from
 *     ATen IR to Triton kernel", section 14.12.2, and "[Inductor] Codegen
 *     Gluon", section 3.2.
 *
 * Arithmetic: every value is widened to double, computed in double, and
 * rounded ONCE to bf16 (or, for the *_fmt forms with f16 = 1, IEEE fp16)
 * with round-to-nearest-even at the end.  Sums run in
 * plain index order.  Compile without -ffast-math and with -ffp-contract=off
 * so the result is the same on every host.
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---- bf16 <-> double ---------------------------------------------------- */

/* bf16 is the top 16 bits of an IEEE binary32; widening is exact. */
double rn_oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), in one step.
 *
 * bf16 has 8 significant bits and binary32's exponent range: normal numbers
 * down to 2^-126, subnormals with a fixed quantum of 2^-133, and a largest
 * finite value of (2 - 2^-7) * 2^127.  For |v| in [2^(e-1), 2^e) the quantum
 * is 2^(e-8).  Dividing by a power of two is exact, so v / quantum rounded to
 * the nearest even integer and multiplied back is the correctly rounded
 * value.  The rounded value fits binary32 exactly, so its top half is the
 * bf16 pattern. */
uint16_t rn_oracle_double_to_bf16(double v)
{
    uint32_t u;
    float f;
    if (isnan(v)) return 0x7FC0u;
    if (v == 0.0) {
        f = (float)v; /* keeps the sign of zero */
        memcpy(&u, &f, sizeof u);
        return (uint16_t)(u >> 16);
    }
    if (isinf(v)) return signbit(v) ? 0xFF80u : 0x7F80u;

    int e;
    (void)frexp(v, &e);              /* |v| in [2^(e-1), 2^e) */
    int qexp = e - 8;
    if (qexp < -133) qexp = -133;    /* subnormal quantum */
    double q = ldexp(1.0, qexp);
    double n = nearbyint(v / q);     /* default mode: nearest, ties to even */
    double r = n * q;
    /* Anything at or above 2^128 after rounding overflows to infinity. */
    if (fabs(r) >= ldexp(1.0, 128)) return signbit(v) ? 0xFF80u : 0x7F80u;
    f = (float)r;                    /* exact: r has <= 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* ---- fp16 (IEEE binary16) <-> double ------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 mantissa bits. */
double rn_oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                  /* zero and subnormals */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return sign ? -v : v;
}

/* Round a double to the nearest binary16 (ties to even), in one step:
 * 11 significant bits, quantum 2^(e-11) for |v| in [2^(e-1), 2^e), fixed
 * subnormal quantum 2^-24, and everything that rounds to 2^16 or beyond is
 * infinity (the largest finite value is 65504). */
uint16_t rn_oracle_double_to_f16(double v)
{
    if (isnan(v)) return 0x7E00u;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7C00u;
    int e;
    (void)frexp(a, &e);                              /* a in [2^(e-1), 2^e) */
    int qexp = e - 11;
    if (qexp < -24) qexp = -24;
    double q = ldexp(1.0, qexp);
    double r = nearbyint(a / q) * q;                 /* ties to even */
    if (r >= 65536.0) return sign | 0x7C00u;
    if (r < ldexp(1.0, -14))                         /* subnormal (or zero) */
        return sign | (uint16_t)(r / ldexp(1.0, -24));
    int ex;
    double m = frexp(r, &ex);                        /* r = m * 2^ex, m in [0.5, 1) */
    int E = ex - 1;                                  /* r = (2m) * 2^E */
    uint16_t mant = (uint16_t)((2.0 * m - 1.0) * 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | mant;
}

/* Element format of the row operations: 0 = bf16, 1 = fp16. */
static double widen(uint16_t b, int f16)
{
    return f16 ? rn_oracle_f16_to_double(b) : rn_oracle_bf16_to_double(b);
}

static uint16_t narrow(double v, int f16)
{
    return f16 ? rn_oracle_double_to_f16(v) : rn_oracle_double_to_bf16(v);
}

/* ---- RMSNorm ------------------------------------------------------------ */

/* y[r, j] = round( x[r, j] * 1/sqrt( (sum_k x[r, k]^2) / N + eps ) * w[j] )
 * for a row-major x[M, N], one row at a time, in bf16 (f16 = 0) or fp16
 * (f16 = 1).  eps is the caller's binary32 value widened exactly.  Follows
 * "[Inductor] Codegen Gluon", section 3.1 (section 3.2 widens it to fp16). */
int rn_oracle_rmsnorm_fmt(const uint16_t *x, const uint16_t *w, float eps,
                          int64_t M, int64_t N, uint16_t *y, int f16)
{
    if (M < 0 || N <= 0) return -3;
    if (M == 0) return 0;
    if (!x || !w || !y) return -1;
    const double deps = (double)eps;
    for (int64_t r = 0; r < M; ++r) {
        const uint16_t *xr = x + r * N;
        uint16_t *yr = y + r * N;
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double v = widen(xr[j], f16);
            ss += v * v;
        }
        double ms = ss / (double)N;
        double rs = 1.0 / sqrt(ms + deps);
        for (int64_t j = 0; j < N; ++j) {
            double v = widen(xr[j], f16);
            double g = widen(w[j], f16);
            yr[j] = narrow(v * rs * g, f16);
        }
    }
    return 0;
}

int rn_oracle_rmsnorm(const uint16_t *x, const uint16_t *w, float eps,
                      int64_t M, int64_t N, uint16_t *y)
{
    return rn_oracle_rmsnorm_fmt(x, w, eps, M, N, y, 0);
}

/* The row statistic alone: rstd[r] = 1/sqrt(mean(x[r,:]^2) + eps), in
 * double.  Used by tests that check invariants of the normalisation. */
int rn_oracle_rms_rstd(const uint16_t *x, float eps, int64_t M, int64_t N,
                       double *rstd)
{
    if (M < 0 || N <= 0) return -3;
    if (M == 0) return 0;
    if (!x || !rstd) return -1;
    for (int64_t r = 0; r < M; ++r) {
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double v = rn_oracle_bf16_to_double(x[r * N + j]);
            ss += v * v;
        }
        rstd[r] = 1.0 / sqrt(ss / (double)N + (double)eps);
    }
    return 0;
}

/* ---- rotary table ------------------------------------------------------- */

/* cos_sin[p, i]         = float(cos(p * f_i)),
 * cos_sin[p, r/2 + i]   = float(sin(p * f_i)),   f_i = theta^(-2i/r),
 * for p in [0, max_pos), i in [0, r/2).  The angle and the trig functions
 * are evaluated in double, then rounded once to binary32 (C's conversion is
 * round-to-nearest-even).  The pages print no table; this is the common neox
 * layout (cos half first) taken as the plain reading. */
int rn_oracle_rope_cos_sin(double theta, int64_t max_pos, int rotary_dim,
                           float *cos_sin)
{
    if (max_pos < 0 || rotary_dim <= 0 || (rotary_dim & 1) || !(theta > 0.0))
        return -3;
    if (max_pos == 0) return 0;
    if (!cos_sin) return -1;
    const int half = rotary_dim / 2;
    for (int64_t p = 0; p < max_pos; ++p) {
        float *row = cos_sin + p * (int64_t)rotary_dim;
        for (int i = 0; i < half; ++i) {
            double f = pow(theta, -2.0 * (double)i / (double)rotary_dim);
            double a = (double)p * f;
            row[i] = (float)cos(a);
            row[half + i] = (float)sin(a);
        }
    }
    return 0;
}

/* The same table with bf16 entries: the angle and the trig functions in
 * double as above, each entry rounded ONCE to bf16 (ties to even), not
 * through binary32 (rounding twice could land on the other neighbour).  A
 * bf16 table is read by the fused kernel widened exactly to fp32, so the
 * fused oracle below takes it as the binary32 values it widens to. */
int rn_oracle_rope_cos_sin_bf16(double theta, int64_t max_pos, int rotary_dim,
                                uint16_t *cos_sin)
{
    if (max_pos < 0 || rotary_dim <= 0 || (rotary_dim & 1) || !(theta > 0.0))
        return -3;
    if (max_pos == 0) return 0;
    if (!cos_sin) return -1;
    const int half = rotary_dim / 2;
    for (int64_t p = 0; p < max_pos; ++p) {
        uint16_t *row = cos_sin + p * (int64_t)rotary_dim;
        for (int i = 0; i < half; ++i) {
            double f = pow(theta, -2.0 * (double)i / (double)rotary_dim);
            double a = (double)p * f;
            row[i] = rn_oracle_double_to_bf16(cos(a));
            row[half + i] = rn_oracle_double_to_bf16(sin(a));
        }
    }
    return 0;
}

/* ---- fused Q/K RMSNorm + neox RoPE ------------------------------------- */

/* In place on qkv[T, (Hq + 2*Hkv) * D] (bf16).  Token t holds Hq query heads,
 * then Hkv key heads, then Hkv value heads, each D contiguous elements.  For
 * every token and every query or key head:
 *   n_j = x_j * 1/sqrt(mean_j(x_j^2) + eps) * w_j,  w = wq (query) or wk (key),
 *         the mean taken over all D elements even when rotary_dim < D;
 *   for i < r/2, with c = cos_sin[pos, i] and s = cos_sin[pos, r/2 + i]:
 *         o_i       = n_i * c - n_{i+r/2} * s
 *         o_{i+r/2} = n_{i+r/2} * c + n_i * s
 *   o_j = n_j for r <= j < D (the non-rotary tail);
 * each o rounded once to bf16.  Value heads are neither read nor written.
 * style 0 is the neox pairing above; style 1 pairs interleaved neighbours
 * (GPT-J): o_{2i} = n_{2i} c - n_{2i+1} s, o_{2i+1} = n_{2i+1} c + n_{2i} s,
 * with the same table row.  Follows "[pretuned] Optimize fused_qk_norm_rope on
 * B200", section "Summary".  A position outside [0, max_pos) is an error (-3) and nothing
 * is written for that token. */
int rn_oracle_qk_norm_rope_ex(uint16_t *qkv, const uint16_t *wq,
                           const uint16_t *wk, const float *cos_sin,
                           const int64_t *positions, int64_t max_pos,
                           int64_t T, int Hq, int Hkv, int D, int rotary_dim,
                           float eps, int style)
{
    if (T < 0 || Hq < 0 || Hkv < 0 || D <= 0 || rotary_dim <= 0 ||
        (rotary_dim & 1) || rotary_dim > D || D > 4096 || (style != 0 && style != 1))
        return -3;
    if (T == 0 || Hq + Hkv == 0) return 0;
    if (!qkv || !wq || !wk || !cos_sin || !positions) return -1;
    const int half = rotary_dim / 2;
    const int64_t token_stride = (int64_t)(Hq + 2 * Hkv) * D;
    const double deps = (double)eps;
    double n[4096];
    double o[4096];
    int bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        int64_t pos = positions[t];
        if (pos < 0 || pos >= max_pos) { bad = 1; continue; }
        const float *cs = cos_sin + pos * (int64_t)rotary_dim;
        for (int h = 0; h < Hq + Hkv; ++h) {
            uint16_t *head = qkv + t * token_stride + (int64_t)h * D;
            const uint16_t *w = (h < Hq) ? wq : wk;
            double ss = 0.0;
            for (int j = 0; j < D; ++j) {
                double v = rn_oracle_bf16_to_double(head[j]);
                ss += v * v;
            }
            double rs = 1.0 / sqrt(ss / (double)D + deps);
            for (int j = 0; j < D; ++j)
                n[j] = rn_oracle_bf16_to_double(head[j]) * rs *
                       rn_oracle_bf16_to_double(w[j]);
            for (int i = 0; i < half; ++i) {
                double c = (double)cs[i];
                double s = (double)cs[half + i];
                /* neox pairs (i, i + r/2); GPT-J pairs (2i, 2i + 1) */
                int a = style ? 2 * i : i;
                int b = style ? 2 * i + 1 : i + half;
                o[a] = n[a] * c - n[b] * s;
                o[b] = n[b] * c + n[a] * s;
            }
            for (int j = rotary_dim; j < D; ++j) o[j] = n[j];
            for (int j = 0; j < D; ++j) head[j] = rn_oracle_double_to_bf16(o[j]);
        }
    }
    return bad ? -3 : 0;
}

/* The neox form of rn_oracle_qk_norm_rope_ex (style 0). */
int rn_oracle_qk_norm_rope(uint16_t *qkv, const uint16_t *wq,
                           const uint16_t *wk, const float *cos_sin,
                           const int64_t *positions, int64_t max_pos,
                           int64_t T, int Hq, int Hkv, int D, int rotary_dim,
                           float eps)
{
    return rn_oracle_qk_norm_rope_ex(qkv, wq, wk, cos_sin, positions, max_pos, T, Hq, Hkv, D,
                                     rotary_dim, eps, 0);
}

/* ---- L2Norm ------------------------------------------------------------- */

/* y[r, j] = bf16( x[r, j] / max(||x[r, :]||_2, eps) ): one reduction, then a
 * scale by the inverse norm ("[Inductor] Codegen Gluon", section 3.2).  The
 * norm is sqrt(sum_j x^2) in double; eps guards rows whose norm is below it. */
int rn_oracle_l2norm_fmt(const uint16_t *x, float eps, int64_t M, int64_t N, uint16_t *y,
                         int f16)
{
    if (M < 0 || N <= 0) return -3;
    if (M == 0) return 0;
    if (!x || !y) return -1;
    for (int64_t r = 0; r < M; ++r) {
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double v = widen(x[r * N + j], f16);
            ss += v * v;
        }
        double nrm = sqrt(ss);
        double d = nrm > (double)eps ? nrm : (double)eps;
        for (int64_t j = 0; j < N; ++j)
            y[r * N + j] = narrow(widen(x[r * N + j], f16) / d, f16);
    }
    return 0;
}

int rn_oracle_l2norm(const uint16_t *x, float eps, int64_t M, int64_t N, uint16_t *y)
{
    return rn_oracle_l2norm_fmt(x, eps, M, N, y, 0);
}

/* ---- fused residual add + RMSNorm ---------------------------------------- */

/* h[r, j] = bf16(x[r, j] + res[r, j])   (the exact sum, rounded once)
 * y[r, :] = rmsnorm(h[r, :]) with the rounded h, exactly as the unfused pair
 * "add, then RMSNorm" would give: fusing the two ops removes HBM round trips
 * and changes nothing else ("TorchInductor: from ATen IR to Triton kernel",
 * sections 14.3 and 14.27: the norm / residual-add chain fused into one
 * kernel). */
int rn_oracle_add_rmsnorm_fmt(const uint16_t *x, const uint16_t *res, const uint16_t *w,
                              float eps, int64_t M, int64_t N, uint16_t *h, uint16_t *y,
                              int f16)
{
    if (M < 0 || N <= 0) return -3;
    if (M == 0) return 0;
    if (!x || !res || !w || !h || !y) return -1;
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t j = 0; j < N; ++j)
            h[r * N + j] = narrow(widen(x[r * N + j], f16) + widen(res[r * N + j], f16), f16);
    }
    return rn_oracle_rmsnorm_fmt(h, w, eps, M, N, y, f16);
}

int rn_oracle_add_rmsnorm(const uint16_t *x, const uint16_t *res, const uint16_t *w,
                          float eps, int64_t M, int64_t N, uint16_t *h, uint16_t *y)
{
    return rn_oracle_add_rmsnorm_fmt(x, res, w, eps, M, N, h, y, 0);
}

/* ---- LayerNorm ---------------------------------------------------------- */

/* y[r, j] = bf16( (x[r, j] - mean_r) / sqrt(var_r + eps) * w[j] + b[j] ),
 * mean and the biased variance (divide by N) taken over the row, as the
 * var_mean -> add(eps) -> rsqrt -> sub -> mul -> mul(weight) -> add(bias)
 * decomposition in "TorchInductor: from ATen IR to Triton kernel", section
 * 14.12.2, spells out.  The variance is the plain two-pass definition here;
 * the one-pass Welford update of that section reaches the same value up to
 * rounding.  b may be NULL (no bias). */
int rn_oracle_layernorm_fmt(const uint16_t *x, const uint16_t *w, const uint16_t *b,
                            float eps, int64_t M, int64_t N, uint16_t *y, int f16)
{
    if (M < 0 || N <= 0) return -3;
    if (M == 0) return 0;
    if (!x || !w || !y) return -1;
    for (int64_t r = 0; r < M; ++r) {
        const uint16_t *xr = x + r * N;
        uint16_t *yr = y + r * N;
        double sum = 0.0;
        for (int64_t j = 0; j < N; ++j) sum += widen(xr[j], f16);
        double mean = sum / (double)N;
        double m2 = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double d = widen(xr[j], f16) - mean;
            m2 += d * d;
        }
        double rs = 1.0 / sqrt(m2 / (double)N + (double)eps);
        for (int64_t j = 0; j < N; ++j) {
            double v = (widen(xr[j], f16) - mean) * rs * widen(w[j], f16);
            if (b) v += widen(b[j], f16);
            yr[j] = narrow(v, f16);
        }
    }
    return 0;
}

int rn_oracle_layernorm(const uint16_t *x, const uint16_t *w, const uint16_t *b, float eps,
                        int64_t M, int64_t N, uint16_t *y)
{
    return rn_oracle_layernorm_fmt(x, w, b, eps, M, N, y, 0);
}
