/*
 * oracle.c - plain, slow, single-threaded fp64 CPU reference for the
 * row-wise LayerNorm and RMSNorm forward and backward passes.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library. The product path
 * (the CUDA library and its Python binding) never links, imports or calls
 * it, and shares no code, header or table with it.
 *
 * Sources (page title, section):
 *   [Ch7]  "第 7 章 LayerNorm 与 RMSNorm" (CUDA 算子工程)
 *   [RMS2] "CUDA算子优化(2)：RMSNorm"
 *   [T3]   "T3 讲解：LayerNorm / RMSNorm 的 forward"
 *
 * Every routine below is the textbook definition written out, accumulating
 * in double precision: no blocking, no fusion, no reordering.
 *
 * Element types of the inputs: 0 = fp32, 1 = bf16 (raw 16-bit patterns),
 * 2 = fp64, 3 = fp16 (raw 16-bit patterns). Every input is widened exactly
 * to double before any arithmetic.
 *
 * Parity pins: each routine is pinned in tests/test_oracle_pins.py against
 * the pages' worked examples, closed forms, exact rational arithmetic on tiny
 * rows and an independent library routine (torch fp64 on the CPU).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2, ORC_F16 = 3 };

/* IEEE binary16 bit pattern to double, from the format's definition:
 * sign, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 holds
 * subnormals (fraction * 2^-24), exponent 31 infinities and NaNs. Exact. */
static double orc_f16_value(uint16_t h)
{
    const int sign = h >> 15, ex = (h >> 10) & 31, fr = h & 1023;
    double v;
    if (ex == 0)
        v = ldexp((double)fr, -24);
    else if (ex == 31)
        v = fr ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + fr), ex - 25);
    return sign ? -v : v;
}

/* Widen element i of a row to double. bf16 is the upper half of an fp32
 * bit pattern; every fp16 value is a double: the widening is exact for all
 * four types. */
static double orc_load(const void *p, int dtype, int64_t i)
{
    if (dtype == ORC_F32)
        return (double)((const float *)p)[i];
    if (dtype == ORC_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)p)[i] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (dtype == ORC_F16)
        return orc_f16_value(((const uint16_t *)p)[i]);
    return ((const double *)p)[i];
}

static int64_t orc_elem_size(int dtype)
{
    return dtype == ORC_F32 ? 4 : (dtype == ORC_BF16 || dtype == ORC_F16) ? 2 : 8;
}

/*
 * Mean and biased variance of one row of N elements, by the two-pass
 * definition: [Ch7] §7.1 (mu = sum/H, sigma^2 = sum (x - mu)^2 / H) and the
 * two-pass algorithm of [Ch7] §7.2; divisor N, not N-1 ([T3] §⑥).
 */
void oracle_row_moments(const void *x, int dtype, int64_t N,
                        double *mean, double *var)
{
    double sum = 0.0;
    for (int64_t i = 0; i < N; ++i)
        sum += orc_load(x, dtype, i);
    const double mu = sum / (double)N;

    double sq = 0.0;
    for (int64_t i = 0; i < N; ++i) {
        const double d = orc_load(x, dtype, i) - mu;
        sq += d * d;
    }
    *mean = mu;
    *var = sq / (double)N;
}

/*
 * LayerNorm forward over an [M, N] row-major matrix ([Ch7] §7.1):
 *   y = (x - mu) / sqrt(var + eps) * gamma + beta,  rstd = 1/sqrt(var + eps).
 * x, gamma and beta share `dtype`. Outputs are double; mean and rstd may be
 * NULL.
 */
void oracle_ln_fwd(const void *x, const void *gamma, const void *beta,
                   int dtype, int64_t M, int64_t N, double eps,
                   double *y, double *mean, double *rstd)
{
    const int64_t es = orc_elem_size(dtype);
    for (int64_t r = 0; r < M; ++r) {
        const void *xr = (const char *)x + r * N * es;
        double mu, var;
        oracle_row_moments(xr, dtype, N, &mu, &var);
        const double rs = 1.0 / sqrt(var + eps);
        for (int64_t i = 0; i < N; ++i) {
            const double xi = orc_load(xr, dtype, i);
            y[r * N + i] = (xi - mu) * rs * orc_load(gamma, dtype, i)
                           + orc_load(beta, dtype, i);
        }
        if (mean)
            mean[r] = mu;
        if (rstd)
            rstd[r] = rs;
    }
}

/*
 * RMSNorm forward over an [M, N] row-major matrix ([Ch7] §7.5; [RMS2] §1):
 *   rstd = 1/sqrt(sum x^2 / N + eps),  y = x * rstd * w.
 * No mean is subtracted and there is no bias. rstd may be NULL.
 */
void oracle_rms_fwd(const void *x, const void *w, int dtype, int64_t M,
                    int64_t N, double eps, double *y, double *rstd)
{
    const int64_t es = orc_elem_size(dtype);
    for (int64_t r = 0; r < M; ++r) {
        const void *xr = (const char *)x + r * N * es;
        double ss = 0.0;
        for (int64_t i = 0; i < N; ++i) {
            const double xi = orc_load(xr, dtype, i);
            ss += xi * xi;
        }
        const double rs = 1.0 / sqrt(ss / (double)N + eps);
        for (int64_t i = 0; i < N; ++i)
            y[r * N + i] = orc_load(xr, dtype, i) * rs * orc_load(w, dtype, i);
        if (rstd)
            rstd[r] = rs;
    }
}

/* Round each double to the nearest fp32, ties to even (C's conversion under
 * the default rounding mode is the single IEEE rounding). */
void oracle_round_f32(const double *v, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)v[i];
}

/* Round one double to bf16 (8 significant bits, fp32 exponent range),
 * nearest with ties to even, returned as the raw 16-bit pattern. The value
 * is scaled onto an integer grid whose spacing is one bf16 ulp of its
 * binade, rounded with rint(), and scaled back; all steps but rint() are
 * exact. */
static uint16_t orc_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    const int neg = signbit(v) != 0;
    const double a = fabs(v);
    if (isinf(a))
        return neg ? 0xFF80 : 0x7F80;
    double res = 0.0;
    if (a != 0.0) {
        int e;
        (void)frexp(a, &e);       /* a = m * 2^e with m in [0.5, 1) */
        int ex = e - 1;           /* floor(log2 a) */
        if (ex < -126)
            ex = -126;            /* subnormal binade keeps the fixed spacing */
        res = ldexp(rint(ldexp(a, 7 - ex)), ex - 7);
    }
    float f = (float)res;
    if (res >= 0x1p128)
        f = INFINITY;
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    bits >>= 16;
    if (neg)
        bits |= 0x8000u;
    return (uint16_t)bits;
}

void oracle_round_bf16(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16(v[i]);
}

/* Round one double to IEEE binary16, nearest with ties to even, returned as
 * the bit pattern: 11 significant bits, normal binades 2^-14 .. 2^15, below
 * them the fixed subnormal spacing 2^-24. As for bf16, the value is scaled
 * onto an integer grid of one ulp of its binade, rounded with rint() and
 * scaled back; a result of 2^16 or more (65520 and up before rounding) is
 * infinity. The pattern is then assembled field by field. */
static uint16_t orc_f16(double v)
{
    if (isnan(v))
        return 0x7E00;
    const uint16_t sign = signbit(v) ? 0x8000 : 0;
    const double a = fabs(v);
    if (isinf(a))
        return sign | 0x7C00;
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);
    int ex = e - 1;                 /* floor(log2 a) */
    if (ex < -14)
        ex = -14;
    const double r = ldexp(rint(ldexp(a, 10 - ex)), ex - 10);
    if (r >= 65536.0)
        return sign | 0x7C00;
    if (r < ldexp(1.0, -14))        /* subnormal (or zero): fraction = r / 2^-24 */
        return sign | (uint16_t)ldexp(r, 24);
    (void)frexp(r, &e);
    const int be = e - 1 + 15;      /* biased exponent of the rounded value */
    const uint16_t frac = (uint16_t)(ldexp(r, 10 - (e - 1)) - 1024.0);
    return sign | (uint16_t)(be << 10) | frac;
}

void oracle_round_f16(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f16(v[i]);
}

/*
 * Welford's running state and Chan's merge, in double precision. They are
 * not used by the reference outputs above (which follow the definition);
 * they exist so that the pins can show, on tiny rows and under every merge
 * order, that the algorithm the GPU path uses reaches the two-pass result.
 */
typedef struct {
    double n, mean, m2;
} orc_welford;

/* One-element update, [Ch7] §7.4: n' = n+1; d = x - mean; mean += d/n';
 * m2 += d * (x - mean'). */
void oracle_welford_update(orc_welford *s, double x)
{
    const double n1 = s->n + 1.0;
    const double d = x - s->mean;
    s->mean += d / n1;
    s->m2 += d * (x - s->mean);
    s->n = n1;
}

/* Parallel merge of two partial states, [Ch7] §7.4.1:
 * n = na+nb; d = mb - ma; mean = ma + d*nb/n; m2 = m2a + m2b + d^2*na*nb/n.
 * The merge of two empty states is empty. */
void oracle_chan_combine(const orc_welford *a, const orc_welford *b,
                         orc_welford *out)
{
    const double n = a->n + b->n;
    if (n == 0.0) {
        out->n = out->mean = out->m2 = 0.0;
        return;
    }
    const double d = b->mean - a->mean;
    orc_welford r;
    r.n = n;
    r.mean = a->mean + d * b->n / n;
    r.m2 = a->m2 + b->m2 + d * d * a->n * b->n / n;
    *out = r;
}

/*
 * Fused residual add ([Ch7] §7.9-7.10, the fused add + norm of the residual
 * stream; [T3] §⑤): h = x + residual, rounded to the row type, as an
 * unfused add that stores h would leave it. The sum is formed in double
 * (exact for two bf16 or fp16 values; for fp32 values exact or carrying more
 * than 2*24+2 bits, so rounding it once more to the row type gives the
 * correctly rounded sum) and rounded to the row type. The norm of the
 * fused op is then the norm of h (oracle_ln_fwd / oracle_rms_fwd on h).
 */
void oracle_add_round(const void *x, const void *r, int dtype, int64_t n, void *h)
{
    for (int64_t i = 0; i < n; ++i) {
        const double v = orc_load(x, dtype, i) + orc_load(r, dtype, i);
        if (dtype == ORC_F32)
            ((float *)h)[i] = (float)v;
        else if (dtype == ORC_BF16)
            ((uint16_t *)h)[i] = orc_bf16(v);
        else if (dtype == ORC_F16)
            ((uint16_t *)h)[i] = orc_f16(v);
        else
            ((double *)h)[i] = v;
    }
}

/*
 * LayerNorm backward over an [M, N] row-major matrix ([Ch7] §7.7), given the
 * upstream gradient dy of the same shape. Per row, with mu, var by the
 * two-pass definition and rstd = 1/sqrt(var + eps):
 *   xhat_i = (x_i - mu) * rstd,  g_i = dy_i * gamma_i,
 *   gbar = sum_j g_j / N,  gxbar = sum_j g_j xhat_j / N,
 *   dx_i = rstd * (g_i - gbar - xhat_i * gxbar)
 * (gamma multiplies dy inside the bracket, element by element), and over
 * rows dgamma_i = sum_n dy_i xhat_i, dbeta_i = sum_n dy_i. dy, x and gamma
 * share `dtype`; every output is double.
 */
void oracle_ln_bwd(const void *dy, const void *x, const void *gamma, int dtype,
                   int64_t M, int64_t N, double eps,
                   double *dx, double *dgamma, double *dbeta)
{
    const int64_t es = orc_elem_size(dtype);
    for (int64_t i = 0; i < N; ++i)
        dgamma[i] = dbeta[i] = 0.0;
    for (int64_t r = 0; r < M; ++r) {
        const void *xr = (const char *)x + r * N * es;
        const void *dyr = (const char *)dy + r * N * es;
        double mu, var;
        oracle_row_moments(xr, dtype, N, &mu, &var);
        const double rs = 1.0 / sqrt(var + eps);
        double sg = 0.0, sgx = 0.0;
        for (int64_t i = 0; i < N; ++i) {
            const double xh = (orc_load(xr, dtype, i) - mu) * rs;
            const double g = orc_load(dyr, dtype, i) * orc_load(gamma, dtype, i);
            sg += g;
            sgx += g * xh;
        }
        const double gbar = sg / (double)N, gxbar = sgx / (double)N;
        for (int64_t i = 0; i < N; ++i) {
            const double xh = (orc_load(xr, dtype, i) - mu) * rs;
            const double d = orc_load(dyr, dtype, i);
            const double g = d * orc_load(gamma, dtype, i);
            dx[r * N + i] = rs * (g - gbar - xh * gxbar);
            dgamma[i] += d * xh;
            dbeta[i] += d;
        }
    }
}

/*
 * RMSNorm backward ([Ch7] §7.7, last paragraph: one row sum, of dy*w*x).
 * With rstd = 1/sqrt(sum x^2 / N + eps) and y_i = x_i * rstd * w_i:
 *   S = sum_j dy_j w_j x_j,
 *   dx_i = rstd * w_i * dy_i - x_i * rstd^3 * S / N,
 *   dw_i = sum_n dy_i x_i rstd.
 * (d rstd / d x_j = -rstd^3 x_j / N.)
 */
void oracle_rms_bwd(const void *dy, const void *x, const void *w, int dtype,
                    int64_t M, int64_t N, double eps, double *dx, double *dw)
{
    const int64_t es = orc_elem_size(dtype);
    for (int64_t i = 0; i < N; ++i)
        dw[i] = 0.0;
    for (int64_t r = 0; r < M; ++r) {
        const void *xr = (const char *)x + r * N * es;
        const void *dyr = (const char *)dy + r * N * es;
        double ss = 0.0, s = 0.0;
        for (int64_t i = 0; i < N; ++i) {
            const double xi = orc_load(xr, dtype, i);
            ss += xi * xi;
            s += orc_load(dyr, dtype, i) * orc_load(w, dtype, i) * xi;
        }
        const double rs = 1.0 / sqrt(ss / (double)N + eps);
        const double c = rs * rs * rs * s / (double)N;
        for (int64_t i = 0; i < N; ++i) {
            const double xi = orc_load(xr, dtype, i);
            const double d = orc_load(dyr, dtype, i);
            dx[r * N + i] = rs * orc_load(w, dtype, i) * d - xi * c;
            dw[i] += d * xi * rs;
        }
    }
}

/*
 * FP8 output for the next GEMM ([Ch7] §7.9: the norm writes the quantised
 * input of the following GEMM, as vLLM's static-scale fused kernels do).
 * Format: OCP FP8 E4M3 ("fn": finite only): sign, 4 exponent bits (bias 7),
 * 3 fraction bits; normal values 2^-6 .. 448, subnormals fraction * 2^-9,
 * the pattern 0x7F / 0xFF is NaN, and there is no infinity. Quantisation
 * with a per-tensor static scale: q = E4M3(y / scale), nearest with ties to
 * even, saturating: values of magnitude 448 or more give +-448.
 */
static uint8_t orc_e4m3(double v)
{
    if (isnan(v))
        return 0x7F;
    const uint8_t sign = signbit(v) ? 0x80 : 0;
    const double a = fabs(v);
    if (a >= 448.0)
        return sign | 0x7E;           /* 448 = 1.75 * 2^8: exponent 15, fraction 110 */
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);
    int ex = e - 1;                   /* floor(log2 a) */
    if (ex < -6)
        ex = -6;                      /* subnormals keep the spacing 2^-9 */
    const double r = ldexp(rint(ldexp(a, 3 - ex)), ex - 3);
    if (r >= 448.0)
        return sign | 0x7E;
    if (r < ldexp(1.0, -6))           /* subnormal (or zero): fraction = r / 2^-9 */
        return sign | (uint8_t)ldexp(r, 9);
    (void)frexp(r, &e);
    const int be = e - 1 + 7;
    const uint8_t frac = (uint8_t)(ldexp(r, 3 - (e - 1)) - 8.0);
    return sign | (uint8_t)(be << 3) | frac;
}

/* q_i = E4M3(y_i / scale) for n values (the division is exact-rounded in
 * double; see orc_e4m3 for the rounding). */
void oracle_quant_e4m3(const double *y, int64_t n, double scale, uint8_t *q)
{
    for (int64_t i = 0; i < n; ++i)
        q[i] = orc_e4m3(y[i] / scale);
}

/* Value of an E4M3 code (exact; NaN for 0x7F and 0xFF). */
double oracle_e4m3_value(uint8_t q)
{
    const int sign = q >> 7, ex = (q >> 3) & 15, fr = q & 7;
    double v;
    if (ex == 15 && fr == 7)
        return NAN;
    if (ex == 0)
        v = ldexp((double)fr, -9);
    else
        v = ldexp((double)(8 + fr), ex - 10);
    return sign ? -v : v;
}

int oracle_abi_version(void) { return 5; }
